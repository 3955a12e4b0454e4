"""GPU parity of d2f_kv_append (bit-exact) and the append-then-attend
consistency of the cache: moving a finished block from the window into its page
leaves the later window blocks' attention unchanged."""
import pytest
import torch

import oracle
from block_causal_kv_gb300 import d2f, synth
from gpu_common import check_attention, device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["dream", "tiny"])
def test_bitwise(name):
    dev = device()
    w = synth.small(name) if name != "tiny" else synth.Workload(
        "t", 1, 4, 4, 64, 16, torch.float32, [64], [2], 1000, appends_per_seq=2, seed=9)
    p = synth.make_problem(w)
    g = p.to(dev)
    d2f.kv_append(g.k_win, g.v_win, g.src_row, g.dst_page, g.k_pool, g.v_pool,
                  block_size=w.block_size)
    torch.cuda.synchronize()
    kp, vp = oracle.kv_append(p.k_win, p.v_win, p.src_row, p.dst_page, p.k_pool, p.v_pool,
                              w.block_size)
    assert torch.equal(g.k_pool.cpu(), kp)
    assert torch.equal(g.v_pool.cpu(), vp)


def test_full_size_dream_appends():
    dev = device()
    p = synth.make_problem(synth.workload("dream"))
    g = p.to(dev)
    d2f.kv_append(g.k_win, g.v_win, g.src_row, g.dst_page, g.k_pool, g.v_pool, block_size=16)
    torch.cuda.synchronize()
    for s, d in zip(p.src_row.tolist(), p.dst_page.tolist()):
        assert torch.equal(g.k_pool[d].cpu(), p.k_win[s:s + 16].transpose(0, 1))
        assert torch.equal(g.v_pool[d].cpu(), p.v_win[s:s + 16].transpose(0, 1))


def test_append_then_attend():
    dev = device()
    B = 16
    w = synth.Workload("aa", 2, 8, 2, 128, B, torch.bfloat16, [64, 112], [3, 2], 64,
                       appends_per_seq=1, permute_pages=True, seed=31)
    p = synth.make_problem(w)
    g = p.to(dev)
    d2f.kv_append(g.k_win, g.v_win, g.src_row, g.dst_page, g.k_pool, g.v_pool, block_size=B)
    keep = []
    qs = p.q_start.tolist()
    new_qs = [0]
    for b in range(w.batch):
        keep += list(range(qs[b] + B, qs[b + 1]))
        new_qs.append(len(keep))
    keep = torch.tensor(keep)
    kd = keep.to(dev)
    nq = torch.tensor(new_qs, dtype=torch.int32)
    after, _ = d2f.block_attn(g.q[kd].contiguous(), g.k_win[kd].contiguous(),
                              g.v_win[kd].contiguous(), g.k_pool, g.v_pool, g.page_table,
                              g.ctx_len + B, nq.to(dev), block_size=B, max_q_per_seq=2 * B,
                              max_ctx=int(max(w.ctx_lens)) + B)
    torch.cuda.synchronize()
    before, _ = oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
                                  p.ctx_len, p.q_start, B)
    check_attention(after, None, before[keep], None, torch.bfloat16, "append-then-attend")


def _attn(g, p, dev, splits=0, append=False):
    kw = dict(append_src_row=g.src_row, append_dst_page=g.dst_page) if append else {}
    out, lse = d2f.block_attn(g.q, g.k_win, g.v_win, g.k_pool, g.v_pool, g.page_table, g.ctx_len,
                              g.q_start, block_size=p.w.block_size, max_q_per_seq=p.max_q_per_seq,
                              max_ctx=p.max_ctx, num_splits=splits, **kw)
    return out, lse


def _fused_case(w, dev, splits):
    p = synth.make_problem(w)
    g1, g2 = p.to(dev), p.to(dev)
    out1, lse1 = _attn(g1, p, dev, splits, append=True)
    out2, lse2 = _attn(g2, p, dev, splits)
    d2f.kv_append(g2.k_win, g2.v_win, g2.src_row, g2.dst_page, g2.k_pool, g2.v_pool,
                  block_size=w.block_size)
    torch.cuda.synchronize()
    # the same attention, bit for bit, and the same pool, bit for bit
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    assert torch.equal(g1.k_pool, g2.k_pool) and torch.equal(g1.v_pool, g2.v_pool)
    kp, vp = oracle.kv_append(p.k_win, p.v_win, p.src_row, p.dst_page, p.k_pool, p.v_pool,
                              w.block_size)
    assert torch.equal(g1.k_pool.cpu(), kp) and torch.equal(g1.v_pool.cpu(), vp)


@pytest.mark.parametrize("B", [8, 16, 32])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_fused_append_matches_separate(B, splits):
    """d2f_block_attn_append: the attention's own window tiles are stored to the
    appended pages; output and pool equal attention followed by d2f_kv_append
    (64- and 128-row tiles, one or two row tiles per group)."""
    dev = device()
    w = synth.Workload("fa", 3, 4, 2, 128, B, torch.bfloat16, [5 * B + 3, 130, 2 * B],
                       [3, 2, 1], 64, permute_pages=True, extra_pages=4,
                       appends_per_seq=1, seed=700 + B)
    _fused_case(w, dev, splits)


@pytest.mark.parametrize("mt", ["1", "0"])
@pytest.mark.parametrize("deep", ["1", "0"])
def test_fused_append_row_tile_variants(mt, deep, monkeypatch):
    """The Dream shape (GQA 7, three 128-row tiles) on two-row-tile CTAs or one
    row tile per CTA, 2- or 6-stage rings: only row group 0 stores."""
    dev = device()
    monkeypatch.setenv("D2F_TC_MT", mt)
    monkeypatch.setenv("D2F_TC_DEEP", deep)
    _fused_case(synth.small("dream"), dev, 0)


def test_fused_append_cuda_core_path():
    """float32 runs the attention on CUDA cores and the append after it."""
    dev = device()
    w = synth.Workload("t", 1, 4, 4, 64, 16, torch.float32, [64], [2], 1000, appends_per_seq=2,
                       seed=9)
    _fused_case(w, dev, 0)


def test_fused_append_full_size_dream():
    dev = device()
    _fused_case(synth.workload("dream"), dev, 0)
