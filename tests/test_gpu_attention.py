"""GPU parity of d2f_block_attn against the CPU oracle (element by element).

Covers every workload at reduced size (several tiles, ragged tails, GQA with
more than 128 packed rows, permuted page tables, contexts that are not a
multiple of the block, empty contexts), forced split counts (the log-space
composition path), both the tensor-core and the CUDA-core path, and the
full-size LLaDA-shaped layer in the launch configuration the benchmark times.
"""
import os

import pytest
import torch

import oracle
from block_causal_kv_gb300 import d2f, synth
from gpu_common import check_attention, device

pytestmark = pytest.mark.gpu


def _run(p, dev, num_splits=0, want_lse=True):
    g = p.to(dev)
    out, lse = d2f.block_attn(g.q, g.k_win, g.v_win, g.k_pool, g.v_pool, g.page_table,
                              g.ctx_len, g.q_start, block_size=p.w.block_size,
                              max_q_per_seq=p.max_q_per_seq, max_ctx=p.max_ctx,
                              num_splits=num_splits, want_lse=want_lse)
    torch.cuda.synchronize()
    return out, lse


_REF = {}


def _ref(p):
    key = (p.w.name, p.w.seed, p.w.block_size, p.w.head_dim, str(p.w.dtype))
    if key not in _REF:
        _REF[key] = oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
                                      p.ctx_len, p.q_start, p.w.block_size)
    return _REF[key]


SMALL = ["tiny", "llada", "ragged", "dream", "long_b8", "long_b16", "long_b32"]


@pytest.mark.parametrize("name", SMALL)
@pytest.mark.parametrize("splits", [0, 1, 3, 6, 8])
def test_small_workloads(name, splits):
    dev = device()
    w = synth.workload("tiny") if name == "tiny" else synth.small(name)
    p = synth.make_problem(w)
    out, lse = _run(p, dev, splits)
    ref, ref_lse = _ref(p)
    check_attention(out, lse, ref, ref_lse, w.dtype, "%s/s%d" % (name, splits))


@pytest.mark.parametrize("name", ["llada", "ragged", "long_b8", "long_b16"])
@pytest.mark.parametrize("splits", [0, 1, 5])
def test_full_row_tiles_where_half_tiles_fit(name, splits, monkeypatch):
    """Workloads with at most 64 rows per sequence run on 64-row tiles (three
    ring stages); D2F_TC_ROWS=128 forces the 128-row tile. Both agree with the
    oracle."""
    dev = device()
    monkeypatch.setenv("D2F_TC_ROWS", "128")
    p = synth.make_problem(synth.small(name))
    assert p.max_q_per_seq * p.w.num_heads_q // p.w.num_heads_kv <= 64
    out, lse = _run(p, dev, splits)
    ref, ref_lse = _ref(p)
    check_attention(out, lse, ref, ref_lse, torch.bfloat16, "rows128/%s/s%d" % (name, splits))


@pytest.mark.parametrize("name", ["dream", "long_b32"])
@pytest.mark.parametrize("splits", [0, 1, 3, 8])
@pytest.mark.parametrize("deep", ["1", "0"])
def test_ring_depth_variants_for_full_row_tiles(name, splits, deep, monkeypatch):
    """head_dim 128 with 128-row tiles runs either a 6-stage ring at one CTA per SM
    (D2F_TC_DEEP=1) or a 2-stage ring at two CTAs per SM (D2F_TC_DEEP=0); both
    agree with the oracle."""
    dev = device()
    monkeypatch.setenv("D2F_TC_DEEP", deep)
    p = synth.make_problem(synth.small(name))
    out, lse = _run(p, dev, splits)
    ref, ref_lse = _ref(p)
    check_attention(out, lse, ref, ref_lse, torch.bfloat16, "deep%s/%s/s%d" % (deep, name, splits))


def _gqa_two_tiles():
    # G = 4, windows of 3 and 2 blocks of 16: 192 and 128 packed rows
    return synth.Workload("gqa2", 2, 16, 4, 128, 16, torch.bfloat16, [700, 333], [3, 2], 64,
                          permute_pages=True, extra_pages=3, seed=515)


def _gqa_mixed_rows():
    # G = 7, windows of 3, 1 and 2 blocks of 16: 336, 112 and 224 packed rows, so
    # the second CTA of a row-tile group holds one row tile, or none
    return synth.Workload("gqa3r", 3, 28, 4, 128, 16, torch.bfloat16, [700, 333, 1500], [3, 1, 2], 64,
                          permute_pages=True, extra_pages=5, seed=516)


@pytest.mark.parametrize("name", ["dream", "gqa2", "gqa3r"])
@pytest.mark.parametrize("splits", [0, 1, 3, 8])
def test_two_row_tiles_per_cta(name, splits, monkeypatch):
    """GQA groups of 2 or 3 row tiles on CTAs of two row tiles with a softmax
    warpgroup each (D2F_TC_MT=1): one K/V stream for both, one accumulator per
    row tile; three tiles leave the second CTA one tile, and shorter sequences
    one idle warpgroup or a CTA without rows. Same result as the oracle."""
    dev = device()
    monkeypatch.setenv("D2F_TC_MT", "1")
    w = {"gqa2": _gqa_two_tiles, "gqa3r": _gqa_mixed_rows}.get(name, lambda: synth.small(name))()
    p = synth.make_problem(w)
    out, lse = _run(p, dev, splits)
    ref, ref_lse = _ref(p)
    check_attention(out, lse, ref, ref_lse, torch.bfloat16, "mt/%s/s%d" % (name, splits))


@pytest.mark.parametrize("splits", [0, 2])
def test_two_row_tiles_longest_first(splits, monkeypatch):
    """Two-row-tile CTAs with the sequences taken longest context first."""
    dev = device()
    monkeypatch.setenv("D2F_TC_MT", "1")
    monkeypatch.setenv("D2F_LONGEST_FIRST", "1")
    p = synth.make_problem(_gqa_mixed_rows())
    out, lse = _run(p, dev, splits)
    ref, ref_lse = _ref(p)
    check_attention(out, lse, ref, ref_lse, torch.bfloat16, "mt-lf/s%d" % splits)


@pytest.mark.parametrize("name", ["ragged", "dream", "long_b32"])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_longest_first_sequence_order(name, splits, monkeypatch):
    """CTAs mapped to sequences longest context first (D2F_LONGEST_FIRST=1, the
    order taken when the grid exceeds one wave): same result as the oracle."""
    dev = device()
    monkeypatch.setenv("D2F_LONGEST_FIRST", "1")
    w = synth.small(name)
    p = synth.make_problem(w)
    out, lse = _run(p, dev, splits)
    ref, ref_lse = _ref(p)
    check_attention(out, lse, ref, ref_lse, torch.bfloat16, "lf/%s/s%d" % (name, splits))


@pytest.mark.parametrize("name", ["llada", "ragged", "dream", "long_b16"])
def test_cuda_core_path_bf16(name, monkeypatch):
    """The CUDA-core kernel on bf16 operands, cross-checked like the main path."""
    dev = device()
    monkeypatch.setenv("D2F_ATTN_PATH", "simt")
    p = synth.make_problem(synth.small(name))
    out, lse = _run(p, dev, 2)
    ref, ref_lse = _ref(p)
    check_attention(out, lse, ref, ref_lse, torch.bfloat16, "simt/" + name)


@pytest.mark.parametrize("B", [8, 16, 32])
@pytest.mark.parametrize("D", [64, 128])
def test_block_and_head_sizes(B, D):
    dev = device()
    w = synth.Workload("bd", 2, 4, 2, D, B, torch.bfloat16, [5 * B + 3, 130], [3, 2], 64,
                       permute_pages=True, extra_pages=2, seed=400 + B + D)
    p = synth.make_problem(w)
    for splits in (1, 2, 5):
        out, lse = _run(p, dev, splits)
        ref, ref_lse = _ref(p)
        check_attention(out, lse, ref, ref_lse, torch.bfloat16, "B%d D%d s%d" % (B, D, splits))


def test_many_splits_more_than_tiles():
    """Requested splits beyond the number of key tiles: each sequence uses only
    as many non-empty splits as it has tiles."""
    dev = device()
    w = synth.Workload("ms", 3, 4, 4, 128, 16, torch.bfloat16, [0, 16, 700], [1, 2, 3], 64,
                       seed=77)
    p = synth.make_problem(w)
    out, lse = _run(p, dev, 64)
    ref, ref_lse = _ref(p)
    check_attention(out, lse, ref, ref_lse, torch.bfloat16, "splits64")


@pytest.mark.parametrize("path", ["tc", "simt"])
def test_lse_optional_and_repeatable(path, monkeypatch):
    """lse_out may be NULL; back-to-back calls with one workspace give identical
    results. The tensor-core path composes its splits in distributed shared
    memory and needs no workspace; the CUDA-core path's merge counters reset
    themselves."""
    dev = device()
    if path == "simt":
        monkeypatch.setenv("D2F_ATTN_PATH", "simt")
    p = synth.make_problem(synth.small("ragged"))
    g = p.to(dev)
    kw = dict(batch=p.w.batch, total_q=p.w.total_q, max_q_per_seq=p.max_q_per_seq,
              max_ctx=p.max_ctx, num_heads_q=p.w.num_heads_q, num_heads_kv=p.w.num_heads_kv,
              head_dim=p.w.head_dim, block_size=p.w.block_size, num_splits=4)
    nbytes = d2f.attn_workspace_size(**kw)
    if path == "tc":
        assert nbytes == 0
    ws = d2f.attn_workspace(dev, **kw)
    outs = []
    for _ in range(3):
        out, lse = d2f.block_attn(g.q, g.k_win, g.v_win, g.k_pool, g.v_pool, g.page_table,
                                  g.ctx_len, g.q_start, block_size=p.w.block_size,
                                  max_q_per_seq=p.max_q_per_seq, max_ctx=p.max_ctx,
                                  num_splits=4, want_lse=False, workspace=ws)
        outs.append(out.clone())
    torch.cuda.synchronize()
    assert lse is None
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    if path == "simt":
        # merge counters (one per sequence x KV head x 16-row group, at offset 0) back at zero
        n_counters = p.w.batch * p.w.num_heads_kv * -(-p.max_q_per_seq * p.w.num_heads_q
                                                       // p.w.num_heads_kv // 16)
        assert int(ws[:4 * n_counters].view(torch.int32).abs().sum()) == 0
    ref, _ = _ref(p)
    check_attention(outs[0], None, ref, None, torch.bfloat16, "repeat/" + path)


def test_full_size_llada_layer():
    """The LLaDA-8B-shaped layer at full size, automatic splits (the benchmark's
    launch configuration), every output element against the oracle."""
    dev = device()
    p = synth.make_problem(synth.workload("llada"))
    out, lse = _run(p, dev, 0)
    ref, ref_lse = _ref(p)
    mx, mean = check_attention(out, lse, ref, ref_lse, torch.bfloat16, "llada full")
    print("llada full: max-abs %.3e mean-abs %.3e" % (mx, mean))


@pytest.mark.parametrize("name", ["dream", "ragged", "long_b8", "long_b16", "long_b32"])
def test_full_size_sampled(name):
    """Full-size workloads: the GPU runs the whole batch; the oracle recomputes
    one sampled sequence (its window rows, all heads) one by one."""
    dev = device()
    p = synth.make_problem(synth.workload(name))
    out, _ = _run(p, dev, 0, want_lse=False)
    b = p.w.batch // 2
    qs = p.q_start.tolist()
    rows = slice(qs[b], qs[b + 1])
    ref, _ = oracle.block_attn(p.q[rows], p.k_win[rows], p.v_win[rows], p.k_pool, p.v_pool,
                               p.page_table[b:b + 1], p.ctx_len[b:b + 1],
                               torch.tensor([0, qs[b + 1] - qs[b]], dtype=torch.int32),
                               p.w.block_size, want_lse=False)
    mx, mean = check_attention(out[rows], None, ref, None, torch.bfloat16, name + " full")
    print("%s full (sequence %d): max-abs %.3e mean-abs %.3e" % (name, b, mx, mean))


def _part(g, p, part, q=None, prev=None, splits=0):
    out, lse = d2f.block_attn(g.q if q is None else q, g.k_win, g.v_win, g.k_pool, g.v_pool,
                              g.page_table, g.ctx_len, g.q_start, block_size=p.w.block_size,
                              max_q_per_seq=p.max_q_per_seq, max_ctx=p.max_ctx,
                              num_splits=splits, part=part,
                              prev_out=None if prev is None else prev[0],
                              prev_lse=None if prev is None else prev[1])
    torch.cuda.synchronize()
    return out, lse


def _ref_part(p, part, q=None, prev=None):
    return oracle.block_attn_part(p.q if q is None else q, p.k_win, p.v_win, p.k_pool, p.v_pool,
                                  p.page_table, p.ctx_len, p.q_start, p.w.block_size, part,
                                  prev_out=None if prev is None else prev[0].double(),
                                  prev_lse=None if prev is None else prev[1].double())


def _cached_ctx_zero(w):
    # a ragged batch whose second sequence has no cached token
    return synth.Workload("pz", 3, 8, 4, 128, 16, torch.bfloat16, [300, 0, 700], [2, 3, 1], 64,
                          permute_pages=True, extra_pages=2, seed=900)


@pytest.mark.parametrize("name", ["llada", "dream", "long_b32", "ragged", "ctx0"])
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_cached_and_window_parts(name, splits):
    """d2f_block_attn_part: the cached part alone and the window part alone match
    the oracle's parts; the window part composed with the kept cached part of the
    same queries matches the full attention; composed with the kept part of
    earlier queries it matches the oracle's composition of that kept part."""
    dev = device()
    w = _cached_ctx_zero(None) if name == "ctx0" else synth.small(name)
    p = synth.make_problem(w)
    g = p.to(dev)
    oc, lc = _part(g, p, d2f.ATTN_CACHED, splits=splits)
    rc, rlc = _ref_part(p, oracle.ATTN_CACHED)
    check_attention(oc, lc, rc, rlc, torch.bfloat16, "cached/%s/s%d" % (name, splits))
    ow, lw = _part(g, p, d2f.ATTN_WINDOW, splits=splits)
    rw, rlw = _ref_part(p, oracle.ATTN_WINDOW)
    check_attention(ow, lw, rw, rlw, torch.bfloat16, "window/%s/s%d" % (name, splits))
    # the same queries: the full attention
    of, lf = _part(g, p, d2f.ATTN_WINDOW, prev=(oc, lc), splits=splits)
    ref, ref_lse = _ref(p)
    check_attention(of, lf, ref, ref_lse, torch.bfloat16, "composed/%s/s%d" % (name, splits))
    # the next step's queries with the kept part: the oracle's composition of it
    q1 = (p.q.float() + 0.25 * torch.randn(p.q.shape, generator=torch.Generator().manual_seed(5))
          ).to(p.q.dtype)
    o1, l1 = _part(g, p, d2f.ATTN_WINDOW, q=q1.to(dev), prev=(oc, lc), splits=splits)
    r1, rl1 = _ref_part(p, oracle.ATTN_WINDOW, q=q1, prev=(oc.cpu(), lc.cpu()))
    check_attention(o1, l1, r1, rl1, torch.bfloat16, "reuse/%s/s%d" % (name, splits))


@pytest.mark.parametrize("name", ["dream", "long_b32"])
def test_full_size_parts_sampled(name):
    """Full-size workloads in the bench's launch configuration: the cached part,
    then the window part composed with it, against the oracle's full attention
    of one sampled sequence (its window rows, all heads)."""
    dev = device()
    p = synth.make_problem(synth.workload(name))
    g = p.to(dev)
    oc, lc = _part(g, p, d2f.ATTN_CACHED)
    of, lf = _part(g, p, d2f.ATTN_WINDOW, prev=(oc, lc))
    b = p.w.batch // 2
    qs = p.q_start.tolist()
    rows = slice(qs[b], qs[b + 1])
    ref, ref_lse = oracle.block_attn(p.q[rows], p.k_win[rows], p.v_win[rows], p.k_pool, p.v_pool,
                                     p.page_table[b:b + 1], p.ctx_len[b:b + 1],
                                     torch.tensor([0, qs[b + 1] - qs[b]], dtype=torch.int32),
                                     p.w.block_size)
    mx, mean = check_attention(of[rows], lf[rows], ref, ref_lse, torch.bfloat16,
                               name + " parts full")
    print("%s parts full (sequence %d): max-abs %.3e mean-abs %.3e" % (name, b, mx, mean))


def test_attention_parts_need_the_tensor_core_path():
    dev = device()
    p = synth.make_problem(synth.workload("tiny"))
    g = p.to(dev)
    with pytest.raises(d2f.D2FError):
        _part(g, p, d2f.ATTN_CACHED)


def _sk_env(monkeypatch, grid=None):
    monkeypatch.setenv("D2F_ATTN_SK", "1")
    monkeypatch.setenv("D2F_TC_DEEP", "1")
    monkeypatch.setenv("D2F_TC_ROWS", "128")
    if grid is not None:
        monkeypatch.setenv("D2F_ATTN_SK_GRID", str(grid))


def _gqa2_small():
    # GQA 8 / 4, window 1-3 blocks of 16: up to 96 rows per (sequence, KV head)
    return synth.Workload("gqa2sk", 3, 8, 4, 128, 16, torch.bfloat16, [700, 0, 1234], [3, 2, 1],
                          64, permute_pages=True, seed=77)


@pytest.mark.parametrize("name", ["llada", "ragged", "long_b8", "long_b16", "long_b32", "gqa2"])
@pytest.mark.parametrize("grid", [None, 1, 3, 7, 40])
def test_stream_k_form(name, grid, monkeypatch):
    """The stream-K form of the one-CTA variant: every (sequence, KV head)'s key
    tiles laid end to end and cut into equal shares, pieces of a pair composed in
    log space by the last CTA to finish one. Grids of 1 (one CTA walks every pair),
    3, 7, 40 and one per SM move every share boundary (pieces that start and end
    inside the cache or the window, pairs over three or more CTAs, CTAs with no
    share). Output and lse against the oracle; two calls in a row on one
    workspace (the pair counters reset themselves)."""
    dev = device()
    _sk_env(monkeypatch, grid)
    w = _gqa2_small() if name == "gqa2" else synth.small(name)
    p = synth.make_problem(w)
    g = p.to(dev)
    ws = d2f.attn_workspace(dev, batch=w.batch, total_q=w.total_q, max_q_per_seq=p.max_q_per_seq,
                            max_ctx=p.max_ctx, num_heads_q=w.num_heads_q,
                            num_heads_kv=w.num_heads_kv, head_dim=w.head_dim,
                            block_size=w.block_size)
    ref, ref_lse = _ref(p)
    for call in range(2):
        out, lse = d2f.block_attn(g.q, g.k_win, g.v_win, g.k_pool, g.v_pool, g.page_table,
                                  g.ctx_len, g.q_start, block_size=w.block_size,
                                  max_q_per_seq=p.max_q_per_seq, max_ctx=p.max_ctx, workspace=ws)
        torch.cuda.synchronize()
        check_attention(out, lse, ref, ref_lse, torch.bfloat16, "sk %s grid %s call %d" % (name, grid, call))


def test_stream_k_falls_back_for_appends_and_parts(monkeypatch):
    """Calls the stream-K form does not compute (a fused append, an attention
    part) take the split layout on the same plan and workspace."""
    dev = device()
    _sk_env(monkeypatch, 5)
    w = synth.Workload("skapp", 2, 4, 4, 128, 16, torch.bfloat16, [300, 500], [3, 2], 64,
                       appends_per_seq=1, permute_pages=True, seed=78)
    p = synth.make_problem(w)
    g = p.to(dev)
    out, _ = d2f.block_attn(g.q, g.k_win, g.v_win, g.k_pool, g.v_pool, g.page_table, g.ctx_len,
                            g.q_start, block_size=16, max_q_per_seq=p.max_q_per_seq,
                            max_ctx=p.max_ctx, want_lse=False, append_src_row=g.src_row,
                            append_dst_page=g.dst_page)
    torch.cuda.synchronize()
    ref, _ = _ref(p)
    check_attention(out, None, ref, None, torch.bfloat16, "sk fallback, fused append")
    for s_, d_ in zip(p.src_row.tolist(), p.dst_page.tolist()):
        assert torch.equal(g.k_pool[d_].cpu(), p.k_win[s_:s_ + 16].transpose(0, 1))
    cached, lse_c = _part(g, p, d2f.ATTN_CACHED)
    ref_c, ref_lse_c = _ref_part(p, oracle.ATTN_CACHED)
    check_attention(cached, lse_c, ref_c, ref_lse_c, torch.bfloat16, "sk fallback, cached part")


@pytest.mark.parametrize("name", ["llada", "ragged", "dream", "long_b16", "long_b32"])
def test_cache_ready_flag(name):
    """D2F_ATTN_CACHE_READY: the producers read the page table and layout and load
    cached tiles before waiting for the preceding kernel. Same results, alone and
    replayed from a CUDA graph where each attention follows a commit (which writes
    no cache) under programmatic dependent launch."""
    dev = device()
    w = synth.small(name)
    p = synth.make_problem(w)
    g = p.to(dev)
    ref, ref_lse = _ref(p)
    kw = dict(block_size=w.block_size, max_q_per_seq=p.max_q_per_seq, max_ctx=p.max_ctx,
              cache_ready=True)
    out, lse = d2f.block_attn(g.q, g.k_win, g.v_win, g.k_pool, g.v_pool, g.page_table, g.ctx_len,
                              g.q_start, **kw)
    torch.cuda.synchronize()
    check_attention(out, lse, ref, ref_lse, w.dtype, "cache_ready " + name)
    ws = d2f.attn_workspace(dev, batch=w.batch, total_q=w.total_q, max_q_per_seq=p.max_q_per_seq,
                            max_ctx=p.max_ctx, num_heads_q=w.num_heads_q,
                            num_heads_kv=w.num_heads_kv, head_dim=w.head_dim,
                            block_size=w.block_size)
    wsc = d2f.commit_workspace(dev, total_q=w.total_q, vocab=w.vocab, block_size=w.block_size)
    outs = [torch.empty_like(g.q) for _ in range(3)]
    lses = [torch.empty(g.q.shape[:2], dtype=torch.float32, device=dev) for _ in range(3)]
    toks = [g.tokens.clone() for _ in range(3)]
    msks = [g.masked.clone() for _ in range(3)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # warm-up outside the capture (function attributes)
        d2f.commit(g.logits, g.tokens.clone(), g.masked.clone(), g.q_start, g.block_phase, g.tau,
                   block_size=w.block_size, mask_id=p.mask_id, workspace=wsc)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for i in range(3):
            d2f.commit(g.logits, toks[i], msks[i], g.q_start, g.block_phase, g.tau,
                       block_size=w.block_size, mask_id=p.mask_id, workspace=wsc)
            d2f.block_attn(g.q, g.k_win, g.v_win, g.k_pool, g.v_pool, g.page_table, g.ctx_len,
                           g.q_start, out=outs[i], lse=lses[i], workspace=ws, **kw)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for i in range(3):
        check_attention(outs[i], lses[i], ref, ref_lse, w.dtype, "cache_ready graph %d" % i)
