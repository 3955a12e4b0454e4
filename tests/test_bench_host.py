"""Host logic of bench.py that needs no GPU: the byte accounting of the attention
parts and the starting state of the device-driven step (--scheduler).
"""
import sys
import os

import pytest
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from block_causal_kv_gb300 import synth  # noqa: E402


def _padded(name):
    # the scheduler takes prompts padded to whole blocks (the full-size workloads are)
    if name == "llada":
        return synth.small("llada")
    return synth.Workload("dream_padded", 3, 14, 2, 128, 16, torch.bfloat16, [512, 304, 96],
                          [3, 3, 3], 256, appends_per_seq=1, permute_pages=True, seed=41)


@pytest.mark.parametrize("name", ["llada", "dream"])
def test_scheduler_snapshot_is_a_consistent_state(oracle, name):
    """The state every device-driven step starts from is one the scheduler accepts.
    Its layout, phases and append list are the workload's. The next call retires
    the blocks appended during the step and nothing else."""
    w = _padded(name)
    p = synth.make_problem(w)
    W = max(w.window_blocks)
    st = bench.sched_state_dict(p, W)
    assert torch.equal(st["q_start"], p.q_start) and torch.equal(st["ctx_len"], p.ctx_len)
    i32, u8, fields, const = bench.sched_snapshot(p, "cpu", W)
    assert torch.equal(u8, p.block_phase)
    off, shape = fields["n_append"]
    assert int(i32[off]) == len(p.src_row)
    off, shape = fields["app_src"]
    assert i32[off:off + len(p.src_row)].tolist() == p.src_row.tolist()
    out = oracle.window_step(st, w.block_size, W, p.mask_id, 0.5, 1.0)
    assert out["err"] == 0
    per_seq = torch.zeros(w.batch, dtype=torch.int32)
    qs = p.q_start.tolist()
    for r in p.src_row.tolist():
        per_seq[next(b for b in range(w.batch) if qs[b] <= r < qs[b + 1])] += 1
    assert torch.equal(out["ctx_len"], p.ctx_len + w.block_size * per_seq)
    # the listed pages stay where the workload put them
    for b in range(w.batch):
        c = int(p.ctx_len[b]) // w.block_size
        n = int(per_seq[b])
        assert torch.equal(out["page_table"][b, c:c + n], p.page_table[b, c:c + n])


def test_part_bytes_add_up():
    """The cached part's and the window part's algorithmic bytes add up to the whole
    attention's, plus the kept part's output and normaliser (written by one, read by
    the other) and Q read twice."""
    w = synth.small("dream")
    p = synth.make_problem(w)
    full = bench.algorithmic_bytes(p)[0]
    cached = bench.algorithmic_bytes(p, "cached")[0]
    window = bench.algorithmic_bytes(p, "window")[0]
    tq, H, D = w.total_q, w.num_heads_q, w.head_dim
    kept = tq * H * D * 2 + tq * H * 4
    q = tq * H * D * 2
    assert cached + window == full + q + 2 * kept


def test_attention_roofline_terms():
    """The attention's two roofline terms from the workload's own byte and flop
    counts: the Dream-shaped layer sits past the ridge (tensor-bound at the
    sustained dense peak), the LLaDA-shaped layer and the long context are
    HBM-bound, and the float32 path has no tensor term."""
    hbm, tf = 6791.7, 1714.0

    def terms(name, tensor=True, us=100.0):
        p = synth.make_problem(synth.workload(name))
        b = bench.algorithmic_bytes(p)[0]
        return b, bench.flops(p), bench.attn_roofline(b, bench.flops(p), hbm, tf, us, tensor)

    b, f, r = terms("dream")
    assert r["bound"] == "tensor"
    assert r["hbm_us"] == pytest.approx(b / (hbm * 1e9) * 1e6)
    assert r["tensor_us"] == pytest.approx(f / (tf * 1e12) * 1e6)
    assert r["frac_of_roofline"] == pytest.approx(r["tensor_us"] / 100.0)
    assert terms("llada")[2]["bound"] == "hbm"
    r = terms("tiny", tensor=False)[2]
    assert r["tensor_us"] is None and r["bound"] == "hbm"
