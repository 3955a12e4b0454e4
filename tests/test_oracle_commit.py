"""Pins for the oracle's confidence commit (CPU only).

Checked against hand-worked closed forms (tests/golden/commit_hand.txt), a
vectorised SciPy/NumPy restatement, and invariants the pages fix: an aggressive
block with a masked position commits at least one; tau >= 1 in the aggressive
phase is LLaDA's low-confidence remasking with one token per step; tau = 0
commits every masked position; committed positions never change.
"""
import math
import os

import numpy as np
import pytest
import torch

import bruteforce
from block_causal_kv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NS = {"__builtins__": {}}
FN = {"ln": math.log, "e": math.e}


def _golden():
    rows, blocks = [], []
    with open(os.path.join(GOLDEN, "commit_hand.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kv = dict((a.strip(), b.strip()) for a, b in (p.split("=", 1) for p in line.split(";")))
            if "row" in kv:
                rows.append(([eval(t, NS, FN) for t in kv["row"].split()],
                             eval(kv["p"], NS, FN), int(kv["a"])))
            else:
                blocks.append(kv)
    return rows, blocks


ROWS, BLOCKS = _golden()


def test_hand_rows_confidence(oracle):
    V = 4
    logits = torch.tensor([r[0] for r in ROWS], dtype=torch.float32)
    n = len(ROWS)
    tokens = torch.full((n,), V, dtype=torch.int32)
    masked = torch.ones(n, dtype=torch.uint8)
    res = oracle.commit(logits, tokens, masked, torch.tensor([0, n], dtype=torch.int32),
                        torch.zeros(n, dtype=torch.uint8), torch.tensor([0.9]), 1, V)
    for i, (_, p, a) in enumerate(ROWS):
        assert res["argmax"][i].item() == a
        # logits are float32 roundings of ln c: p is exact to ~1e-7 relative
        assert abs(res["conf"][i].item() - p) <= 2e-7 * p, (i, res["conf"][i].item(), p)


@pytest.mark.parametrize("k", range(len(BLOCKS)))
def test_hand_blocks(oracle, k):
    blk = BLOCKS[k]
    V, B = 4, 4
    rows = blk["rows"].split()
    logits = torch.zeros(B, V)
    tokens = torch.full((B,), V, dtype=torch.int32)
    masked = torch.ones(B, dtype=torch.uint8)
    for u, spec in enumerate(rows):
        if spec.startswith("c"):
            masked[u] = 0
            tokens[u] = int(spec[1:])
            logits[u] = float("nan")  # a committed position is never read
        else:
            logits[u] = torch.tensor(ROWS[int(spec)][0])
    phase = torch.tensor([1 if blk["block"] == "aggressive" else 0], dtype=torch.uint8)
    res = oracle.commit(logits, tokens, masked, torch.tensor([0, B], dtype=torch.int32),
                        phase, torch.tensor([0.9]), B, V)
    assert res["tokens"].tolist() == [int(t) for t in blk["tokens"].split()]
    assert res["block_remaining"].tolist() == [int(blk["remaining"])]
    assert res["masked"].tolist() == [int(t == V) for t in res["tokens"].tolist()]


def test_threshold_is_strict_on_the_boundary(oracle):
    """ln 27 gives p = 0.9 exactly in real arithmetic; in float it rounds to the
    same float as tau = 0.9, and "above the threshold" is strict."""
    logits = torch.tensor([[math.log(27), 0, 0, 0]], dtype=torch.float32)
    p = oracle.commit(logits, torch.tensor([4], dtype=torch.int32), torch.ones(1, dtype=torch.uint8),
                      torch.tensor([0, 1], dtype=torch.int32), torch.zeros(1, dtype=torch.uint8),
                      torch.tensor([0.9]), 1, 4)
    conf = p["conf"][0].item()
    tau32 = torch.tensor(0.9).item()
    assert abs(conf - 0.9) < 1e-6
    assert (p["masked"][0].item() == 0) == (conf > tau32)


def _problem(seed, **over):
    base = dict(batch=3, num_heads_q=1, num_heads_kv=1, head_dim=4, block_size=8,
                ctx_lens=[0, 0, 0], window_blocks=[2, 1, 3], vocab=257, masked_frac=0.6,
                taus=(0.05, 0.2, 0.5), logit_sigma=2.0)
    base.update(over)
    w = synth.Workload("c", dtype=torch.bfloat16, seed=seed, **base)
    p = synth.make_problem(w)
    phase = torch.randint(0, 2, p.block_phase.shape, generator=torch.Generator().manual_seed(seed),
                          dtype=torch.uint8)
    return p, phase


@pytest.mark.parametrize("seed", range(10))
def test_against_vectorised_restatement(oracle, seed):
    p, phase = _problem(seed)
    B = p.w.block_size
    res = oracle.commit(p.logits, p.tokens, p.masked, p.q_start, phase, p.tau, B, p.mask_id)
    ref = bruteforce.commit(p.logits, p.tokens, p.masked, p.q_start, phase, p.tau, B, p.mask_id)
    np.testing.assert_array_equal(res["argmax"].numpy(), ref["argmax"])
    # both round a double-precision value to float: equal, or one ulp apart
    c, rc = res["conf"].numpy(), ref["conf"]
    assert np.all(np.abs(c - rc) <= np.spacing(np.abs(rc)))
    near = np.abs(rc - p.tau.numpy()[np.searchsorted(p.q_start.numpy(), np.arange(len(rc)), "right") - 1]) < 1e-6
    ok = ~near
    np.testing.assert_array_equal(res["tokens"].numpy()[ok], ref["tokens"][ok])
    np.testing.assert_array_equal(res["masked"].numpy()[ok], ref["masked"][ok])


@pytest.mark.parametrize("seed", range(6))
def test_invariants(oracle, seed):
    p, phase = _problem(seed, masked_frac=0.7)
    B = p.w.block_size
    res = oracle.commit(p.logits, p.tokens, p.masked, p.q_start, phase, p.tau, B, p.mask_id)
    m0 = p.masked.view(-1, B).bool()
    m1 = res["masked"].view(-1, B).bool()
    # committed positions never change
    was_committed = ~p.masked.bool()
    assert torch.equal(res["tokens"][was_committed], p.tokens[was_committed])
    assert not torch.any(m1 & ~m0)
    # still-masked rows carry the mask token; newly committed rows carry their argmax
    assert torch.all(res["tokens"][res["masked"].bool()] == p.mask_id)
    new = p.masked.bool() & ~res["masked"].bool()
    assert torch.equal(res["tokens"][new], res["argmax"][new])
    # remaining count
    assert torch.equal(res["block_remaining"], m1.sum(1).to(torch.int32))
    # aggressive blocks with a masked position commit at least one
    aggressive = phase.bool()
    has_masked = m0.any(1)
    committed = (m0 & ~m1).sum(1)
    assert torch.all(committed[aggressive & has_masked] >= 1)


@pytest.mark.parametrize("seed", range(4))
def test_tau_one_aggressive_is_single_top_confidence(oracle, seed):
    """tau >= 1 and every block aggressive: exactly one commit per block with a
    masked position, at its most confident masked position (LLaDA low-confidence
    remasking, one token per step per block)."""
    p, _ = _problem(seed, taus=(1.0,))
    B = p.w.block_size
    phase = torch.ones_like(p.block_phase)
    res = oracle.commit(p.logits, p.tokens, p.masked, p.q_start, phase, p.tau, B, p.mask_id)
    m0 = p.masked.view(-1, B).bool()
    m1 = res["masked"].view(-1, B).bool()
    conf = res["conf"].view(-1, B)
    for jb in range(m0.shape[0]):
        if not m0[jb].any():
            assert torch.equal(m0[jb], m1[jb])
            continue
        newly = (m0[jb] & ~m1[jb]).nonzero().flatten().tolist()
        assert len(newly) == 1
        c = torch.where(m0[jb], conf[jb], torch.tensor(-2.0))
        assert newly[0] == int(torch.argmax(c))  # torch.argmax: first maximum


def test_tau_zero_commits_everything(oracle):
    p, phase = _problem(3, taus=(0.0,))
    res = oracle.commit(p.logits, p.tokens, p.masked, p.q_start, phase, p.tau, p.w.block_size,
                        p.mask_id)
    assert int(res["masked"].sum()) == 0
    assert int(res["block_remaining"].sum()) == 0


def test_argmax_ties_take_lowest_index(oracle):
    """Rows quantised to a handful of values: the maximum repeats; the greedy token
    is its first occurrence."""
    g = torch.Generator().manual_seed(9)
    n, V = 16, 300
    logits = (torch.randint(0, 4, (n, V), generator=g).float() * 0.5).to(torch.bfloat16)
    res = oracle.commit(logits, torch.full((n,), V, dtype=torch.int32),
                        torch.ones(n, dtype=torch.uint8), torch.tensor([0, n], dtype=torch.int32),
                        torch.zeros(n // 8, dtype=torch.uint8), torch.tensor([0.9]), 8, V)
    x = logits.float().numpy()
    for r in range(n):
        first = int(np.nonzero(x[r] == x[r].max())[0][0])
        assert res["argmax"][r].item() == first
        cnt = int((x[r] == x[r].max()).sum())
        assert cnt > 1  # the test really exercises ties


def test_equal_confidence_ties_take_lowest_position(oracle):
    """Aggressive top-1 among equally confident masked positions: the lowest one."""
    V, B = 8, 4
    row = torch.tensor([1.0, 0, 0, 0, 0, 0, 0, 0])
    logits = torch.stack([row, row, row, row])
    masked = torch.tensor([0, 1, 1, 1], dtype=torch.uint8)
    tokens = torch.tensor([5, V, V, V], dtype=torch.int32)
    res = oracle.commit(logits, tokens, masked, torch.tensor([0, B], dtype=torch.int32),
                        torch.ones(1, dtype=torch.uint8), torch.tensor([0.99]), B, V)
    assert res["masked"].tolist() == [0, 0, 1, 1]
    assert res["tokens"].tolist() == [5, 0, V, V]


def test_logit_row_indirection_and_row_stride(oracle):
    """Dream-style shift (position r predicted by logit row r - 1 of the window
    hidden states, "확산 언어 모델(Diffusion LLM)이란 무엇인가" §Dream 7B와 Dream-Coder)
    and a padded row stride: padding (NaN) is never read."""
    w = synth.Workload("s", 1, 1, 1, 4, 8, torch.bfloat16, [0], [2], 101, logit_row_pad=13,
                       seed=5, masked_frac=0.8)
    p = synth.make_problem(w)
    n = p.tokens.shape[0]
    shift = torch.clamp(torch.arange(n, dtype=torch.int32) - 1, min=0)
    phase = torch.tensor([1, 0], dtype=torch.uint8)
    res = oracle.commit(p.logits, p.tokens, p.masked, p.q_start, phase, p.tau, 8, p.mask_id,
                        logit_row=shift)
    dense = p.logits[shift.long()].contiguous()
    ref = oracle.commit(dense, p.tokens, p.masked, p.q_start, phase, p.tau, 8, p.mask_id)
    for k in ("tokens", "masked", "conf", "argmax", "block_remaining"):
        assert torch.equal(res[k], ref[k]), k
    assert not torch.isnan(res["conf"]).any()
