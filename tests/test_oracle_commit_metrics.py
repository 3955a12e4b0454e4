"""Pins for the oracle's alternative confidences (CPU only): negative entropy,
top-1 / top-2 probability margin and logit gap.

Checked against hand-worked closed forms (tests/golden/commit_metrics_hand.txt),
against an independent SciPy / NumPy restatement on seeded random rows (softmax,
entropy and a sort for the top two), and on commit decisions where the metrics
rank the same two positions differently.
"""
import math
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NS = {"__builtins__": {}}
FN = {"ln": math.log, "e": math.e}
METRICS = {"negent": 1, "margin": 2, "gap": 3}


def _golden():
    rows = []
    with open(os.path.join(GOLDEN, "commit_metrics_hand.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kv = dict((a.strip(), b.strip()) for a, b in (p.split("=", 1) for p in line.split(";")))
            rows.append(([eval(t, NS, FN) for t in kv["row"].split()],
                         {k: eval(kv[k], NS, FN) for k in METRICS}, int(kv["a"])))
    return rows


ROWS = _golden()


def _conf(oracle, logits, metric):
    n = logits.shape[0]
    res = oracle.commit(logits, torch.zeros(n, dtype=torch.int32), torch.ones(n, dtype=torch.uint8),
                        torch.tensor([0, n], dtype=torch.int32), torch.zeros(n, dtype=torch.uint8),
                        torch.tensor([1e9]), 1, logits.shape[1], metric=metric)
    return res["conf"], res["argmax"], res


@pytest.mark.parametrize("name", list(METRICS))
@pytest.mark.parametrize("k", range(len(ROWS)))
def test_hand_rows(oracle, name, k):
    row, want, a = ROWS[k]
    logits = torch.tensor([row], dtype=torch.float32)
    conf, amax, _ = _conf(oracle, logits, METRICS[name])
    assert amax[0].item() == a
    # logits are float32 roundings of ln c: a few 1e-7 of slack
    assert abs(conf[0].item() - want[name]) <= 1e-6 * max(1.0, abs(want[name])), (conf[0].item(), want)


def _restated(x):
    """Independent NumPy / SciPy restatement in float64."""
    from scipy.special import softmax
    from scipy.stats import entropy
    x = x.astype(np.float64)
    p = softmax(x, axis=1)
    top = np.sort(x, axis=1)[:, ::-1]
    ps = np.sort(p, axis=1)[:, ::-1]
    return {"negent": -entropy(p, axis=1), "margin": ps[:, 0] - ps[:, 1], "gap": top[:, 0] - top[:, 1],
            "argmax": np.argmax(x, axis=1)}


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_against_scipy_restatement(oracle, seed, dtype):
    pytest.importorskip("scipy")
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(24, 3001, generator=g) * 3.0
    x[::3, 17] += 9.0  # planted peaks on some rows
    x[1::5, 5] = x[1::5, 9]  # exact ties at (possibly) the top
    x = x.to(dtype)
    ref = _restated(x.float().numpy())
    for name, m in METRICS.items():
        conf, amax, _ = _conf(oracle, x, m)
        np.testing.assert_allclose(conf.numpy(), ref[name], rtol=2e-6, atol=2e-6, err_msg=name)
        assert (amax.numpy() == ref["argmax"]).all()


def test_metrics_rank_positions_differently(oracle):
    """Rows A = [ln 4, 0, 0, 0] and B = [ln 4, ln 3, -30, -30] have (almost) the
    same largest probability 4/7, but B has the lower entropy and A the larger
    margin and gap: an aggressive block {A, B} with an unreachable threshold
    commits B under negative entropy and A under margin, gap and probability."""
    ln = math.log
    logits = torch.tensor([[ln(4), 0, 0, 0], [ln(4), ln(3), -30.0, -30.0]], dtype=torch.float32)
    want = {0: 0, 1: 1, 2: 0, 3: 0}  # metric -> committed position
    for metric, pos in want.items():
        res = oracle.commit(logits, torch.zeros(2, dtype=torch.int32), torch.ones(2, dtype=torch.uint8),
                            torch.tensor([0, 2], dtype=torch.int32), torch.ones(1, dtype=torch.uint8),
                            torch.tensor([1e9]), 2, 4, metric=metric)
        assert res["masked"].tolist() == [int(pos != 0), int(pos != 1)], (metric, res["masked"])
        assert res["block_remaining"].tolist() == [1]


@pytest.mark.parametrize("metric", [1, 2, 3])
def test_threshold_in_metric_units_is_strict(oracle, metric):
    """Conservative blocks commit c > tau, in the metric's own units: tau equal to
    a row's confidence leaves it masked, tau just below commits it."""
    logits = torch.tensor([[math.log(6), math.log(3), 0]], dtype=torch.float32)
    conf, _, _ = _conf(oracle, logits, metric)
    c = conf[0].item()
    for tau, committed in ((c, False), (float(np.nextafter(np.float32(c), np.float32(-np.inf))), True)):
        res = oracle.commit(logits, torch.zeros(1, dtype=torch.int32), torch.ones(1, dtype=torch.uint8),
                            torch.tensor([0, 1], dtype=torch.int32), torch.zeros(1, dtype=torch.uint8),
                            torch.tensor([tau]), 1, 3, metric=metric)
        assert res["masked"].item() == (0 if committed else 1)


def _early_problem():
    """Two sequences of two blocks of 2 (vocab 4, float32 logits). Sequence 0:
    masked rows with logit gaps 3, 5 and 4 (row 1 committed earlier); sequence 1:
    gaps 6, 6, 0.5 and 7."""
    rows = [[3, 0, 0, 0], [0, 0, 0, 0], [0, 5, 0, 0], [0, 0, 4, -1],
            [6, 0, 0, 0], [0, 6, 0, 0], [0.5, 0, 0, 0], [0, 0, 0, 7]]
    logits = torch.tensor(rows, dtype=torch.float32)
    tokens = torch.full((8,), 4, dtype=torch.int32)
    tokens[1] = 2
    masked = torch.ones(8, dtype=torch.uint8)
    masked[1] = 0
    q_start = torch.tensor([0, 4, 8], dtype=torch.int32)
    return logits, tokens, masked, q_start


@pytest.mark.parametrize("metric", [0, 2, 3])
def test_early_commit_of_whole_sequences(oracle, metric):
    """Prophet's early commit: a sequence whose smallest logit gap over its masked
    positions exceeds its threshold commits them all with their greedy tokens
    (stopped = 1, block_remaining = 0); a sequence with one position at or below
    the threshold keeps the block rule (here: nothing passes tau)."""
    logits, tokens, masked, q_start = _early_problem()
    phase = torch.zeros(4, dtype=torch.uint8)
    tau = torch.tensor([1e9, 1e9])
    for gap0, gap1, stop in ((2.5, 0.4, (1, 1)), (3.0, 0.5, (0, 0)), (2.9, 5.0, (1, 0))):
        res = oracle.commit(logits, tokens, masked, q_start, phase, tau, 2, 4, metric=metric,
                            early_gap=torch.tensor([gap0, gap1]))
        assert res["stopped"].tolist() == list(stop), (gap0, gap1, res["stopped"])
        want_tok = [0, 2, 1, 2] if stop[0] else [4, 2, 4, 4]
        want_tok += [0, 1, 0, 3] if stop[1] else [4, 4, 4, 4]
        assert res["tokens"].tolist() == want_tok
        assert res["masked"].tolist() == ([0, 0, 0, 0] if stop[0] else [1, 0, 1, 1]) + \
            ([0, 0, 0, 0] if stop[1] else [1, 1, 1, 1])
        assert res["block_remaining"].tolist() == ([0, 0] if stop[0] else [1, 2]) + \
            ([0, 0] if stop[1] else [2, 2])


def test_early_commit_leaves_the_block_rule_otherwise(oracle):
    """Without early_gap the result equals the plain commit; a sequence with
    nothing masked never stops."""
    logits, tokens, masked, q_start = _early_problem()
    phase = torch.tensor([1, 0, 1, 0], dtype=torch.uint8)
    tau = torch.tensor([4.5, 6.5])
    plain = oracle.commit(logits, tokens, masked, q_start, phase, tau, 2, 4, metric=3)
    off = oracle.commit(logits, tokens, masked, q_start, phase, tau, 2, 4, metric=3,
                        early_gap=torch.tensor([1e9, 1e9]))
    for k in ("tokens", "masked", "block_remaining", "conf", "argmax"):
        assert torch.equal(plain[k], off[k]), k
    assert off["stopped"].tolist() == [0, 0]
    none = torch.zeros(8, dtype=torch.uint8)
    res = oracle.commit(logits, tokens, none, q_start, phase, tau, 2, 4, metric=3,
                        early_gap=torch.tensor([-1.0, -1.0]))
    assert res["stopped"].tolist() == [0, 0]
    assert torch.equal(res["tokens"], tokens)
