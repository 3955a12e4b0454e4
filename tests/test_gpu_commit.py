"""GPU parity of d2f_commit against the CPU oracle.

Greedy tokens bit-exact; confidence within 1e-5 relative; committed tokens and
masks bit-exact outside the reported |p - tau| < 1e-5 band and aggressive
near-ties. Covers every workload's logits (full size for LLaDA, Dream and the
ragged batch), tie-heavy rows, tau = 0 / 1, Dream's shifted logit rows, padded
and unaligned row strides, float32 logits, split counts, block sizes 1..32.
"""
import pytest
import torch

import oracle
from block_causal_kv_gb300 import d2f, synth
from gpu_common import commit_compare, device

pytestmark = pytest.mark.gpu


def _gpu_commit(p, dev, phase=None, tau=None, num_splits=0, logit_row=None, logits=None,
                metric=0):
    g = p.to(dev)
    phase = g.block_phase if phase is None else phase.to(dev)
    tau = g.tau if tau is None else tau.to(dev)
    lg = g.logits if logits is None else logits.to(dev)
    lr = None if logit_row is None else logit_row.to(dev)
    res = d2f.commit(lg, g.tokens, g.masked, g.q_start, phase, tau, block_size=p.w.block_size,
                     mask_id=p.mask_id, logit_row=lr, num_splits=num_splits, metric=metric)
    torch.cuda.synchronize()
    return g, res, phase, tau


# per metric: (absolute slack on the confidence, |c - tau| band excluded from
# the bit-exact decisions); the logit gap is exact
METRIC_TOL = {0: (0.0, None), 1: (2e-5, 1e-4), 2: (2e-6, 1e-5), 3: (0.0, 1e-6)}


def _check(p, dev, phase=None, tau=None, num_splits=0, logit_row=None, logits=None, metric=0,
           label=None, max_frac=None):
    g, res, phase, tau = _gpu_commit(p, dev, phase, tau, num_splits, logit_row, logits, metric)
    ref = oracle.commit(p.logits if logits is None else logits, p.tokens, p.masked, p.q_start,
                        phase.cpu(), tau.cpu(), p.w.block_size, p.mask_id,
                        logit_row=logit_row, metric=metric)
    atol, band = METRIC_TOL[metric]
    return commit_compare(p, g.tokens, g.masked, res["conf"], res["argmax"],
                          res["block_remaining"], phase, tau, ref, band=band, atol=atol,
                          label=label, max_frac=max_frac)


@pytest.mark.parametrize("name", ["tiny", "llada", "ragged", "dream", "long_b8", "long_b32"])
@pytest.mark.parametrize("splits", [0, 1, 7])
def test_small_workloads(name, splits):
    dev = device()
    w = synth.workload("tiny") if name == "tiny" else synth.small(name)
    nb, nt = _check(synth.make_problem(w), dev, num_splits=splits,
                    label="%s small, splits %d" % (name, splits), max_frac=0.02)
    print("%s s%d: band %d tie %d" % (name, splits, nb, nt))


@pytest.mark.parametrize("name", ["llada", "ragged", "dream", "long_b8", "long_b16", "long_b32"])
def test_full_size(name):
    """Every full-size workload in the bench's launch configuration (automatic
    plan): the excluded positions are recorded and stay below 2 % of the masked
    ones."""
    dev = device()
    p = synth.make_problem(synth.workload(name))
    nb, nt = _check(p, dev, label="%s full size" % name, max_frac=0.02)
    print("%s full: rows %d, excluded band %d tie %d" % (name, p.w.total_q, nb, nt))


def _tiny_vocab(seed, B=8, vocab=300, **over):
    kw = dict(masked_frac=0.6, taus=(0.05, 0.3, 0.6), logit_sigma=1.5)
    kw.update(over)
    w = synth.Workload("c", 3, 1, 1, 8, B, torch.bfloat16, [0, 0, 0], [2, 1, 3], vocab,
                       seed=seed, **kw)
    return synth.make_problem(w)


@pytest.mark.parametrize("seed", range(4))
def test_random_phases_and_thresholds(seed):
    dev = device()
    p = _tiny_vocab(seed)
    phase = torch.randint(0, 2, p.block_phase.shape, generator=torch.Generator().manual_seed(seed),
                          dtype=torch.uint8)
    _check(p, dev, phase=phase)


def test_argmax_ties_take_lowest_index():
    dev = device()
    p = _tiny_vocab(3, vocab=4096)
    g = torch.Generator().manual_seed(5)
    tied = (torch.randint(0, 3, p.logits.shape, generator=g).float() * 0.5).to(torch.bfloat16)
    _check(p, dev, logits=tied, num_splits=5)


def test_tau_zero_and_one():
    dev = device()
    p = _tiny_vocab(8)
    all_aggr = torch.ones_like(p.block_phase)
    _check(p, dev, phase=all_aggr, tau=torch.ones_like(p.tau))
    _check(p, dev, tau=torch.zeros_like(p.tau))


def test_logit_row_shift_and_padded_stride():
    dev = device()
    w = synth.Workload("s", 2, 1, 1, 8, 16, torch.bfloat16, [0, 0], [2, 1], 1001,
                       logit_row_pad=24, masked_frac=0.8, seed=21)
    p = synth.make_problem(w)
    shift = torch.clamp(torch.arange(p.w.total_q, dtype=torch.int32) - 1, min=0)
    _check(p, dev, logit_row=shift)


def test_unaligned_rows_use_the_scalar_path():
    dev = device()
    w = synth.Workload("u", 1, 1, 1, 8, 8, torch.bfloat16, [0], [2], 999, logit_row_pad=2,
                       seed=22)
    p = synth.make_problem(w)  # row stride 1001 elements: rows not 16-byte aligned
    _check(p, dev, num_splits=3)


@pytest.mark.parametrize("splits", [0, 3, 7])
def test_vector_path_with_a_ragged_row_end(splits):
    # vocab 1001 with a 1008-element row stride: rows start 16-byte aligned (the
    # 128-bit path), and each row ends inside a vector, so the last slice of every
    # row finishes with scalar loads
    dev = device()
    w = synth.Workload("v", 2, 1, 1, 8, 8, torch.bfloat16, [0, 0], [3, 2], 1001,
                       logit_row_pad=7, masked_frac=0.7, seed=23)
    p = synth.make_problem(w)
    assert (p.logits.stride(0) * 2) % 16 == 0 and p.w.vocab % 8 != 0
    _check(p, dev, num_splits=splits)


@pytest.mark.parametrize("B", [1, 4, 8])
@pytest.mark.parametrize("metric", [0, 3])
def test_small_vocabulary_many_blocks(B, metric):
    # a 96-entry vocabulary over 224 rows: one slice per row, 28 to 224 blocks
    # decided by their last-arriving CTAs, random phases
    dev = device()
    w = synth.Workload("m", 4, 1, 1, 8, B, torch.bfloat16, [0] * 4, [64 // B, 40 // B, 96 // B, 24 // B],
                       96, masked_frac=0.6, taus=(0.05, 0.3, 0.6), logit_sigma=1.5, seed=40 + B)
    p = synth.make_problem(w)
    phase = torch.randint(0, 2, p.block_phase.shape, generator=torch.Generator().manual_seed(B),
                          dtype=torch.uint8)
    _check(p, dev, phase=phase, metric=metric)


def test_float32_logits():
    dev = device()
    p = synth.make_problem(synth.workload("tiny"))
    _check(p, dev, num_splits=2)


@pytest.mark.parametrize("B", [1, 4, 32])
def test_block_sizes(B):
    dev = device()
    p = _tiny_vocab(30 + B, B=B)
    phase = torch.randint(0, 2, p.block_phase.shape, generator=torch.Generator().manual_seed(B),
                          dtype=torch.uint8)
    _check(p, dev, phase=phase, num_splits=2)


def test_nothing_masked_and_repeated_calls():
    """Three calls in a row on the evolving state match the oracle applied three
    times (counters reset themselves); a batch with every position committed
    commits nothing, also with a different split count on the same workspace."""
    dev = device()
    p = _tiny_vocab(11)
    g = p.to(dev)
    ws = d2f.commit_workspace(dev, total_q=p.w.total_q, vocab=p.w.vocab, block_size=p.w.block_size,
                              num_splits=4)
    ref = {"tokens": p.tokens, "masked": p.masked}
    for _ in range(3):
        d2f.commit(g.logits, g.tokens, g.masked, g.q_start, g.block_phase, g.tau,
                   block_size=p.w.block_size, mask_id=p.mask_id, num_splits=4, workspace=ws)
        ref = oracle.commit(p.logits, ref["tokens"], ref["masked"], p.q_start, p.block_phase,
                            p.tau, p.w.block_size, p.mask_id)
    torch.cuda.synchronize()
    assert torch.equal(g.tokens.cpu(), ref["tokens"])
    assert torch.equal(g.masked.cpu(), ref["masked"])
    done = torch.zeros_like(g.masked)
    res = d2f.commit(g.logits, g.tokens, done, g.q_start, torch.ones_like(g.block_phase), g.tau,
                     block_size=p.w.block_size, mask_id=p.mask_id, num_splits=2, workspace=ws)
    torch.cuda.synchronize()
    assert int(res["block_remaining"].sum()) == 0
    assert torch.all(res["conf"] == -1)


# tau in each metric's units, near the middle of its range on these logits
METRIC_TAU = {1: (-2.5, -0.5, -0.05), 2: (0.3, 0.6, 0.9), 3: (1.0, 3.0, 6.0)}


@pytest.mark.parametrize("metric", [1, 2, 3])
@pytest.mark.parametrize("name", ["tiny", "llada", "ragged", "dream"])
@pytest.mark.parametrize("splits", [0, 5])
def test_confidence_metrics(metric, name, splits):
    """Negative entropy, probability margin and logit gap in the same streaming
    pass (d2f_commit_metric): confidence, greedy token and commit decisions match
    the oracle's on every workload shape (float32 Tiny on the scalar path),
    with tau drawn in the metric's own units and random phases."""
    dev = device()
    w = synth.workload("tiny") if name == "tiny" else synth.small(name)
    p = synth.make_problem(w)
    g = torch.Generator().manual_seed(100 + metric)
    taus = torch.tensor(METRIC_TAU[metric], dtype=torch.float32)
    tau = taus[torch.randint(0, len(taus), (p.w.batch,), generator=g)]
    phase = torch.randint(0, 2, p.block_phase.shape, generator=g, dtype=torch.uint8)
    lr = None
    if name == "dream":  # Dream's one-position shift of the logit rows
        lr = torch.clamp(torch.arange(p.w.total_q, dtype=torch.int32) - 1, min=0)
    nb, nt = _check(p, dev, phase=phase, tau=tau, num_splits=splits, logit_row=lr, metric=metric)
    print("%s m%d s%d: band %d tie %d" % (name, metric, splits, nb, nt))


@pytest.mark.parametrize("metric", [1, 2, 3])
def test_confidence_metrics_ties_and_unaligned_rows(metric):
    """Tie-heavy logits (repeated maxima: margin and gap 0) and rows that are not
    16-byte aligned (scalar path)."""
    dev = device()
    p = _tiny_vocab(3, vocab=4096)
    g = torch.Generator().manual_seed(7)
    tied = (torch.randint(0, 3, p.logits.shape, generator=g).float() * 0.5).to(torch.bfloat16)
    _check(p, dev, logits=tied, num_splits=5, metric=metric,
           tau=torch.full_like(p.tau, METRIC_TAU[metric][1]))
    w = synth.Workload("u", 1, 1, 1, 8, 8, torch.bfloat16, [0], [2], 999, logit_row_pad=2, seed=23)
    _check(synth.make_problem(w), dev, num_splits=3, metric=metric,
           tau=torch.full((1,), METRIC_TAU[metric][0]))


def test_unknown_metric_is_rejected():
    dev = device()
    p = _tiny_vocab(2)
    with pytest.raises(d2f.D2FError):
        _gpu_commit(p, dev, metric=7)


def _early_hand_problem():
    rows = [[3, 0, 0, 0], [0, 0, 0, 0], [0, 5, 0, 0], [0, 0, 4, -1],
            [6, 0, 0, 0], [0, 6, 0, 0], [0.5, 0, 0, 0], [0, 0, 0, 7]]
    w = synth.Workload("e", 2, 1, 1, 8, 2, torch.float32, [0, 0], [2, 2], 4, seed=30)
    p = synth.make_problem(w)
    p.logits = torch.tensor(rows, dtype=torch.float32)
    p.tokens = torch.full((8,), 4, dtype=torch.int32)
    p.tokens[1] = 2
    p.masked = torch.ones(8, dtype=torch.uint8)
    p.masked[1] = 0
    p.mask_id = 4
    return p


def _early_check(p, dev, metric, early_gap, phase=None, tau=None, num_splits=0):
    g = p.to(dev)
    phase = g.block_phase if phase is None else phase.to(dev)
    tau = g.tau if tau is None else tau.to(dev)
    stopped = torch.full((p.w.batch,), 9, dtype=torch.uint8, device=dev)
    res = d2f.commit(g.logits, g.tokens, g.masked, g.q_start, phase, tau, block_size=p.w.block_size,
                     mask_id=p.mask_id, num_splits=num_splits, metric=metric,
                     early_gap=early_gap.to(dev), stopped=stopped)
    torch.cuda.synchronize()
    ref = oracle.commit(p.logits, p.tokens, p.masked, p.q_start, phase.cpu(), tau.cpu(),
                        p.w.block_size, p.mask_id, metric=metric, early_gap=early_gap)
    assert torch.equal(stopped.cpu(), ref["stopped"]), (stopped.cpu(), ref["stopped"])
    atol, band = METRIC_TOL[metric]
    commit_compare(p, g.tokens, g.masked, res["conf"], res["argmax"], res["block_remaining"],
                   phase, tau, ref, band=band, atol=atol)
    return ref["stopped"]


@pytest.mark.parametrize("metric", [0, 2, 3])
def test_early_commit_hand_sequences(metric):
    """Prophet's early commit on hand-built sequences (gaps 3/5/4 and 6/6/0.5/7):
    stopped flags, tokens, masks and block_remaining as the oracle's."""
    dev = device()
    p = _early_hand_problem()
    tau = torch.tensor([1e9, 1e9])
    for gaps, stop in (((2.5, 0.4), [1, 1]), ((3.0, 0.5), [0, 0]), ((2.9, 5.0), [1, 0])):
        got = _early_check(p, dev, metric, torch.tensor(gaps), tau=tau)
        assert got.tolist() == stop


@pytest.mark.parametrize("metric", [0, 3])
@pytest.mark.parametrize("name", ["llada", "ragged", "dream"])
@pytest.mark.parametrize("splits", [0, 3])
def test_early_commit_workloads(metric, name, splits):
    """Thresholds just below / above each sequence's smallest logit gap (from the
    oracle), alternating: half the sequences stop. Random phases."""
    dev = device()
    p = synth.make_problem(synth.small(name))
    gaps = oracle.commit(p.logits, p.tokens, p.masked, p.q_start, p.block_phase, p.tau,
                         p.w.block_size, p.mask_id, metric=3)["conf"]
    m0 = p.masked.bool()
    thr = []
    for b in range(p.w.batch):
        r0, r1 = int(p.q_start[b]), int(p.q_start[b + 1])
        g = gaps[r0:r1][m0[r0:r1]]
        gmin = float(g.min()) if len(g) else 0.0
        thr.append(gmin - 0.25 if b % 2 == 0 else gmin + 0.25)
    g = torch.Generator().manual_seed(41)
    phase = torch.randint(0, 2, p.block_phase.shape, generator=g, dtype=torch.uint8)
    stop = _early_check(p, dev, metric, torch.tensor(thr, dtype=torch.float32), phase=phase,
                        num_splits=splits)
    print("%s m%d s%d: stopped %s" % (name, metric, splits, stop.tolist()))


@pytest.mark.parametrize("B", [1, 4])
def test_early_commit_small_vocabulary_many_blocks(B):
    """The early commit over many small blocks (a 96-entry vocabulary, 224 rows):
    thresholds 0.1 below / above each sequence's smallest gap, alternating."""
    dev = device()
    w = synth.Workload("m", 4, 1, 1, 8, B, torch.bfloat16, [0] * 4, [64 // B, 40 // B, 96 // B, 24 // B],
                       96, masked_frac=0.6, taus=(0.05, 0.3, 0.6), logit_sigma=1.5, seed=50 + B)
    p = synth.make_problem(w)
    gaps = oracle.commit(p.logits, p.tokens, p.masked, p.q_start, p.block_phase, p.tau,
                         p.w.block_size, p.mask_id, metric=3)["conf"]
    m0 = p.masked.bool()
    thr = []
    for b in range(p.w.batch):
        r0, r1 = int(p.q_start[b]), int(p.q_start[b + 1])
        g = gaps[r0:r1][m0[r0:r1]]
        thr.append((float(g.min()) if len(g) else 0.0) + (-0.1 if b % 2 == 0 else 0.1))
    stop = _early_check(p, dev, 3, torch.tensor(thr, dtype=torch.float32))
    assert stop.tolist() == [1, 0, 1, 0]


def test_early_commit_rejects_entropy():
    dev = device()
    p = _tiny_vocab(2)
    g = p.to(dev)
    with pytest.raises(d2f.D2FError):
        d2f.commit(g.logits, g.tokens, g.masked, g.q_start, g.block_phase, g.tau,
                   block_size=p.w.block_size, mask_id=p.mask_id, metric=1,
                   early_gap=torch.zeros(p.w.batch, device=dev))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_planted_threshold_boundary(dtype):
    """Rows planted just outside the reported band: every sequence holds one
    block whose row 0 is the planted row, and its tau is that row's confidence
    (from the oracle) moved by +-2e-5 or +-1e-4, in conservative and aggressive
    blocks (in aggressive blocks row 1 is made clearly more confident, so the
    planted row's fate is the threshold test), at the full LLaDA vocabulary.
    Every decision outside the 1e-5 band is bit-exact, and each planted row
    commits exactly when tau lies below its confidence."""
    dev = device()
    V, B = 126464, 16
    deltas = [2e-5, -2e-5, 1e-4, -1e-4]
    nseq = 2 * 2 * len(deltas)
    w = synth.Workload("plant", nseq, 1, 1, 8, B, dtype, [0] * nseq, [1] * nseq, V,
                       masked_frac=0.75, seed=77)
    p = synth.make_problem(w)
    p.masked[0::B] = 1          # the planted row is masked
    p.tokens[0::B] = p.mask_id
    phase = torch.tensor([(b // len(deltas)) % 2 for b in range(nseq)], dtype=torch.uint8)
    for b in range(nseq):
        if phase[b] == 1:       # a clearly more confident row ahead of the planted one
            r = b * B
            row = p.logits[r].clone()
            row[int(torch.argmax(row.float()))] += 8
            p.logits[r + 1] = row
            p.masked[r + 1] = 1
            p.tokens[r + 1] = p.mask_id
    conf = oracle.commit(p.logits, p.tokens, p.masked, p.q_start, phase,
                         torch.full((nseq,), 2.0), B, p.mask_id)["conf"]
    d = torch.tensor([deltas[b % len(deltas)] for b in range(nseq)], dtype=torch.float64)
    tau = (conf[0::B].double() + d).float()
    assert bool(((tau.double() - conf[0::B].double()).abs() >= 1.5e-5).all())
    p.tau = tau
    p.block_phase = phase
    g, res, _, _ = _gpu_commit(p, dev, phase=phase, tau=tau)
    ref = oracle.commit(p.logits, p.tokens, p.masked, p.q_start, phase, tau, B, p.mask_id)
    nb, nt = commit_compare(p, g.tokens, g.masked, res["conf"], res["argmax"],
                            res["block_remaining"], phase, tau, ref,
                            label="planted boundary %s" % str(dtype).split(".")[-1])
    planted = torch.arange(nseq) * B
    gm = g.masked.cpu()[planted]
    expect_commit = d < 0        # tau below p: p > tau holds
    assert torch.equal(gm == 0, expect_commit), (gm, d)
    assert torch.equal(g.tokens.cpu()[planted][expect_commit], ref["argmax"][planted][expect_commit])
