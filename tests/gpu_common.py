"""Helpers shared by the GPU parity tests: build/load, tolerances, oracle runs.

Tolerances
  attention, bf16 operands: max |gpu - oracle| <= 2e-2 and mean <= 2e-3 on the
      output (the hot path's stated bar); lse within 1.1e-2: P is exponentiated
      from a bf16-rounded argument x (relative rounding 2^-9), and with the lazy
      rescale x reaches +8 (log2 units) before the reference moves, so a dominant
      term can be off by 8 * 2^-9 * ln 2 relative: ln(1 + 0.0108) = 0.0108 on the
      natural-log normaliser.
  attention, float32 operands: the CUDA-core path accumulates in float32 over at
      most a few thousand keys of unit-scale values, so its error is ~1e-6; the
      bar is 1e-4 max / 1e-5 mean.
  commit: greedy tokens bit-exact; confidence relative error <= 1e-5; tokens and
      masks bit-exact except positions with |p - tau| < 1e-5 and, in aggressive
      blocks, the rows within 1e-5 of the block's best masked confidence when
      there are several (their commit count must still match); both reported.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

ATTN_TOL = {torch.bfloat16: (2e-2, 2e-3), torch.float32: (1e-4, 1e-5)}
LSE_TOL = 1.1e-2
CONF_RTOL = 1e-5
BAND = 1e-5


def device():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def attn_errors(out, ref):
    err = (out.double().cpu() - ref).abs()
    return float(err.max()), float(err.mean())


def check_attention(out, lse, ref, ref_lse, dtype, label=""):
    mx, mean = attn_errors(out, ref)
    tmax, tmean = ATTN_TOL[dtype]
    assert mx <= tmax and mean <= tmean, "%s max %.3g mean %.3g" % (label, mx, mean)
    if lse is not None:
        lg, lr = lse.double().cpu(), ref_lse
        # rows without any visible key carry lse = -inf on both sides
        inf = torch.isneginf(lr)
        assert torch.equal(torch.isneginf(lg), inf), "%s lse -inf rows differ" % label
        le = float((lg[~inf] - lr[~inf]).abs().max()) if (~inf).any() else 0.0
        assert le <= LSE_TOL, "%s lse err %.3g" % (label, le)
    return mx, mean


def record_excluded(label, n_masked, n_band, n_tie, max_frac=None, n_tie_blocks=0):
    """The positions a commit comparison left out of the bit-exact check are
    reported separately: appended as one JSON line to the file named by
    D2F_PARITY_LOG (when set). With max_frac they are also bounded: band
    positions at most that fraction of the masked ones (at least one allowed),
    near-tied rows at most four per aggressive block that has them."""
    path = os.environ.get("D2F_PARITY_LOG")
    if path and label:
        with open(path, "a") as f:
            f.write(json.dumps({"case": label, "masked": n_masked, "band": n_band,
                                "near_tie_rows": n_tie, "near_tie_blocks": n_tie_blocks}) + "\n")
    if max_frac is not None:
        lim = max(1, int(max_frac * n_masked))
        assert n_band <= lim, "%s: %d band positions excluded of %d masked" % (
            label, n_band, n_masked)
        assert n_tie <= 4 * n_tie_blocks, "%s: %d near-tied rows in %d blocks" % (
            label, n_tie, n_tie_blocks)


def commit_compare(p, gpu_tokens, gpu_masked, gpu_conf, gpu_arg, gpu_rem, phase, tau, ref,
                   band=None, atol=0.0, label=None, max_frac=None):
    """Compare a GPU commit with the oracle's. Returns (n_band, n_tie) positions
    excluded from the bit-exact check. band: the |c - tau| (and top-two) band
    excluded from it (default BAND); atol: absolute slack on the confidence
    besides CONF_RTOL (for metrics that can be near 0); label / max_frac: see
    record_excluded."""
    BAND_ = BAND if band is None else band
    m0 = p.masked.cpu().bool()
    conf = gpu_conf.cpu()
    arg = gpu_arg.cpu()
    # greedy token and confidence of every row masked on entry
    assert torch.equal(arg[m0], ref["argmax"][m0]), "argmax mismatch"
    assert torch.equal(arg[~m0], torch.full_like(arg[~m0], -1))
    rc = ref["conf"][m0].double()
    err = ((conf[m0].double() - rc).abs() - atol).clamp(min=0.0)
    rel = (err / (rc.abs() + 1e-30)).max().item() if m0.any() else 0.0
    assert rel <= CONF_RTOL, "conf rel err %.3g" % rel
    # excluded positions: the |c - tau| band, and in aggressive blocks the masked
    # rows within the band of the block's most confident row when there are
    # several (which of them is the extra top-1 commit depends on rounding)
    B = p.w.block_size
    q_start = p.q_start.cpu()
    seq = torch.searchsorted(q_start, torch.arange(len(m0), dtype=torch.int32), right=True) - 1
    t_row = tau.cpu()[seq]
    band = m0 & ((ref["conf"] - t_row).abs() < BAND_)
    tie_rows = torch.zeros_like(m0)
    nb = len(m0) // B
    ph = phase.cpu()
    tie_blocks = []
    for jb in range(nb):
        if ph[jb] != 1:
            continue
        sl = slice(jb * B, (jb + 1) * B)
        if m0[sl].sum() < 2:
            continue
        c = torch.where(m0[sl], ref["conf"][sl], torch.tensor(float("-inf")))
        tied = m0[sl] & (c >= c.max() - BAND_)
        if tied.sum() >= 2:
            tie_rows[sl] |= tied
            tie_blocks.append(jb)
    excl = band | tie_rows
    tok = gpu_tokens.cpu()
    msk = gpu_masked.cpu()
    assert torch.equal(tok[~excl], ref["tokens"][~excl]), "token mismatch"
    assert torch.equal(msk[~excl], ref["masked"][~excl]), "mask mismatch"
    # near-tied rows: as many commits among them as the oracle makes, each with
    # its greedy token; the others stay masked
    for jb in tie_blocks:
        sl = slice(jb * B, (jb + 1) * B)
        t = tie_rows[sl] & ~band[sl]
        assert int((msk[sl][t] == 0).sum()) == int((ref["masked"][sl][t] == 0).sum()), \
            "block %d: commits among near-tied rows differ" % jb
        com = t & (msk[sl] == 0)
        assert torch.equal(tok[sl][com], ref["argmax"][sl][com])
        assert bool((tok[sl][t & (msk[sl] != 0)] == p.mask_id).all())
    blk_ok = ~band.view(-1, B).any(1)
    assert torch.equal(gpu_rem.cpu()[blk_ok], ref["block_remaining"][blk_ok])
    n_band, n_tie = int(band.sum()), int((tie_rows & ~band).sum())
    record_excluded(label, int(m0.sum()), n_band, n_tie, max_frac, len(tie_blocks))
    return n_band, n_tie
