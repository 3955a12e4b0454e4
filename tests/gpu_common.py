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
      masks bit-exact except positions with |p - tau| < 1e-5 and aggressive
      blocks whose two best masked confidences differ by < 1e-5 (both reported).
"""
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


def commit_compare(p, gpu_tokens, gpu_masked, gpu_conf, gpu_arg, gpu_rem, phase, tau, ref,
                   band=None, atol=0.0):
    """Compare a GPU commit with the oracle's. Returns (n_band, n_tie) positions
    excluded from the bit-exact check. band: the |c - tau| (and top-two) band
    excluded from it (default BAND); atol: absolute slack on the confidence
    besides CONF_RTOL (for metrics that can be near 0)."""
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
    # excluded positions
    B = p.w.block_size
    q_start = p.q_start.cpu()
    seq = torch.searchsorted(q_start, torch.arange(len(m0), dtype=torch.int32), right=True) - 1
    t_row = tau.cpu()[seq]
    band = m0 & ((ref["conf"] - t_row).abs() < BAND_)
    tie_rows = torch.zeros_like(m0)
    nb = len(m0) // B
    ph = phase.cpu()
    for jb in range(nb):
        if ph[jb] != 1:
            continue
        sl = slice(jb * B, (jb + 1) * B)
        c = torch.where(m0[sl], ref["conf"][sl], torch.tensor(float("-inf")))
        top = torch.sort(c, descending=True).values
        if m0[sl].sum() >= 2 and float(top[0] - top[1]) < BAND_:
            tie_rows[sl] = True
    excl = band | tie_rows
    tok = gpu_tokens.cpu()
    msk = gpu_masked.cpu()
    assert torch.equal(tok[~excl], ref["tokens"][~excl]), "token mismatch"
    assert torch.equal(msk[~excl], ref["masked"][~excl]), "mask mismatch"
    blk_ok = ~excl.view(-1, B).any(1)
    assert torch.equal(gpu_rem.cpu()[blk_ok], ref["block_remaining"][blk_ok])
    return int(band.sum()), int(tie_rows.sum())
