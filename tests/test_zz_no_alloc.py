"""d2f_commit_noalloc: the commit for callers that cannot allocate device memory.

Some callers of this library may not allocate: a plugin or callback that may
only use the buffers its host framework hands it, or a runtime that must not
allocate once it is serving. For them d2f_commit_noalloc takes no workspace and
keeps its scratch in a fixed array inside the library. These tests call it
through the C ABI and check it against d2f_commit (which takes a caller
workspace) on identical inputs, two calls in a row, within the commit tolerance
the other tests use. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

from block_causal_kv_gb300 import d2f, synth
from gpu_common import CONF_RTOL, device

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, g, logits, tokens, masked, conf, amax, rem, num_splits=0):
    st = lib.d2f_commit_noalloc(
        logits.data_ptr(), logits.stride(0), d2f.BF16, logits.shape[1], logits.shape[0], None,
        tokens.data_ptr(), masked.data_ptr(), g.q_start.data_ptr(), g.block_phase.data_ptr(),
        g.tau.data_ptr(), g.q_start.shape[0] - 1, tokens.shape[0], g.w.block_size,
        ctypes.c_int32(g.mask_id), conf.data_ptr(), amax.data_ptr(), rem.data_ptr(), num_splits,
        None, torch.cuda.current_stream().cuda_stream)
    return st


@pytest.mark.parametrize("name", ["llada", "ragged"])
def test_matches_workspace_commit_two_calls(name):
    dev = device()
    lib = d2f.load()
    p = synth.make_problem(synth.small(name))
    g = p.to(dev)
    B = p.w.block_size
    n = p.w.total_q
    # two identical decode states: one for each entry point
    tok_a, msk_a = g.tokens.clone(), g.masked.clone()
    tok_b, msk_b = g.tokens.clone(), g.masked.clone()
    out_a = [torch.empty(n, dtype=torch.float32, device=dev), torch.empty(n, dtype=torch.int32, device=dev),
             torch.empty(n // B, dtype=torch.int32, device=dev)]
    out_b = [torch.empty_like(t) for t in out_a]
    ws = d2f.commit_workspace(dev, total_q=n, vocab=p.w.vocab, block_size=B)
    for call in range(2):
        assert _call_noalloc(lib, g, g.logits, tok_a, msk_a, *out_a) == 0, \
            lib.d2f_last_error_string().decode()
        d2f.commit(g.logits, tok_b, msk_b, g.q_start, g.block_phase, g.tau, block_size=B,
                   mask_id=p.mask_id, conf=out_b[0], argmax=out_b[1], block_remaining=out_b[2],
                   workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(tok_a, tok_b), "tokens differ on call %d" % call
        assert torch.equal(msk_a, msk_b), "masks differ on call %d" % call
        assert torch.equal(out_a[1], out_b[1]), "argmax differs on call %d" % call
        assert torch.equal(out_a[2], out_b[2]), "block_remaining differs on call %d" % call
        m = out_b[0] > 0
        rel = ((out_a[0][m] - out_b[0][m]).abs() / out_b[0][m]).max().item() if m.any() else 0.0
        assert rel <= CONF_RTOL
        assert torch.equal(out_a[0][~m], out_b[0][~m])


def test_rejects_requests_beyond_its_scratch():
    device()
    lib = d2f.load()
    # 8192 rows x 64 vocabulary slices need more than the fixed scratch holds;
    # the request is refused on the host before anything is enqueued.
    st = lib.d2f_commit_noalloc(None, 126464, d2f.BF16, 126464, 8192, None, None, None, None,
                                None, None, 1, 8192, 16, ctypes.c_int32(0), None, None, None, 64,
                                None, None)
    assert st == 6
    assert b"scratch" in lib.d2f_last_error_string()


def _random_problem(dev, total_q, vocab, B, seed):
    """A decode state over `total_q` rows (every row masked, random phases and
    thresholds) with N(0, 3) logits drawn on the device."""
    g = torch.Generator(device=dev).manual_seed(seed)
    logits = (torch.randn((total_q, vocab), generator=g, device=dev) * 3).to(torch.bfloat16)
    tokens = torch.full((total_q,), vocab, dtype=torch.int32, device=dev)
    masked = torch.ones(total_q, dtype=torch.uint8, device=dev)
    q_start = torch.tensor([0, total_q], dtype=torch.int32, device=dev)
    phase = torch.randint(0, 2, (total_q // B,), generator=g, device=dev).to(torch.uint8)
    tau = torch.full((1,), 1e-4, dtype=torch.float32, device=dev)
    return logits, tokens, masked, q_start, phase, tau


@pytest.mark.parametrize("num_splits,total_q,vocab", [(64, 2032, 126464), (1, 65520, 2048)])
def test_largest_requests_that_fit(num_splits, total_q, vocab):
    """At block size 16 the scratch holds 2,032 rows at 64 vocabulary slices (the
    largest multiple of the block that fits) and the API's largest row count at
    one slice; both run and match d2f_commit. Sixteen rows more at 64 slices are
    refused before anything is enqueued."""
    dev = device()
    B = 16
    logits, tokens, masked, q_start, phase, tau = _random_problem(dev, total_q, vocab, B, 5)
    need = d2f.commit_workspace_size(total_q, vocab, B, d2f.BF16, num_splits)
    assert need <= 2 << 20
    tok_a, msk_a, tok_b, msk_b = tokens.clone(), masked.clone(), tokens.clone(), masked.clone()
    kw = dict(block_size=B, mask_id=vocab, num_splits=num_splits)
    res_a = {k: torch.empty(n, dtype=t, device=dev) for k, n, t in (
        ("conf", total_q, torch.float32), ("argmax", total_q, torch.int32),
        ("block_remaining", total_q // B, torch.int32))}
    d2f.commit_noalloc(logits, tok_a, msk_a, q_start, phase, tau, conf=res_a["conf"],
                       argmax=res_a["argmax"], block_remaining=res_a["block_remaining"], **kw)
    res_b = d2f.commit(logits, tok_b, msk_b, q_start, phase, tau, **kw)
    torch.cuda.synchronize()
    assert torch.equal(tok_a, tok_b) and torch.equal(msk_a, msk_b)
    assert torch.equal(res_a["argmax"], res_b["argmax"])
    assert torch.equal(res_a["block_remaining"], res_b["block_remaining"])
    rel = ((res_a["conf"] - res_b["conf"]).abs() / res_b["conf"]).max().item()
    assert rel <= CONF_RTOL
    if num_splits == 64:
        lib = d2f.load()
        st = lib.d2f_commit_noalloc(None, vocab, d2f.BF16, vocab, total_q + 16, None, None, None,
                                    None, None, None, 1, total_q + 16, B, ctypes.c_int32(0), None,
                                    None, None, num_splits, None, None)
        assert st == 6


def test_python_wrapper_across_shapes():
    """d2f.commit_noalloc (the binding) on three differently shaped calls in a row
    on the one shared scratch -- each call clears only the counters it needs --
    against d2f_commit with its own workspace."""
    dev = device()
    for name in ("llada", "ragged", "dream", "llada"):
        p = synth.make_problem(synth.small(name))
        g = p.to(dev)
        B = p.w.block_size
        n = p.w.total_q
        tok_a, msk_a, tok_b, msk_b = g.tokens.clone(), g.masked.clone(), g.tokens.clone(), g.masked.clone()
        outs = [torch.empty(n, dtype=torch.float32, device=dev),
                torch.empty(n, dtype=torch.int32, device=dev),
                torch.empty(n // B, dtype=torch.int32, device=dev)]
        d2f.commit_noalloc(g.logits, tok_a, msk_a, g.q_start, g.block_phase, g.tau, block_size=B,
                           mask_id=p.mask_id, conf=outs[0], argmax=outs[1],
                           block_remaining=outs[2])
        ref = d2f.commit(g.logits, tok_b, msk_b, g.q_start, g.block_phase, g.tau, block_size=B,
                         mask_id=p.mask_id)
        torch.cuda.synchronize()
        assert torch.equal(tok_a, tok_b) and torch.equal(msk_a, msk_b), name
        assert torch.equal(outs[1], ref["argmax"]) and torch.equal(outs[2], ref["block_remaining"])
