"""Pins for the oracle's block-causal attention (CPU only).

Each test checks the oracle against something other than itself: hand-worked
values, a dense explicit-mask brute force, PyTorch SDPA in the special cases the
mask reduces to (block size 1 = causal, one block = bidirectional), and the
split/merge closed form of the log-space composition.
"""
import math
import os

import numpy as np
import pytest
import torch

import bruteforce
from block_causal_kv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _vals(s):
    s = s.strip()
    if not s:
        return []
    return [float(eval(tok, {"__builtins__": {}}, {"ln": math.log, "e": math.e}))
            for tok in s.split()]


def _cases():
    out = []
    with open(os.path.join(GOLDEN, "attn_hand.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kv = dict((a.strip(), b.strip()) for a, b in (p.split("=", 1) for p in line.split(";")))
            out.append(kv)
    return out


def _single_head_problem(B, ctx, k_cache, v_cache, k_win, v_win, pool_pages=4, cache_page=2):
    """One sequence, one head, head_dim 1, the cached block in a chosen physical page;
    every other pool slot holds NaN so a wrong page lookup poisons the output."""
    n = len(k_win)
    q = torch.ones(n, 1, 1, dtype=torch.float32)
    kw = torch.tensor(k_win, dtype=torch.float32).view(n, 1, 1)
    vw = torch.tensor(v_win, dtype=torch.float32).view(n, 1, 1)
    kp = torch.full((pool_pages, 1, B, 1), float("nan"))
    vp = torch.full((pool_pages, 1, B, 1), float("nan"))
    pt = torch.full((1, pool_pages), -1, dtype=torch.int32)
    for t in range(ctx):
        page = cache_page + t // B
        kp[page, 0, t % B, 0] = k_cache[t]
        vp[page, 0, t % B, 0] = v_cache[t]
        pt[0, t // B] = page
    return dict(q=q, k_win=kw, v_win=vw, k_pool=kp, v_pool=vp, page_table=pt,
                ctx_len=torch.tensor([ctx], dtype=torch.int32),
                q_start=torch.tensor([0, n], dtype=torch.int32))


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["case"])
def test_hand_worked_examples(oracle, case):
    B, ctx = int(case["B"]), int(case["ctx"])
    p = _single_head_problem(B, ctx, _vals(case["k_cache"]), _vals(case["v_cache"]),
                             _vals(case["k_win"]), _vals(case["v_win"]))
    out, _ = oracle.block_attn(**p, block_size=B, scale=1.0)
    expect = np.array(_vals(case["expect"]))
    # inputs are float32 roundings of ln(w); the weights are exact to ~1e-7 relative
    np.testing.assert_allclose(out[:, 0, 0].numpy(), expect, rtol=2e-6, atol=0)


def _random_problem(seed, batch=3, H=4, Hk=2, D=8, B=4, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    ctx = [int(x) for x in torch.randint(0, 23, (batch,), generator=g)]
    ctx[0] = 0  # always include an empty cache
    win = [int(x) for x in torch.randint(1, 4, (batch,), generator=g)]
    w = synth.Workload("rand", batch, H, Hk, D, B, dtype, ctx, win, 17, planted_peak=False,
                       permute_pages=True, extra_pages=3, seed=seed)
    return synth.make_problem(w)


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("B", [1, 2, 4])
def test_against_dense_explicit_mask(oracle, seed, B):
    p = _random_problem(seed, B=B)
    out, lse = oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
                                 p.ctx_len, p.q_start, B)
    ref, ref_lse = bruteforce.attention(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool,
                                        p.page_table, p.ctx_len, p.q_start, B)
    np.testing.assert_allclose(out.numpy(), ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse.numpy(), ref_lse, rtol=0, atol=1e-12)


def test_bf16_inputs_widen_exactly(oracle):
    p = _random_problem(11, dtype=torch.bfloat16)
    out, _ = oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
                               p.ctx_len, p.q_start, 4)
    out32, _ = oracle.block_attn(p.q.float(), p.k_win.float(), p.v_win.float(),
                                 p.k_pool.float(), p.v_pool.float(), p.page_table,
                                 p.ctx_len, p.q_start, 4)
    assert torch.equal(out, out32)


def _sdpa(q, k, v, mask, scale):
    return torch.nn.functional.scaled_dot_product_attention(
        q.double(), k.double(), v.double(), attn_mask=mask, scale=scale)


@pytest.mark.parametrize("ctx", [0, 5])
def test_block_size_one_is_causal(oracle, ctx):
    """B = 1: every window row is its own block, so the mask is the causal mask
    over [cache ; window] (autoregressive decoding)."""
    n, H, D = 7, 3, 16
    w = synth.Workload("b1", 1, H, H, D, 1, torch.float32, [ctx], [n], 11,
                       planted_peak=False, seed=77 + ctx)
    p = synth.make_problem(w)
    out, _ = oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
                               p.ctx_len, p.q_start, 1)
    # dense sequence in logical order
    pages = p.page_table[0, :ctx].long()
    kc = p.k_pool[pages, :, 0, :]
    vc = p.v_pool[pages, :, 0, :]
    K = torch.cat([kc, p.k_win], 0).transpose(0, 1)  # [H, C+n, D]
    V = torch.cat([vc, p.v_win], 0).transpose(0, 1)
    Q = p.q.transpose(0, 1)
    # explicit boolean mask: the whole cache, then lower-triangular over the window
    mask = torch.cat([torch.ones(n, ctx, dtype=torch.bool),
                      torch.tril(torch.ones(n, n, dtype=torch.bool))], 1)
    ref = _sdpa(Q, K, V, mask, 1.0 / math.sqrt(D)).transpose(0, 1)
    torch.testing.assert_close(out, ref, rtol=0, atol=1e-12)


def test_single_block_no_cache_is_bidirectional(oracle):
    """One window block and no cache: full bidirectional attention (vanilla dLLM)."""
    B, H, D = 8, 2, 16
    w = synth.Workload("bi", 1, H, H, D, B, torch.float32, [0], [1], 11, planted_peak=False,
                       seed=91)
    p = synth.make_problem(w)
    out, _ = oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
                               p.ctx_len, p.q_start, B)
    ref = _sdpa(p.q.transpose(0, 1), p.k_win.transpose(0, 1), p.v_win.transpose(0, 1), None,
                1.0 / math.sqrt(D)).transpose(0, 1)
    torch.testing.assert_close(out, ref, rtol=0, atol=1e-12)


def test_gqa_grouping_is_consecutive(oracle):
    """q head h reads KV head h // (Hq / Hkv): swapping KV heads 0 and 1 must swap
    the outputs of q-head groups {0,1} and {2,3}."""
    p = _random_problem(3, H=4, Hk=2)
    out, _ = oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
                               p.ctx_len, p.q_start, 4)
    sw = [1, 0]
    q2 = p.q[:, [2, 3, 0, 1], :]
    out2, _ = oracle.block_attn(q2, p.k_win[:, sw], p.v_win[:, sw], p.k_pool[:, sw],
                                p.v_pool[:, sw], p.page_table, p.ctx_len, p.q_start, 4)
    torch.testing.assert_close(out2[:, [2, 3, 0, 1]], out, rtol=0, atol=1e-12)


def test_log_space_merge_of_key_partitions(oracle):
    """Log-space composition ("확산 언어 모델(Diffusion LLM)이란 무엇인가", §FlashBlock):
    attention over a union of disjoint key sets equals the merge of the parts,
    O = sum_s e^{lse_s - L} O_s with L = log sum_s e^{lse_s}. Split the key list of a
    one-block window at every page boundary, attend to each part densely, compose
    the parts, and compare with the oracle's single pass (output and lse)."""
    B, H, D, C = 4, 2, 8, 24
    w = synth.Workload("m", 1, H, H, D, B, torch.float32, [C], [1], 11, planted_peak=False,
                       seed=123)
    p = synth.make_problem(w)
    full, full_lse = oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
                                       p.ctx_len, p.q_start, B)
    n = p.q.shape[0]
    # Every row of a one-block window sees the same keys [cache ; window]; split that
    # key list at page boundaries and compose the parts.
    q = p.q.double().numpy()
    pages = p.page_table[0, : C // B].long()
    kc = p.k_pool[pages].permute(0, 2, 1, 3).reshape(C, H, D).double().numpy()
    vc = p.v_pool[pages].permute(0, 2, 1, 3).reshape(C, H, D).double().numpy()
    K = np.concatenate([kc, p.k_win.double().numpy()], 0)
    V = np.concatenate([vc, p.v_win.double().numpy()], 0)
    scale = 1.0 / math.sqrt(D)
    for cut in range(0, C + n + 1, B):
        parts = [(0, cut), (cut, C + n)]
        Os, Ls = [], []
        for a, b in parts:
            if a == b:
                continue
            S = scale * np.einsum("qhd,khd->hqk", q, K[a:b])
            m = S.max(-1, keepdims=True)
            P = np.exp(S - m)
            l = P.sum(-1, keepdims=True)
            Os.append(np.einsum("hqk,khd->qhd", P / l, V[a:b]))
            Ls.append((m + np.log(l))[..., 0].T)
        L = np.logaddexp.reduce(np.stack(Ls), axis=0)
        O = sum(np.exp(Ls[i] - L)[..., None] * Os[i] for i in range(len(Os)))
        np.testing.assert_allclose(O, full.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(L, full_lse.numpy(), rtol=0, atol=1e-12)


def test_rejects_bad_page_id(oracle):
    p = _random_problem(4)
    pt = p.page_table.clone()
    b = int(torch.argmax(p.ctx_len))
    pt[b, 0] = p.k_pool.shape[0]
    with pytest.raises(ValueError):
        oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, pt, p.ctx_len, p.q_start, 4)
