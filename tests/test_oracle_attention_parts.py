"""Pins for the oracle's attention parts and their log-space composition (CPU only).

"확산 언어 모델(Diffusion LLM)이란 무엇인가", §FlashBlock: 블록 외부 어텐션 캐싱:
the output and normaliser over the keys outside the blocks being decoded are
kept from one step and recombined in log space with the attention recomputed
inside. Checked against the full attention (composition of the cached part and
the window part of the same queries), against a dense brute-force restatement
with an explicit mask for the cached part alone, and, for reuse across steps,
against one softmax whose cached scores use the earlier queries and whose window
scores use the current ones.
"""
import numpy as np
import pytest
import torch

import bruteforce
from block_causal_kv_gb300 import synth


def _problem(seed, ctx=(37, 0, 96), win=(2, 3, 1), B=8, H=(4, 2), D=32):
    w = synth.Workload("p", len(ctx), H[0], H[1], D, B, torch.float32, list(ctx), list(win), 64,
                       permute_pages=True, extra_pages=3, seed=seed)
    return synth.make_problem(w)


def _args(p, q=None):
    return ((p.q if q is None else q), p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
            p.ctx_len, p.q_start, p.w.block_size)


@pytest.mark.parametrize("seed", range(3))
def test_cached_and_window_parts_compose_to_the_full_attention(oracle, seed):
    p = _problem(seed)
    full, lse = oracle.block_attn(*_args(p))
    oc, lc = oracle.block_attn_part(*_args(p), part=oracle.ATTN_CACHED)
    out, l2 = oracle.block_attn_part(*_args(p), part=oracle.ATTN_WINDOW, prev_out=oc, prev_lse=lc)
    assert torch.allclose(out, full, rtol=0, atol=1e-12)
    assert torch.allclose(l2, lse, rtol=0, atol=1e-12)


def test_cached_part_of_a_sequence_without_context(oracle):
    """No cached token: output 0 and lse -inf, and composing it with the window
    part gives the window part itself."""
    p = _problem(5)
    oc, lc = oracle.block_attn_part(*_args(p), part=oracle.ATTN_CACHED)
    r0, r1 = int(p.q_start[1]), int(p.q_start[2])  # sequence 1 has ctx 0
    assert torch.all(oc[r0:r1] == 0) and torch.all(torch.isneginf(lc[r0:r1]))
    ow, lw = oracle.block_attn_part(*_args(p), part=oracle.ATTN_WINDOW)
    oc2, lc2 = oracle.block_attn_part(*_args(p), part=oracle.ATTN_WINDOW, prev_out=oc, prev_lse=lc)
    assert torch.equal(oc2[r0:r1], ow[r0:r1]) and torch.equal(lc2[r0:r1], lw[r0:r1])


@pytest.mark.parametrize("seed", range(2))
def test_cached_part_against_brute_force(oracle, seed):
    """The cached part is the dense attention with every window key masked."""
    p = _problem(10 + seed)
    oc, lc = oracle.block_attn_part(*_args(p), part=oracle.ATTN_CACHED)
    q, kp, vp = (x.double().numpy() for x in (p.q, p.k_pool, p.v_pool))
    B, H, Hk = p.w.block_size, p.w.num_heads_q, p.w.num_heads_kv
    for b in range(p.w.batch):
        C = int(p.ctx_len[b])
        if C == 0:
            continue
        t = np.arange(C)
        pages = p.page_table[b].numpy()[t // B]
        for r in range(int(p.q_start[b]), int(p.q_start[b + 1])):
            for h in range(H):
                K, V = kp[pages, h // (H // Hk), t % B], vp[pages, h // (H // Hk), t % B]
                s = K @ q[r, h] / np.sqrt(q.shape[-1])
                pr = np.exp(s - s.max())
                np.testing.assert_allclose(oc[r, h].numpy(), pr @ V / pr.sum(), rtol=1e-10, atol=1e-12)
                np.testing.assert_allclose(lc[r, h].item(), s.max() + np.log(pr.sum()), rtol=1e-12)


def test_reuse_across_steps_is_one_softmax_with_mixed_queries(oracle):
    """Composing a cached part computed with earlier queries q0 with the window
    part of the current queries q1 equals one softmax over all visible keys whose
    cached scores use q0 and whose window scores use q1 (dense, per row)."""
    p = _problem(21)
    q0 = p.q
    q1 = p.q + 0.3 * torch.randn(p.q.shape, generator=torch.Generator().manual_seed(3))
    oc, lc = oracle.block_attn_part(*_args(p, q0), part=oracle.ATTN_CACHED)
    out, lse = oracle.block_attn_part(*_args(p, q1), part=oracle.ATTN_WINDOW, prev_out=oc,
                                      prev_lse=lc)
    a0, a1, kw, vw, kp, vp = (x.double().numpy() for x in (q0, q1, p.k_win, p.v_win, p.k_pool,
                                                             p.v_pool))
    B, H, Hk, D = p.w.block_size, p.w.num_heads_q, p.w.num_heads_kv, p.w.head_dim
    for b in range(p.w.batch):
        C, r0, r1 = int(p.ctx_len[b]), int(p.q_start[b]), int(p.q_start[b + 1])
        t = np.arange(C)
        pages = p.page_table[b].numpy()[t // B]
        for r in range(r0, r1):
            vis = [w for w in range(r0, r1) if (w - r0) // B <= (r - r0) // B]
            for h in range(H):
                g = h // (H // Hk)
                s = np.concatenate([kp[pages, g, t % B] @ a0[r, h], kw[vis, g] @ a1[r, h]]) / np.sqrt(D)
                V = np.concatenate([vp[pages, g, t % B], vw[vis, g]])
                pr = np.exp(s - s.max())
                np.testing.assert_allclose(out[r, h].numpy(), pr @ V / pr.sum(), rtol=1e-10,
                                           atol=1e-12)
                np.testing.assert_allclose(lse[r, h].item(), s.max() + np.log(pr.sum()), rtol=1e-12)
