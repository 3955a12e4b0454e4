"""Pins for the oracle's KV append (CPU only).

"D2F: 확산 언어 모델이 KV 캐시를 얻고 자기회귀 모델보다 2.5배 빨라지는 방법",
§블록 단위 인과 어텐션 and §운영 관점: a finished block's K/V never change and are
kept in the cache, a page holding one block. Pinned by a NumPy gather and by the
consequence that matters: moving a block from the window into the cache leaves
the attention of the later window blocks unchanged.
"""
import numpy as np
import torch

import bruteforce
from block_causal_kv_gb300 import synth


def test_bitwise_copy_matches_numpy(oracle):
    w = synth.Workload("a", 2, 4, 2, 16, 8, torch.bfloat16, [16, 8], [3, 2], 11,
                       appends_per_seq=2, extra_pages=2, seed=3)
    p = synth.make_problem(w)
    kp, vp = oracle.kv_append(p.k_win, p.v_win, p.src_row, p.dst_page, p.k_pool, p.v_pool, 8)
    ek = p.k_pool.clone().view(torch.int16).numpy()
    ev = p.v_pool.clone().view(torch.int16).numpy()
    kw = p.k_win.view(torch.int16).numpy()
    vw = p.v_win.view(torch.int16).numpy()
    for s, d in zip(p.src_row.tolist(), p.dst_page.tolist()):
        ek[d] = np.transpose(kw[s:s + 8], (1, 0, 2))
        ev[d] = np.transpose(vw[s:s + 8], (1, 0, 2))
    np.testing.assert_array_equal(kp.view(torch.int16).numpy(), ek)
    np.testing.assert_array_equal(vp.view(torch.int16).numpy(), ev)
    # pages that were not targets are untouched
    others = sorted(set(range(p.k_pool.shape[0])) - set(p.dst_page.tolist()))
    assert torch.equal(kp[others], p.k_pool[others])


def test_append_then_attend_is_unchanged(oracle):
    """Attention of window block 1.. with block 0 in the window equals the attention
    with block 0 appended to the cache and removed from the window."""
    B, H, Hk, D = 4, 4, 2, 8
    w = synth.Workload("a", 2, H, Hk, D, B, torch.float32, [8, 12], [3, 2], 11,
                       appends_per_seq=1, permute_pages=True, seed=17)
    p = synth.make_problem(w)
    before, lse_b = oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
                                      p.ctx_len, p.q_start, B)
    kp, vp = oracle.kv_append(p.k_win, p.v_win, p.src_row, p.dst_page, p.k_pool, p.v_pool, B)
    # drop block 0 of each sequence from the window, extend the context by B
    keep = []
    qs = p.q_start.tolist()
    new_qs = [0]
    for b in range(w.batch):
        rows = list(range(qs[b] + B, qs[b + 1]))
        keep += rows
        new_qs.append(new_qs[-1] + len(rows))
    keep_t = torch.tensor(keep)
    after, lse_a = oracle.block_attn(p.q[keep_t], p.k_win[keep_t], p.v_win[keep_t], kp, vp,
                                     p.page_table, p.ctx_len + B,
                                     torch.tensor(new_qs, dtype=torch.int32), B)
    np.testing.assert_allclose(after.numpy(), before[keep_t].numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse_a.numpy(), lse_b[keep_t].numpy(), rtol=0, atol=1e-12)
    # and the dense brute force agrees on the appended layout
    ref, _ = bruteforce.attention(p.q[keep_t], p.k_win[keep_t], p.v_win[keep_t], kp, vp,
                                  p.page_table, p.ctx_len + B,
                                  torch.tensor(new_qs, dtype=torch.int32), B)
    np.testing.assert_allclose(after.numpy(), ref, rtol=0, atol=1e-12)
