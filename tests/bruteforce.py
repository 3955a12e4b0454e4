"""Independent brute-force restatements used to pin the oracle.

Written in NumPy/SciPy with dense matrices and an explicit mask matrix, so a
mistake in the oracle's index-range formulation (a dropped key, a wrong block
boundary, a transposed page lookup) shows up as a mismatch. Shares no code with
oracle/ or with the CUDA library.

Sources: "D2F: 확산 언어 모델이 KV 캐시를 얻고 자기회귀 모델보다 2.5배 빨라지는
방법" §블록 단위 인과 어텐션 (block-wise causal mask); "D2F 논문 리뷰" §쉽게
이해하기 (conservative / aggressive commit); "확산 언어 모델(Diffusion LLM)이란
무엇인가" §양방향 어텐션과 사라진 KV 캐시 (max-probability confidence).
"""
import numpy as np
from scipy.special import logsumexp


def _f64(t):
    return t.detach().to("cpu").double().numpy()


def block_ids_mask(ctx, n_win, B):
    """Explicit (n_win x (ctx + n_win)) visibility matrix.

    Cached tokens carry block id -1, window row i carries id i // B; query row i
    may see key k iff id(k) <= i // B.
    """
    ids = np.concatenate([np.full(ctx, -1), np.arange(n_win) // B])
    qid = np.arange(n_win) // B
    return ids[None, :] <= qid[:, None]


def attention(q, k_win, v_win, k_pool, v_pool, page_table, ctx_len, q_start, B, scale=None):
    """Dense masked softmax attention per sequence and head (float64)."""
    q, k_win, v_win, k_pool, v_pool = (_f64(x) for x in (q, k_win, v_win, k_pool, v_pool))
    page_table = page_table.cpu().numpy()
    ctx_len = ctx_len.cpu().numpy()
    q_start = q_start.cpu().numpy()
    total_q, H, D = q.shape
    Hk = k_win.shape[1]
    G = H // Hk
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    out = np.zeros((total_q, H, D))
    lse = np.zeros((total_q, H))
    for b in range(len(ctx_len)):
        s0, s1 = q_start[b], q_start[b + 1]
        n = s1 - s0
        if n == 0:
            continue
        C = int(ctx_len[b])
        # Gather the cached context into logical token order: [C, Hk, D].
        t = np.arange(C)
        pages = page_table[b, t // B] if C else np.zeros(0, dtype=np.int64)
        kc = k_pool[pages, :, t % B, :] if C else np.zeros((0, Hk, D))
        vc = v_pool[pages, :, t % B, :] if C else np.zeros((0, Hk, D))
        K = np.concatenate([kc, k_win[s0:s1]], axis=0)  # [C+n, Hk, D]
        V = np.concatenate([vc, v_win[s0:s1]], axis=0)
        M = block_ids_mask(C, n, B)
        for h in range(H):
            g = h // G
            S = scale * (q[s0:s1, h, :] @ K[:, g, :].T)
            S = np.where(M, S, -np.inf)
            L = logsumexp(S, axis=1)
            P = np.exp(S - L[:, None])
            out[s0:s1, h, :] = P @ V[:, g, :]
            lse[s0:s1, h] = L
    return out, lse


def confidence(logits_row_f32):
    """(p_max as float32, greedy token) of one logit row via SciPy logsumexp."""
    x = np.asarray(logits_row_f32, dtype=np.float32).astype(np.float64)
    a = int(np.argmax(x))  # NumPy returns the first (lowest) index of the maximum
    p = np.float32(np.exp(x[a] - logsumexp(x)))
    return p, a


def commit(logits, tokens, masked, q_start, block_phase, tau, B, mask_id, logit_row=None):
    """Vectorised restatement of the commit rule (returns numpy arrays)."""
    L = logits.detach().to("cpu").float().numpy()
    tokens = tokens.cpu().numpy().astype(np.int64).copy()
    masked = masked.cpu().numpy().astype(bool).copy()
    q_start = q_start.cpu().numpy()
    phase = block_phase.cpu().numpy()
    tau = tau.cpu().numpy().astype(np.float32)
    total_q = tokens.shape[0]
    rows = np.arange(total_q) if logit_row is None else logit_row.cpu().numpy()
    conf = np.full(total_q, -1.0, dtype=np.float32)
    amax = np.full(total_q, -1, dtype=np.int64)
    for r in np.nonzero(masked)[0]:
        conf[r], amax[r] = confidence(L[rows[r]])
    seq_of_row = np.searchsorted(q_start, np.arange(total_q), side="right") - 1
    rem = np.zeros(total_q // B, dtype=np.int64)
    for jb in range(total_q // B):
        sl = slice(jb * B, (jb + 1) * B)
        m = masked[sl]
        c = conf[sl]
        t = tau[seq_of_row[jb * B]]
        take = m & (c > t)
        if phase[jb] == 1 and m.any():
            take[int(np.argmax(np.where(m, c, -np.inf)))] = True
        tok = tokens[sl]
        tok[take] = amax[sl][take]
        tok[m & ~take] = mask_id
        tokens[sl] = tok
        masked[sl] = m & ~take
        rem[jb] = int(masked[sl].sum())
    return {"tokens": tokens, "masked": masked.astype(np.uint8), "conf": conf,
            "argmax": amax, "block_remaining": rem}
