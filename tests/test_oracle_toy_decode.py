"""Cache invariant of block-causal decoding on a toy transformer (CPU only).

"D2F: 확산 언어 모델이 KV 캐시를 얻고 자기회귀 모델보다 2.5배 빨라지는 방법",
§블록 단위 인과 어텐션: because a block only sees itself and earlier blocks, the
K/V of a finished block never change, so decoding with a KV cache is exact (no
approximation, unlike periodic-refresh caches, §기존 근사 캐싱의 한계).
"D2F 논문 리뷰", §쉽게 이해하기: a window of active blocks, a new block joins when
the last block has progressed past a threshold, conservative / aggressive commit.

A 2-layer random float64 transformer decodes several blocks with the oracle's
paged attention, commit and append. At every step the window logits must equal a
full recomputation over [prompt ; all blocks] with the explicit block-causal mask,
and cached pages must stay bitwise unchanged. No trained weights are needed: the
invariant is structural.

Readings: the prompt is one bidirectional block (block id -1); a block whose last
masked token committed stays in the window for one more step (its K/V are then
computed from final tokens) and is appended at the end of that step.
"""
import numpy as np
import torch

VOCAB, MASK = 50, 50
DM, HEADS, HD, LAYERS, HID = 32, 2, 16, 2, 64
B, PROMPT, NBLOCKS, WMAX = 4, 8, 5, 3
TAU, GROW_AT = 0.3, 0.5


class Toy:
    def __init__(self, seed=0):
        r = np.random.default_rng(seed)
        s = 1.0 / np.sqrt(DM)
        self.emb = r.normal(0, 1, (VOCAB + 1, DM))
        self.pos = r.normal(0, 0.5, (PROMPT + NBLOCKS * B, DM))
        self.Wq = r.normal(0, s, (LAYERS, DM, HEADS * HD))
        self.Wk = r.normal(0, s, (LAYERS, DM, HEADS * HD))
        self.Wv = r.normal(0, s, (LAYERS, DM, HEADS * HD))
        self.Wo = r.normal(0, s, (LAYERS, HEADS * HD, DM))
        self.W1 = r.normal(0, s, (LAYERS, DM, HID))
        self.W2 = r.normal(0, 1.0 / np.sqrt(HID), (LAYERS, HID, DM))
        self.Wlm = r.normal(0, 3 * s, (DM, VOCAB))

    def embed(self, tokens, positions):
        return self.emb[tokens] + self.pos[positions]

    def qkv(self, x, l):
        n = x.shape[0]
        return ((x @ self.Wq[l]).reshape(n, HEADS, HD), (x @ self.Wk[l]).reshape(n, HEADS, HD),
                (x @ self.Wv[l]).reshape(n, HEADS, HD))

    def post(self, x, att, l):
        x = x + att.reshape(x.shape[0], HEADS * HD) @ self.Wo[l]
        return x + np.maximum(x @ self.W1[l], 0) @ self.W2[l]


def dense_attention(q, k, v, mask):
    s = np.einsum("qhd,khd->hqk", q, k) / np.sqrt(HD)
    s = np.where(mask[None], s, -np.inf)
    s = s - s.max(-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(-1, keepdims=True)
    return np.einsum("hqk,khd->qhd", p, v)


def full_recompute(model, tokens, block_id):
    """All positions from scratch with the explicit block-causal mask.
    Returns (logits of every position, per-layer K and V)."""
    pos = np.arange(len(tokens))
    x = model.embed(tokens, pos)
    mask = block_id[None, :] <= block_id[:, None]
    ks, vs = [], []
    for l in range(LAYERS):
        q, k, v = model.qkv(x, l)
        ks.append(k)
        vs.append(v)
        x = model.post(x, dense_attention(q, k, v, mask), l)
    return x @ model.Wlm, ks, vs


def test_cached_decode_equals_full_recompute(oracle):
    model = Toy(0)
    rng = np.random.default_rng(1)
    prompt = rng.integers(0, VOCAB, PROMPT)
    gen = np.full((NBLOCKS, B), MASK)  # tokens of generated blocks

    # Paged cache per layer: physical pages permuted, one block per page.
    n_pages = PROMPT // B + NBLOCKS + 2
    phys = rng.permutation(n_pages)
    k_pool = [torch.zeros(n_pages, HEADS, B, HD, dtype=torch.float64) for _ in range(LAYERS)]
    v_pool = [torch.zeros(n_pages, HEADS, B, HD, dtype=torch.float64) for _ in range(LAYERS)]
    page_table = torch.tensor(phys[None, :], dtype=torch.int32)

    def f64(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))

    # Prefill the prompt (one bidirectional block) and store its K/V.
    pid = np.full(PROMPT, -1)
    _, pk, pv = full_recompute(model, prompt, pid)
    for l in range(LAYERS):
        for t in range(PROMPT):
            k_pool[l][phys[t // B], :, t % B] = f64(pk[l][t])
            v_pool[l][phys[t // B], :, t % B] = f64(pv[l][t])
    ctx = PROMPT
    window = [0]
    done_at = {}
    appended = []
    snapshots = {}
    step = 0
    while (window or len(appended) < NBLOCKS) and step < 60:
        step += 1
        rows_tok = np.concatenate([gen[j] for j in window])
        rows_pos = np.concatenate([PROMPT + j * B + np.arange(B) for j in window])
        x = model.embed(rows_tok, rows_pos)
        win_k, win_v = [], []
        n = len(rows_tok)
        for l in range(LAYERS):
            q, k, v = model.qkv(x, l)
            q, k, v = (f64(a) for a in (q, k, v))
            win_k.append(k)
            win_v.append(v)
            out, _ = oracle.block_attn(q, k, v, k_pool[l], v_pool[l], page_table,
                                       torch.tensor([ctx], dtype=torch.int32),
                                       torch.tensor([0, n], dtype=torch.int32), B)
            x = model.post(x, out.numpy(), l)
        logits = x @ model.Wlm

        # Invariant 1: equal to the full recomputation with the explicit mask.
        last = max(window)
        all_tok = np.concatenate([prompt] + [gen[j] for j in range(last + 1)])
        ids = np.concatenate([np.full(PROMPT, -1), np.repeat(np.arange(last + 1), B)])
        ref_logits, _, _ = full_recompute(model, all_tok, ids)
        sel = rows_pos
        np.testing.assert_allclose(logits, ref_logits[sel], rtol=0, atol=1e-12)

        # Invariant 2: cached pages never change.
        for key, (kk, vv) in snapshots.items():
            l, page = key
            assert torch.equal(k_pool[l][page], kk) and torch.equal(v_pool[l][page], vv)

        # Append the oldest block if it was complete before this step.
        if window and window[0] in done_at and done_at[window[0]] < step:
            j = window.pop(0)
            page = phys[ctx // B]
            for l in range(LAYERS):
                kp, vp = oracle.kv_append(win_k[l], win_v[l], torch.tensor([0], dtype=torch.int32),
                                          torch.tensor([page], dtype=torch.int32), k_pool[l],
                                          v_pool[l], B)
                k_pool[l], v_pool[l] = kp, vp
                snapshots[(l, page)] = (kp[page].clone(), vp[page].clone())
            ctx += B
            appended.append(j)
            rows_tok = rows_tok[B:]
            logits = logits[B:]
        if not window:
            if len(appended) < NBLOCKS:
                window.append(len(appended))
            continue

        # Commit: the oldest window block aggressive, the others conservative.
        n = len(window) * B
        phase = torch.zeros(len(window), dtype=torch.uint8)
        phase[0] = 1
        masked = torch.tensor((rows_tok == MASK).astype(np.uint8))
        res = oracle.commit(torch.from_numpy(logits.astype(np.float32)),
                            torch.tensor(rows_tok, dtype=torch.int32), masked,
                            torch.tensor([0, n], dtype=torch.int32), phase,
                            torch.tensor([TAU]), B, MASK)
        new_tok = res["tokens"].numpy()
        for u, j in enumerate(window):
            gen[j] = new_tok[u * B:(u + 1) * B]
            if res["block_remaining"][u].item() == 0 and j not in done_at:
                done_at[j] = step
        # Grow the window when the last block has progressed enough.
        lastj = window[-1]
        progress = float((gen[lastj] != MASK).mean())
        if progress >= GROW_AT and len(window) < WMAX and lastj + 1 < NBLOCKS:
            window.append(lastj + 1)

    assert appended == list(range(NBLOCKS)), (appended, step)
    # Invariant 3: cached K/V equal the full recomputation of the final sequence.
    all_tok = np.concatenate([prompt] + [gen[j] for j in range(NBLOCKS)])
    ids = np.concatenate([np.full(PROMPT, -1), np.repeat(np.arange(NBLOCKS), B)])
    _, ks, vs = full_recompute(model, all_tok, ids)
    for l in range(LAYERS):
        for t in range(len(all_tok)):
            page = phys[t // B]
            np.testing.assert_allclose(k_pool[l][page, :, t % B].numpy(), ks[l][t], rtol=0, atol=1e-12)
            np.testing.assert_allclose(v_pool[l][page, :, t % B].numpy(), vs[l][t], rtol=0, atol=1e-12)


def test_scheduled_decode_equals_full_recompute(oracle):
    """The same toy decode with the window driven by the window scheduler
    (oracle.window_step): block entry on the progress threshold, phases, positions,
    the one-step-delayed append list, pages off a free list and the page table. The
    invariants are the pages' own: every step's logits equal a full recomputation
    with the explicit block-causal mask, cached pages never change, and at the end
    the cache holds the full recomputation's K/V of the final sequence."""
    model = Toy(0)
    rng = np.random.default_rng(2)
    prompt = rng.integers(0, VOCAB, PROMPT)
    n_pages = PROMPT // B + NBLOCKS + 3
    phys = rng.permutation(n_pages)
    prompt_pages = [int(x) for x in phys[:PROMPT // B]]
    free = [int(x) for x in phys[PROMPT // B:]]
    k_pool = [torch.zeros(n_pages, HEADS, B, HD, dtype=torch.float64) for _ in range(LAYERS)]
    v_pool = [torch.zeros(n_pages, HEADS, B, HD, dtype=torch.float64) for _ in range(LAYERS)]

    def f64(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))

    _, pk, pv = full_recompute(model, prompt, np.full(PROMPT, -1))
    for l in range(LAYERS):
        for t in range(PROMPT):
            k_pool[l][prompt_pages[t // B], :, t % B] = f64(pk[l][t])
            v_pool[l][prompt_pages[t // B], :, t % B] = f64(pv[l][t])
    max_pages = PROMPT // B + NBLOCKS
    pt = torch.full((1, max_pages), -1, dtype=torch.int32)
    pt[0, :len(prompt_pages)] = torch.tensor(prompt_pages, dtype=torch.int32)
    cap = WMAX * B
    st = {"q_start": torch.zeros(2, dtype=torch.int32),
          "tokens": torch.full((cap,), MASK, dtype=torch.int32),
          "masked": torch.zeros(cap, dtype=torch.uint8),
          "ctx_len": torch.tensor([PROMPT], dtype=torch.int32), "page_table": pt,
          "next_block": torch.zeros(1, dtype=torch.int32),
          "gen_blocks": torch.tensor([NBLOCKS], dtype=torch.int32),
          "n_leaving": torch.zeros(1, dtype=torch.int32), "stopped": None,
          "free_pages": torch.tensor(free, dtype=torch.int32), "free_count": len(free)}
    tau_add, tau_act = 0.5, 1.0
    st = oracle.window_step(st, B, WMAX, MASK, tau_add, tau_act)
    committed = {}                       # position -> token
    snapshots = {}
    steps = 0
    while int(st["q_start"][1]) > 0:
        steps += 1
        assert steps < 80 and st["err"] == 0
        n = int(st["q_start"][1])
        rows_tok = st["tokens"][:n].numpy()
        rows_pos = st["row_pos"][:n].numpy()
        ctx = int(st["ctx_len"][0])
        assert rows_pos[0] == ctx and (np.diff(rows_pos) == 1).all()
        x = model.embed(rows_tok, rows_pos)
        win_k, win_v = [], []
        for l in range(LAYERS):
            q, k, v = (f64(a) for a in model.qkv(x, l))
            win_k.append(k)
            win_v.append(v)
            out, _ = oracle.block_attn(q, k, v, k_pool[l], v_pool[l], st["page_table"],
                                       st["ctx_len"], torch.tensor([0, n], dtype=torch.int32), B)
            x = model.post(x, out.numpy(), l)
        logits = x @ model.Wlm
        # the full recomputation over [prompt ; every block up to the window's last]
        last = (int(rows_pos[-1]) - PROMPT) // B
        toks = [committed.get(PROMPT + t, MASK) for t in range((last + 1) * B)]
        all_tok = np.concatenate([prompt, np.array(toks)])
        ids = np.concatenate([np.full(PROMPT, -1), np.repeat(np.arange(last + 1), B)])
        ref_logits, _, _ = full_recompute(model, all_tok, ids)
        np.testing.assert_allclose(logits, ref_logits[rows_pos], rtol=0, atol=1e-12)
        for (l, page), (kk, vv) in snapshots.items():
            assert torch.equal(k_pool[l][page], kk) and torch.equal(v_pool[l][page], vv)
        # the appends listed for this step read this step's K/V (final tokens)
        for src, page in zip(st["app_src"].tolist(), st["app_dst"].tolist()):
            assert not st["masked"][src:src + B].any()
            for l in range(LAYERS):
                kp, vp = oracle.kv_append(win_k[l], win_v[l], torch.tensor([src], dtype=torch.int32),
                                          torch.tensor([page], dtype=torch.int32), k_pool[l],
                                          v_pool[l], B)
                k_pool[l], v_pool[l] = kp, vp
                snapshots[(l, page)] = (kp[page].clone(), vp[page].clone())
        # commit on this step's logits, then the scheduler
        res = oracle.commit(torch.from_numpy(logits.astype(np.float32)), st["tokens"][:n],
                            st["masked"][:n], st["q_start"], st["block_phase"][:n // B],
                            torch.tensor([TAU]), B, MASK)
        tok, msk = st["tokens"].clone(), st["masked"].clone()
        tok[:n], msk[:n] = res["tokens"], res["masked"]
        for r in range(n):
            if st["masked"][r] and not msk[r]:
                committed[int(rows_pos[r])] = int(tok[r])
        st = oracle.window_step(dict(st, tokens=tok, masked=msk), B, WMAX, MASK, tau_add, tau_act)

    assert int(st["ctx_len"][0]) == PROMPT + NBLOCKS * B and len(committed) == NBLOCKS * B
    final = np.concatenate([prompt, np.array([committed[PROMPT + t] for t in range(NBLOCKS * B)])])
    ids = np.concatenate([np.full(PROMPT, -1), np.repeat(np.arange(NBLOCKS), B)])
    _, ks, vs = full_recompute(model, final, ids)
    for l in range(LAYERS):
        for t in range(len(final)):
            page = int(st["page_table"][0, t // B])
            np.testing.assert_allclose(k_pool[l][page, :, t % B].numpy(), ks[l][t], rtol=0, atol=1e-12)
            np.testing.assert_allclose(v_pool[l][page, :, t % B].numpy(), vs[l][t], rtol=0, atol=1e-12)
