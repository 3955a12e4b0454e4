"""GPU parity of the device window scheduler (d2f_window_step) and of a whole
decode loop replayed from one CUDA graph per step.

The scheduler is integer work: every output is compared bit for bit with the
oracle's, step by step, over randomised decodes (more sequences than the kernel
has threads, ragged prompts, early stops, a free list that runs dry). The loop
test runs attention (with the device-counted fused append), commit and scheduler
from one captured graph with no host readback between steps, and compares the
decode state, the cache pages and a sampled attention output with a host loop
over the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import device, check_attention
from block_causal_kv_gb300 import d2f

pytestmark = pytest.mark.gpu

STATE_KEYS = ("q_start", "tokens", "masked", "ctx_len", "page_table", "next_block",
              "gen_blocks", "n_leaving", "stopped", "free_pages")


def _make(dev, rng, batch, B, W, gen, ctx0, n_free, mask_id=1000, stopped=False):
    max_pages = max(ctx0) // B + max(gen) + 1
    st = d2f.WindowState(dev, batch=batch, block_size=B, max_blocks=W,
                         max_pages_per_seq=max_pages, num_free=n_free, mask_id=mask_id)
    pt = torch.full((batch, max_pages), -1, dtype=torch.int32)
    nxt = 0
    for b, c in enumerate(ctx0):
        pt[b, :c // B] = torch.arange(nxt, nxt + c // B, dtype=torch.int32)
        nxt += c // B
    free = torch.from_numpy(rng.permutation(np.arange(nxt, nxt + n_free)).astype(np.int32))
    st.page_table.copy_(pt)
    st.ctx_len.copy_(torch.tensor(ctx0, dtype=torch.int32))
    st.gen_blocks.copy_(torch.tensor(gen, dtype=torch.int32))
    st.free_pages[:n_free].copy_(free)
    st.free_count.fill_(n_free)
    if not stopped:
        st.stopped = None
    return st


def _host(st):
    d = {k: getattr(st, k).cpu() for k in STATE_KEYS if getattr(st, k) is not None}
    if st.stopped is None:
        d["stopped"] = None
    d["free_count"] = int(st.free_count.item())
    return d


def _compare(st, ref, err, label):
    B = st.block_size
    for k in ("q_start", "tokens", "masked", "ctx_len", "page_table", "next_block",
              "n_leaving", "row_pos", "block_phase"):
        got = getattr(st, k).cpu()
        exp = ref[k]
        if k == "block_phase":
            got = got[:st.capacity // B]
        assert torch.equal(got, exp), "%s: %s differs" % (label, k)
    assert int(st.free_count.item()) == ref["free_count"], label
    n = int(st.n_append.item())
    assert n == ref["n_append"], label
    assert torch.equal(st.app_src[:n].cpu(), ref["app_src"]), label
    assert torch.equal(st.app_dst[:n].cpu(), ref["app_dst"]), label
    assert int(err.item()) == ref["err"], "%s: err %d vs %d" % (label, int(err.item()), ref["err"])


def _play_commit(rng, host, p_commit, stop_at, step, B):
    """The test's stand-in for the commit: random masked positions, at least one in
    an aggressive block; a sequence past its stop step commits everything."""
    qs = host["q_start"].tolist()
    tok, msk = host["tokens"].clone(), host["masked"].clone()
    stopped = None if host["stopped"] is None else host["stopped"].clone()
    for b in range(len(qs) - 1):
        stop = stop_at is not None and stop_at[b] is not None and step >= stop_at[b]
        for r in range(qs[b], qs[b + 1], B):
            m = [u for u in range(B) if msk[r + u]]
            if not m:
                continue
            pick = m if stop else [u for u in m if rng.random() < p_commit]
            if not pick and host["block_phase"][r // B]:
                pick = [m[-1]]
            for u in pick:
                tok[r + u] = int(rng.integers(0, 999))
                msk[r + u] = 0
        if stop and stopped is not None:
            stopped[b] = 1
    return tok, msk, stopped


CASES = [
    # batch, B, W, tau_add, tau_act, p_commit, pages short, early stop
    (3, 16, 3, 0.25, 0.75, 0.3, False, False),
    (7, 8, 2, 0.5, 1.0, 0.4, False, True),
    (600, 4, 3, 0.0, 0.5, 0.5, False, False),   # more sequences than threads
    (40, 32, 4, 0.9, 0.75, 0.2, True, False),   # the free list runs dry
    (5, 16, 1, 1.0, 0.75, 0.5, False, True),    # one block at a time
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_window_step_matches_oracle(case):
    dev = device()
    batch, B, W, tau_add, tau_act, p_commit, short, early = CASES[case]
    rng = np.random.default_rng(100 + case)
    gen = [int(rng.integers(1, 6)) for _ in range(batch)]
    ctx0 = [B * int(rng.integers(0, 5)) for _ in range(batch)]
    n_free = sum(gen) // 2 if short else sum(gen) + 2
    st = _make(dev, rng, batch, B, W, gen, ctx0, n_free, stopped=early)
    stop_at = [int(rng.integers(1, 6)) if early and rng.random() < 0.5 else None
               for _ in range(batch)]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ref_state = _host(st)
    for step in range(400):
        err.zero_()
        d2f.window_step(st, tau_add=tau_add, tau_act=tau_act, err=err,
                        use_stopped=st.stopped is not None)
        ref = oracle.window_step(ref_state, B, W, st.mask_id, tau_add, tau_act)
        torch.cuda.synchronize()
        _compare(st, ref, err, "case %d step %d" % (case, step))
        if int(ref["q_start"][-1]) == 0:
            break
        if short and step == 30:  # give the starved sequences pages again
            more = torch.arange(10000, 10000 + sum(gen), dtype=torch.int32)
            st.free_pages = more.to(dev)
            st.free_count.fill_(len(more))
            ref["free_pages"], ref["free_count"] = more.clone(), len(more)
        tok, msk, stopped = _play_commit(rng, ref, p_commit, stop_at, step, B)
        st.tokens.copy_(tok)
        st.masked.copy_(msk)
        if stopped is not None:
            st.stopped.copy_(stopped)
        ref_state = dict(ref, tokens=tok, masked=msk, stopped=stopped)
    else:
        raise AssertionError("decode did not finish")
    assert int(st.q_start[-1]) == 0


def test_window_step_refuses_an_inconsistent_state():
    dev = device()
    rng = np.random.default_rng(3)
    st = _make(dev, rng, 4, 8, 2, [2, 2, 2, 2], [8, 0, 16, 8], 12)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    d2f.window_step(st, tau_add=0.25, tau_act=0.75, err=err, use_stopped=False)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    st.n_leaving[2] = 5                       # more than the window holds
    before = {k: getattr(st, k).clone() for k in ("q_start", "tokens", "masked", "ctx_len",
                                                  "page_table", "next_block", "row_pos",
                                                  "free_count", "n_append")}
    d2f.window_step(st, tau_add=0.25, tau_act=0.75, err=err, use_stopped=False)
    torch.cuda.synchronize()
    assert int(err.item()) == 1               # D2F_ERR_INVALID_ARG
    for k, v in before.items():
        assert torch.equal(getattr(st, k), v), k   # nothing written


def test_window_step_host_checks():
    dev = device()
    rng = np.random.default_rng(4)
    st = _make(dev, rng, 2, 8, 2, [1, 1], [0, 0], 4)
    st.capacity = 20                           # not a multiple of the block size
    with pytest.raises(d2f.D2FError):
        d2f.window_step(st, tau_add=0.25, tau_act=0.75, use_stopped=False)
    st.capacity = 16                           # < batch * max_blocks * block_size = 32
    with pytest.raises(d2f.D2FError):
        d2f.window_step(st, tau_add=0.25, tau_act=0.75, use_stopped=False)
    big = _make(dev, rng, 2, 8, 2, [1, 1], [0, 0], 4)
    big.capacity = 60000                       # past one CTA's shared memory
    with pytest.raises(d2f.D2FError):
        d2f.window_step(big, tau_add=0.25, tau_act=0.75, use_stopped=False)


# ---------------------------------------------------------------------------
# a whole decode from one CUDA graph per step
# ---------------------------------------------------------------------------
def _loop_problem(seed, batch, B, W, Hq, Hkv, D, V, ctx0, gen):
    g = torch.Generator().manual_seed(seed)
    cap = batch * W * B
    prompt_pages = sum(c // B for c in ctx0)
    n_free = sum(gen) + 3
    num_pages = prompt_pages + n_free
    k_pool = torch.randn(num_pages, Hkv, B, D, generator=g).to(torch.bfloat16)
    v_pool = torch.randn(num_pages, Hkv, B, D, generator=g).to(torch.bfloat16)
    q = torch.randn(cap, Hq, D, generator=g).to(torch.bfloat16)
    k_win = torch.randn(cap, Hkv, D, generator=g).to(torch.bfloat16)
    v_win = torch.randn(cap, Hkv, D, generator=g).to(torch.bfloat16)
    # logits: a row is either confident (one logit 0, the rest -100, whose terms
    # vanish in float and in double: p = 1 exactly) or flat (p = 1/V exactly), far
    # from tau = 0.5 either way, so no rounding can move a decision; equal
    # confidences tie on both sides alike, broken by the lowest position
    logits = torch.zeros(cap, V)
    conf_rows = torch.rand(cap, generator=g) < 0.35
    peak = torch.randint(0, V, (cap,), generator=g)
    logits[conf_rows] = -100.0
    logits[conf_rows, peak[conf_rows]] = 0.0
    return dict(k_pool=k_pool, v_pool=v_pool, q=q, k_win=k_win, v_win=v_win,
                logits=logits.to(torch.bfloat16), num_pages=num_pages, n_free=n_free,
                prompt_pages=prompt_pages)


def test_decode_loop_from_one_graph_matches_the_oracle_loop():
    dev = device()
    batch, B, W, Hq, Hkv, D, V = 5, 16, 3, 8, 2, 128, 64
    ctx0, gen = [0, 16, 64, 32, 128], [4, 2, 6, 3, 1]
    tau_add, tau_act, mask_id = 0.25, 0.75, V
    pr = _loop_problem(7, batch, B, W, Hq, Hkv, D, V, ctx0, gen)
    rng = np.random.default_rng(7)
    st = _make(dev, rng, batch, B, W, gen, ctx0, pr["n_free"], mask_id=mask_id)
    # the generator above numbered prompt pages 0.. and free pages after them
    g = {k: pr[k].to(dev) for k in ("k_pool", "v_pool", "q", "k_win", "v_win", "logits")}
    tau = torch.full((batch,), 0.5, dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    cap = st.capacity
    max_ctx = max(c + n * B for c, n in zip(ctx0, gen))
    out = torch.empty_like(g["q"])
    conf = torch.empty(cap, dtype=torch.float32, device=dev)
    amax = torch.empty(cap, dtype=torch.int32, device=dev)
    rem = torch.empty(cap // B, dtype=torch.int32, device=dev)
    ws_a = d2f.attn_workspace(dev, batch=batch, total_q=cap, max_q_per_seq=W * B, max_ctx=max_ctx,
                              num_heads_q=Hq, num_heads_kv=Hkv, head_dim=D, block_size=B)
    ws_c = d2f.commit_workspace(dev, total_q=cap, vocab=V, block_size=B)

    def step():
        d2f.block_attn(g["q"], g["k_win"], g["v_win"], g["k_pool"], g["v_pool"], st.page_table,
                       st.ctx_len, st.q_start, block_size=B, max_q_per_seq=W * B,
                       max_ctx=max_ctx, out=out, want_lse=False, workspace=ws_a, err=err,
                       append_src_row=st.app_src, append_dst_page=st.app_dst,
                       append_n_dev=st.n_append)
        d2f.commit(g["logits"], st.tokens, st.masked, st.q_start, st.block_phase, tau,
                   block_size=B, mask_id=mask_id, conf=conf, argmax=amax, block_remaining=rem,
                   workspace=ws_c, err=err)
        d2f.window_step(st, tau_add=tau_add, tau_act=tau_act, err=err, use_stopped=False)

    # the oracle loop, on the host
    ref = _host(st)
    ref["stopped"] = None
    pool_k, pool_v = pr["k_pool"].clone(), pr["v_pool"].clone()
    ref = oracle.window_step(ref, B, W, mask_id, tau_add, tau_act)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        d2f.window_step(st, tau_add=tau_add, tau_act=tau_act, err=err, use_stopped=False)
        stream.synchronize()
        _compare(st, ref, err, "first window")
        graph = torch.cuda.CUDAGraph()
        snapshot = [t.clone() for t in (st.q_start, st.tokens, st.masked, st.block_phase,
                                        st.row_pos, st.ctx_len, st.page_table, st.next_block,
                                        st.n_leaving, st.free_count, st.app_src, st.app_dst,
                                        st.n_append, g["k_pool"], g["v_pool"])]
        step()                                   # warm-up (function attributes, plans)
        stream.synchronize()
        for t, s0 in zip((st.q_start, st.tokens, st.masked, st.block_phase, st.row_pos,
                          st.ctx_len, st.page_table, st.next_block, st.n_leaving,
                          st.free_count, st.app_src, st.app_dst, st.n_append, g["k_pool"],
                          g["v_pool"]), snapshot):
            t.copy_(s0)
        with torch.cuda.graph(graph, stream=stream):
            step()
    sampled = False
    for i in range(200):
        live = int(ref["q_start"][-1])
        if live == 0:
            break
        graph.replay()
        stream.synchronize()
        assert int(err.item()) == 0, "step %d: device error %d" % (i, int(err.item()))
        # the attention of this step against the oracle, once, on a full window
        if not sampled and live >= 3 * B:
            rows = slice(0, live)
            r_out, _ = oracle.block_attn(pr["q"][rows], pr["k_win"][rows], pr["v_win"][rows],
                                         pool_k, pool_v, ref["page_table"], ref["ctx_len"],
                                         ref["q_start"], B, want_lse=False)
            check_attention(out[:live], None, r_out, None, torch.bfloat16, "loop step %d" % i)
            sampled = True
        # the oracle's step: append the listed blocks, commit, schedule
        if ref["n_append"]:
            pool_k, pool_v = oracle.kv_append(pr["k_win"], pr["v_win"], ref["app_src"],
                                              ref["app_dst"], pool_k, pool_v, B)
        c = oracle.commit(pr["logits"][:live], ref["tokens"][:live], ref["masked"][:live],
                          ref["q_start"], ref["block_phase"][:live // B], tau.cpu(), B, mask_id)
        tok, msk = ref["tokens"].clone(), ref["masked"].clone()
        tok[:live], msk[:live] = c["tokens"], c["masked"]
        ref = oracle.window_step(dict(ref, tokens=tok, masked=msk, stopped=None), B, W, mask_id,
                                 tau_add, tau_act)
        _compare(st, ref, err, "loop step %d" % i)
    else:
        raise AssertionError("decode did not finish")
    assert sampled
    assert torch.equal(st.ctx_len.cpu(), torch.tensor([c + n * B for c, n in zip(ctx0, gen)],
                                                      dtype=torch.int32))
    assert torch.equal(g["k_pool"].cpu(), pool_k) and torch.equal(g["v_pool"].cpu(), pool_v)
