"""Pins for the oracle's pipelined window scheduler (CPU only).

"D2F 논문 리뷰: 확산 LLM이 자기회귀 모델보다 빠른 추론을 처음으로 달성한 방식",
§쉽게 이해하기: an active window of blocks; a new block is added behind the last one
when its progress passes a threshold; a new block starts conservative and turns
aggressive once the block before it has progressed enough. "D2F: 확산 언어 모델이
KV 캐시를 얻고 자기회귀 모델보다 2.5배 빨라지는 방법", §운영 관점: a completed block
is persisted to the paged cache.

Pinned by a hand-worked run (tests/golden/window_hand.txt), by thresholds that
reduce the scheduler to known decoders (one block at a time; a window filled at
once), by hand-derived edge cases (early stop, running out of pages, refused
states), and by invariants over whole randomised decodes: the window shows every
position exactly where the bookkeeping says, committed tokens never change,
blocks enter and reach the cache once each and in order, the cache holds exactly
the committed tokens, pages come off the free list in order.
"""
import os

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "window_hand.txt")


def _state(batch, B, W, ctx, gen, pages, free_pages, max_pages, mask_id, stopped=None):
    cap = batch * W * B
    pt = torch.full((batch, max_pages), -1, dtype=torch.int32)
    for b, row in enumerate(pages):
        pt[b, :len(row)] = torch.tensor(row, dtype=torch.int32)
    return {"q_start": torch.zeros(batch + 1, dtype=torch.int32),
            "tokens": torch.full((cap,), mask_id, dtype=torch.int32),
            "masked": torch.zeros(cap, dtype=torch.uint8),
            "ctx_len": torch.tensor(ctx, dtype=torch.int32),
            "page_table": pt,
            "next_block": torch.zeros(batch, dtype=torch.int32),
            "gen_blocks": torch.tensor(gen, dtype=torch.int32),
            "n_leaving": torch.zeros(batch, dtype=torch.int32),
            "stopped": None if stopped is None else torch.tensor(stopped, dtype=torch.uint8),
            "free_pages": torch.tensor(free_pages, dtype=torch.int32),
            "free_count": len(free_pages)}


def _ints(words):
    return [int(w) for w in words if w != "|"]


def _parse_golden():
    cfg, seqs, steps, free = {}, [], [], []
    cur = None
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *rest = line.split()
            if key == "config":
                cfg = dict(kv.split("=") for kv in rest)
            elif key == "free_pages":
                free = _ints(rest)
            elif key == "seq":
                d = dict(kv.split("=") for kv in rest[1:])
                seqs.append((int(d["ctx"]), [int(x) for x in d["pages"].split(",")],
                             int(d["gen"])))
            elif key == "step":
                cur = {"name": rest[0], "page_table": {}}
                steps.append(cur)
            elif key == "commit":
                cur["commit"] = [] if rest == ["-"] else [tuple(map(int, w.split("=")))
                                                          for w in rest]
            elif key == "append":
                cur["append"] = [] if rest == ["-"] else [tuple(map(int, w.split(":")))
                                                          for w in rest]
            elif key == "page_table":
                cur["page_table"][int(rest[0])] = _ints(rest[1:])
            else:
                cur[key] = _ints(rest)
    return cfg, seqs, free, steps


def test_hand_worked_run(oracle):
    cfg, seqs, free, steps = _parse_golden()
    B, W, mask_id = int(cfg["B"]), int(cfg["W"]), int(cfg["mask_id"])
    cap, max_pages = int(cfg["capacity"]), int(cfg["max_pages"])
    st = _state(len(seqs), B, W, [s[0] for s in seqs], [s[2] for s in seqs],
                [s[1] for s in seqs], free, max_pages, mask_id)
    assert st["tokens"].shape[0] == cap
    for step in steps:
        for r, t in step["commit"]:
            st["tokens"][r] = t
            st["masked"][r] = 0
        st = oracle.window_step(st, B, W, mask_id, float(cfg["tau_add"]), float(cfg["tau_act"]))
        name = step["name"]
        assert st["err"] == 0, name
        assert st["q_start"].tolist() == step["q_start"], name
        live = int(st["q_start"][-1])
        assert st["tokens"][:live].tolist() == step["tokens"], name
        assert st["masked"][:live].tolist() == step["masked"], name
        assert st["row_pos"][:live].tolist() == step["row_pos"], name
        assert st["block_phase"][:live // B].tolist() == step["phase"], name
        assert (st["tokens"][live:] == mask_id).all() and (st["masked"][live:] == 0).all()
        assert (st["row_pos"][live:] == -1).all() and (st["block_phase"][live // B:] == 0).all()
        assert st["ctx_len"].tolist() == step["ctx_len"], name
        assert st["next_block"].tolist() == step["next_block"], name
        assert st["n_leaving"].tolist() == step["n_leaving"], name
        assert list(zip(st["app_src"].tolist(), st["app_dst"].tolist())) == step["append"], name
        assert st["free_count"] == step["free_count"][0], name
        for b, row in step["page_table"].items():
            assert st["page_table"][b].tolist() == row, name


# ---------------------------------------------------------------------------
# whole decodes: a driver that plays the commit (random subsets of the masked
# positions, respecting the aggressive rule's "at least one"), and bookkeeping of
# its own: the tokens by position and the cache by logical page
# ---------------------------------------------------------------------------
def _decode(oracle, rng, batch, B, W, tau_add, tau_act, gen, ctx0, n_free, p_commit=0.3,
            stop_at=None, check=None, max_steps=2000):
    mask_id = 1000
    max_pages = max(ctx0) // B + max(gen) + 1
    prompt_pages = sum(c // B for c in ctx0)
    pages = []
    nxt = 0
    for c in ctx0:
        pages.append(list(range(nxt, nxt + c // B)))
        nxt += c // B
    free = list(range(prompt_pages, prompt_pages + n_free))
    rng.shuffle(free)
    st = _state(batch, B, W, ctx0, gen, pages, free, max_pages, mask_id,
                stopped=[0] * batch)
    truth = [dict() for _ in range(batch)]      # position -> committed token
    cache = [dict() for _ in range(batch)]      # logical page -> tokens appended there
    pending = []                                # append list of the coming step
    for step in range(max_steps):
        old = {k: (v.clone() if torch.is_tensor(v) else v) for k, v in st.items()}
        st = oracle.window_step(st, B, W, mask_id, tau_add, tau_act)
        if check:
            check(old, st, truth, pending)
        # the appends of this step read the window's rows (final tokens)
        pending = []
        qs = st["q_start"].tolist()
        for src, dst in zip(st["app_src"].tolist(), st["app_dst"].tolist()):
            b = next(i for i in range(batch) if qs[i] <= src < qs[i + 1])
            pos = int(st["row_pos"][src])
            pending.append((b, src, dst, pos))
            cache[b][pos // B] = (dst, st["tokens"][src:src + B].tolist())
        if qs[-1] == 0:
            return st, truth, cache, step
        # the commit of this step: random masked positions; an aggressive block
        # with masked positions commits at least one
        for b in range(batch):
            for r in range(qs[b], qs[b + 1], B):
                m = [u for u in range(B) if st["masked"][r + u]]
                if not m:
                    continue
                pick = [u for u in m if rng.random() < p_commit]
                if not pick and st["block_phase"][r // B]:
                    pick = [m[0]]
                if stop_at is not None and stop_at[b] is not None and step >= stop_at[b]:
                    pick = m
                    st["stopped"][b] = 1
                for u in pick:
                    tok = int(rng.integers(0, 999))
                    st["tokens"][r + u] = tok
                    st["masked"][r + u] = 0
                    truth[b][int(st["row_pos"][r + u])] = tok
    raise AssertionError("decode did not finish")


def _invariants(B, W, tau_act, mask_id=1000):
    def check(old, st, truth, pending):
        assert st["err"] == 0
        qs = st["q_start"].tolist()
        batch = len(qs) - 1
        assert qs[0] == 0
        for b in range(batch):
            n = qs[b + 1] - qs[b]
            assert n >= 0 and n % B == 0 and n // B <= W
            # blocks that were appended during the step just run left the window
            assert int(st["ctx_len"][b]) == int(old["ctx_len"][b]) + B * int(old["n_leaving"][b])
            # the window starts right after the cache, positions consecutive
            pos = st["row_pos"][qs[b]:qs[b + 1]].tolist()
            assert pos == list(range(int(st["ctx_len"][b]), int(st["ctx_len"][b]) + n))
            # every shown position carries the committed token, or is masked
            for r, p in zip(range(qs[b], qs[b + 1]), pos):
                if p in truth[b]:
                    assert not st["masked"][r] and int(st["tokens"][r]) == truth[b][p]
                else:
                    assert st["masked"][r] and int(st["tokens"][r]) == mask_id
            # blocks enter one at a time
            assert int(st["next_block"][b]) - int(old["next_block"][b]) in (0, 1)
            # the oldest block is aggressive (the cache precedes it) when tau_act <= 1
            if n:
                assert st["block_phase"][qs[b] // B] == (1 if 1.0 >= tau_act else 0)
        live = qs[-1]
        assert (st["masked"][live:] == 0).all() and (st["row_pos"][live:] == -1).all()
        # the append list: complete oldest blocks, pages off the top of the list
        fc_old = int(old["free_count"])
        got = st["app_dst"].tolist()
        assert got == old["free_pages"][fc_old - len(got):fc_old].flip(0).tolist()
        assert st["free_count"] == fc_old - len(got)
        per_seq = {}
        for src, dst in zip(st["app_src"].tolist(), got):
            b = next(i for i in range(batch) if qs[i] <= src < qs[i + 1])
            i = per_seq.get(b, 0)
            assert src == qs[b] + i * B                    # a prefix of the window
            assert not st["masked"][src:src + B].any()      # complete
            assert int(st["page_table"][b][int(st["ctx_len"][b]) // B + i]) == dst
            per_seq[b] = i + 1
        for b in range(batch):
            assert int(st["n_leaving"][b]) == per_seq.get(b, 0)
    return check


@pytest.mark.parametrize("seed", range(6))
def test_whole_decodes_keep_their_invariants(oracle, seed):
    rng = np.random.default_rng(seed)
    B = int(rng.choice([4, 8]))
    W = int(rng.integers(1, 4))
    batch = int(rng.integers(1, 6))
    tau_add = float(rng.choice([0.0, 0.25, 0.5, 0.9]))
    tau_act = float(rng.choice([0.5, 0.75, 1.0]))
    gen = [int(rng.integers(1, 7)) for _ in range(batch)]
    ctx0 = [B * int(rng.integers(0, 4)) for _ in range(batch)]
    st, truth, cache, steps = _decode(oracle, rng, batch, B, W, tau_add, tau_act, gen, ctx0,
                                      n_free=sum(gen) + 3, check=_invariants(B, W, tau_act))
    used = []
    for b in range(batch):
        # every generated block reached the cache once, in order, with its tokens
        assert int(st["ctx_len"][b]) == ctx0[b] + gen[b] * B
        assert sorted(cache[b]) == list(range(ctx0[b] // B, ctx0[b] // B + gen[b]))
        for lp, (page, toks) in cache[b].items():
            assert toks == [truth[b][lp * B + u] for u in range(B)]
            assert int(st["page_table"][b][lp]) == page
            used.append(page)
        assert int(st["next_block"][b]) == gen[b]
    assert len(set(used)) == len(used)


def test_threshold_one_is_one_block_at_a_time(oracle):
    """tau_add >= 1: no block is ever past the threshold, so a block enters only
    into an empty window: plain block-by-block decoding (each block completes,
    is appended, and only then does the next one start)."""
    rng = np.random.default_rng(11)
    B, W = 4, 3

    def check(old, st, truth, pending):
        qs = st["q_start"].tolist()
        for b in range(len(qs) - 1):
            n = (qs[b + 1] - qs[b]) // B
            assert n <= 1
            if int(st["next_block"][b]) > int(old["next_block"][b]):
                # the new block is alone (the previous one left): all of it masked
                assert n == 1 and bool(st["masked"][qs[b]:qs[b] + B].all())

    st, truth, cache, steps = _decode(oracle, rng, 3, B, W, 1.0, 0.75, [3, 2, 4], [0, 4, 8],
                                      n_free=12, check=check)
    assert [int(c) for c in st["ctx_len"]] == [12, 12, 24]


def test_negative_threshold_fills_the_window_at_once(oracle):
    """tau_add < 0: every block is past the threshold, so one block enters per
    step until the window holds W blocks."""
    B, W = 4, 3
    st = _state(1, B, W, [0], [5], [[]], list(range(8)), 8, 99)
    sizes = []
    for _ in range(4):
        st = oracle.window_step(st, B, W, 99, -1.0, 0.75)
        sizes.append(int(st["q_start"][1]) // B)
    assert sizes == [1, 2, 3, 3]
    # nothing committed: only the oldest block is aggressive (tau_act = 0.75)
    assert st["block_phase"][:3].tolist() == [1, 0, 0]
    st2 = oracle.window_step(st, B, W, 99, -1.0, 0.0)
    assert st2["block_phase"][:3].tolist() == [1, 1, 1]       # tau_act = 0: all aggressive
    st3 = oracle.window_step(st, B, W, 99, -1.0, 1.5)
    assert st3["block_phase"][:3].tolist() == [0, 0, 0]       # tau_act > 1: none


def test_stopped_sequence_takes_no_new_block_and_drains(oracle):
    rng = np.random.default_rng(5)
    st, truth, cache, steps = _decode(oracle, rng, 2, 4, 2, 0.25, 0.75, [6, 3], [4, 0],
                                      n_free=12, stop_at=[3, None])
    # sequence 0 stopped early: fewer blocks than asked for, all of them cached
    n0 = int(st["next_block"][0])
    assert n0 < 6 and int(st["ctx_len"][0]) == 4 + 4 * n0
    assert int(st["ctx_len"][1]) == 12


def test_out_of_pages(oracle):
    """Two sequences each with a complete block and one page left: the first
    sequence (in order) gets it, the second keeps its block in the window and the
    error word says 7; a later call with a page appends it."""
    B, W = 4, 2
    st = _state(2, B, W, [4, 4], [1, 1], [[0], [1]], [7], 4, 99)
    st = oracle.window_step(st, B, W, 99, 0.25, 0.75)        # both take a block
    st["tokens"][0:8] = torch.arange(8, dtype=torch.int32)
    st["masked"][0:8] = 0
    st = oracle.window_step(st, B, W, 99, 2.0, 0.75)         # no new block (tau_add 2)
    assert st["err"] == 7
    assert list(zip(st["app_src"].tolist(), st["app_dst"].tolist())) == [(0, 7)]
    assert st["n_leaving"].tolist() == [1, 0]
    assert st["page_table"][0].tolist()[:2] == [0, 7] and st["page_table"][1].tolist()[1] == -1
    st["free_pages"] = torch.tensor([9], dtype=torch.int32)
    st["free_count"] = 1
    st = oracle.window_step(st, B, W, 99, 2.0, 0.75)
    assert st["err"] == 0 and st["ctx_len"].tolist() == [8, 4]
    assert list(zip(st["app_src"].tolist(), st["app_dst"].tolist())) == [(0, 9)]
    assert st["q_start"].tolist() == [0, 0, 4]


def test_full_page_table_row(oracle):
    B, W = 4, 1
    st = _state(1, B, W, [4], [3], [[0]], [5, 6, 7], 1, 99)   # one slot, the prompt's
    st = oracle.window_step(st, B, W, 99, 0.25, 0.75)
    st["masked"][:4] = 0
    st = oracle.window_step(st, B, W, 99, 0.25, 0.75)
    assert st["err"] == 7 and st["n_append"] == 0 and st["free_count"] == 3


@pytest.mark.parametrize("bad", ["leaving", "ctx", "partial", "too_many", "start"])
def test_inconsistent_state_is_refused(oracle, bad):
    B, W = 4, 2
    st = _state(1, B, W, [4], [3], [[0]], [5, 6], 4, 99)
    st = oracle.window_step(st, B, W, 99, 0.25, 0.75)
    if bad == "leaving":
        st["n_leaving"][0] = 2
    elif bad == "ctx":
        st["ctx_len"][0] = 6
    elif bad == "partial":
        st["q_start"][1] = 3
    elif bad == "too_many":
        st["q_start"][1] = 12
    else:
        st["q_start"][0] = 4
    with pytest.raises(ValueError):
        oracle.window_step(st, B, W, 99, 0.25, 0.75)
