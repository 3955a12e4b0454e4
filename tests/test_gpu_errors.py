"""Device-side error reporting and buffer bounds, on the GPU.

Bad indices planted on the host (a page-table entry or an append destination
outside the pool, a logit row outside the logits) must set the caller's error
word to D2F_ERR_BAD_INDEX while every access stays in bounds: the kernels check
each index before they use it and skip the work it names, so the other
sequences' results still match the oracle. None of these cases faults or hangs
a GPU: the checks precede every access.

Canary bytes: outputs and workspaces are views into larger buffers whose
margins hold a fixed byte pattern; after each call the margins must be intact
(no write outside the buffers the call was given).
"""
import pytest
import torch

import oracle
from block_causal_kv_gb300 import d2f, synth
from gpu_common import check_attention, commit_compare, device

pytestmark = pytest.mark.gpu

ERR_BAD_INDEX = 4
CANARY = 0xA5
PAD = 4096  # canary bytes on each side


def _guarded(nbytes, dev):
    """A uint8 buffer of nbytes (256-byte aligned start) between two canary margins."""
    buf = torch.full((nbytes + 2 * PAD,), CANARY, dtype=torch.uint8, device=dev)
    return buf, buf[PAD:PAD + nbytes]


def _guarded_like(shape, dtype, dev, fill=None):
    elt = torch.empty((), dtype=dtype).element_size()
    n = 1
    for s in shape:
        n *= s
    buf, mid = _guarded(n * elt, dev)
    t = mid.view(dtype).view(shape)
    if fill is not None:
        t.fill_(fill)
    return buf, t


def _canary_intact(buf, label):
    head, tail = buf[:PAD].cpu(), buf[-PAD:].cpu()
    assert bool((head == CANARY).all()) and bool((tail == CANARY).all()), \
        "%s: bytes written outside the buffer" % label


def _attn(g, p, splits=0, err=None, out=None, lse=None, workspace=None, **kw):
    o, l = d2f.block_attn(g.q, g.k_win, g.v_win, g.k_pool, g.v_pool, g.page_table, g.ctx_len,
                          g.q_start, block_size=p.w.block_size, max_q_per_seq=p.max_q_per_seq,
                          max_ctx=p.max_ctx, num_splits=splits, err=err, out=out, lse=lse,
                          workspace=workspace, **kw)
    torch.cuda.synchronize()
    return o, l


def _check_others(out, p, skip_seq, label):
    ref, _ = oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
                               p.ctx_len, p.q_start, p.w.block_size)
    qs = p.q_start.tolist()
    keep = torch.ones(p.w.total_q, dtype=torch.bool)
    keep[qs[skip_seq]:qs[skip_seq + 1]] = False
    check_attention(out.cpu()[keep], None, ref[keep], None, torch.bfloat16, label)


@pytest.mark.parametrize("path", ["tc", "simt"])
@pytest.mark.parametrize("bad_id", [10 ** 6, -7])
@pytest.mark.parametrize("splits", [0, 3])
def test_bad_page_id_sets_the_error_word(path, bad_id, splits, monkeypatch):
    dev = device()
    if path == "simt":
        monkeypatch.setenv("D2F_ATTN_PATH", "simt")
    p = synth.make_problem(synth.small("ragged"))
    g = p.to(dev)
    # sequence 1 holds 200 cached tokens (13 pages): its page 3 points outside the pool
    g.page_table[1, 3] = bad_id
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out, _ = _attn(g, p, splits, err=err)
    assert int(err.item()) == ERR_BAD_INDEX
    # the other sequences are untouched by the bad id
    _check_others(out, p, 1, "%s bad page %d" % (path, bad_id))
    # a clean call afterwards (error word cleared by the caller) is exact again
    err.zero_()
    g.page_table[1, 3] = p.page_table[1, 3].to(dev)
    out, _ = _attn(g, p, splits, err=err)
    assert int(err.item()) == 0
    ref, _ = oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
                               p.ctx_len, p.q_start, p.w.block_size)
    check_attention(out, None, ref, None, torch.bfloat16, path + " after")


@pytest.mark.parametrize("bad_dst", [10 ** 6, -1])
def test_bad_append_destination_sets_the_error_word(bad_dst):
    dev = device()
    p = synth.make_problem(synth.small("dream"))
    g = p.to(dev)
    dst = g.dst_page.clone()
    dst[0] = bad_dst
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kp0, vp0 = g.k_pool.clone(), g.v_pool.clone()
    d2f.kv_append(g.k_win, g.v_win, g.src_row, dst, g.k_pool, g.v_pool, block_size=16, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == ERR_BAD_INDEX
    # the good append landed; no other page changed
    s, d = int(p.src_row[1]), int(p.dst_page[1])
    assert torch.equal(g.k_pool[d].cpu(), p.k_win[s:s + 16].transpose(0, 1))
    assert torch.equal(g.v_pool[d].cpu(), p.v_win[s:s + 16].transpose(0, 1))
    other = torch.ones(g.k_pool.shape[0], dtype=torch.bool)
    other[d] = False
    assert torch.equal(g.k_pool[other.to(dev)], kp0[other.to(dev)])
    assert torch.equal(g.v_pool[other.to(dev)], vp0[other.to(dev)])


def test_bad_src_row_sets_the_error_word():
    dev = device()
    p = synth.make_problem(synth.small("dream"))
    g = p.to(dev)
    src = g.src_row.clone()
    src[1] = p.w.total_q - 3  # the block would run past the window rows
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    d2f.kv_append(g.k_win, g.v_win, src, g.dst_page, g.k_pool, g.v_pool, block_size=16, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == ERR_BAD_INDEX
    s, d = int(p.src_row[0]), int(p.dst_page[0])
    assert torch.equal(g.k_pool[d].cpu(), p.k_win[s:s + 16].transpose(0, 1))


@pytest.mark.parametrize("bad_dst", [10 ** 6, -3])
def test_bad_fused_append_destination_sets_the_error_word(bad_dst):
    """d2f_block_attn_append: a bad destination is skipped and reported; the
    attention output of every sequence and the other append are exact."""
    dev = device()
    p = synth.make_problem(synth.small("dream"))
    g = p.to(dev)
    dst = g.dst_page.clone()
    dst[1] = bad_dst
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out, _ = _attn(g, p, 0, err=err, want_lse=False, append_src_row=g.src_row,
                   append_dst_page=dst)
    assert int(err.item()) == ERR_BAD_INDEX
    ref, _ = oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
                               p.ctx_len, p.q_start, p.w.block_size)
    check_attention(out, None, ref, None, torch.bfloat16, "fused append, bad dst")
    s, d = int(p.src_row[0]), int(p.dst_page[0])
    assert torch.equal(g.k_pool[d].cpu(), p.k_win[s:s + 16].transpose(0, 1))
    assert torch.equal(g.v_pool[d].cpu(), p.v_win[s:s + 16].transpose(0, 1))


@pytest.mark.parametrize("splits", [0, 3])
def test_bad_logit_row_sets_the_error_word(splits):
    """A logit row index outside the logits is reported and read as nothing; the
    blocks without it decide exactly as the oracle."""
    dev = device()
    p = synth.make_problem(synth.small("ragged"))
    g = p.to(dev)
    n = p.w.total_q
    B = p.w.block_size
    lr = torch.arange(n, dtype=torch.int32)
    masked_rows = torch.nonzero(p.masked).flatten().tolist()
    bad_row = masked_rows[0]
    lr[bad_row] = n + 5
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    res = d2f.commit(g.logits, g.tokens, g.masked, g.q_start, g.block_phase, g.tau, block_size=B,
                     mask_id=p.mask_id, logit_row=lr.to(dev), num_splits=splits, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == ERR_BAD_INDEX
    ref = oracle.commit(p.logits, p.tokens, p.masked, p.q_start, p.block_phase, p.tau, B,
                        p.mask_id)
    jb = bad_row // B
    keep = torch.ones(n, dtype=torch.bool)
    keep[jb * B:(jb + 1) * B] = False
    tok, msk = g.tokens.cpu(), g.masked.cpu()
    assert torch.equal(tok[keep], ref["tokens"][keep])
    assert torch.equal(msk[keep], ref["masked"][keep])
    assert torch.equal(res["argmax"].cpu()[keep], ref["argmax"][keep])


# ---------------------------------------------------------------------------
# canary bytes around outputs and workspaces
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("path", ["tc", "simt", "sk"])
@pytest.mark.parametrize("name", ["ragged", "dream", "long_b32"])
@pytest.mark.parametrize("splits", [0, 3])
def test_attention_writes_stay_inside_its_buffers(path, name, splits, monkeypatch):
    dev = device()
    if path == "simt":
        monkeypatch.setenv("D2F_ATTN_PATH", "simt")
    if path == "sk":
        if name == "dream" or splits:
            pytest.skip("the stream-K form takes one 128-row tile per (sequence, KV head), auto splits")
        monkeypatch.setenv("D2F_ATTN_SK", "1")
        monkeypatch.setenv("D2F_ATTN_SK_GRID", "7")
        monkeypatch.setenv("D2F_TC_DEEP", "1")
        monkeypatch.setenv("D2F_TC_ROWS", "128")
    p = synth.make_problem(synth.small(name))
    g = p.to(dev)
    w = p.w
    ob, out = _guarded_like(tuple(p.q.shape), p.q.dtype, dev)
    lb, lse = _guarded_like((w.total_q, w.num_heads_q), torch.float32, dev)
    need = d2f.attn_workspace_size(w.batch, w.total_q, p.max_q_per_seq, p.max_ctx, w.num_heads_q,
                                   w.num_heads_kv, w.head_dim, w.block_size, d2f.BF16, splits)
    wb, ws = _guarded(max(need, 1), dev)
    ws.zero_()
    for _ in range(2):  # the workspace is reused as the second call finds it
        o, l = _attn(g, p, splits, out=out, lse=lse, workspace=ws)
    _canary_intact(ob, "out")
    _canary_intact(lb, "lse")
    _canary_intact(wb, "workspace")
    ref, ref_lse = oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
                                     p.ctx_len, p.q_start, p.w.block_size)
    check_attention(out, lse, ref, ref_lse, torch.bfloat16, "canary " + name)


@pytest.mark.parametrize("name", ["llada", "ragged", "dream"])
@pytest.mark.parametrize("splits", [0, 5])
def test_commit_writes_stay_inside_its_buffers(name, splits):
    dev = device()
    p = synth.make_problem(synth.small(name))
    g = p.to(dev)
    n, B = p.w.total_q, p.w.block_size
    tb, tokens = _guarded_like((n,), torch.int32, dev)
    tokens.copy_(g.tokens)
    mb, masked = _guarded_like((n,), torch.uint8, dev)
    masked.copy_(g.masked)
    cb, conf = _guarded_like((n,), torch.float32, dev)
    ab, amax = _guarded_like((n,), torch.int32, dev)
    rb, rem = _guarded_like((n // B,), torch.int32, dev)
    need = d2f.commit_workspace_size(n, p.w.vocab, B, d2f.BF16, splits)
    wb, ws = _guarded(need, dev)
    ws.zero_()
    res = d2f.commit(g.logits, tokens, masked, g.q_start, g.block_phase, g.tau, block_size=B,
                     mask_id=p.mask_id, num_splits=splits, conf=conf, argmax=amax,
                     block_remaining=rem, workspace=ws)
    torch.cuda.synchronize()
    for buf, label in ((tb, "tokens"), (mb, "masked"), (cb, "conf"), (ab, "argmax"),
                       (rb, "block_remaining"), (wb, "workspace")):
        _canary_intact(buf, label)
    ref = oracle.commit(p.logits, p.tokens, p.masked, p.q_start, p.block_phase, p.tau, B,
                        p.mask_id)
    commit_compare(p, tokens, masked, conf, amax, rem, p.block_phase, p.tau, ref)


def test_append_writes_stay_inside_the_pool():
    dev = device()
    p = synth.make_problem(synth.small("dream"))
    g = p.to(dev)
    kb, kpool = _guarded_like(tuple(p.k_pool.shape), p.k_pool.dtype, dev)
    vb, vpool = _guarded_like(tuple(p.v_pool.shape), p.v_pool.dtype, dev)
    kpool.copy_(g.k_pool)
    vpool.copy_(g.v_pool)
    d2f.kv_append(g.k_win, g.v_win, g.src_row, g.dst_page, kpool, vpool, block_size=16)
    torch.cuda.synchronize()
    _canary_intact(kb, "k_pool")
    _canary_intact(vb, "v_pool")
    kp, vp = oracle.kv_append(p.k_win, p.v_win, p.src_row, p.dst_page, p.k_pool, p.v_pool, 16)
    assert torch.equal(kpool.cpu(), kp) and torch.equal(vpool.cpu(), vp)


ERR_TIMEOUT = 5


@pytest.mark.parametrize("name,deep", [("llada", None), ("dream", "0"), ("dream", "1"),
                                       ("long_b32", "1"), ("long_b32", "sk")])
@pytest.mark.parametrize("splits", [1, 3])
def test_wait_budget_runs_out_cleanly(name, deep, splits, monkeypatch):
    """The tensor-core attention's waits on another role's work are bounded. With
    their budget cut to one cycle (D2F_WAIT_CYCLES, a test switch) they run out:
    the kernel records D2F_ERR_TIMEOUT, every CTA drains the copies and MMAs it
    issued (those waits keep their own budget) and returns, cluster peers still
    exchange their partials; the launch completes. A normal call right after, on
    the same buffers, matches the oracle. Single-split and cluster-composed
    launches, the one-issuer and the split-issuer variants."""
    dev = device()
    if deep == "sk":  # the stream-K form: five CTAs over every (sequence, KV head)
        monkeypatch.setenv("D2F_ATTN_SK", "1")
        monkeypatch.setenv("D2F_ATTN_SK_GRID", "5")
        monkeypatch.setenv("D2F_TC_DEEP", "1")
        splits = 0
    elif deep is not None:
        monkeypatch.setenv("D2F_TC_DEEP", deep)
    p = synth.make_problem(synth.small(name))
    g = p.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    monkeypatch.setenv("D2F_WAIT_CYCLES", "1")
    _attn(g, p, splits, err=err)
    assert int(err.item()) == ERR_TIMEOUT
    monkeypatch.delenv("D2F_WAIT_CYCLES")
    err.zero_()
    out, lse = _attn(g, p, splits, err=err)  # a fresh (zeroed) workspace, as after any device error
    assert int(err.item()) == 0
    ref, ref_lse = oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
                                     p.ctx_len, p.q_start, p.w.block_size)
    check_attention(out, lse, ref, ref_lse, torch.bfloat16, "after the timeout " + name)
