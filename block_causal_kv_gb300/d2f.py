"""Python binding of libd2f (ctypes): argument marshalling only.

Every function takes torch CUDA tensors, passes their device pointers, sizes
and the current CUDA stream to the C entry point of the same name, and raises
D2FError on a non-OK status. No computation happens here; there is no CPU
fallback: if libd2f.so is missing the import fails.

    from block_causal_kv_gb300 import d2f
    out, lse = d2f.block_attn(q, k_win, v_win, k_pool, v_pool, page_table, ctx_len,
                              q_start, block_size=16, max_q_per_seq=48, max_ctx=1024)
    res = d2f.commit(logits, tokens, masked, q_start, block_phase, tau,
                     block_size=16, mask_id=126464)
    d2f.kv_append(k_win, v_win, src_row, dst_page, k_pool, v_pool, block_size=16)
"""
import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libd2f.so")

BF16 = 0
F32 = 1
PHASE_CONSERVATIVE = 0
PHASE_AGGRESSIVE = 1

STATUS = {0: "D2F_OK", 1: "D2F_ERR_INVALID_ARG", 2: "D2F_ERR_UNSUPPORTED", 3: "D2F_ERR_CUDA",
          4: "D2F_ERR_BAD_INDEX", 5: "D2F_ERR_TIMEOUT", 6: "D2F_ERR_WORKSPACE",
          7: "D2F_ERR_NO_PAGE"}

# Every symbol include/d2f.h declares.
EXPORTS = ("d2f_version", "d2f_status_string", "d2f_last_error_string",
           "d2f_block_attn_workspace_size", "d2f_block_attn", "d2f_block_attn_flags",
           "d2f_block_attn_append", "d2f_block_attn_part",
           "d2f_commit_workspace_size",
           "d2f_commit", "d2f_commit_metric", "d2f_commit_noalloc", "d2f_kv_append",
           "d2f_kv_append_dev", "d2f_block_attn_append_dev", "d2f_window_step")

# attention parts of block_attn(part=...) (include/d2f.h D2F_ATTN_*)
ATTN_ALL, ATTN_CACHED, ATTN_WINDOW = 0, 1, 2
# d2f_block_attn_flags: the cache and window layout are final before the preceding kernel
CACHE_READY = 1
# confidence metrics of commit(metric=...) (include/d2f.h D2F_CONF_*)
CONF_PMAX, CONF_NEG_ENTROPY, CONF_MARGIN, CONF_LOGIT_GAP = 0, 1, 2, 3


class D2FError(RuntimeError):
    def __init__(self, status, message):
        super().__init__("%s: %s" % (STATUS.get(status, status), message))
        self.status = status


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t


def load(path=LIB_PATH):
    """Load libd2f.so (built in-tree by __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError("libd2f.so is not built (%s); run __graft_entry__.build()" % path)
    lib = ctypes.CDLL(path)
    lib.d2f_version.restype = _I
    lib.d2f_status_string.restype = ctypes.c_char_p
    lib.d2f_status_string.argtypes = [_I]
    lib.d2f_last_error_string.restype = ctypes.c_char_p
    lib.d2f_block_attn_workspace_size.restype = _I
    lib.d2f_block_attn_workspace_size.argtypes = [_I] * 10 + [ctypes.POINTER(_SZ)]
    lib.d2f_block_attn.restype = _I
    lib.d2f_block_attn.argtypes = ([_P] * 6 + [_I] + [_P] * 2 + [_P, _P] + [_I] * 10 +
                                   [ctypes.c_float, _I, _P, _SZ, _P, _P])
    lib.d2f_block_attn_flags.restype = _I
    lib.d2f_block_attn_flags.argtypes = ([_P] * 6 + [_I] + [_P] * 2 + [_P, _P] + [_I] * 10 +
                                         [ctypes.c_float, _I, _P, _SZ, ctypes.c_uint, _P, _P])
    lib.d2f_block_attn_append.restype = _I
    lib.d2f_block_attn_append.argtypes = ([_P] * 6 + [_I] + [_P] * 2 + [_P, _P] + [_I] * 10 +
                                          [ctypes.c_float, _I, _P, _SZ, _P, _P, _I, _P, _P])
    lib.d2f_block_attn_part.restype = _I
    lib.d2f_block_attn_part.argtypes = ([_P] * 6 + [_I] + [_P] * 2 + [_P, _P] + [_I] * 10 +
                                        [ctypes.c_float, _I, _P, _SZ, _I, _P, _P, _P, _P])
    lib.d2f_commit_workspace_size.restype = _I
    lib.d2f_commit_workspace_size.argtypes = [_I] * 5 + [ctypes.POINTER(_SZ)]
    lib.d2f_commit.restype = _I
    lib.d2f_commit.argtypes = ([_P, ctypes.c_int64, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I,
                                ctypes.c_int32, _P, _P, _P, _I, _P, _SZ, _P, _P])
    lib.d2f_commit_metric.restype = _I
    lib.d2f_commit_metric.argtypes = ([_P, ctypes.c_int64, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I,
                                       _I, _I, ctypes.c_int32, _I, _P, _P, _P, _P, _P, _I, _P, _SZ,
                                       _P, _P])
    lib.d2f_commit_noalloc.restype = _I
    lib.d2f_commit_noalloc.argtypes = ([_P, ctypes.c_int64, _I, _I, _I, _P, _P, _P, _P, _P, _P, _I,
                                        _I, _I, ctypes.c_int32, _P, _P, _P, _I, _P, _P])
    lib.d2f_kv_append.restype = _I
    lib.d2f_kv_append.argtypes = [_P, _P, _P, _P, _I, _I, _P, _P, _I, _I, _I, _I, _I, _P, _P]
    lib.d2f_kv_append_dev.restype = _I
    lib.d2f_kv_append_dev.argtypes = [_P, _P, _P, _P, _P, _I, _I, _P, _P, _I, _I, _I, _I, _I,
                                      _P, _P]
    lib.d2f_block_attn_append_dev.restype = _I
    lib.d2f_block_attn_append_dev.argtypes = ([_P] * 6 + [_I] + [_P] * 2 + [_P, _P] + [_I] * 10 +
                                              [ctypes.c_float, _I, _P, _SZ, _P, _P, _P, _I, _P,
                                               _P])
    lib.d2f_window_step.restype = _I
    lib.d2f_window_step.argtypes = ([_I] * 5 + [ctypes.c_int32, ctypes.c_float, ctypes.c_float] +
                                    [_P] * 18)
    _lib = lib
    return lib


def _check(status):
    if status != 0:
        raise D2FError(status, _lib.d2f_last_error_string().decode())


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError("libd2f takes bfloat16 or float32 tensors, got %s" % t.dtype)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _dev(t, name, dtype=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))


def status_string(status):
    return load().d2f_status_string(status).decode()


def version():
    return load().d2f_version()


# ---------------------------------------------------------------------------
# block attention
# ---------------------------------------------------------------------------
def attn_workspace_size(batch, total_q, max_q_per_seq, max_ctx, num_heads_q, num_heads_kv,
                        head_dim, block_size, dtype=BF16, num_splits=0):
    lib = load()
    n = _SZ(0)
    _check(lib.d2f_block_attn_workspace_size(batch, total_q, max_q_per_seq, max_ctx, num_heads_q,
                                             num_heads_kv, head_dim, block_size, dtype,
                                             num_splits, ctypes.byref(n)))
    return n.value


def attn_workspace(device, **kw):
    """A zero-filled workspace of the size attn_workspace_size(**kw) returns."""
    return torch.zeros(max(attn_workspace_size(**kw), 1), dtype=torch.uint8, device=device)


def block_attn(q, k_win, v_win, k_pool, v_pool, page_table, ctx_len, q_start, *, block_size,
               max_q_per_seq, max_ctx, softmax_scale=None, num_splits=0, out=None, lse=None,
               want_lse=True, workspace=None, err=None, stream=None, append_src_row=None,
               append_dst_page=None, part=ATTN_ALL, prev_out=None, prev_lse=None,
               append_n_dev=None, cache_ready=False):
    """Block-causal attention of the window over [paged cache ; window] (one layer).
    With append_src_row / append_dst_page (int32 [n_append]) the finished blocks
    are appended to their pages in the same launch (d2f_block_attn_append).
    With append_n_dev (int32 [1] on the device, d2f_block_attn_append_dev) the list's
    length is read there, at most len(append_src_row).
    part ATTN_CACHED / ATTN_WINDOW (d2f_block_attn_part): one part of the keys; the
    window part composes a kept cached part given as prev_out / prev_lse.
    cache_ready=True (d2f_block_attn_flags with D2F_ATTN_CACHE_READY, the whole
    attention only): page_table, ctx_len, q_start and the cached pages are not
    written by the kernel that precedes this call in the stream.

    Returns (out [total_q, Hq, D] like q, lse [total_q, Hq] float32 or None)."""
    lib = load()
    for name, t in (("q", q), ("k_win", k_win), ("v_win", v_win), ("k_pool", k_pool),
                    ("v_pool", v_pool)):
        _dev(t, name, q.dtype)
    _dev(page_table, "page_table", torch.int32)
    _dev(ctx_len, "ctx_len", torch.int32)
    _dev(q_start, "q_start", torch.int32)
    total_q, hq, d = q.shape
    hkv = k_win.shape[1]
    batch = ctx_len.shape[0]
    dt = _dtype_code(q)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _dev(out, "out", q.dtype)
    if lse is None and want_lse:
        lse = torch.empty((total_q, hq), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = attn_workspace(q.device, batch=batch, total_q=total_q,
                                   max_q_per_seq=max_q_per_seq, max_ctx=max_ctx,
                                   num_heads_q=hq, num_heads_kv=hkv, head_dim=d,
                                   block_size=block_size, dtype=dt, num_splits=num_splits)
    args = (_ptr(q), _ptr(k_win), _ptr(v_win), _ptr(k_pool), _ptr(v_pool), _ptr(page_table),
            page_table.shape[1] if page_table is not None else 0, _ptr(ctx_len), _ptr(q_start),
            _ptr(out), _ptr(lse), batch, total_q, max_q_per_seq, max_ctx, hq, hkv, d, block_size,
            k_pool.shape[0] if k_pool is not None else 0, dt, float(softmax_scale), num_splits,
            _ptr(workspace), workspace.numel() * workspace.element_size())
    if cache_ready and (part != ATTN_ALL or append_src_row is not None):
        raise ValueError("cache_ready goes with the whole attention, without an append")
    if part != ATTN_ALL:
        if append_src_row is not None:
            raise ValueError("an append goes with the whole attention (part ATTN_ALL)")
        _dev(prev_out, "prev_out", q.dtype)
        _dev(prev_lse, "prev_lse", torch.float32)
        _check(lib.d2f_block_attn_part(*args, int(part), _ptr(prev_out), _ptr(prev_lse), _ptr(err),
                                       _stream(stream)))
    elif append_src_row is None and cache_ready:
        _check(lib.d2f_block_attn_flags(*args, CACHE_READY, _ptr(err), _stream(stream)))
    elif append_src_row is None:
        _check(lib.d2f_block_attn(*args, _ptr(err), _stream(stream)))
    elif append_n_dev is not None:
        _dev(append_src_row, "append_src_row", torch.int32)
        _dev(append_dst_page, "append_dst_page", torch.int32)
        _dev(append_n_dev, "append_n_dev", torch.int32)
        _check(lib.d2f_block_attn_append_dev(*args, _ptr(append_src_row), _ptr(append_dst_page),
                                             _ptr(append_n_dev), append_src_row.shape[0],
                                             _ptr(err), _stream(stream)))
    else:
        _dev(append_src_row, "append_src_row", torch.int32)
        _dev(append_dst_page, "append_dst_page", torch.int32)
        _check(lib.d2f_block_attn_append(*args, _ptr(append_src_row), _ptr(append_dst_page),
                                         append_src_row.shape[0], _ptr(err), _stream(stream)))
    return out, lse


# ---------------------------------------------------------------------------
# commit
# ---------------------------------------------------------------------------
def commit_workspace_size(total_q, vocab, block_size, dtype=BF16, num_splits=0):
    lib = load()
    n = _SZ(0)
    _check(lib.d2f_commit_workspace_size(total_q, vocab, dtype, block_size, num_splits,
                                         ctypes.byref(n)))
    return n.value


def commit_workspace(device, **kw):
    return torch.zeros(max(commit_workspace_size(**kw), 1), dtype=torch.uint8, device=device)


def commit(logits, tokens, masked, q_start, block_phase, tau, *, block_size, mask_id,
           logit_row=None, num_splits=0, conf=None, argmax=None, block_remaining=None,
           want_outputs=True, workspace=None, err=None, stream=None, metric=CONF_PMAX,
           early_gap=None, stopped=None):
    """Confidence commit + remask, in place on tokens / masked.

    logits may be a row-strided view ([rows, vocab] with stride(1) == 1).
    metric: CONF_PMAX (d2f_commit) or another CONF_* (d2f_commit_metric; tau in
    the metric's units). early_gap (float32 [batch]) turns on the early commit
    of whole sequences; stopped (uint8 [batch]) receives its flags. Returns
    dict(conf, argmax, block_remaining, stopped) (device tensors, or None)."""
    lib = load()
    if not logits.is_cuda or logits.stride(-1) != 1:
        raise ValueError("logits must be a CUDA tensor with unit stride along the vocabulary")
    _dev(tokens, "tokens", torch.int32)
    _dev(masked, "masked", torch.uint8)
    _dev(q_start, "q_start", torch.int32)
    _dev(block_phase, "block_phase", torch.uint8)
    _dev(tau, "tau", torch.float32)
    _dev(logit_row, "logit_row", torch.int32)
    total_q = tokens.shape[0]
    rows, vocab = logits.shape
    dt = _dtype_code(logits)
    dev = tokens.device
    if want_outputs:
        if conf is None:
            conf = torch.empty(total_q, dtype=torch.float32, device=dev)
        if argmax is None:
            argmax = torch.empty(total_q, dtype=torch.int32, device=dev)
        if block_remaining is None:
            block_remaining = torch.empty(max(total_q // block_size, 1), dtype=torch.int32,
                                          device=dev)
    if workspace is None:
        workspace = commit_workspace(dev, total_q=total_q, vocab=vocab, block_size=block_size,
                                     dtype=dt, num_splits=num_splits)
    _dev(early_gap, "early_gap", torch.float32)
    _dev(stopped, "stopped", torch.uint8)
    if metric == CONF_PMAX and early_gap is None:
        _check(lib.d2f_commit(
            _ptr(logits), logits.stride(0), dt, vocab, rows, _ptr(logit_row), _ptr(tokens),
            _ptr(masked), _ptr(q_start), _ptr(block_phase), _ptr(tau), q_start.shape[0] - 1,
            total_q, block_size, int(mask_id), _ptr(conf), _ptr(argmax), _ptr(block_remaining),
            num_splits, _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(err),
            _stream(stream)))
    else:
        _check(lib.d2f_commit_metric(
            _ptr(logits), logits.stride(0), dt, vocab, rows, _ptr(logit_row), _ptr(tokens),
            _ptr(masked), _ptr(q_start), _ptr(block_phase), _ptr(tau), q_start.shape[0] - 1,
            total_q, block_size, int(mask_id), int(metric), _ptr(early_gap), _ptr(stopped),
            _ptr(conf), _ptr(argmax), _ptr(block_remaining), num_splits, _ptr(workspace),
            workspace.numel() * workspace.element_size(), _ptr(err), _stream(stream)))
    return {"conf": conf, "argmax": argmax, "block_remaining": block_remaining,
            "stopped": stopped}


def commit_noalloc(logits, tokens, masked, q_start, block_phase, tau, *, block_size, mask_id,
                   logit_row=None, num_splits=0, conf=None, argmax=None, block_remaining=None,
                   err=None, stream=None):
    """d2f_commit_noalloc: the commit without a workspace, for callers that cannot
    allocate device memory; its scratch is a fixed array inside the library (see
    include/d2f.h for the size limit and the rule that calls must not overlap)."""
    lib = load()
    if not logits.is_cuda or logits.stride(-1) != 1:
        raise ValueError("logits must be a CUDA tensor with unit stride along the vocabulary")
    total_q = tokens.shape[0]
    rows, vocab = logits.shape
    _check(lib.d2f_commit_noalloc(
        _ptr(logits), logits.stride(0), _dtype_code(logits), vocab, rows, _ptr(logit_row),
        _ptr(tokens), _ptr(masked), _ptr(q_start), _ptr(block_phase), _ptr(tau),
        q_start.shape[0] - 1, total_q, block_size, int(mask_id), _ptr(conf), _ptr(argmax),
        _ptr(block_remaining), num_splits, _ptr(err), _stream(stream)))
    return {"conf": conf, "argmax": argmax, "block_remaining": block_remaining}


# ---------------------------------------------------------------------------
# KV append
# ---------------------------------------------------------------------------
def kv_append(k_win, v_win, src_row, dst_page, k_pool, v_pool, *, block_size, err=None,
              stream=None, n_append_dev=None):
    """Copy finished blocks (rows src_row[a] .. +B of the window K/V) into pages dst_page[a].
    n_append_dev (int32 [1] on the device, d2f_kv_append_dev): the list's length is
    read there, at most len(src_row)."""
    lib = load()
    for name, t in (("k_win", k_win), ("v_win", v_win), ("k_pool", k_pool), ("v_pool", v_pool)):
        _dev(t, name, k_win.dtype)
    _dev(src_row, "src_row", torch.int32)
    _dev(dst_page, "dst_page", torch.int32)
    total_q, hkv, d = k_win.shape
    if n_append_dev is not None:
        _dev(n_append_dev, "n_append_dev", torch.int32)
        _check(lib.d2f_kv_append_dev(
            _ptr(k_win), _ptr(v_win), _ptr(src_row), _ptr(dst_page), _ptr(n_append_dev),
            src_row.shape[0], total_q, _ptr(k_pool), _ptr(v_pool), hkv, d, block_size,
            k_pool.shape[0], _dtype_code(k_win), _ptr(err), _stream(stream)))
        return
    _check(lib.d2f_kv_append(
        _ptr(k_win), _ptr(v_win), _ptr(src_row), _ptr(dst_page), src_row.shape[0], total_q,
        _ptr(k_pool), _ptr(v_pool), hkv, d, block_size, k_pool.shape[0], _dtype_code(k_win),
        _ptr(err), _stream(stream)))


# ---------------------------------------------------------------------------
# pipelined window scheduler
# ---------------------------------------------------------------------------
class WindowState:
    """Device buffers of the window scheduler (d2f_window_step), one attribute per
    argument of that name: q_start, tokens, masked, block_phase, row_pos,
    ctx_len, page_table, next_block, gen_blocks, n_leaving, stopped, free_pages,
    free_count, app_src, app_dst, n_append. Created empty (no window, nothing
    listed); the caller fills ctx_len / page_table (prompt pages), gen_blocks
    and the free list."""

    def __init__(self, device, *, batch, block_size, max_blocks, max_pages_per_seq, num_free,
                 mask_id, capacity=None):
        i32 = dict(dtype=torch.int32, device=device)
        u8 = dict(dtype=torch.uint8, device=device)
        cap = batch * max_blocks * block_size if capacity is None else capacity
        self.batch, self.block_size, self.max_blocks, self.capacity = (batch, block_size,
                                                                       max_blocks, cap)
        self.mask_id = mask_id
        self.q_start = torch.zeros(batch + 1, **i32)
        self.tokens = torch.full((cap,), mask_id, **i32)
        self.masked = torch.zeros(cap, **u8)
        self.block_phase = torch.zeros(max(cap // block_size, 1), **u8)
        self.row_pos = torch.full((cap,), -1, **i32)
        self.ctx_len = torch.zeros(batch, **i32)
        self.page_table = torch.full((batch, max_pages_per_seq), -1, **i32)
        self.next_block = torch.zeros(batch, **i32)
        self.gen_blocks = torch.zeros(batch, **i32)
        self.n_leaving = torch.zeros(batch, **i32)
        self.stopped = torch.zeros(batch, **u8)
        self.free_pages = torch.zeros(max(num_free, 1), **i32)
        self.free_count = torch.zeros(1, **i32)
        self.app_src = torch.zeros(max(cap // block_size, 1), **i32)
        self.app_dst = torch.zeros_like(self.app_src)
        self.n_append = torch.zeros(1, **i32)


def window_step(st, *, tau_add, tau_act, err=None, stream=None, use_stopped=True):
    """One call of the device window scheduler on WindowState `st` (in place)."""
    lib = load()
    _check(lib.d2f_window_step(
        st.batch, st.block_size, st.max_blocks, st.capacity, st.page_table.shape[1],
        int(st.mask_id), float(tau_add), float(tau_act), _ptr(st.q_start), _ptr(st.tokens),
        _ptr(st.masked), _ptr(st.block_phase), _ptr(st.row_pos), _ptr(st.ctx_len),
        _ptr(st.page_table), _ptr(st.next_block), _ptr(st.gen_blocks), _ptr(st.n_leaving),
        _ptr(st.stopped) if use_stopped else None, _ptr(st.free_pages), _ptr(st.free_count),
        _ptr(st.app_src), _ptr(st.app_dst), _ptr(st.n_append), _ptr(err), _stream(stream)))
