"""CPU oracle for the D2F block-diffusion decoding hot path.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package; the product
path (the CUDA library and its binding) never does. The arithmetic lives in
``d2f_oracle.c`` (plain C, double precision); this module only marshals
torch CPU tensors into pointers.

Functions:
  block_attn  -- block-causal attention over [paged cache ; window], fp64.
  commit      -- per-position max-probability confidence, threshold /
                 aggressive commit per block, remasking.
  kv_append   -- bitwise copy of finished blocks into their pages.
  window_step -- the pipelined window scheduler between two steps (block
                 entry, phases, append list, pages, repacked window).
"""
import ctypes
import os

import torch

from . import build as _build

_lib = None
_P = ctypes.c_void_p

DT_BF16 = 0
DT_F32 = 1
DT_F64 = 2


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        lib.d2f_oracle_block_attn.restype = ctypes.c_int
        lib.d2f_oracle_block_attn.argtypes = [
            _P, _P, _P, _P, _P, _P, ctypes.c_int, _P, _P,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, _P, _P, ctypes.c_int]
        lib.d2f_oracle_block_attn_part.restype = ctypes.c_int
        lib.d2f_oracle_block_attn_part.argtypes = [
            _P, _P, _P, _P, _P, _P, ctypes.c_int, _P, _P,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int, _P, _P,
            _P, _P, ctypes.c_int]
        lib.d2f_oracle_commit.restype = ctypes.c_int
        lib.d2f_oracle_commit.argtypes = [
            _P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P,
            _P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int32,
            _P, _P, _P, ctypes.c_int]
        lib.d2f_oracle_commit_metric.restype = ctypes.c_int
        lib.d2f_oracle_commit_metric.argtypes = [
            _P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P,
            _P, _P, _P, _P, _P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int32,
            _P, _P, _P, ctypes.c_int, _P, _P, ctypes.c_int]
        lib.d2f_oracle_window_step.restype = ctypes.c_int
        lib.d2f_oracle_window_step.argtypes = [
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int32,
            ctypes.c_float, ctypes.c_float] + [_P] * 17
        lib.d2f_oracle_kv_append.restype = ctypes.c_int
        lib.d2f_oracle_kv_append.argtypes = [
            _P, _P, _P, _P, ctypes.c_int, ctypes.c_int, _P, _P,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DT_BF16
    if t.dtype == torch.float32:
        return DT_F32
    if t.dtype == torch.float64:
        return DT_F64
    raise TypeError("oracle supports bfloat16, float32 and float64 inputs, got %s" % t.dtype)


def _cpu(t, dtype=None):
    if t is None:
        return None
    t = t.detach().to("cpu")
    if dtype is not None:
        t = t.to(dtype)
    return t.contiguous()


def _ptr(t):
    return None if t is None else t.data_ptr()


def block_attn(q, k_win, v_win, k_pool, v_pool, page_table, ctx_len, q_start,
               block_size, scale=None, nthreads=None, want_lse=True):
    """Block-causal attention, fp64.

    q [total_q, Hq, D]; k_win/v_win [total_q, Hkv, D]; k_pool/v_pool
    [num_pages, Hkv, B, D]; page_table [batch, max_pages] int32; ctx_len [batch];
    q_start [batch+1]. Returns (out [total_q, Hq, D] float64, lse [total_q, Hq]
    float64 or None).
    """
    lib = _load()
    q, k_win, v_win, k_pool, v_pool = (_cpu(x) for x in (q, k_win, v_win, k_pool, v_pool))
    dt = _dt(q)
    for x in (k_win, v_win, k_pool, v_pool):
        if x.dtype != q.dtype:
            raise TypeError("all attention operands must share one dtype")
    page_table = _cpu(page_table, torch.int32)
    ctx_len = _cpu(ctx_len, torch.int32)
    q_start = _cpu(q_start, torch.int32)
    total_q, hq, d = q.shape
    hkv = k_win.shape[1]
    num_pages = k_pool.shape[0]
    batch = ctx_len.shape[0]
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    out = torch.zeros((total_q, hq, d), dtype=torch.float64)
    lse = torch.zeros((total_q, hq), dtype=torch.float64) if want_lse else None
    rc = lib.d2f_oracle_block_attn(
        _ptr(q), _ptr(k_win), _ptr(v_win), _ptr(k_pool), _ptr(v_pool), _ptr(page_table),
        page_table.shape[1] if page_table.dim() == 2 else 0, _ptr(ctx_len), _ptr(q_start),
        batch, total_q, hq, hkv, d, block_size, num_pages, dt, float(scale),
        _ptr(out), _ptr(lse), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle block_attn rejected its input (code %d)" % rc)
    return out, lse


# attention parts of block_attn_part(): all keys, cached tokens only, window only
ATTN_ALL, ATTN_CACHED, ATTN_WINDOW = 0, 1, 2


def block_attn_part(q, k_win, v_win, k_pool, v_pool, page_table, ctx_len, q_start, block_size,
                    part, prev_out=None, prev_lse=None, scale=None, nthreads=None):
    """Attention over one part of the keys (fp64); part ATTN_WINDOW with
    prev_out / prev_lse (a cached-part result) composes the two in log space.
    Returns (out [total_q, Hq, D] float64, lse [total_q, Hq] float64)."""
    lib = _load()
    q, k_win, v_win, k_pool, v_pool = (_cpu(x) for x in (q, k_win, v_win, k_pool, v_pool))
    dt = _dt(q)
    page_table = _cpu(page_table, torch.int32)
    ctx_len = _cpu(ctx_len, torch.int32)
    q_start = _cpu(q_start, torch.int32)
    prev_out = _cpu(prev_out, torch.float64)
    prev_lse = _cpu(prev_lse, torch.float64)
    total_q, hq, d = q.shape
    if scale is None:
        scale = 1.0 / (d ** 0.5)
    out = torch.zeros((total_q, hq, d), dtype=torch.float64)
    lse = torch.zeros((total_q, hq), dtype=torch.float64)
    rc = lib.d2f_oracle_block_attn_part(
        _ptr(q), _ptr(k_win), _ptr(v_win), _ptr(k_pool), _ptr(v_pool), _ptr(page_table),
        page_table.shape[1] if page_table.dim() == 2 else 0, _ptr(ctx_len), _ptr(q_start),
        ctx_len.shape[0], total_q, hq, k_win.shape[1], d, block_size, k_pool.shape[0], dt,
        float(scale), int(part), _ptr(prev_out), _ptr(prev_lse), _ptr(out), _ptr(lse),
        nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle attention part rejected its input (code %d)" % rc)
    return out, lse


# confidence metrics of commit(): largest probability, negative entropy,
# top-1 - top-2 probability margin, top-1 - top-2 logit gap
CONF_PMAX, CONF_NEG_ENTROPY, CONF_MARGIN, CONF_LOGIT_GAP = 0, 1, 2, 3


def commit(logits, tokens, masked, q_start, block_phase, tau, block_size, mask_id,
           logit_row=None, row_stride=None, nthreads=None, metric=CONF_PMAX, early_gap=None):
    """Confidence commit + remask. Returns a dict of new CPU tensors:
    tokens (int32), masked (uint8), conf (float32), argmax (int32),
    block_remaining (int32), stopped (uint8 per sequence). Inputs are not
    modified. `metric` picks the confidence (tau in its units); early_gap (per
    sequence) turns on the early commit of whole sequences."""
    lib = _load()
    logits = _cpu(logits)
    dt = _dt(logits)
    if dt == DT_F64:
        raise TypeError("commit logits are bfloat16 or float32")
    tokens = _cpu(tokens, torch.int32).clone()
    masked = _cpu(masked, torch.uint8).clone()
    q_start = _cpu(q_start, torch.int32)
    block_phase = _cpu(block_phase, torch.uint8)
    tau = _cpu(tau, torch.float32)
    logit_row = _cpu(logit_row, torch.int32)
    total_q = tokens.shape[0]
    batch = q_start.shape[0] - 1
    vocab = logits.shape[-1]
    n_rows = logits.shape[0]
    if row_stride is None:
        row_stride = logits.stride(0)
    conf = torch.empty(total_q, dtype=torch.float32)
    amax = torch.empty(total_q, dtype=torch.int32)
    rem = torch.empty(max(total_q // block_size, 0), dtype=torch.int32)
    early_gap = _cpu(early_gap, torch.float32)
    stopped = torch.zeros(max(batch, 1), dtype=torch.uint8)
    if metric == CONF_PMAX and early_gap is None:
        rc = lib.d2f_oracle_commit(
            _ptr(logits), int(row_stride), dt, vocab, n_rows, _ptr(logit_row), _ptr(tokens),
            _ptr(masked), _ptr(q_start), _ptr(block_phase), _ptr(tau), batch, total_q,
            block_size, int(mask_id), _ptr(conf), _ptr(amax), _ptr(rem),
            nthreads or default_threads())
    else:
        rc = lib.d2f_oracle_commit_metric(
            _ptr(logits), int(row_stride), dt, vocab, n_rows, _ptr(logit_row), _ptr(tokens),
            _ptr(masked), _ptr(q_start), _ptr(block_phase), _ptr(tau), batch, total_q,
            block_size, int(mask_id), _ptr(conf), _ptr(amax), _ptr(rem), int(metric),
            _ptr(early_gap), _ptr(stopped), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle commit rejected its input (code %d)" % rc)
    return {"tokens": tokens, "masked": masked, "conf": conf, "argmax": amax,
            "block_remaining": rem, "stopped": stopped[:batch]}


def kv_append(k_win, v_win, src_row, dst_page, k_pool, v_pool, block_size):
    """Returns new (k_pool, v_pool) CPU tensors with the blocks appended."""
    lib = _load()
    k_win, v_win = _cpu(k_win), _cpu(v_win)
    k_pool, v_pool = _cpu(k_pool).clone(), _cpu(v_pool).clone()
    src_row = _cpu(src_row, torch.int32)
    dst_page = _cpu(dst_page, torch.int32)
    total_q, hkv, d = k_win.shape
    rc = lib.d2f_oracle_kv_append(
        _ptr(k_win), _ptr(v_win), _ptr(src_row), _ptr(dst_page), src_row.shape[0], total_q,
        _ptr(k_pool), _ptr(v_pool), hkv, d, block_size, k_pool.shape[0], k_win.element_size())
    if rc != 0:
        raise ValueError("oracle kv_append rejected its input (code %d)" % rc)
    return k_pool, v_pool


# keys of the window scheduler's state (see window_step)
WINDOW_STATE = ("q_start", "tokens", "masked", "ctx_len", "page_table", "next_block",
                "gen_blocks", "n_leaving", "stopped", "free_pages", "free_count")


def window_step(state, block_size, max_blocks, mask_id, tau_add, tau_act):
    """One call of the pipelined window scheduler on a copy of `state` (a dict of
    CPU tensors: q_start int32 [batch+1], tokens int32 [capacity], masked uint8
    [capacity], ctx_len / next_block / gen_blocks / n_leaving int32 [batch],
    page_table int32 [batch, max_pages], stopped uint8 [batch] or None,
    free_pages int32 [F], free_count int). Returns the new state plus
    block_phase uint8 [capacity / B], row_pos int32 [capacity], app_src /
    app_dst int32 [n_append], n_append and err (ints). Raises on bad sizes or an
    inconsistent state (the oracle writes nothing then)."""
    lib = _load()
    st = {}
    for k in ("q_start", "tokens", "ctx_len", "page_table", "next_block", "gen_blocks",
              "n_leaving", "free_pages"):
        st[k] = _cpu(state[k], torch.int32).clone().contiguous()
    st["masked"] = _cpu(state["masked"], torch.uint8).clone().contiguous()
    stopped = state.get("stopped")
    st["stopped"] = None if stopped is None else _cpu(stopped, torch.uint8).clone().contiguous()
    batch = st["q_start"].shape[0] - 1
    capacity = st["tokens"].shape[0]
    max_pages = st["page_table"].shape[1] if st["page_table"].dim() == 2 else 0
    free_count = torch.tensor([int(state["free_count"])], dtype=torch.int32)
    phase = torch.zeros(max(capacity // block_size, 1), dtype=torch.uint8)
    row_pos = torch.empty(max(capacity, 1), dtype=torch.int32)
    app_src = torch.empty(max(capacity // block_size, 1), dtype=torch.int32)
    app_dst = torch.empty_like(app_src)
    n_append = torch.zeros(1, dtype=torch.int32)
    err = torch.zeros(1, dtype=torch.int32)
    rc = lib.d2f_oracle_window_step(
        batch, block_size, max_blocks, capacity, max_pages, int(mask_id), float(tau_add),
        float(tau_act), _ptr(st["q_start"]), _ptr(st["tokens"]), _ptr(st["masked"]), _ptr(phase),
        _ptr(row_pos), _ptr(st["ctx_len"]), _ptr(st["page_table"]), _ptr(st["next_block"]),
        _ptr(st["gen_blocks"]), _ptr(st["n_leaving"]), _ptr(st["stopped"]),
        _ptr(st["free_pages"]), _ptr(free_count), _ptr(app_src), _ptr(app_dst), _ptr(n_append),
        _ptr(err))
    if rc != 0:
        raise ValueError("oracle window_step rejected its input (code %d)" % rc)
    n = int(n_append.item())
    st["free_count"] = int(free_count.item())
    st.update(block_phase=phase[:capacity // block_size], row_pos=row_pos[:capacity],
              app_src=app_src[:n].clone(), app_dst=app_dst[:n].clone(), n_append=n,
              err=int(err.item()))
    return st
