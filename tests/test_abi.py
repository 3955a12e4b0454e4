"""The C-ABI library loads and exports every declared entry point; host-side
validation (no GPU needed) returns the documented status codes."""
import ctypes
import os
import re

import pytest

from block_causal_kv_gb300 import d2f

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "d2f.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return d2f.load()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(d2f_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_hot_path():
    names = _declared()
    for n in ("d2f_block_attn", "d2f_commit", "d2f_kv_append"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)
    assert set(_declared()) <= set(d2f.EXPORTS)


def test_version_and_status_strings(lib):
    assert d2f.version() >= 100
    assert d2f.status_string(0) == "ok"
    assert "workspace" in d2f.status_string(6)


def _attn_ws(**over):
    kw = dict(batch=1, total_q=48, max_q_per_seq=48, max_ctx=1024, num_heads_q=32,
              num_heads_kv=32, head_dim=128, block_size=16, dtype=d2f.BF16, num_splits=4)
    kw.update(over)
    return d2f.attn_workspace_size(**kw)


def test_attention_workspace_size(lib, monkeypatch):
    # tensor-core path: splits compose in distributed shared memory, no workspace
    monkeypatch.setenv("D2F_ATTN_SK", "0")
    assert _attn_ws() == 0
    monkeypatch.delenv("D2F_ATTN_SK")
    # CUDA-core path: counters + 4 splits x (max, sum) + 4 splits x fp32 partial rows
    monkeypatch.setenv("D2F_ATTN_PATH", "simt")
    n4 = _attn_ws()
    assert n4 >= 4 * 48 * 32 * (128 * 4 + 8)
    assert _attn_ws(num_splits=1) < 4096
    assert _attn_ws(dtype=d2f.F32) == n4


@pytest.mark.parametrize("over,status", [
    (dict(num_heads_q=30, num_heads_kv=4), 1),
    (dict(head_dim=96), 2),
    (dict(dtype=7), 1),
    (dict(max_q_per_seq=49), 1),
    (dict(batch=-1), 1),
    (dict(num_splits=-2), 1),
])
def test_attention_rejects_bad_sizes(lib, over, status):
    with pytest.raises(d2f.D2FError) as e:
        _attn_ws(**over)
    assert e.value.status == status


def test_commit_workspace_and_rejections(lib):
    assert d2f.commit_workspace_size(48, 126464, 16, num_splits=8) > 48 * 8 * 16
    with pytest.raises(d2f.D2FError) as e:
        d2f.commit_workspace_size(47, 126464, 16)
    assert e.value.status == 1
    with pytest.raises(d2f.D2FError) as e:
        d2f.commit_workspace_size(64, 126464, 64)
    assert e.value.status == 2


def test_null_pointers_are_rejected_before_any_launch(lib):
    st = lib.d2f_kv_append(None, None, None, None, 1, 16, None, None, 4, 128, 16, 8, 0, None, None)
    assert st == 1
    assert b"NULL" in lib.d2f_last_error_string()
    st = lib.d2f_block_attn(None, None, None, None, None, None, 4, None, None, None, None,
                            1, 16, 16, 0, 4, 4, 64, 16, 4, 0, ctypes.c_float(0.125), 1, None, 0,
                            None, None)
    assert st == 1


def _window(lib, batch=2, B=16, W=3, cap=None, maxp=8, tau_add=0.5, tau_act=1.0, ptr=1):
    """d2f_window_step with every pointer set to `ptr` (never dereferenced: each call
    here must be refused on the host)."""
    cap = batch * W * B if cap is None else cap
    p = ctypes.c_void_p(ptr) if ptr else None
    return lib.d2f_window_step(batch, B, W, cap, maxp, 99, ctypes.c_float(tau_add),
                               ctypes.c_float(tau_act), *([p] * 18))


def test_window_step_host_checks(lib):
    assert _window(lib, cap=100) == 1                  # not a multiple of block_size
    assert _window(lib, cap=64) == 1                   # < batch * max_blocks * block_size
    assert _window(lib, B=256, cap=2 * 3 * 256) == 2   # block_size > 128
    assert _window(lib, batch=1, W=1, B=16, cap=64000) == 2   # past one CTA's shared memory
    assert _window(lib, tau_add=float("nan")) == 1
    assert _window(lib, W=0) == 1
    assert _window(lib, ptr=0) == 1                    # NULL state
    assert b"NULL" in lib.d2f_last_error_string()


def test_device_count_appends_need_the_count(lib):
    st = lib.d2f_kv_append_dev(None, None, None, None, None, 4, 16, None, None, 4, 128, 16, 8,
                               0, None, None)
    assert st == 1 and b"n_append_dev" in lib.d2f_last_error_string()
    st = lib.d2f_block_attn_append_dev(None, None, None, None, None, None, 4, None, None, None,
                                       None, 1, 16, 16, 0, 4, 4, 64, 16, 4, 0,
                                       ctypes.c_float(0.125), 1, None, 0, None, None, None, 4,
                                       None, None)
    assert st == 1 and b"n_append_dev" in lib.d2f_last_error_string()


def test_attention_flags_are_checked(lib):
    """d2f_block_attn_flags refuses unknown flag bits before any launch."""
    st = lib.d2f_block_attn_flags(None, None, None, None, None, None, 4, None, None, None, None,
                                  1, 16, 16, 0, 4, 4, 64, 16, 4, 0, ctypes.c_float(0.125), 1, None,
                                  0, 2, None, None)
    assert st == 1
    assert b"flags" in lib.d2f_last_error_string()
