"""GPU parity of the appends whose list length lives in device memory
(d2f_kv_append_dev, and the CUDA-core attention path of d2f_block_attn_append_dev,
which appends after the attention): exactly the first n entries are applied, n
read on the device and bounded by the list's capacity."""
import pytest
import torch

import oracle
from block_causal_kv_gb300 import d2f, synth
from gpu_common import check_attention, device

pytestmark = pytest.mark.gpu


def _problem(dtype):
    w = synth.Workload("dc", 2, 4, 4, 64, 16, dtype, [64, 32], [3, 2], 1000,
                       appends_per_seq=2, seed=17)
    return w, synth.make_problem(w)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("count", [0, 1, 3, 4, 9, -2])
def test_kv_append_reads_its_count_on_the_device(dtype, count):
    dev = device()
    w, p = _problem(dtype)
    g = p.to(dev)
    n_dev = torch.tensor([count], dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    d2f.kv_append(g.k_win, g.v_win, g.src_row, g.dst_page, g.k_pool, g.v_pool,
                  block_size=w.block_size, err=err, n_append_dev=n_dev)
    torch.cuda.synchronize()
    n = max(0, min(count, len(p.src_row)))
    kp, vp = oracle.kv_append(p.k_win, p.v_win, p.src_row[:n], p.dst_page[:n], p.k_pool,
                              p.v_pool, w.block_size)
    assert int(err.item()) == 0
    assert torch.equal(g.k_pool.cpu(), kp) and torch.equal(g.v_pool.cpu(), vp)


@pytest.mark.parametrize("count", [0, 2, 4])
def test_float32_attention_appends_after_with_a_device_count(count):
    """float32 takes the CUDA-core attention, which appends after itself."""
    dev = device()
    w, p = _problem(torch.float32)
    g = p.to(dev)
    n_dev = torch.tensor([count], dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out, lse = d2f.block_attn(g.q, g.k_win, g.v_win, g.k_pool, g.v_pool, g.page_table,
                              g.ctx_len, g.q_start, block_size=w.block_size,
                              max_q_per_seq=p.max_q_per_seq, max_ctx=p.max_ctx, err=err,
                              append_src_row=g.src_row, append_dst_page=g.dst_page,
                              append_n_dev=n_dev)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref, ref_lse = oracle.block_attn(p.q, p.k_win, p.v_win, p.k_pool, p.v_pool, p.page_table,
                                     p.ctx_len, p.q_start, w.block_size)
    check_attention(out, lse, ref, ref_lse, torch.float32, "f32 append count %d" % count)
    kp, vp = oracle.kv_append(p.k_win, p.v_win, p.src_row[:count], p.dst_page[:count],
                              p.k_pool, p.v_pool, w.block_size)
    assert torch.equal(g.k_pool.cpu(), kp) and torch.equal(g.v_pool.cpu(), vp)
