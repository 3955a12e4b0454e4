"""The seeded synthetic inputs have the shapes, sizes and value distributions of the
workloads the pages' configurations describe (CPU only).

Tiny: batch 1, 4 MHA heads, head_dim 64, float32, a 32-token prompt plus two
committed blocks in the cache, a window of two 16-token blocks (the first
aggressive, the second conservative), float32 logits N(0, 2) over 1000 tokens with
30% of the positions committed. LLaDA-8B layer: 32 MHA heads, head_dim 128, bf16,
1024 cached tokens, a 3-block window, bf16 logits N(0, 3) over 126464 tokens with
one planted peak per position, 2 to 12 above the row's maximum. Ragged: 16
sequences, contexts uniform in [256, 4096] in steps of 16, windows of 1 to 3
blocks, permuted pages, half the positions masked, tau from {0.7, 0.9, 0.95}.
Dream-7B layer: 28 / 4 GQA heads, batch 8, 8192 cached tokens, a 3-block window,
one appended block per sequence, vocab 152064. Long context: batch 4, 32 MHA heads,
32768 cached tokens, a 4-block window, B in {8, 16, 32}.
"""
import pytest
import torch

from block_causal_kv_gb300 import synth


def test_tiny():
    w = synth.workload("tiny")
    assert (w.batch, w.num_heads_q, w.num_heads_kv, w.head_dim, w.block_size) == (1, 4, 4, 64, 16)
    assert w.dtype == torch.float32 and w.ctx_lens == [32 + 2 * 16] and w.window_blocks == [2]
    assert w.vocab == 1000
    p = synth.make_problem(w)
    assert p.block_phase.tolist() == [1, 0]
    assert float(p.tau[0]) == pytest.approx(0.9)
    committed = 1.0 - float(p.masked.float().mean())
    assert abs(committed - 0.3) < 0.05
    assert abs(float(p.logits.float().std()) - 2.0) < 0.05
    assert abs(float(p.q.float().std()) - 1.0) < 0.05


def test_llada():
    w = synth.workload("llada")
    assert (w.batch, w.num_heads_q, w.num_heads_kv, w.head_dim, w.block_size) == (1, 32, 32, 128, 16)
    assert w.dtype == torch.bfloat16 and w.ctx_lens == [1024] and w.window_blocks == [3]
    assert w.vocab == 126464
    p = synth.make_problem(w)
    assert p.logits.shape == (48, 126464) and p.logits.dtype == torch.bfloat16
    assert bool(p.masked.all()) and float(p.tau[0]) == pytest.approx(0.9)
    z = p.logits.float()
    top2 = z.topk(2, dim=1).values
    gap = top2[:, 0] - top2[:, 1]
    # the planted peak stands 2..12 above the rest (bf16 rounding of values near 15-25
    # moves each side by at most 0.0625)
    assert float(gap.min()) > 2.0 - 0.13 and float(gap.max()) < 12.0 + 0.13
    body = z.clone()
    body[torch.arange(48), z.argmax(1)] = 0.0
    assert abs(float(body.std()) - 3.0) < 0.05
    assert p.page_table.shape == (1, 64)


def test_ragged_descriptor():
    w = synth.workload("ragged")
    assert w.batch == 16 and (w.num_heads_q, w.num_heads_kv, w.head_dim) == (32, 32, 128)
    assert all(256 <= c <= 4096 and c % 16 == 0 for c in w.ctx_lens)
    assert len(set(w.ctx_lens)) > 4
    assert all(1 <= n <= 3 for n in w.window_blocks) and len(set(w.window_blocks)) > 1
    assert w.permute_pages and w.masked_frac == 0.5 and tuple(w.taus) == (0.7, 0.9, 0.95)
    assert w.vocab == 126464


def test_dream_descriptor():
    w = synth.workload("dream")
    assert (w.batch, w.num_heads_q, w.num_heads_kv, w.head_dim, w.block_size) == (8, 28, 4, 128, 16)
    assert w.ctx_lens == [8192] * 8 and w.window_blocks == [3] * 8
    assert w.appends_per_seq == 1 and w.vocab == 152064 and w.dtype == torch.bfloat16


@pytest.mark.parametrize("B", [8, 16, 32])
def test_long_descriptor(B):
    w = synth.workload("long_b%d" % B)
    assert (w.batch, w.num_heads_q, w.num_heads_kv, w.head_dim, w.block_size) == (4, 32, 32, 128, B)
    assert w.ctx_lens == [32768] * 4 and w.window_blocks == [4] * 4 and w.vocab == 126464


def test_inputs_are_seeded():
    a = synth.make_problem(synth.workload("tiny"))
    b = synth.make_problem(synth.workload("tiny"))
    for f in ("q", "k_win", "k_pool", "logits", "masked", "tokens"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f
    c = synth.make_problem(synth.workload("tiny", seed=99))
    assert not torch.equal(a.q, c.q)
