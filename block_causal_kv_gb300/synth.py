"""Seeded synthetic inputs for the D2F decoding hot path.

This module only draws random numbers and lays out metadata (window rows, page
tables, masked/committed state, phases, thresholds). It holds none of the
method's arithmetic, and it is the one module that both the CUDA path's tests
and the CPU oracle's tests take their inputs from.

Shapes and distributions follow the five workloads of the hot path:
  tiny         batch 1, 4 MHA heads, D=64, float32, context 64, window 2x16
  llada        LLaDA-8B-shaped layer: batch 1, 32 MHA heads, D=128, bf16,
               context 1024 (16-token pages), window 3 blocks, vocab 126464
  ragged       16 sequences of the LLaDA shape, ragged context / window,
               permuted page table, 50% masked, tau in {0.7, 0.9, 0.95}
  dream        Dream-7B-shaped layer: GQA 28/4, D=128, bf16, batch 8,
               context 8192, window 3x16, one append per sequence, vocab 152064
  long_b{8,16,32}  batch 4, LLaDA shape, context 32768, window 4 blocks of B
No dataset is involved; these shapes stand in for the pages' GSM8K/HumanEval
decoding runs.
"""
from dataclasses import dataclass, field, replace
from typing import List, Optional, Sequence

import torch

PHASE_CONSERVATIVE = 0
PHASE_AGGRESSIVE = 1


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    block_size: int
    dtype: torch.dtype
    ctx_lens: Sequence[int]          # cached tokens per sequence (prompt + committed blocks)
    window_blocks: Sequence[int]     # active window blocks per sequence
    vocab: int
    logit_sigma: float = 3.0
    planted_peak: bool = True        # one peak per row, max + U(2,12)
    masked_frac: Optional[float] = None   # Bernoulli masked fraction; None = all masked
    committed_count: Optional[int] = None  # exact number of committed positions (Tiny)
    taus: Sequence[float] = (0.9,)   # per-sequence tau drawn uniformly from this set
    permute_pages: bool = True
    appends_per_seq: int = 0
    extra_pages: int = 0             # unused pool pages (page-table indirection check)
    logit_row_pad: int = 0           # logits row stride = vocab + pad
    seed: int = 1234

    @property
    def total_q(self) -> int:
        return sum(w * self.block_size for w in self.window_blocks)


def _uniform_ctx(gen, batch, lo, hi, step):
    n = (hi - lo) // step + 1
    idx = torch.randint(0, n, (batch,), generator=gen)
    return [lo + int(i) * step for i in idx]


def workload(name: str, seed: Optional[int] = None) -> Workload:
    """The named full-size workload."""
    if name == "tiny":
        w = Workload("tiny", 1, 4, 4, 64, 16, torch.float32, [64], [2], 1000,
                     logit_sigma=2.0, planted_peak=False, committed_count=10,
                     seed=1234)
    elif name == "llada":
        w = Workload("llada", 1, 32, 32, 128, 16, torch.bfloat16, [1024], [3], 126464,
                     permute_pages=False, seed=1235)
    elif name == "ragged":
        g = torch.Generator().manual_seed(1236 if seed is None else seed)
        ctx = _uniform_ctx(g, 16, 256, 4096, 16)
        win = [int(x) for x in torch.randint(1, 4, (16,), generator=g)]
        w = Workload("ragged", 16, 32, 32, 128, 16, torch.bfloat16, ctx, win, 126464,
                     masked_frac=0.5, taus=(0.7, 0.9, 0.95), permute_pages=True, seed=1236)
    elif name == "dream":
        w = Workload("dream", 8, 28, 4, 128, 16, torch.bfloat16, [8192] * 8, [3] * 8, 152064,
                     appends_per_seq=1, permute_pages=False, seed=1237)
    elif name == "long_b32_ctx8k":
        # the long-context layout at a quarter of the context: a case small enough
        # for multi-pass profiler captures of the same kernels (0.5 GB of K/V)
        w = Workload(name, 4, 32, 32, 128, 32, torch.bfloat16, [8192] * 4, [4] * 4, 126464,
                     permute_pages=False, seed=1239)
    elif name.startswith("long_b"):
        B = int(name[len("long_b"):])
        if B not in (8, 16, 32):
            raise ValueError(name)
        w = Workload(name, 4, 32, 32, 128, B, torch.bfloat16, [32768] * 4, [4] * 4, 126464,
                     permute_pages=False, seed=1238)
    else:
        raise KeyError(name)
    if seed is not None:
        w = replace(w, seed=seed)
    return w


WORKLOADS = ("tiny", "llada", "ragged", "dream", "long_b8", "long_b16", "long_b32")


@dataclass
class Problem:
    w: Workload
    q: torch.Tensor
    k_win: torch.Tensor
    v_win: torch.Tensor
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    page_table: torch.Tensor      # int32 [batch, max_pages_per_seq], -1 where unused
    ctx_len: torch.Tensor         # int32 [batch]
    q_start: torch.Tensor         # int32 [batch+1]
    logits: torch.Tensor          # [total_q, vocab] view of a [total_q, vocab+pad] buffer
    tokens: torch.Tensor          # int32 [total_q]
    masked: torch.Tensor          # uint8 [total_q]
    block_phase: torch.Tensor     # uint8 [total_q / B]
    tau: torch.Tensor             # float32 [batch]
    src_row: torch.Tensor         # int32 [n_append]
    dst_page: torch.Tensor        # int32 [n_append]
    mask_id: int
    max_q_per_seq: int
    max_ctx: int
    fields: List[str] = field(default_factory=list)

    @property
    def num_pages(self) -> int:
        return self.k_pool.shape[0]

    def to(self, device) -> "Problem":
        kw = {}
        for name in self.fields:
            t = getattr(self, name)
            if name == "logits":
                base = t.as_strided((t.shape[0], t.stride(0)), (t.stride(0), 1)).to(device)
                kw[name] = base[:, : t.shape[1]]
            else:
                kw[name] = t.to(device)
        return replace(self, **kw)


def _randn(shape, gen, dtype, device, chunk_rows=None):
    """Standard normal draws (float32) cast to dtype, generated in chunks along dim 0."""
    out = torch.empty(shape, dtype=dtype, device=device)
    n0 = shape[0]
    per_row = 1
    for s in shape[1:]:
        per_row *= s
    if chunk_rows is None:
        chunk_rows = max(1, (1 << 24) // max(per_row, 1))
    for r0 in range(0, n0, chunk_rows):
        r1 = min(n0, r0 + chunk_rows)
        out[r0:r1] = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=gen,
                                 dtype=torch.float32, device=device).to(dtype)
    return out


def make_problem(w: Workload, device="cpu") -> Problem:
    """Draw one seeded problem for workload w on `device` (CPU by default).

    The same workload and device always give the same tensors.
    """
    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(w.seed)
    cpu_gen = torch.Generator().manual_seed(w.seed + 7919)
    B = w.block_size
    batch = w.batch
    assert len(w.ctx_lens) == batch and len(w.window_blocks) == batch
    nq = [wb * B for wb in w.window_blocks]
    q_start = [0]
    for n in nq:
        q_start.append(q_start[-1] + n)
    total_q = q_start[-1]

    # Page pool: every sequence's cached pages, its append targets, and spares.
    used = [(c + B - 1) // B for c in w.ctx_lens]
    per_seq = [u + w.appends_per_seq for u in used]
    num_pages = sum(per_seq) + w.extra_pages
    if w.permute_pages:
        phys = torch.randperm(num_pages, generator=cpu_gen).tolist()
    else:
        phys = list(range(num_pages))
    max_pages = max(per_seq) if per_seq else 1
    page_table = torch.full((batch, max(max_pages, 1)), -1, dtype=torch.int32)
    src_row, dst_page = [], []
    cur = 0
    for b in range(batch):
        for p in range(per_seq[b]):
            page_table[b, p] = phys[cur]
            cur += 1
        for a in range(w.appends_per_seq):
            src_row.append(q_start[b] + a * B)
            dst_page.append(int(page_table[b, used[b] + a]))

    H, Hk, D = w.num_heads_q, w.num_heads_kv, w.head_dim
    q = _randn((total_q, H, D), gen, w.dtype, dev)
    k_win = _randn((total_q, Hk, D), gen, w.dtype, dev)
    v_win = _randn((total_q, Hk, D), gen, w.dtype, dev)
    k_pool = _randn((num_pages, Hk, B, D), gen, w.dtype, dev)
    v_pool = _randn((num_pages, Hk, B, D), gen, w.dtype, dev)

    # Logits: N(0, sigma) drawn in float32, optional planted peak, cast once.
    V = w.vocab
    stride = V + w.logit_row_pad
    buf = torch.empty((total_q, stride), dtype=w.dtype, device=dev)
    rows_per_chunk = max(1, (1 << 24) // stride)
    for r0 in range(0, total_q, rows_per_chunk):
        r1 = min(total_q, r0 + rows_per_chunk)
        z = torch.randn((r1 - r0, V), generator=gen, dtype=torch.float32, device=dev) * w.logit_sigma
        if w.planted_peak:
            peak = torch.randint(0, V, (r1 - r0,), generator=gen, device=dev)
            delta = torch.rand((r1 - r0,), generator=gen, device=dev) * 10.0 + 2.0
            top = z.max(dim=1).values
            z[torch.arange(r1 - r0, device=dev), peak] = top + delta
        buf[r0:r1, :V] = z.to(w.dtype)
        if w.logit_row_pad:
            buf[r0:r1, V:] = float("nan")  # padding must never be read
    logits = buf[:, :V]

    # Masked / committed state.
    mask_id = V
    if w.committed_count is not None:
        masked = torch.ones(total_q, dtype=torch.uint8)
        perm = torch.randperm(total_q, generator=cpu_gen)[: w.committed_count]
        masked[perm] = 0
    elif w.masked_frac is not None:
        masked = (torch.rand(total_q, generator=cpu_gen) < w.masked_frac).to(torch.uint8)
    else:
        masked = torch.ones(total_q, dtype=torch.uint8)
    tokens = torch.randint(0, V, (total_q,), generator=cpu_gen, dtype=torch.int32)
    tokens[masked.bool()] = mask_id

    # Phases: the oldest window block of each sequence is aggressive, the rest
    # conservative; thresholds drawn per sequence from the workload's set.
    block_phase = torch.zeros(total_q // B, dtype=torch.uint8)
    for b in range(batch):
        block_phase[q_start[b] // B] = PHASE_AGGRESSIVE
    tau_idx = torch.randint(0, len(w.taus), (batch,), generator=cpu_gen)
    tau = torch.tensor([w.taus[int(i)] for i in tau_idx], dtype=torch.float32)

    fields = ["q", "k_win", "v_win", "k_pool", "v_pool", "page_table", "ctx_len", "q_start",
              "logits", "tokens", "masked", "block_phase", "tau", "src_row", "dst_page"]
    prob = Problem(
        w=w, q=q, k_win=k_win, v_win=v_win, k_pool=k_pool, v_pool=v_pool,
        page_table=page_table.to(dev), ctx_len=torch.tensor(w.ctx_lens, dtype=torch.int32).to(dev),
        q_start=torch.tensor(q_start, dtype=torch.int32).to(dev), logits=logits,
        tokens=tokens.to(dev), masked=masked.to(dev), block_phase=block_phase.to(dev),
        tau=tau.to(dev), src_row=torch.tensor(src_row, dtype=torch.int32).to(dev),
        dst_page=torch.tensor(dst_page, dtype=torch.int32).to(dev), mask_id=mask_id,
        max_q_per_seq=max(nq) if nq else 0, max_ctx=max(w.ctx_lens) if batch else 0,
        fields=fields)
    return prob


def small(name: str, **over) -> Workload:
    """A reduced-size variant of a workload (same structure, oracle finishes in seconds)."""
    base = workload(name)
    defaults = {
        "tiny": {},
        "llada": dict(num_heads_q=4, num_heads_kv=4, ctx_lens=[256], vocab=5003),
        "ragged": dict(batch=5, num_heads_q=4, num_heads_kv=4, ctx_lens=[16, 200, 0, 96, 333],
                       window_blocks=[1, 3, 2, 1, 2], vocab=3001),
        "dream": dict(batch=2, num_heads_q=14, num_heads_kv=2, ctx_lens=[512, 300],
                      window_blocks=[3, 3], vocab=4099, appends_per_seq=1),
        "long_b8": dict(batch=2, num_heads_q=2, num_heads_kv=2, ctx_lens=[1000, 1024],
                         window_blocks=[4, 4], vocab=2048),
        "long_b16": dict(batch=2, num_heads_q=2, num_heads_kv=2, ctx_lens=[1000, 1024],
                         window_blocks=[4, 4], vocab=2048),
        "long_b32": dict(batch=2, num_heads_q=2, num_heads_kv=2, ctx_lens=[1000, 1024],
                         window_blocks=[4, 4], vocab=2048),
    }[name]
    defaults.update(over)
    return replace(base, name=name + "_small", **defaults)
