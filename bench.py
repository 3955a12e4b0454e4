#!/usr/bin/env python
"""Benchmark of the D2F decoding hot path: block-attn + commit steps/s.

One step = d2f_block_attn (one layer, the whole active window) + d2f_commit
(every still-masked window position), + d2f_kv_append where the workload
appends, preceded by a 2-copy reset of the decode state (tokens, masked) so that
every step does the same work.

By default every workload is measured, each on its own: tiny, llada, ragged,
dream, long_b8, long_b16, long_b32. The line's headline fields (value, roofline,
kernels, e2e, cpu_baseline) are those of long_b32, the largest configuration
that fits one GPU (batch 4, 32 MHA heads, head_dim 128, context 32768, window 4
blocks of 32, vocabulary 126464), timed over exactly --steps steps; per_config
holds the same fields for every workload (the others timed over at least a few
hundred milliseconds of steps).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload all|llada|...]
    python bench.py --impl reference ...   # the CPU oracle, timed the same way

Timing: inputs resident in HBM; the step cycles through enough independent
input sets (> 4x L2) that no step finds its inputs in L2; K steps replayed from
CUDA graphs between CUDA events, barrier + synchronize on both sides, max over
ranks. Per-kernel durations come from graphs of each kernel over the same input
sets. Prints one JSON line (rank 0).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "block-attn + commit steps/sec and achieved HBM GB/s (% of GB300 roofline)"
PROFILES = os.path.join(ROOT, "profiles")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="all",
                    help="one workload, or all (default): the headline on %s and per_config "
                         "results for every workload" % "long_b32")
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--commit-splits", type=int, default=0)
    ap.add_argument("--conf-metric", default="pmax", choices=list(CONF_METRICS),
                    help="confidence of the commit: largest probability (d2f_commit), negative "
                         "entropy, probability margin or logit gap (d2f_commit_metric)")
    ap.add_argument("--fused-append", action="store_true",
                    help="append finished blocks inside the attention (d2f_block_attn_append) "
                         "instead of d2f_kv_append after it")
    ap.add_argument("--early-gap", type=float, default=None,
                    help="early commit of whole sequences at this logit-gap threshold "
                         "(d2f_commit_metric; every sequence)")
    ap.add_argument("--reuse-cached", action="store_true",
                    help="steps inside a block's denoising: the window part of the attention "
                         "composed with a kept cached part (d2f_block_attn_part); the cached "
                         "part is computed once per input set, before the timed region, and "
                         "timed on its own")
    ap.add_argument("--scheduler", action="store_true",
                    help="the step of a device-driven decode: attention (appending the listed "
                         "blocks, d2f_block_attn_append_dev), commit and the window scheduler "
                         "(d2f_window_step), the scheduler's state reset per step")
    ap.add_argument("--tau-add", type=float, default=0.5,
                    help="window scheduler: progress of the last block that lets a block enter")
    ap.add_argument("--tau-act", type=float, default=1.0,
                    help="window scheduler: progress of the block before that makes a block "
                         "aggressive")
    ap.add_argument("--cache-ready", type=int, default=1, choices=[0, 1],
                    help="pass D2F_ATTN_CACHE_READY with the plain step's attention (the cache "
                         "is written by no kernel of the step)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=4.0,
                    help="time budget of the oracle on all host cores, per workload")
    ap.add_argument("--cpu-seconds-1t", type=float, default=3.0,
                    help="time budget of the oracle on one host thread, per workload")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="oracle time budget of the reference arm")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="run this many eager steps and exit (for ncu captures)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU, replicas: no data-path collective)
# ---------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# workload accounting
# ---------------------------------------------------------------------------
def algorithmic_bytes(p, part="all"):
    """Bytes a step must move at minimum: cached K+V once per (sequence, KV
    head), window K/V, Q, O, page ids; logits of masked rows; appended blocks.
    part "window" (composed with a kept cached part): window K/V, Q, O and the
    kept part's output and normaliser, no cached page; part "cached": cached K+V,
    page ids, Q, and its output and normaliser."""
    w = p.w
    elt = 2 if w.dtype == torch.bfloat16 else 4
    Hk, H, D = w.num_heads_kv, w.num_heads_q, w.head_dim
    ctx = sum(w.ctx_lens)
    tq = w.total_q
    pages = sum((c + w.block_size - 1) // w.block_size for c in w.ctx_lens)
    if part == "window":
        attn = 2 * tq * Hk * D * elt + 3 * tq * H * D * elt + tq * H * 4
    elif part == "cached":
        attn = 2 * ctx * Hk * D * elt + pages * 4 * Hk + 2 * tq * H * D * elt + tq * H * 4
    else:
        attn = 2 * ctx * Hk * D * elt + 2 * tq * Hk * D * elt + 2 * tq * H * D * elt + pages * 4 * Hk
    masked_rows = int(p.masked.sum())
    commit = masked_rows * w.vocab * elt + tq * 6
    append = 2 * 2 * len(p.src_row) * w.block_size * Hk * D * elt
    return attn, commit, append


def flops(p, reuse=False):
    w = p.w
    f = 0
    for c, nb in zip(w.ctx_lens, w.window_blocks):
        n = nb * w.block_size
        c = 0 if reuse else c
        keys = sum(c + (i // w.block_size + 1) * w.block_size for i in range(n))
        f += 4 * w.num_heads_q * w.head_dim * keys
    return f


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def sustained_tflops():
    """Dense bf16 TF/s sustained over seconds (the step loop is seconds long), else
    the fallback's sustained figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1700.0, "fallback"


def attn_roofline(bytes_, flops_, hbm_gbs, tflops, us, tensor=True):
    """The attention's two roofline terms (µs): its bytes at the HBM peak and its
    flops at the dense bf16 peak (none on the CUDA-core path); the larger one
    bounds it, and frac_of_roofline is that bound over the measured time."""
    t_hbm = bytes_ / hbm_gbs / 1e3
    t_tensor = flops_ / tflops / 1e6 if tensor else None
    bound = "tensor" if (t_tensor or 0.0) > t_hbm else "hbm"
    t_roof = max(t_hbm, t_tensor or 0.0)
    return {"hbm_us": t_hbm, "tensor_us": t_tensor, "bound": bound,
            "frac_of_roofline": t_roof / us if us else None}


def source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "attn": ["block_causal_kv_gb300/csrc/attn_tc.cu", "block_causal_kv_gb300/csrc/attn_common.cuh",
             "block_causal_kv_gb300/csrc/d2f_internal.cuh"],
    "attn_window": ["block_causal_kv_gb300/csrc/attn_tc.cu",
                    "block_causal_kv_gb300/csrc/attn_common.cuh",
                    "block_causal_kv_gb300/csrc/d2f_internal.cuh"],
    "commit": ["block_causal_kv_gb300/csrc/commit.cu", "block_causal_kv_gb300/csrc/d2f_internal.cuh"],
}


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu capture, if the kernel source is
    unchanged since the counters were taken; else None."""
    path = os.path.join(PROFILES, "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel + ":" + workload]
    except Exception:
        return None
    if rec.get("source_sha") != source_sha(KERNEL_SOURCES[kernel]):
        return None
    return rec.get("bytes_per_launch")


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
CLOCK_FIELDS = ("timestamp,index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,"
                "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
                "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                "clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, out_path=None):
        self.proc = None
        self.out_path = out_path or os.path.join("/tmp", "d2f_clocks_%d.csv" % os.getpid())

    def start(self):
        try:
            self.fh = open(self.out_path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + CLOCK_FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, bus_id=None):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.out_path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 11:
                    continue
                if bus_id is not None:
                    try:  # "DDDDDDDD:BB:DD.F" -> bus number
                        if int(parts[2].split(":")[1], 16) != int(bus_id):
                            continue
                    except (ValueError, IndexError):
                        pass
                try:
                    rows.append(dict(sm=float(parts[3]), smax=float(parts[4]),
                                     power=float(parts[5]) if parts[5] not in ("[N/A]", "") else None,
                                     hw=parts[7], hwt=parts[8], swt=parts[9], swp=parts[10]))
                except ValueError:
                    continue
        if not rows:
            return None
        busy = [r for r in rows if r["power"] is None or r["power"] > 0] or rows
        reasons = set()
        for r in busy:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                            ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[k].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["smax"] for r in busy), "reasons": sorted(reasons),
                "samples": len(busy)}


# ---------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------
def time_oracle(p, seconds, nthreads, metric=0, reuse=False, sched=None):
    """Time the CPU oracle on a bounded sample of one step and extrapolate to
    full steps: attention over a subset of KV heads (its cost is linear in heads)
    and the commit over a subset of rows (linear in rows), with the commit's
    confidence `metric`. reuse: the attention is the window part composed with a
    cached part that is computed once per sample size, untimed. sched (tau_add,
    tau_act): each step also runs the oracle's window scheduler over the whole
    batch, from the state the device-driven step starts from."""
    import oracle
    w = p.w
    Hk, G = w.num_heads_kv, w.num_heads_q // w.num_heads_kv
    kept = {}

    # calibrate with one KV head and one block of rows
    def attn_sample(nh):
        hk = list(range(nh))
        hq = [h for g in hk for h in range(g * G, (g + 1) * G)]
        args = (p.q[:, hq], p.k_win[:, hk], p.v_win[:, hk], p.k_pool[:, hk], p.v_pool[:, hk],
                p.page_table, p.ctx_len, p.q_start, w.block_size)
        if reuse and nh not in kept:
            kept[nh] = oracle.block_attn_part(*args, oracle.ATTN_CACHED, nthreads=nthreads)
        t0 = time.perf_counter()
        if reuse:
            oracle.block_attn_part(*args, oracle.ATTN_WINDOW, prev_out=kept[nh][0],
                                   prev_lse=kept[nh][1], nthreads=nthreads)
        else:
            oracle.block_attn(*args, nthreads=nthreads, want_lse=False)
        return time.perf_counter() - t0

    def commit_sample(nb):
        B = w.block_size
        rows = nb * B
        qs = torch.tensor([0, rows], dtype=torch.int32)
        t0 = time.perf_counter()
        oracle.commit(p.logits[:rows], p.tokens[:rows], p.masked[:rows], qs,
                      p.block_phase[:nb], p.tau[:1], B, p.mask_id, nthreads=nthreads,
                      metric=metric)
        return time.perf_counter() - t0

    t_window = 0.0
    if sched is not None:
        W = max(w.window_blocks)
        state = sched_state_dict(p, W)
        t0 = time.perf_counter()
        n_win = 0
        while n_win < 3 or time.perf_counter() - t0 < 0.05:
            oracle.window_step(state, w.block_size, W, p.mask_id, sched[0], sched[1])
            n_win += 1
        t_window = (time.perf_counter() - t0) / n_win

    ta1 = attn_sample(1)
    tc1 = commit_sample(1)
    n_blocks = w.total_q // w.block_size
    # grow the sample so that the whole measurement takes about `seconds`
    est_step = ta1 * Hk + tc1 * n_blocks
    nh = max(1, min(Hk, int(Hk * min(1.0, seconds / 2 / max(est_step, 1e-9)))))
    nb = max(1, min(n_blocks, int(n_blocks * min(1.0, seconds / 2 / max(est_step, 1e-9)))))
    reps = 0
    ta = tc = 0.0
    t_start = time.perf_counter()
    while True:
        ta += attn_sample(nh)
        tc += commit_sample(nb)
        reps += 1
        if time.perf_counter() - t_start >= seconds:
            break
    step_s = (ta / reps) * Hk / nh + (tc / reps) * n_blocks / nb + t_window
    sample = ("%d x [%s for %d of %d KV heads + commit for %d of %d window blocks], "
              "extrapolated linearly to full steps" % (
                  reps, "window-part attention with a kept cached part" if reuse else "attention",
                  nh, Hk, nb, n_blocks))
    if sched is not None:
        sample += " + the window scheduler over the whole batch (%.1f us)" % (t_window * 1e6)
    return 1.0 / step_s, sample


def oracle_threads():
    return max(1, len(os.sched_getaffinity(0)))


def run_reference(args, world, rank):
    if rank != 0:
        return
    from block_causal_kv_gb300 import synth
    import oracle
    oracle._load()
    w = synth.workload(HEADLINE if args.workload == "all" else args.workload)
    p = synth.make_problem(w)
    nthreads = oracle_threads()
    # bounded: the whole run takes about --ref-seconds regardless of K
    budget = args.ref_seconds
    sched = (args.tau_add, args.tau_act) if args.scheduler else None
    for _ in range(max(0, min(args.warmup, 1))):
        time_oracle(p, 0.1, nthreads, CONF_METRICS[args.conf_metric], args.reuse_cached, sched)
    value, sample = time_oracle(p, budget, nthreads, CONF_METRICS[args.conf_metric],
                                args.reuse_cached, sched)
    ms = 1000.0 / value
    cfg = workload_config(p, args)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": value, "unit": "steps/s", "cores": nthreads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# confidence metric -> D2F_CONF_* value
CONF_METRICS = {"pmax": 0, "negent": 1, "margin": 2, "gap": 3}


def workload_config(p, args):
    w = p.w
    extra = {} if args.conf_metric == "pmax" else {
        "confidence": "%s (d2f_commit_metric; tau as drawn for the workload)" % args.conf_metric}
    if args.early_gap is not None:
        extra["early_commit_gap"] = args.early_gap
    if args.fused_append and w.appends_per_seq:
        extra["append"] = "fused into the attention (d2f_block_attn_append)"
    if args.scheduler:
        extra["scheduler"] = ("d2f_window_step after the commit (tau_add %g, tau_act %g); the "
                              "append of listed blocks inside the attention "
                              "(d2f_block_attn_append_dev); the scheduler's state starts every "
                              "step from the same device snapshot" % (args.tau_add, args.tau_act))
    if args.reuse_cached:
        extra["attention"] = ("window part composed with a kept cached part (d2f_block_attn_part): "
                              "a step inside a block's denoising, no append; the cached part of "
                              "each input set is computed before the timed region and timed on "
                              "its own in kernels.cached_part")
    return {**extra,"workload": "%s: batch %d, Hq %d / Hkv %d, head_dim %d, block %d, context %s, "
                        "window %s blocks, vocab %d" % (
                            w.name, w.batch, w.num_heads_q, w.num_heads_kv, w.head_dim,
                            w.block_size, "/".join(str(c) for c in sorted(set(w.ctx_lens))),
                            "/".join(str(x) for x in sorted(set(w.window_blocks))), w.vocab),
            "batch": w.batch, "window_queries": w.total_q, "context": max(w.ctx_lens),
            "parallelism": "replica per GPU (no collective)"}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class StepSet:
    """Device buffers of one independent input set (its decode state is a row of a
    buffer shared by all sets, so one copy resets every set's state)."""

    def __init__(self, p, dev, clone_from=None):
        src = clone_from
        for name in ("q", "k_win", "v_win", "k_pool", "v_pool", "page_table", "ctx_len", "q_start",
                     "block_phase", "tau", "src_row", "dst_page"):
            if src is None:
                setattr(self, name, getattr(p, name).to(dev))
            else:
                setattr(self, name, getattr(src, name).clone())
        if src is None:
            self.logits = p.logits.contiguous().to(dev)
        else:
            self.logits = src.logits.clone()
        self.out = torch.empty_like(self.q)

    def nbytes(self):
        return sum(t.numel() * t.element_size() for t in
                   (self.q, self.k_win, self.v_win, self.k_pool, self.v_pool, self.logits, self.out))


def sched_snapshot(p, dev, W):
    """The window scheduler's state at the start of a step of problem `p`: its
    layout, its phases, its cache bookkeeping and the appends listed for the step.
    Returns (int32 row, uint8 row, {field: (offset, shape)}, constants)."""
    w = p.w
    B, batch, cap = w.block_size, w.batch, w.total_q
    maxp = p.page_table.shape[1] + W + 1
    pt = torch.full((batch, maxp), -1, dtype=torch.int32)
    pt[:, :p.page_table.shape[1]] = p.page_table.cpu()
    src, dst = p.src_row.cpu(), p.dst_page.cpu()
    qs = p.q_start.cpu()
    leaving = torch.zeros(batch, dtype=torch.int32)
    for r in src.tolist():
        leaving[int(torch.searchsorted(qs, torch.tensor(r), right=True)) - 1] += 1
    app_src = torch.zeros(cap // B, dtype=torch.int32)
    app_dst = torch.zeros(cap // B, dtype=torch.int32)
    app_src[:len(src)], app_dst[:len(dst)] = src, dst
    parts = [("q_start", qs.to(torch.int32)), ("ctx_len", p.ctx_len.cpu().to(torch.int32)),
             ("page_table", pt),
             ("next_block", torch.tensor(w.window_blocks, dtype=torch.int32)),
             ("n_leaving", leaving), ("free_count", torch.tensor([p.k_pool.shape[0]],
                                                                 dtype=torch.int32)),
             ("app_src", app_src), ("app_dst", app_dst),
             ("n_append", torch.tensor([len(src)], dtype=torch.int32)),
             ("row_pos", torch.full((cap,), -1, dtype=torch.int32))]
    fields, off, rows = {}, 0, []
    for name, t in parts:
        fields[name] = (off, tuple(t.shape))
        off += t.numel()
        rows.append(t.reshape(-1))
    const = {"gen_blocks": torch.tensor([wb + 10 ** 6 for wb in w.window_blocks],
                                        dtype=torch.int32, device=dev),
             "free_pages": torch.arange(p.k_pool.shape[0], dtype=torch.int32, device=dev)}
    return (torch.cat(rows).to(dev), p.block_phase.cpu().to(torch.uint8).to(dev), fields, const)


def sched_state_dict(p, W):
    """The same starting state as sched_snapshot, as the oracle's window_step takes it
    (CPU tensors)."""
    i32, u8, fields, const = sched_snapshot(p, "cpu", W)
    st = {}
    for name, (off, shape) in fields.items():
        n = 1
        for x in shape:
            n *= x
        st[name] = i32[off:off + n].view(shape).clone()
    st.update(tokens=p.tokens.cpu().clone(), masked=p.masked.cpu().clone(), stopped=None,
              gen_blocks=const["gen_blocks"].cpu(), free_pages=const["free_pages"].cpu(),
              free_count=int(st.pop("free_count")[0]))
    for k in ("app_src", "app_dst", "n_append", "row_pos"):
        st.pop(k)
    return st


def sched_views(tokens, masked, i32, u8, fields, const, p, W):
    """A d2f.window_step state whose fields are views of one int32 and one uint8 row."""
    from types import SimpleNamespace
    w = p.w
    st = SimpleNamespace(batch=w.batch, block_size=w.block_size, max_blocks=W,
                         capacity=w.total_q, mask_id=p.mask_id, tokens=tokens, masked=masked,
                         block_phase=u8, stopped=None, **const)
    for name, (off, shape) in fields.items():
        n = 1
        for x in shape:
            n *= x
        setattr(st, name, i32[off:off + n].view(shape))
    return st


def measure(args, name, K, W, world, rank, dev, cpu=True):
    """Time K steps of workload `name` (after W warm-up steps) on `dev`; returns
    the workload's result object (the JSON line's fields for it)."""
    from block_causal_kv_gb300 import d2f, synth
    w = synth.workload(name)
    big = w.name.startswith("long") or w.name in ("dream", "ragged")
    p = synth.make_problem(w, device="cuda" if big else "cpu")
    base = StepSet(p, dev)
    B = w.block_size
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    per_set = base.nbytes()
    n_sets = max(1, min(64, -(-4 * l2 // per_set)))
    sets = [base] + [StepSet(p, dev, clone_from=base) for _ in range(n_sets - 1)]
    # decode state of every set in one buffer: one copy per graph replay resets all
    tokens0 = p.tokens.to(dev).repeat(n_sets, 1)
    masked0 = p.masked.to(dev).repeat(n_sets, 1)
    tokens_all, masked_all = tokens0.clone(), masked0.clone()
    for i, st in enumerate(sets):
        st.tokens, st.masked = tokens_all[i], masked_all[i]
    reuse = args.reuse_cached
    sched = args.scheduler
    if reuse and args.fused_append:
        raise SystemExit("--reuse-cached times steps without an append: drop --fused-append")
    if sched and (reuse or args.fused_append):
        raise SystemExit("--scheduler appends inside the attention by itself; it goes alone")
    if sched and w.total_q != w.batch * max(w.window_blocks) * B:
        raise SystemExit("--scheduler takes workloads whose windows all hold the same blocks")
    if sched and any(c % B for c in w.ctx_lens):
        raise SystemExit("--scheduler takes prompts padded to whole blocks")
    fused = (args.fused_append or sched) and len(p.src_row) > 0
    appends = len(p.src_row) > 0 and not fused and not reuse

    dcode = d2f.F32 if w.dtype == torch.float32 else d2f.BF16
    ws_attn = d2f.attn_workspace(dev, batch=w.batch, total_q=w.total_q, dtype=dcode,
                                 max_q_per_seq=p.max_q_per_seq, max_ctx=p.max_ctx,
                                 num_heads_q=w.num_heads_q, num_heads_kv=w.num_heads_kv,
                                 head_dim=w.head_dim, block_size=B, num_splits=args.num_splits)
    ws_commit = d2f.commit_workspace(dev, total_q=w.total_q, vocab=w.vocab, block_size=B, dtype=dcode,
                                     num_splits=args.commit_splits)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    conf = torch.empty(w.total_q, dtype=torch.float32, device=dev)
    amax = torch.empty(w.total_q, dtype=torch.int32, device=dev)
    rem = torch.empty(w.total_q // B, dtype=torch.int32, device=dev)

    # the scheduler's state (one int32 and one uint8 row per input set, so that one
    # copy of each resets every set)
    if sched:
        Wmax = max(w.window_blocks)
        sched_i32_0, sched_u8_0, sched_fields, sched_const = sched_snapshot(p, dev, Wmax)
        sched_i32_rep = sched_i32_0.repeat(n_sets, 1)
        sched_u8_rep = sched_u8_0.repeat(n_sets, 1)
        sched_i32_all, sched_u8_all = sched_i32_rep.clone(), sched_u8_rep.clone()
        for i, st in enumerate(sets):
            st.ws = sched_views(st.tokens, st.masked, sched_i32_all[i], sched_u8_all[i],
                                sched_fields, sched_const, p, Wmax)

    def attn(s):
        pt, cl, qs = s.page_table, s.ctx_len, s.q_start
        if reuse:
            kw = dict(part=d2f.ATTN_WINDOW, prev_out=s.prev_out, prev_lse=s.prev_lse)
        elif sched:
            pt, cl, qs = s.ws.page_table, s.ws.ctx_len, s.ws.q_start
            kw = dict(append_src_row=s.ws.app_src, append_dst_page=s.ws.app_dst,
                      append_n_dev=s.ws.n_append)
        elif fused:
            kw = dict(append_src_row=s.src_row, append_dst_page=s.dst_page)
        else:
            # without an append the cache, page table and layout are written by
            # no kernel of the step: the attention may load cached tiles before
            # its dependency wait
            kw = dict(cache_ready=bool(args.cache_ready) and not appends)
        d2f.block_attn(s.q, s.k_win, s.v_win, s.k_pool, s.v_pool, pt, cl, qs, block_size=B,
                       max_q_per_seq=p.max_q_per_seq, max_ctx=p.max_ctx,
                       num_splits=args.num_splits, out=s.out, want_lse=False, workspace=ws_attn,
                       err=err, **kw)

    def window(s):
        d2f.window_step(s.ws, tau_add=args.tau_add, tau_act=args.tau_act, err=err,
                        use_stopped=False)

    def cached_part(s):
        d2f.block_attn(s.q, s.k_win, s.v_win, s.k_pool, s.v_pool, s.page_table, s.ctx_len,
                       s.q_start, block_size=B, max_q_per_seq=p.max_q_per_seq, max_ctx=p.max_ctx,
                       num_splits=args.num_splits, out=s.prev_out, lse=s.prev_lse,
                       workspace=ws_attn, err=err, part=d2f.ATTN_CACHED)

    if reuse:
        for s in sets:
            s.prev_out = torch.empty_like(s.q)
            s.prev_lse = torch.empty(s.q.shape[:2], dtype=torch.float32, device=dev)
            cached_part(s)
        torch.cuda.synchronize()

    early_gap = stopped = None
    if args.early_gap is not None:
        early_gap = torch.full((w.batch,), args.early_gap, dtype=torch.float32, device=dev)
        stopped = torch.zeros(w.batch, dtype=torch.uint8, device=dev)

    def commit(s):
        qs, ph = (s.ws.q_start, s.ws.block_phase) if sched else (s.q_start, s.block_phase)
        d2f.commit(s.logits, s.tokens, s.masked, qs, ph, s.tau, block_size=B,
                   mask_id=p.mask_id, num_splits=args.commit_splits, conf=conf, argmax=amax,
                   block_remaining=rem, workspace=ws_commit, err=err,
                   metric=CONF_METRICS[args.conf_metric], early_gap=early_gap, stopped=stopped)

    def append(s):
        d2f.kv_append(s.k_win, s.v_win, s.src_row, s.dst_page, s.k_pool, s.v_pool, block_size=B,
                      err=err)

    def reset_all():
        tokens_all.copy_(tokens0)
        masked_all.copy_(masked0)
        if sched:
            sched_i32_all.copy_(sched_i32_rep)
            sched_u8_all.copy_(sched_u8_rep)

    def reset(s):
        i = sets.index(s)
        s.tokens.copy_(tokens0[i])
        s.masked.copy_(masked0[i])
        if sched:
            sched_i32_all[i].copy_(sched_i32_0)
            sched_u8_all[i].copy_(sched_u8_0)

    def step_kernels(s):
        attn(s)
        commit(s)
        if appends:
            append(s)
        if sched:
            window(s)

    if args.profile_steps:
        for i in range(args.profile_steps):
            s = sets[i % n_sets]
            reset(s)
            step_kernels(s)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, "device error %d" % int(err.item())
        return

    stream = torch.cuda.Stream(device=dev)
    # warm-up (library init, function attributes) outside capture
    with torch.cuda.stream(stream):
        for i in range(max(3, min(W, n_sets))):
            s = sets[i % n_sets]
            reset(s)
            step_kernels(s)
    stream.synchronize()

    def capture(indices):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            if len(indices) == n_sets:
                reset_all()
            for i in indices:
                s = sets[i]
                if len(indices) != n_sets:
                    reset(s)
                step_kernels(s)
        return g

    g_all = capture(range(n_sets))
    singles = [capture([i]) for i in range(n_sets)]

    full, rest = divmod(K, n_sets)

    # warm-up replays (untimed) plus a short pre-roll so clock samples overlap load
    with torch.cuda.stream(stream):
        for i in range(W):
            singles[i % n_sets].replay()
    stream.synchronize()
    sampler = ClockSampler()
    sampler.start()
    t_pre = time.time()
    with torch.cuda.stream(stream):
        while time.time() - t_pre < 0.6:
            g_all.replay()
            stream.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(full):
            g_all.replay()
        for i in range(rest):
            singles[i].replay()
        stop.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    bus = getattr(props, "pci_bus_id", None)
    clocks = sampler.stop(bus if isinstance(bus, int) else None)
    elapsed_ms = start.elapsed_time(stop)
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    if int(err.item()) != 0:
        raise RuntimeError("device error word %d after the timed region" % int(err.item()))

    # Per-kernel durations. The commit (and the append) run as graphs of that
    # kernel only over the same rotating input sets, launched back to back as in
    # the step (no programmatic early launch), timed with CUDA events around whole
    # replays: the average launch duration including the gap to the next launch.
    # The attention's duration is the step time less those: its share of the
    # step. (An attention-only graph chains attention launches through
    # programmatic dependent launch, which the step never does: for grids that
    # fill the GPU the next launch's early CTAs take slots from the current one,
    # so that number is reported for reference only. Events between kernels
    # would add their own latency to every bracket.)
    per_kernel = {}
    kernel_fns = [("attn", attn), ("commit", commit)] + ([("append", append)] if appends else []) \
        + ([("cached_part", cached_part)] if reuse else []) \
        + ([("window", window)] if sched else [])
    for which, fn in kernel_fns:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            if which in ("commit", "window"):
                reset_all()
            for i in range(n_sets):
                fn(sets[i])
        reps = max(3, min(50, 20000 // n_sets))
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(reps):
                g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        per_kernel[which] = a.elapsed_time(b) * 1000.0 / (reps * n_sets)
    # Hot-L2 step (reported, never the headline): the same inputs every step, so
    # they stay in L2, where one input set fits in half of L2. Like the timed
    # graph, one graph runs many steps and resets their decode state once; each
    # step has its own copy of that small state (the commit rewrites it), all
    # other inputs are input set 0's. Plain steps only.
    hot = None
    if per_set <= l2 // 2 and not (reuse or sched or fused or appends):
        import copy as _copy
        n_hot = max(8, n_sets)
        tok_h0, msk_h0 = tokens0[0].repeat(n_hot, 1), masked0[0].repeat(n_hot, 1)
        tok_h, msk_h = tok_h0.clone(), msk_h0.clone()
        hsets = []
        for i in range(n_hot):
            h = _copy.copy(sets[0])
            h.tokens, h.masked = tok_h[i], msk_h[i]
            hsets.append(h)
        g_hot = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_hot, stream=stream, capture_error_mode="relaxed"):
            tok_h.copy_(tok_h0)
            msk_h.copy_(msk_h0)
            for h in hsets:
                step_kernels(h)
        reps_hot = max(3, min(200, 20000 // n_hot))
        with torch.cuda.stream(stream):
            for _ in range(3):
                g_hot.replay()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for _ in range(reps_hot):
                g_hot.replay()
            b.record(stream)
        torch.cuda.synchronize()
        hot_us = a.elapsed_time(b) * 1000.0 / (reps_hot * n_hot)
        hot = {"us_per_step": hot_us, "steps_per_s": 1e6 / hot_us, "set_bytes": per_set,
               "note": "input set 0 every step (L2-resident), decode state reset per graph "
                       "as in the timed region: not counted"}
    step_us = elapsed_ms * 1000.0 / K
    attn_in_step = (step_us - per_kernel["commit"] - per_kernel.get("append", 0.0)
                    - per_kernel.get("window", 0.0))
    attn_us, commit_us = [attn_in_step], [per_kernel["commit"]]

    steps_total = K * world
    value = steps_total / (elapsed_ms / 1000.0)
    ms_per_step = elapsed_ms / K
    attn_b, commit_b, append_b = algorithmic_bytes(p, "window" if reuse else "all")
    if fused:  # the appended pages' writes (their window rows are read by the attention anyway)
        attn_b += append_b // 2
    hbm, tflops, peak_kind = peaks()
    t_attn = statistics.mean(attn_us) if attn_us else None
    t_commit = statistics.mean(commit_us) if commit_us else None
    kernels = {}
    if t_attn:
        tf_sus, tf_kind = sustained_tflops()
        kernels["block_attn"] = {"us": t_attn, "bytes": attn_b, "GB/s": attn_b / t_attn / 1e3,
                                 "frac": attn_b / t_attn / 1e3 / hbm,
                                 "TFLOP/s": flops(p, reuse) / t_attn / 1e6,
                                 "roofline": dict(attn_roofline(attn_b, flops(p, reuse), hbm, tf_sus,
                                                                t_attn, dcode == d2f.BF16),
                                                  tensor_peak_tflops=tf_sus,
                                                  tensor_peak_kind=tf_kind + " sustained"),
                                 "us_attention_only_graph": per_kernel["attn"]}
    if t_commit:
        kernels["commit"] = {"us": t_commit, "bytes": commit_b, "GB/s": commit_b / t_commit / 1e3,
                             "frac": commit_b / t_commit / 1e3 / hbm}
    if reuse:
        cb = algorithmic_bytes(p, "cached")[0]
        t_cp = per_kernel["cached_part"]
        kernels["cached_part"] = {"us": t_cp, "bytes": cb, "GB/s": cb / t_cp / 1e3,
                                  "frac": cb / t_cp / 1e3 / hbm,
                                  "note": "once per cache change (a finished block), not per step"}
    if sched:
        kernels["window_step"] = {"us": per_kernel["window"],
                                  "note": "one CTA; integer work on a few KB of state"}
    if appends:
        t_app = per_kernel["append"]
        kernels["kv_append"] = {"us": t_app, "bytes": append_b, "GB/s": append_b / t_app / 1e3,
                                "frac": append_b / t_app / 1e3 / hbm}
    dom = "block_attn" if (t_attn or 0) >= (t_commit or 0) else "commit"
    dk = kernels.get(dom, {})
    roofline = {"bound": "hbm", "kernel": dom,
                "duration": ("step time less the commit%s: commit-only%s graphs over the "
                             "rotating input sets, CUDA events around whole replays" % (
                                 " and append" if appends else "", " and append-only" if appends
                                 else "")) if dom == "block_attn" else
                            "average launch of a commit-only CUDA graph over the rotating input "
                            "sets, CUDA events around whole replays",
                "achieved": dk.get("GB/s"), "peak": hbm,
                "unit": "GB/s", "frac": dk.get("frac"), "peak_kind": peak_kind,
                "traffic": recorded_traffic(("attn_window" if reuse else "attn")
                                            if dom == "block_attn" else "commit", w.name)}

    # end to end through the C ABI from pinned host buffers
    e2e = None
    if not args.no_e2e:
        hooks = None
        if sched:
            def make_ws(d):
                d.ws_i32, d.ws_u8 = sched_i32_0.clone(), sched_u8_0.clone()
                d.ws = sched_views(d.tokens, d.masked, d.ws_i32, d.ws_u8, sched_fields,
                                   sched_const, p, Wmax)

            def pre_step(d):
                d.ws_i32.copy_(sched_i32_0)
                d.ws_u8.copy_(sched_u8_0)

            hooks = (make_ws, pre_step, window)
        e2e = run_e2e(p, dev, sets[0], attn, commit, append if appends else None, K, stream,
                      tokens0[0], masked0[0], hooks)

    line = {"metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == torch.bfloat16 else "f32",
            "data": "synthetic (seeded; no dataset, no weights)",
            "config": dict(workload_config(p, args),
                           l2="%d rotating input sets of %.1f MB (%.0f MB > 4x L2 %.0f MB)" % (
                               n_sets, per_set / 1e6, n_sets * per_set / 1e6, l2 / 1e6),
                           state_reset="2 device copies of the decode state (%d B per step) "
                                       "at the start of each %d-step graph" % (5 * w.total_q,
                                                                              n_sets),
                           attn_splits=args.num_splits or "auto",
                           commit_splits=args.commit_splits or "auto",
                           cache_ready=bool(args.cache_ready) and not (reuse or fused or
                                                                       appends)),
            "roofline": roofline, "kernels": kernels,
            "gpu_launches": K * (2 + (1 if appends else 0) + (1 if sched else 0)),
            "clocks": clocks, "e2e": e2e}
    if hot:
        line["hot_l2"] = hot
    # free the device buffers before the CPU legs (and the next workload)
    del sets, base
    torch.cuda.synchronize()
    if rank == 0 and cpu and not args.no_cpu_baseline:
        pc = p if p.q.device.type == "cpu" else p.to("cpu")
        del p
        torch.cuda.empty_cache()
        line["cpu_baseline"] = cpu_baseline(pc, args, reuse, sched)
    return line


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(p, args, reuse, sched):
    """The oracle as it stands on this host: all cores, then one thread, each on
    a bounded sample of the step (time_oracle)."""
    metric = CONF_METRICS[args.conf_metric]
    sch = (args.tau_add, args.tau_act) if sched else None
    n = oracle_threads()
    v_all, s_all = time_oracle(p, args.cpu_seconds, n, metric, reuse, sch)
    res = {"value": v_all, "unit": "steps/s", "cores": n, "kind": "oracle", "sample": s_all,
           "cpu_model": cpu_model()}
    if n > 1 and args.cpu_seconds_1t > 0:
        v1, s1 = time_oracle(p, args.cpu_seconds_1t, 1, metric, reuse, sch)
        res["one_thread"] = {"value": v1, "unit": "steps/s", "cores": 1, "sample": s1}
    return res


# Order of the per-workload results; the headline is the largest configuration
# that fits one GPU (long context, block size 32: 2.16 GB of cached K/V and
# 129.5 MB of logits per step).
HEADLINE = "long_b32"
ALL_WORKLOADS = ("tiny", "llada", "ragged", "dream", "long_b8", "long_b16", "long_b32")
# steps timed for the workloads other than the headline (which times exactly
# --steps): enough for a timed region of a few hundred milliseconds
MIN_STEPS = {"tiny": 20000, "llada": 20000, "ragged": 3000, "dream": 3000, "long_b8": 1000,
             "long_b16": 1000, "long_b32": 1000}
# per-workload fields kept in the per_config object
PER_CONFIG_KEYS = ("value", "unit", "steps", "ms_per_step", "dtype", "config", "roofline",
                   "kernels", "clocks", "e2e", "cpu_baseline", "hot_l2")


def run_ours(args, world, rank, local):
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    K, W = args.steps, args.warmup
    if args.profile_steps and args.workload == "all":
        raise SystemExit("--profile-steps takes one --workload")
    if args.workload != "all":
        line = measure(args, args.workload, K, W, world, rank, dev)
        if rank == 0 and line is not None:
            print(json.dumps(line), flush=True)
        return
    per = {}
    for name in ALL_WORKLOADS:
        k = K if name == HEADLINE else max(K, MIN_STEPS[name])
        per[name] = measure(args, name, k, W, world, rank, dev)
        torch.cuda.empty_cache()
    line = dict(per[HEADLINE])
    line["per_config"] = {n: {k: v for k, v in r.items() if k in PER_CONFIG_KEYS}
                          for n, r in per.items()}
    line["config"] = dict(line["config"], headline=(
        "%s: the largest configuration that fits one GPU; per_config holds every workload, each "
        "timed on its own" % HEADLINE))
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(p, dev, s, attn, commit, append, K, stream, tokens0, masked0, hooks=None):
    """Same step through the public API with host inputs: every step copies its
    inputs (Q, window K/V, logits, decode state) from pinned host memory and
    reads back its results (output, tokens, masked). The inputs of a step travel
    as one packed host-to-device copy into one of two device input sets, on a copy
    stream, so the copy of step i+1 overlaps the kernels of step i; each step's
    results are read back on the compute stream right after its kernels."""
    import copy as _copy
    names = ("q", "k_win", "v_win", "logits", "tokens", "masked")
    src = {"q": s.q, "k_win": s.k_win, "v_win": s.v_win, "logits": s.logits,
           "tokens": tokens0, "masked": masked0}
    align = 256
    offs, total = {}, 0
    for nm in names:
        offs[nm] = total
        total += -(-src[nm].numel() * src[nm].element_size() // align) * align
    h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
    for nm in names:
        t = src[nm].detach().to("cpu").contiguous()
        nb = t.numel() * t.element_size()
        h_in[offs[nm]:offs[nm] + nb].copy_(t.view(-1).view(torch.uint8))

    def view(buf, nm):
        t = src[nm]
        nb = t.numel() * t.element_size()
        return buf[offs[nm]:offs[nm] + nb].view(t.dtype).view(t.shape)

    dsets = []
    for _ in range(2):
        d = _copy.copy(s)  # shares the cache, page table and metadata tensors
        buf = torch.empty(total, dtype=torch.uint8, device=dev)
        for nm in names:
            setattr(d, nm, view(buf, nm))
        d.buf = buf
        d.out = torch.empty_like(s.out)
        d.ready = torch.cuda.Event()   # inputs landed
        d.read = torch.cuda.Event()    # results read back
        if hooks:
            hooks[0](d)                # its own scheduler state over its tokens / masked
        dsets.append(d)
    h_out = torch.empty(s.out.shape, dtype=s.out.dtype).pin_memory()
    h_tok_o = torch.empty(tokens0.shape, dtype=tokens0.dtype).pin_memory()
    h_msk_o = torch.empty(masked0.shape, dtype=masked0.dtype).pin_memory()
    h2d = sum(src[nm].numel() * src[nm].element_size() for nm in names)
    d2h = sum(t.numel() * t.element_size() for t in (h_out, h_tok_o, h_msk_o))
    n = max(10, min(K, 2000))
    cstream = torch.cuda.Stream(device=dev)

    def step(i):
        d = dsets[i % 2]
        with torch.cuda.stream(cstream):
            if i >= 2:
                cstream.wait_event(d.read)      # its previous results are read back
            d.buf.copy_(h_in, non_blocking=True)
            d.ready.record(cstream)
        with torch.cuda.stream(stream):
            stream.wait_event(d.ready)
            if hooks:
                hooks[1](d)            # the scheduler's state of the step (device copy)
            attn(d)
            commit(d)
            if append:
                append(d)
            if hooks:
                hooks[2](d)
            # results back right after the kernels (on this stream, so the copy
            # stream stays free for the next step's inputs)
            h_out.copy_(d.out, non_blocking=True)
            h_tok_o.copy_(d.tokens, non_blocking=True)
            h_msk_o.copy_(d.masked, non_blocking=True)
            d.read.record(stream)

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    cstream.wait_event(a)
    for i in range(n):
        step(i)
    stream.wait_stream(cstream)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    return {"value": n / (ms / 1000.0), "unit": "steps/s", "steps": n,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "overlap": "one packed input copy per step on a copy stream, two device input "
                       "sets: step i+1's copy overlaps step i's kernels and result reads"}


def main():
    args = parse()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
