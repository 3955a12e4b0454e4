// d2f_commit kernel: one streaming pass over the logits of every still-masked
// window position, fused with the block-level commit decision.
//
// Sources: "확산 언어 모델(Diffusion LLM)이란 무엇인가", §양방향 어텐션과 사라진 KV
// 캐시 and §토큰 순서의 이론 (confidence = largest softmax probability);
// "D2F 논문 리뷰: 확산 LLM이 자기회귀 모델보다 빠른 추론을 처음으로 달성한 방식",
// §쉽게 이해하기 (conservative threshold commit, aggressive top-1, remask).
//
// Grid (slices, rows): CTA (s, r) reduces vocabulary slice s of row r to
// (max, first argmax, sum of exp(l - max)) with 128-bit streaming loads, four
// in flight per thread (scalar loads where rows are not 16-byte aligned). The
// slices are long (a few CTAs per SM over the whole grid): measured on GB300,
// staging slices in shared memory with bulk copies, or persistent CTAs streaming
// many slices through a ring of bulk copies, were slower (Dream-shaped layer:
// 42.8 and 39-42 us against 34.5 us for this form).
// Every CTA of a window block then bumps one arrival counter; the last one to
// arrive composes the slices of all rows of the block and decides the block with
// one warp (lane = row). The decision's metadata (sequence, tau, phase) is
// fetched while the slice streams. There is no spin-wait on another CTA: the
// counter hands the work to whoever arrives last and is reset by it.
#include <mutex>

#include "d2f_internal.cuh"

namespace d2f {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr float kLog2e = 1.4426950408889634f;

// Per-row terms beyond (max, argmax, sum) by metric kind: MK 0 none (largest
// probability), MK 1 e = sum of exp(l - m) (l - m) (negative entropy), MK 2
// e = the second largest logit, counted with multiplicity (margin, logit gap).
constexpr int kMkNone = 0, kMkEntropy = 1, kMkTop2 = 2;
__host__ __device__ constexpr int metric_kind(int metric) {
  return metric == D2F_CONF_NEG_ENTROPY ? kMkEntropy
         : (metric == D2F_CONF_MARGIN || metric == D2F_CONF_LOGIT_GAP) ? kMkTop2 : kMkNone;
}

struct RowState {
  float m;    // running maximum
  int idx;    // lowest index attaining m
  float s;    // sum of exp(l - m)
  float e;    // metric term (see metric_kind)
};

template <int MK>
__device__ __forceinline__ RowState combine(RowState a, RowState b) {
  if (MK == kMkTop2) {  // second largest of the union (before a state is dropped as empty)
    const float e = fmaxf(fminf(a.m, b.m), fmaxf(a.e, b.e));
    a.e = e;
    b.e = e;
  }
  if (b.m == -INFINITY) return a;
  if (a.m == -INFINITY) return b;
  RowState r;
  if (a.m > b.m) {
    r.m = a.m;
    r.idx = a.idx;
  } else if (b.m > a.m) {
    r.m = b.m;
    r.idx = b.idx;
  } else {
    r.m = a.m;
    r.idx = min(a.idx, b.idx);
  }
  const float wa = fast_exp2((a.m - r.m) * kLog2e), wb = fast_exp2((b.m - r.m) * kLog2e);
  r.s = a.s * wa + b.s * wb;
  // sum exp(l - M)(l - M) = w (E + (m - M) S) for each part
  r.e = MK == kMkEntropy ? wa * (a.e + (a.m - r.m) * a.s) + wb * (b.e + (b.m - r.m) * b.s) : a.e;
  return r;
}

template <int MK>
__device__ __forceinline__ RowState warp_combine(RowState v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    RowState w;
    w.m = __shfl_xor_sync(0xffffffffu, v.m, o);
    w.idx = __shfl_xor_sync(0xffffffffu, v.idx, o);
    w.s = __shfl_xor_sync(0xffffffffu, v.s, o);
    w.e = MK != kMkNone ? __shfl_xor_sync(0xffffffffu, v.e, o) : 0.f;
    v = combine<MK>(v, w);
  }
  return v;
}

// Confidence of a composed row state.
__device__ __forceinline__ float row_conf(const RowState &r, int metric) {
  if (metric == D2F_CONF_NEG_ENTROPY) return r.e / r.s - __logf(r.s);
  if (metric == D2F_CONF_MARGIN) return (1.0f - fast_exp2((r.e - r.m) * kLog2e)) / r.s;
  if (metric == D2F_CONF_LOGIT_GAP) return r.m - r.e;
  return 1.0f / r.s;
}

// Fold N consecutive values starting at index v0 into the thread state. The
// per-lane sums keep N independent accumulation chains; MK adds the entropy
// numerator (one accumulator, rescaled with the sums) or the second largest value.
template <int N, int MK>
__device__ __forceinline__ void fold(const float (&x)[N], int v0, float &m, int &idx,
                                     float (&acc)[N], float &acc_e, float &m2) {
  if (MK == kMkTop2) {  // top two with multiplicity, before m takes this vector in
    float t1 = m, t2 = m2;
#pragma unroll
    for (int j = 0; j < N; ++j) {
      t2 = fmaxf(t2, fminf(t1, x[j]));
      t1 = fmaxf(t1, x[j]);
    }
    m2 = t2;
  }
  float vm = x[0];
#pragma unroll
  for (int j = 1; j < N; ++j) vm = fmaxf(vm, x[j]);
  if (vm > m) {
    int first = 0;
#pragma unroll
    for (int j = N - 1; j >= 0; --j)
      if (x[j] == vm) first = j;
    const float alpha = fast_exp2((m - vm) * kLog2e);
    if (MK == kMkEntropy) {
      // sum exp(l - vm)(l - vm) = alpha (E + (m - vm) S); nothing to carry from m = -inf
      float S = 0.f;
#pragma unroll
      for (int j = 0; j < N; ++j) S += acc[j];
      acc_e = m == -INFINITY ? 0.f : alpha * (acc_e + (m - vm) * S);
    }
#pragma unroll
    for (int j = 0; j < N; ++j) acc[j] *= alpha;
    m = vm;
    idx = v0 + first;
  }
  // x - m is exact in float for bf16 inputs; one rounding in the scale.
#pragma unroll
  for (int j = 0; j < N; ++j) {
    if (MK == kMkEntropy) {
      const float d = fmaxf(x[j] - m, -1e30f);  // a -inf logit adds 0 (not 0 * inf)
      const float t = fast_exp2(d * kLog2e);
      acc[j] += t;
      acc_e = fmaf(t, d, acc_e);
    } else {
      acc[j] += fast_exp2((x[j] - m) * kLog2e);
    }
  }
}

template <int DT>
__device__ __forceinline__ void unpack(const uint4 raw, float (&x)[DT == D2F_BF16 ? 8 : 4]) {
  if (DT == D2F_BF16) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = __uint_as_float(w[j] << 16);
      x[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  } else {
    x[0] = __uint_as_float(raw.x);
    x[1] = __uint_as_float(raw.y);
    x[2] = __uint_as_float(raw.z);
    x[3] = __uint_as_float(raw.w);
  }
}

template <int DT>
__device__ __forceinline__ float load_scalar(const void *base, int64_t i) {
  if (DT == D2F_BF16) return bf16_bits_to_float(((const uint16_t *)base)[i]);
  return ((const float *)base)[i];
}

// One warp (lane u = row u of the block) decides block jb from the composed row
// results in shared memory.
__device__ void decide_block(const CommitArgs &a, int jb, const float *conf_s, const int *arg_s,
                             float t, int phase, bool m) {
  const int lane = threadIdx.x & 31;
  const int r = jb * a.block_size + lane;
  const bool in = lane < a.block_size;
  const float c = m ? conf_s[lane] : -1.0f;
  const int am = m ? arg_s[lane] : -1;
  bool take = m && (c > t);
  const unsigned any_masked = __ballot_sync(0xffffffffu, m);
  if (phase == D2F_PHASE_AGGRESSIVE && any_masked) {
    float bv = m ? c : -INFINITY;
    int bl = m ? lane : 64;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int ol = __shfl_xor_sync(0xffffffffu, bl, o);
      if (ov > bv || (ov == bv && ol < bl)) {
        bv = ov;
        bl = ol;
      }
    }
    take = take || (lane == bl);
  }
  if (m) {
    if (take) {
      a.tokens[r] = am;
      a.masked[r] = 0;
    } else {
      a.tokens[r] = a.mask_id;
    }
  }
  const unsigned left = __ballot_sync(0xffffffffu, m && !take);
  if (in) {
    if (a.conf_out) a.conf_out[r] = c;
    if (a.argmax_out) a.argmax_out[r] = am;
  }
  if (lane == 0 && a.block_remaining) a.block_remaining[jb] = __popc(left);
}

// Early commit of whole sequences ("확산 언어 모델(Diffusion LLM)이란 무엇인가",
// §답을 미리 안다: 조기 확정 디코딩(Prophet): once the gap between the largest and
// the second largest logit over the answer region exceeds a threshold, every
// remaining mask is filled with its argmax). Reading: the region is the
// sequence's window and its gap the smallest over the rows masked on entry. One
// warp, after decide_block for block jb of sequence b: record the block's
// smallest gap and its rows' greedy tokens, arrive on the sequence's counter
// (at its first block); the last block of the sequence to arrive decides it and
// commits the rows still masked in every block of it.
__device__ void early_commit(const CommitArgs &a, int jb, int b, const float *gap_s,
                             const int *arg_s, bool m) {
  const int lane = threadIdx.x & 31;
  const int B = a.block_size;
  const int r = jb * B + lane;
  float g = m ? gap_s[lane] : INFINITY;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) g = fminf(g, __shfl_xor_sync(0xffffffffu, g, o));
  if (m) a.row_arg[r] = arg_s[lane];
  if (lane == 0) a.blk_gap[jb] = g;
  const int q0 = __ldg(a.q_start + b), q1 = __ldg(a.q_start + b + 1);
  const int jb0 = q0 / B, nblk = (q1 - q0) / B;
  __threadfence();  // this block's decision, gap and tokens before the arrival
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomic_add_acq_rel(a.seq_cnt + jb0, 1) == nblk - 1;
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();
  float gs = INFINITY;
  for (int j = jb0 + lane; j < jb0 + nblk; j += 32) gs = fminf(gs, __ldcg(a.blk_gap + j));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) gs = fminf(gs, __shfl_xor_sync(0xffffffffu, gs, o));
  const bool stop = gs < INFINITY && gs > __ldg(a.early_gap + b);  // strict, in float
  if (stop) {
    for (int rr = q0 + lane; rr < q1; rr += 32) {
      if (__ldcg(a.masked + rr)) {
        a.tokens[rr] = __ldcg(a.row_arg + rr);
        a.masked[rr] = 0;
      }
    }
    if (a.block_remaining)
      for (int j = jb0 + lane; j < jb0 + nblk; j += 32) a.block_remaining[j] = 0;
  }
  if (lane == 0) {
    if (a.stopped) a.stopped[b] = stop ? 1 : 0;
    a.seq_cnt[jb0] = 0;
  }
}

template <int DT, int PATH, int MK>  // PATH 0: scalar loads, 1: 128-bit loads; MK: metric_kind
__global__ void __launch_bounds__(kThreads) commit_kernel(const CommitArgs a) {
  constexpr int N = (DT == D2F_BF16) ? 8 : 4;  // values per 16-byte vector
  __shared__ RowState red[kThreads / 32];
  __shared__ float conf_s[32];
  __shared__ float gap_s[32];  // logit gap of each row (top-two state only)
  __shared__ int arg_s[32];
  __shared__ int is_last;

  const int s = blockIdx.x;
  const int r = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int B = a.block_size;
  const int jb = r / B;

  if (tid == 0) D2F_TRACE_MARK(1, 0);
  // The next kernel in the stream may be scheduled from here on (it waits for
  // this grid before reading anything); triggering first gives it the most time
  // to become resident.
  grid_launch_dependents();
  grid_dependency_wait();  // logits / state may come from the previous kernel
  if (tid == 0) D2F_TRACE_MARK(1, 1);

  // Decision metadata of this block, fetched now, used only by the last arriver:
  // lane u of warp 0 holds row u's masked flag, thread 0 the block's tau and phase.
  float tau_b = 0.f;
  int phase = 0, seq_b = 0;
  bool live = true;  // thread 0: the block lies inside the window layout
  const bool blk_masked = warp == 0 && lane < B && a.masked[jb * B + lane] != 0;
  if (tid == 0) {
    int lo = 0, hi = a.batch - 1;
    const int r0 = jb * B;
    while (lo < hi) {  // largest b with q_start[b] <= r0 (blocks never straddle sequences)
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(a.q_start + mid) <= r0) lo = mid; else hi = mid - 1;
    }
    tau_b = __ldg(a.tau + lo);
    phase = __ldg(a.block_phase + jb);
    seq_b = lo;
    // Rows past the last window (a launch sized for a capacity, the layout written
    // on the device) are not masked, so they fold nothing; their block must not
    // arrive either, or it would decide for a sequence it does not belong to.
    live = r0 < __ldg(a.q_start + a.batch);
  }
  const bool is_masked = a.masked[r] != 0;

  if (is_masked) {
    int lr = a.logit_row ? a.logit_row[r] : r;
    const bool row_ok = lr >= 0 && lr < a.num_logit_rows;
    if (!row_ok) {
      if (tid == 0 && s == 0) set_err(a.err, D2F_ERR_BAD_INDEX);
      lr = 0;
    }
    const int v0 = s * a.chunk;
    const int v1 = min(a.vocab, v0 + a.chunk);
    const char *row = (const char *)a.logits + (int64_t)lr * a.row_stride * (DT == D2F_BF16 ? 2 : 4);
    float m = -INFINITY, m2 = -INFINITY;
    int idx = 0x7fffffff;
    float acc[N], acc_e = 0.f;
#pragma unroll
    for (int j = 0; j < N; ++j) acc[j] = 0.f;
    int v_tail = v0;  // first index left for the scalar loop

    if (PATH == 1 && row_ok) {
      // v0 and chunk are multiples of N and the row start is 16-byte aligned.
      const uint4 *vec = reinterpret_cast<const uint4 *>(row);
      const int nvec_end = v1 / N;  // vectors fully inside [v0, v1)
      int k = v0 / N + tid;
      for (; k + (kUnroll - 1) * kThreads < nvec_end; k += kUnroll * kThreads) {
        uint4 raw[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) raw[u] = __ldcs(vec + k + u * kThreads);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          float x[N];
          unpack<DT>(raw[u], x);
          fold<N, MK>(x, (k + u * kThreads) * N, m, idx, acc, acc_e, m2);
        }
      }
      for (; k < nvec_end; k += kThreads) {
        float x[N];
        unpack<DT>(__ldcs(vec + k), x);
        fold<N, MK>(x, k * N, m, idx, acc, acc_e, m2);
      }
      v_tail = max(v0, nvec_end * N);
    }
    // scalar part: the whole slice on the scalar path, else the ragged tail
    if (row_ok) {
      for (int e = v_tail + tid; e < v1; e += kThreads) {
        const float x = load_scalar<DT>(row, e);
        if (MK == kMkTop2) m2 = fmaxf(m2, fminf(m, x));
        if (x > m) {  // new maximum: rescale every lane accumulator
          const float alpha = fast_exp2((m - x) * kLog2e);
          if (MK == kMkEntropy) {
            float S = 0.f;
#pragma unroll
            for (int j = 0; j < N; ++j) S += acc[j];
            acc_e = m == -INFINITY ? 0.f : alpha * (acc_e + (m - x) * S);
          }
#pragma unroll
          for (int j = 0; j < N; ++j) acc[j] *= alpha;
          m = x;
          idx = e;
        }
        if (MK == kMkEntropy) {
          const float d = fmaxf(x - m, -1e30f);
          const float t = fast_exp2(d * kLog2e);
          acc[0] += t;
          acc_e = fmaf(t, d, acc_e);
        } else {
          acc[0] += fast_exp2((x - m) * kLog2e);
        }
      }
    }
    float tot = 0.f;
#pragma unroll
    for (int j = 0; j < N; ++j) tot += acc[j];
    if (tid == 0) D2F_TRACE_MARK(1, 4);
    RowState st = {m, idx, tot, MK == kMkEntropy ? acc_e : MK == kMkTop2 ? m2 : 0.f};
    const RowState empty = {-INFINITY, 0x7fffffff, 0.f, MK == kMkTop2 ? -INFINITY : 0.f};
    st = warp_combine<MK>(st);
    if (lane == 0) red[warp] = st;
    __syncthreads();
    if (warp == 0) {
      st = lane < kThreads / 32 ? red[lane] : empty;
      st = warp_combine<MK>(st);
      if (lane == 0) {
        if (!row_ok) st = empty;
        a.partial[(int64_t)r * a.splits + s] = make_float4(st.m, __int_as_float(st.idx), st.s, st.e);
      }
    }
  }

  // ---- arrival on the block's counter ----------------------------------------
  if (tid == 0) D2F_TRACE_MARK(1, 5);
  if (tid == 0) is_last = live && atomic_add_acq_rel(a.blk_cnt + jb, 1) == B * a.splits - 1;
  __syncthreads();
  if (tid == 0) D2F_TRACE_MARK(1, 6);
  if (!is_last) return;
  // Compose the slices of every masked row of the block at once: half a warp per
  // row (lanes 0-15 row 2w, lanes 16-31 row 2w+1 of warp w), slices strided by 16.
  for (int u0 = 2 * warp; u0 < B; u0 += 2 * (kThreads / 32)) {
    const int u = u0 + (lane >> 4);
    const int sub = lane & 15;
    RowState acc2 = {-INFINITY, 0x7fffffff, 0.f, MK == kMkTop2 ? -INFINITY : 0.f};
    if (u < B) {
      const int rr = jb * B + u;
      for (int j = sub; j < a.splits; j += 16) {
        const float4 p = __ldcg(a.partial + (int64_t)rr * a.splits + j);
        acc2 = combine<MK>(acc2, RowState{p.x, __float_as_int(p.y), p.z, p.w});
      }
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {  // reduce within each 16-lane half
      RowState w;
      w.m = __shfl_xor_sync(0xffffffffu, acc2.m, o);
      w.idx = __shfl_xor_sync(0xffffffffu, acc2.idx, o);
      w.s = __shfl_xor_sync(0xffffffffu, acc2.s, o);
      w.e = __shfl_xor_sync(0xffffffffu, acc2.e, o);
      acc2 = combine<MK>(acc2, w);
    }
    if (sub == 0 && u < B) {
      // rows not masked on entry have no partials (their slots are stale)
      const bool ok = acc2.s > 0.f;
      conf_s[u] = ok ? row_conf(acc2, a.metric) : -1.0f;
      gap_s[u] = ok && MK == kMkTop2 ? acc2.m - acc2.e : INFINITY;
      arg_s[u] = ok ? acc2.idx : -1;
    }
  }
  __syncthreads();
  if (warp == 0) {
    tau_b = __shfl_sync(0xffffffffu, tau_b, 0);
    phase = __shfl_sync(0xffffffffu, phase, 0);
    decide_block(a, jb, conf_s, arg_s, tau_b, phase, blk_masked);
    if (lane == 0) a.blk_cnt[jb] = 0;
    if (MK == kMkTop2 && a.early_gap) early_commit(a, jb, __shfl_sync(0xffffffffu, seq_b, 0),
                                                   gap_s, arg_s, blk_masked);
    if (lane == 0) D2F_TRACE_MARK(1, 7);
  }
}

// Keep the L1 / shared-memory split at its shared-memory maximum, as the
// attention kernel needs it: alternating kernels then never make an SM drain and
// reconfigure between launches. Set once per device.
template <int DT, int PATH, int MK>
cudaError_t ensure_carveout() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(commit_kernel<DT, PATH, MK>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

template <int DT, int PATH, int MK>
cudaError_t launch_path(const CommitArgs &a, cudaStream_t stream) {
  cudaError_t ce = ensure_carveout<DT, PATH, MK>();
  if (ce != cudaSuccess) return ce;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.splits, a.total_q);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  // No programmatic early launch for the commit: measured on GB300, its CTAs
  // scheduled during the previous kernel's tail cost more than they saved. The
  // kernel still waits on its dependencies (a no-op without the attribute).
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, commit_kernel<DT, PATH, MK>, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int MK>
cudaError_t launch_kind(const CommitArgs &a, int dtype, int path, cudaStream_t stream) {
  if (dtype == D2F_BF16) {
    if (path == 1) return launch_path<D2F_BF16, 1, MK>(a, stream);
    return launch_path<D2F_BF16, 0, MK>(a, stream);
  }
  if (path == 1) return launch_path<D2F_F32, 1, MK>(a, stream);
  return launch_path<D2F_F32, 0, MK>(a, stream);
}

}  // namespace

cudaError_t launch_commit(const CommitArgs &a, int dtype, int path, cudaStream_t stream) {
  if (a.total_q == 0) return cudaSuccess;
  // the early commit needs every row's logit gap: the top-two state
  if (a.early_gap && a.metric != D2F_CONF_NEG_ENTROPY)
    return launch_kind<kMkTop2>(a, dtype, path, stream);
  switch (metric_kind(a.metric)) {
    case kMkEntropy: return launch_kind<kMkEntropy>(a, dtype, path, stream);
    case kMkTop2: return launch_kind<kMkTop2>(a, dtype, path, stream);
    default: return launch_kind<kMkNone>(a, dtype, path, stream);
  }
}

}  // namespace d2f

#ifdef D2F_TRACE
namespace d2f {
D2F_TRACE_COPY_FN(d2f_trace_copy_commit)
}  // namespace d2f
#endif
