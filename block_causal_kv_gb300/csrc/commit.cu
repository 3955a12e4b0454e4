// d2f_commit kernel: one streaming pass over the logits of every still-masked
// window position, fused with the block-level commit decision.
//
// Sources: "확산 언어 모델(Diffusion LLM)이란 무엇인가", §양방향 어텐션과 사라진 KV
// 캐시 and §토큰 순서의 이론 (confidence = largest softmax probability);
// "D2F 논문 리뷰: 확산 LLM이 자기회귀 모델보다 빠른 추론을 처음으로 달성한 방식",
// §쉽게 이해하기 (conservative threshold commit, aggressive top-1, remask).
//
// Grid (splits, total_q): CTA (s, r) reduces vocabulary slice s of row r to a
// running (max, first argmax, sum of exp(l - max)) with 128-bit streaming loads.
// The last CTA of a row (arrival counter) composes the slices; the last row of a
// block (second counter) makes the block's commit decision with one warp. There
// is no spin-wait anywhere: arrival counters hand the work to whoever arrives
// last, and every counter is reset by its last arriver so the next call (or a
// graph replay) starts from zero.
#include "d2f_internal.cuh"

namespace d2f {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr float kLog2e = 1.4426950408889634f;

struct RowState {
  float m;    // running maximum
  int idx;    // lowest index attaining m
  float s;    // sum of exp(l - m)
};

__device__ __forceinline__ RowState combine(RowState a, RowState b) {
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
  r.s = a.s * fast_exp2((a.m - r.m) * kLog2e) + b.s * fast_exp2((b.m - r.m) * kLog2e);
  return r;
}

__device__ __forceinline__ RowState warp_combine(RowState v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    RowState w;
    w.m = __shfl_xor_sync(0xffffffffu, v.m, o);
    w.idx = __shfl_xor_sync(0xffffffffu, v.idx, o);
    w.s = __shfl_xor_sync(0xffffffffu, v.s, o);
    v = combine(v, w);
  }
  return v;
}

// Fold N consecutive values starting at index v0 into the thread state. The
// per-lane sums keep N independent accumulation chains.
template <int N>
__device__ __forceinline__ void fold(const float (&x)[N], int v0, float &m, int &idx,
                                     float (&acc)[N]) {
  float vm = x[0];
#pragma unroll
  for (int j = 1; j < N; ++j) vm = fmaxf(vm, x[j]);
  if (vm > m) {
    int first = 0;
#pragma unroll
    for (int j = N - 1; j >= 0; --j)
      if (x[j] == vm) first = j;
    const float alpha = fast_exp2((m - vm) * kLog2e);
#pragma unroll
    for (int j = 0; j < N; ++j) acc[j] *= alpha;
    m = vm;
    idx = v0 + first;
  }
  // x - m is exact in float for bf16 inputs; one rounding in the scale.
#pragma unroll
  for (int j = 0; j < N; ++j) acc[j] += fast_exp2((x[j] - m) * kLog2e);
}

template <int DT>
__device__ __forceinline__ float load_scalar(const void *base, int64_t i) {
  if (DT == D2F_BF16)
    return bf16_bits_to_float(((const uint16_t *)base)[i]);
  return ((const float *)base)[i];
}

// One warp (lane u = row u of the block) decides block jb. Called by all 32
// lanes of one warp after every row of the block has its result.
__device__ void decide_block(const CommitArgs &a, int jb) {
  const int lane = threadIdx.x & 31;
  const int B = a.block_size;
  const int r = jb * B + lane;
  const bool in = lane < B;
  const bool m = in && a.masked[r] != 0;
  float c = -1.0f;
  int am = -1;
  if (m) {
    c = __ldcg(a.row_conf + r);
    am = __ldcg(a.row_arg + r);
  }
  // sequence of the block (q_start values are multiples of B, blocks never straddle)
  int b = 0;
  if (lane == 0) {
    int lo = 0, hi = a.batch - 1;
    const int r0 = jb * B;
    while (lo < hi) {  // largest b with q_start[b] <= r0
      const int mid = (lo + hi + 1) >> 1;
      if (a.q_start[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  b = __shfl_sync(0xffffffffu, b, 0);
  const float t = a.tau[b];
  bool take = m && (c > t);
  const unsigned any_masked = __ballot_sync(0xffffffffu, m);
  if (a.block_phase[jb] == D2F_PHASE_AGGRESSIVE && any_masked) {
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
    if (a.conf_out) a.conf_out[r] = m ? c : -1.0f;
    if (a.argmax_out) a.argmax_out[r] = m ? am : -1;
  }
  if (lane == 0 && a.block_remaining) a.block_remaining[jb] = __popc(left);
}

// Called by warp 0 of the CTA that completed row r.
__device__ void row_done(const CommitArgs &a, int r) {
  const int lane = threadIdx.x & 31;
  const int jb = r / a.block_size;
  int old = 0;
  if (lane == 0) {
    __threadfence();
    old = atomicAdd(a.blk_cnt + jb, 1);
  }
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old != a.block_size - 1) return;
  __threadfence();
  decide_block(a, jb);
  if (lane == 0) a.blk_cnt[jb] = 0;
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads) commit_kernel(const CommitArgs a) {
  const int s = blockIdx.x;
  const int r = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  __shared__ RowState red[kThreads / 32];
  __shared__ int is_last;

  if (a.masked[r] == 0) {
    if (s == 0 && warp == 0) row_done(a, r);
    return;
  }
  int lr = a.logit_row ? a.logit_row[r] : r;
  const bool row_ok = lr >= 0 && lr < a.num_logit_rows;
  if (!row_ok) {
    if (tid == 0 && s == 0) set_err(a.err, D2F_ERR_BAD_INDEX);
    lr = 0;
  }

  // ---- streaming reduction of this CTA's vocabulary slice ------------------
  constexpr int N = (DT == D2F_BF16) ? 8 : 4;  // values per 16-byte vector
  const int v0 = s * a.chunk;
  const int v1 = min(a.vocab, v0 + a.chunk);
  float m = -INFINITY;
  int idx = 0x7fffffff;
  float acc[N];
#pragma unroll
  for (int j = 0; j < N; ++j) acc[j] = 0.f;
  const char *row = (const char *)a.logits + (int64_t)lr * a.row_stride * (DT == D2F_BF16 ? 2 : 4);

  if (row_ok && v0 < v1) {
    int v = v0;
    if (VEC) {
      // v0 and chunk are multiples of N, the row start is 16-byte aligned.
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
          if (DT == D2F_BF16) {
            const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              x[2 * j] = __uint_as_float(w[j] << 16);
              x[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
            }
          } else {
            x[0] = __uint_as_float(raw[u].x);
            x[1] = __uint_as_float(raw[u].y);
            x[2] = __uint_as_float(raw[u].z);
            x[3] = __uint_as_float(raw[u].w);
          }
          fold<N>(x, (k + u * kThreads) * N, m, idx, acc);
        }
      }
      for (; k < nvec_end; k += kThreads) {
        const uint4 raw = __ldcs(vec + k);
        float x[N];
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
        fold<N>(x, k * N, m, idx, acc);
      }
      v = max(v0, nvec_end * N);
    }
    // scalar part (whole slice when not vectorised, else the ragged tail)
    for (int e = v + tid; e < v1; e += kThreads) {
      const float x = load_scalar<DT>(row, e);
      if (x > m) {  // new maximum: rescale every lane accumulator
        const float alpha = fast_exp2((m - x) * kLog2e);
#pragma unroll
        for (int j = 0; j < N; ++j) acc[j] *= alpha;
        m = x;
        idx = e;
      }
      acc[0] += fast_exp2((x - m) * kLog2e);
    }
  }
  float tot = 0.f;
#pragma unroll
  for (int j = 0; j < N; ++j) tot += acc[j];
  RowState st = {m, idx, tot};
  st = warp_combine(st);
  if (lane == 0) red[warp] = st;
  __syncthreads();
  if (warp != 0) return;
  st = lane < kThreads / 32 ? red[lane] : RowState{-INFINITY, 0x7fffffff, 0.f};
  st = warp_combine(st);

  // ---- compose the slices of the row --------------------------------------
  if (a.splits > 1) {
    if (lane == 0) {
      a.partial[(int64_t)r * a.splits + s] =
          make_float4(st.m, __int_as_float(st.idx), st.s, 0.f);
      __threadfence();
      is_last = atomicAdd(a.row_cnt + r, 1) == a.splits - 1;
    }
    __syncwarp();
    if (!__shfl_sync(0xffffffffu, is_last, 0)) return;
    __threadfence();
    RowState acc2 = {-INFINITY, 0x7fffffff, 0.f};
    for (int j = lane; j < a.splits; j += 32) {
      const float4 p = __ldcg(a.partial + (int64_t)r * a.splits + j);
      acc2 = combine(acc2, RowState{p.x, __float_as_int(p.y), p.z});
    }
    st = warp_combine(acc2);
    if (lane == 0) a.row_cnt[r] = 0;
  }
  if (lane == 0) {
    const bool ok = row_ok && st.s > 0.f;
    a.row_conf[r] = ok ? 1.0f / st.s : -1.0f;
    a.row_arg[r] = ok ? st.idx : -1;
  }
  __syncwarp();
  row_done(a, r);
}

}  // namespace

cudaError_t launch_commit(const CommitArgs &a, int dtype, bool vec_ok, cudaStream_t stream) {
  if (a.total_q == 0) return cudaSuccess;
  dim3 grid(a.splits, a.total_q), block(kThreads);
  if (dtype == D2F_BF16) {
    if (vec_ok)
      commit_kernel<D2F_BF16, true><<<grid, block, 0, stream>>>(a);
    else
      commit_kernel<D2F_BF16, false><<<grid, block, 0, stream>>>(a);
  } else {
    if (vec_ok)
      commit_kernel<D2F_F32, true><<<grid, block, 0, stream>>>(a);
    else
      commit_kernel<D2F_F32, false><<<grid, block, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace d2f
