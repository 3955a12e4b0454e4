// CUDA-core path of d2f_block_attn: float32 operands (and bf16 when the
// tensor-core path is not selected). Plain FFMA dot products, one warp per query
// row, keys staged through shared memory 32 at a time, online softmax in log2
// units, split-KV with log-space composition by the last-arriving CTA.
//
// Source of the mask: "D2F: 확산 언어 모델이 KV 캐시를 얻고 자기회귀 모델보다
// 2.5배 빨라지는 방법", §블록 단위 인과 어텐션 (bidirectional inside a block,
// causal between blocks, finished blocks cached).
#include "attn_common.cuh"

namespace d2f {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int KT = kSimtKeys;
constexpr int RPC = kSimtRows;
constexpr int kRowsPerWarp = RPC / kWarps;

template <typename T>
__device__ __forceinline__ float ld_elem(const T *p, int64_t i);
template <>
__device__ __forceinline__ float ld_elem<float>(const float *p, int64_t i) {
  return p[i];
}
template <>
__device__ __forceinline__ float ld_elem<uint16_t>(const uint16_t *p, int64_t i) {
  return bf16_bits_to_float(p[i]);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) attn_simt_kernel(const AttnArgs a) {
  constexpr int DPL = D / 32;
  __shared__ float q_s[RPC][D];
  __shared__ float k_s[KT][D + 1];
  __shared__ float v_s[KT][D];
  __shared__ int kvalid[KT];
  __shared__ int kwin[KT];  // window index of the key, or -1 for a cached key
  __shared__ int is_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = blockIdx.x, split = blockIdx.y;
  const int b = blockIdx.z / a.num_heads_kv, g = blockIdx.z % a.num_heads_kv;
  int q0, n, C;
  if (!load_seq_meta(a, b, q0, n, C)) {
    if (tid == 0 && mt == 0 && split == 0 && g == 0) set_err(a.err, D2F_ERR_INVALID_ARG);
    return;
  }
  const int G = a.group, B = a.block_size, H = a.num_heads_q, Hk = a.num_heads_kv;
  const int rows_total = G * n;
  const int r_begin = mt * RPC;
  if (r_begin >= rows_total) return;
  const int nrows = min(RPC, rows_total - r_begin);
  const int Tc = (C + KT - 1) / KT, Tw = (n + KT - 1) / KT;
  int t0, t1, s_eff;
  if (!split_range(Tc + Tw, a.num_splits, split, t0, t1, s_eff)) return;

  const T *Q = reinterpret_cast<const T *>(a.q);
  const T *Kw = reinterpret_cast<const T *>(a.k_win);
  const T *Vw = reinterpret_cast<const T *>(a.v_win);
  const T *Kp = reinterpret_cast<const T *>(a.k_pool);
  const T *Vp = reinterpret_cast<const T *>(a.v_pool);

  // Query rows of this CTA, pre-scaled into log2 units. Row r -> query i = r / G,
  // head h = g*G + r % G.
  for (int e = tid; e < RPC * D; e += kThreads) {
    const int rr = e / D, d = e % D;
    float v = 0.f;
    if (rr < nrows) {
      const int r = r_begin + rr;
      const int64_t off = ((int64_t)(q0 + r / G) * H + g * G + r % G) * D + d;
      v = ld_elem(Q, off) * a.scale_log2;
    }
    q_s[rr][d] = v;
  }

  float m[kRowsPerWarp], l[kRowsPerWarp], o[kRowsPerWarp][DPL];
  int win_end[kRowsPerWarp];
#pragma unroll
  for (int ri = 0; ri < kRowsPerWarp; ++ri) {
    m[ri] = -INFINITY;
    l[ri] = 0.f;
#pragma unroll
    for (int j = 0; j < DPL; ++j) o[ri][j] = 0.f;
    const int r = r_begin + warp + kWarps * ri;
    const int i = r / G;
    win_end[ri] = (i / B + 1) * B;  // window keys visible to query i: [0, win_end)
  }

  for (int t = t0; t < t1; ++t) {
    __syncthreads();
    if (tid < KT) {
      const int c = tid;
      int ok = 0, w = -1;
      if (t < Tc) {
        const int kk = t * KT + c;
        if (kk < C) {
          const int page = a.page_table[(int64_t)b * a.max_pages_per_seq + kk / B];
          if (page >= 0 && page < a.num_pages) ok = 1;
          else set_err(a.err, D2F_ERR_BAD_INDEX);
        }
      } else {
        w = (t - Tc) * KT + c;
        ok = w < n;
      }
      kvalid[c] = ok;
      kwin[c] = w;
    }
    __syncthreads();
    for (int e = tid; e < KT * D; e += kThreads) {
      const int c = e / D, d = e % D;
      float kv = 0.f, vv = 0.f;
      if (kvalid[c]) {
        int64_t off;
        if (t < Tc) {
          const int kk = t * KT + c;
          const int page = a.page_table[(int64_t)b * a.max_pages_per_seq + kk / B];
          off = (((int64_t)page * Hk + g) * B + kk % B) * D + d;
          kv = ld_elem(Kp, off);
          vv = ld_elem(Vp, off);
        } else {
          off = ((int64_t)(q0 + kwin[c]) * Hk + g) * D + d;
          kv = ld_elem(Kw, off);
          vv = ld_elem(Vw, off);
        }
      }
      k_s[c][d] = kv;
      v_s[c][d] = vv;
    }
    __syncthreads();

#pragma unroll
    for (int ri = 0; ri < kRowsPerWarp; ++ri) {
      const int rr = warp + kWarps * ri;
      if (rr >= nrows) continue;  // warp-uniform
      const int c = lane;
      const bool ok = kvalid[c] && (kwin[c] < 0 || kwin[c] < win_end[ri]);
      float sc = -INFINITY;
      if (ok) {
        float dot = 0.f;
#pragma unroll 8
        for (int d = 0; d < D; ++d) dot = fmaf(q_s[rr][d], k_s[c][d], dot);
        sc = dot;
      }
      float tmax = sc;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
      if (tmax == -INFINITY) continue;  // no visible key in this tile for this row
      const float m_new = fmaxf(m[ri], tmax);
      const float alpha = fast_exp2(m[ri] - m_new);  // 0 when m was -inf
      const float p = ok ? fast_exp2(sc - m_new) : 0.f;
      float ps = p;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l[ri] = l[ri] * alpha + ps;
#pragma unroll
      for (int j = 0; j < DPL; ++j) o[ri][j] *= alpha;
#pragma unroll 4
      for (int cc = 0; cc < KT; ++cc) {
        const float pc = __shfl_sync(0xffffffffu, p, cc);
#pragma unroll
        for (int j = 0; j < DPL; ++j) o[ri][j] = fmaf(pc, v_s[cc][lane + 32 * j], o[ri][j]);
      }
      m[ri] = m_new;
    }
  }

  // ---- epilogue: final output, or a partial plus the log-space composition ----
  const int64_t n_hr = (int64_t)a.total_q * H;
#pragma unroll
  for (int ri = 0; ri < kRowsPerWarp; ++ri) {
    const int rr = warp + kWarps * ri;
    if (rr >= nrows) continue;
    const int r = r_begin + rr;
    const int64_t hr = (int64_t)(q0 + r / G) * H + g * G + r % G;
    if (s_eff == 1) {
      const float inv = 1.0f / l[ri];
      T *dst = reinterpret_cast<T *>(a.out) + hr * D;
#pragma unroll
      for (int j = 0; j < DPL; ++j) store_out<T>(dst + lane + 32 * j, o[ri][j] * inv);
      if (lane == 0 && a.lse_out) a.lse_out[hr] = (m[ri] + __log2f(l[ri])) * 0.6931471805599453f;
    } else {
      float *dst = a.ws_o + ((int64_t)split * n_hr + hr) * D;
#pragma unroll
      for (int j = 0; j < DPL; ++j) dst[lane + 32 * j] = o[ri][j];
      if (lane == 0) a.ws_ml[split * n_hr + hr] = make_float2(m[ri], l[ri]);
    }
  }
  if (s_eff == 1) return;
  __threadfence();
  __syncthreads();
  int32_t *cnt = a.counters + ((int64_t)blockIdx.z * a.m_tiles + mt);
  if (tid == 0) is_last = atomicAdd(cnt, 1) == s_eff - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int rr = warp; rr < nrows; rr += kWarps) {
    const int r = r_begin + rr;
    const int64_t hr = (int64_t)(q0 + r / G) * H + g * G + r % G;
    merge_head_row<T, D>(a, hr, s_eff);
  }
  if (tid == 0) *cnt = 0;
}

template <typename T>
cudaError_t launch_t(const AttnArgs &a, cudaStream_t s) {
  dim3 grid(a.m_tiles, a.num_splits, a.batch * a.num_heads_kv), block(kThreads);
  switch (a.head_dim) {
    case 32: attn_simt_kernel<T, 32><<<grid, block, 0, s>>>(a); break;
    case 64: attn_simt_kernel<T, 64><<<grid, block, 0, s>>>(a); break;
    case 128: attn_simt_kernel<T, 128><<<grid, block, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_simt(const AttnArgs &a, int dtype, cudaStream_t s) {
  if (a.batch == 0 || a.total_q == 0) return cudaSuccess;
  return dtype == D2F_BF16 ? launch_t<uint16_t>(a, s) : launch_t<float>(a, s);
}

}  // namespace d2f
