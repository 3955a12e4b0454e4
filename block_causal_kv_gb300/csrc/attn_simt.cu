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

constexpr int kThreads = 256;
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

// Four consecutive elements (16-byte aligned for float, 8-byte for bf16: the
// offset is a multiple of 4 elements and rows start 16-byte aligned).
__device__ __forceinline__ void ld4(const float *p, int64_t i, float (&x)[4]) {
  const float4 v = *reinterpret_cast<const float4 *>(p + i);
  x[0] = v.x;
  x[1] = v.y;
  x[2] = v.z;
  x[3] = v.w;
}
__device__ __forceinline__ void ld4(const uint16_t *p, int64_t i, float (&x)[4]) {
  const uint2 v = *reinterpret_cast<const uint2 *>(p + i);
  x[0] = bf16_bits_to_float(v.x & 0xffffu);
  x[1] = bf16_bits_to_float(v.x >> 16);
  x[2] = bf16_bits_to_float(v.y & 0xffffu);
  x[3] = bf16_bits_to_float(v.y >> 16);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) attn_simt_kernel(const AttnArgs a) {
  constexpr int DPL = D / 32;
  __shared__ float q_s[RPC][D];
  __shared__ float k_s[KT][D + 1];
  __shared__ float v_s[KT][D];
  __shared__ int kvalid[KT];
  __shared__ int kwin[KT];  // window index of the key, or -1 for a cached key
  __shared__ int kpage[KT];  // physical page of a cached key
  __shared__ int is_last;
  __shared__ long long hr_s[RPC];  // head-row of each row of the CTA (composition)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = blockIdx.x, split = blockIdx.y;
  if (tid == 0) D2F_TRACE_MARK(2, 0);
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
  // head h = g*G + r % G. Four elements per load, every load issued up front.
  constexpr int kQv = (RPC * D / 4 + kThreads - 1) / kThreads;  // vector loads per thread
  {
    float qv[kQv][4];
#pragma unroll
    for (int k = 0; k < kQv; ++k) {
      const int e = tid + k * kThreads;
      const int rr = e / (D / 4), d = (e % (D / 4)) * 4;
#pragma unroll
      for (int j = 0; j < 4; ++j) qv[k][j] = 0.f;
      if (e < RPC * D / 4 && rr < nrows) {
        const int r = r_begin + rr;
        ld4(Q, ((int64_t)(q0 + r / G) * H + g * G + r % G) * D + d, qv[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < kQv; ++k) {
      const int e = tid + k * kThreads;
      const int rr = e / (D / 4), d = (e % (D / 4)) * 4;
      if (e < RPC * D / 4) {
#pragma unroll
        for (int j = 0; j < 4; ++j) q_s[rr][d + j] = qv[k][j] * a.scale_log2;
      }
    }
  }

  if (tid == 0) D2F_TRACE_MARK(2, 1);
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
      int ok = 0, w = -1, page = 0;
      if (t < Tc) {
        const int kk = t * KT + c;
        if (kk < C) {
          page = a.page_table[(int64_t)b * a.max_pages_per_seq + kk / B];
          if (page >= 0 && page < a.num_pages) ok = 1;
          else set_err(a.err, D2F_ERR_BAD_INDEX);
        }
      } else {
        w = (t - Tc) * KT + c;
        ok = w < n;
      }
      kvalid[c] = ok;
      kwin[c] = w;
      kpage[c] = page;
    }
    __syncthreads();
    if (tid == 0 && t == t0) D2F_TRACE_MARK(2, 2);
    // Stage the tile four elements at a time; every load's address comes from
    // shared memory, so the loads of a thread are independent of one another.
#pragma unroll
    for (int e = tid; e < KT * (D / 4); e += kThreads) {
      const int c = e / (D / 4), d = (e % (D / 4)) * 4;
      float kv[4] = {0.f, 0.f, 0.f, 0.f}, vv[4] = {0.f, 0.f, 0.f, 0.f};
      if (kvalid[c]) {
        int64_t off;
        const T *ks, *vs;
        if (t < Tc) {
          const int kk = t * KT + c;
          off = (((int64_t)kpage[c] * Hk + g) * B + kk % B) * D + d;
          ks = Kp;
          vs = Vp;
        } else {
          off = ((int64_t)(q0 + kwin[c]) * Hk + g) * D + d;
          ks = Kw;
          vs = Vw;
        }
        ld4(ks, off, kv);
        ld4(vs, off, vv);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        k_s[c][d + j] = kv[j];
        v_s[c][d + j] = vv[j];
      }
    }
    __syncthreads();

    if (tid == 0 && t == t0) D2F_TRACE_MARK(2, 3);
    // The warp's kRowsPerWarp rows advance together (independent chains per lane):
    // lane = key for the scores, lane = output column for P.V.
    const int c = lane;
    float dot[kRowsPerWarp];
#pragma unroll
    for (int ri = 0; ri < kRowsPerWarp; ++ri) dot[ri] = 0.f;
#pragma unroll 8
    for (int d = 0; d < D; ++d) {
      const float kd = k_s[c][d];
#pragma unroll
      for (int ri = 0; ri < kRowsPerWarp; ++ri)
        dot[ri] = fmaf(q_s[warp + kWarps * ri][d], kd, dot[ri]);
    }
    float p[kRowsPerWarp];
#pragma unroll
    for (int ri = 0; ri < kRowsPerWarp; ++ri) {
      const int rr = warp + kWarps * ri;
      const bool ok = rr < nrows && kvalid[c] && (kwin[c] < 0 || kwin[c] < win_end[ri]);
      const float sc = ok ? dot[ri] : -INFINITY;
      float tmax = sc;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
      // a row with no visible key in this tile keeps its state (alpha 1, p 0)
      const bool any = tmax != -INFINITY;
      const float m_new = any ? fmaxf(m[ri], tmax) : m[ri];
      const float alpha = (any && m[ri] != -INFINITY) ? fast_exp2(m[ri] - m_new) : (any ? 0.f : 1.f);
      p[ri] = ok ? fast_exp2(sc - m_new) : 0.f;
      float ps = p[ri];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l[ri] = l[ri] * alpha + ps;
#pragma unroll
      for (int j = 0; j < DPL; ++j) o[ri][j] *= alpha;
      m[ri] = m_new;
    }
#pragma unroll 4
    for (int cc = 0; cc < KT; ++cc) {
      float vv[DPL];
#pragma unroll
      for (int j = 0; j < DPL; ++j) vv[j] = v_s[cc][lane + 32 * j];
#pragma unroll
      for (int ri = 0; ri < kRowsPerWarp; ++ri) {
        const float pc = __shfl_sync(0xffffffffu, p[ri], cc);
#pragma unroll
        for (int j = 0; j < DPL; ++j) o[ri][j] = fmaf(pc, vv[j], o[ri][j]);
      }
    }
  }

  if (tid == 0) D2F_TRACE_MARK(2, 4);
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
  if (tid == 0) D2F_TRACE_MARK(2, 5);
  if (tid == 0) is_last = atomicAdd(cnt, 1) == s_eff - 1;
  __syncthreads();
  if (tid == 0) D2F_TRACE_MARK(2, 6);
  if (!is_last) return;
  __threadfence();
  // Compose every row of the CTA at once: (max, sum) of each (row, split) into
  // shared memory, then one thread per output element, all loads in flight.
  {
    // Scratch over the key/value tiles (every warp is past its last tile):
    // wts [RPC][kMaxMergeSplits + 1] in k_s (weights, then the row's total),
    // mls [RPC * s_eff] (max, sum) pairs in v_s.
    constexpr int kWtsMax = KT * (D + 1) / RPC - 1, kMlsMax = KT * D / (2 * RPC);
    constexpr int kMaxMergeSplits = kWtsMax < kMlsMax ? kWtsMax : kMlsMax;
    float *wts = &k_s[0][0];
    float *mls = &v_s[0][0];
    if (s_eff <= kMaxMergeSplits) {
      for (int e = tid; e < RPC * s_eff; e += kThreads) {
        const int rr = e / s_eff, sp = e % s_eff;
        float2 ml = make_float2(-INFINITY, 0.f);
        if (rr < nrows) {
          const int r = r_begin + rr;
          const int64_t hr = (int64_t)(q0 + r / G) * H + g * G + r % G;
          ml = __ldcg(&a.ws_ml[sp * n_hr + hr]);
        }
        mls[e * 2] = ml.x;
        mls[e * 2 + 1] = ml.y;
      }
      __syncthreads();
      if (tid < RPC) {  // per row: max, weights 2^(m_s - M), total sum, lse
        float M = -INFINITY;
        for (int sp = 0; sp < s_eff; ++sp) M = fmaxf(M, mls[(tid * s_eff + sp) * 2]);
        float L = 0.f;
        for (int sp = 0; sp < s_eff; ++sp) {
          const float m_s = mls[(tid * s_eff + sp) * 2];
          const float w = m_s == -INFINITY ? 0.f : fast_exp2(m_s - M);
          wts[tid * (kMaxMergeSplits + 1) + sp] = w;
          L += w * mls[(tid * s_eff + sp) * 2 + 1];
        }
        wts[tid * (kMaxMergeSplits + 1) + kMaxMergeSplits] = L;
        const int r = r_begin + tid;
        const int64_t hr = (int64_t)(q0 + r / G) * H + g * G + r % G;
        hr_s[tid] = hr;
        if (tid < nrows && a.lse_out) a.lse_out[hr] = (M + __log2f(L)) * 0.6931471805599453f;
      }
      __syncthreads();
      // each thread: kE output elements, four splits per batch of loads
      constexpr int kE = RPC * D / kThreads;
      float acc[kE];
#pragma unroll
      for (int k = 0; k < kE; ++k) acc[k] = 0.f;
      for (int s0 = 0; s0 < s_eff; s0 += 4) {
        float ov[kE][4];
#pragma unroll
        for (int k = 0; k < kE; ++k) {
          const int e = tid + k * kThreads, rr = e / D, d = e % D;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int sp = s0 + q;
            ov[k][q] = (rr < nrows && sp < s_eff)
                           ? __ldcg(a.ws_o + (sp * n_hr + hr_s[rr]) * D + d) : 0.f;
          }
        }
#pragma unroll
        for (int k = 0; k < kE; ++k) {
          const int rr = (tid + k * kThreads) / D;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (s0 + q < s_eff) acc[k] = fmaf(wts[rr * (kMaxMergeSplits + 1) + s0 + q], ov[k][q], acc[k]);
        }
      }
#pragma unroll
      for (int k = 0; k < kE; ++k) {
        const int e = tid + k * kThreads, rr = e / D, d = e % D;
        if (rr < nrows)
          store_out<T>(reinterpret_cast<T *>(a.out) + hr_s[rr] * D + d,
                       acc[k] / wts[rr * (kMaxMergeSplits + 1) + kMaxMergeSplits]);
      }
    } else {
      for (int rr = warp; rr < nrows; rr += kWarps) {
        const int r = r_begin + rr;
        const int64_t hr = (int64_t)(q0 + r / G) * H + g * G + r % G;
        merge_head_row<T, D>(a, hr, s_eff);
      }
    }
  }
  if (tid == 0) *cnt = 0;
  if (tid == 0) D2F_TRACE_MARK(2, 7);
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

#ifdef D2F_TRACE
D2F_TRACE_COPY_FN(d2f_trace_copy_simt)
#endif

}  // namespace d2f
