// Pieces shared by the two attention paths (tensor-core and CUDA-core):
// how a sequence's key tiles are split among CTAs, and the log-space
// composition of the split partials.
//
// Composition rule ("확산 언어 모델(Diffusion LLM)이란 무엇인가", §FlashBlock:
// attention parts computed separately are recombined in log space, as in
// FlashAttention): with each part s holding a reference maximum m_s (log2
// units), a sum l_s = sum 2^(x - m_s) and an unnormalised output
// O_s = sum 2^(x - m_s) v, the whole is
//   M = max_s m_s,  L = sum_s 2^(m_s - M) l_s,  out = sum_s 2^(m_s - M) O_s / L,
//   lse = (M + log2 L) * ln 2.
#pragma once

#include "d2f_internal.cuh"

namespace d2f {

// Key tiles of one (sequence, KV head) are [0, Tc) over the cache and
// [Tc, Tc + Tw) over the window. Split s of num_splits takes a contiguous run of
// tiles; every split that exists is non-empty. Returns false for a CTA whose
// split does not exist.
__device__ __forceinline__ bool split_range(int T, int num_splits, int s, int &t0, int &t1,
                                            int &s_eff) {
  const int tps = (T + num_splits - 1) / num_splits;
  s_eff = (T + tps - 1) / tps;
  if (s >= s_eff) return false;
  t0 = s * tps;
  t1 = min(T, t0 + tps);
  return true;
}

template <typename OutT>
__device__ __forceinline__ void store_out(OutT *p, float v);
template <>
__device__ __forceinline__ void store_out<float>(float *p, float v) {
  *p = v;
}
template <>
__device__ __forceinline__ void store_out<uint16_t>(uint16_t *p, float v) {
  *p = float_to_bf16_bits(v);
}

// One warp composes the s_eff partials of head-row hr (= window row * Hq + head)
// and writes the normalised output and lse. Lanes cover head_dim. Every load is
// issued before any is used: lane s reads split s's (max, sum); the partial rows
// of up to kMergeBatch splits are read together.
constexpr int kMergeBatch = 8;
template <typename OutT, int D>
__device__ void merge_head_row(const AttnArgs &a, int64_t hr, int s_eff) {
  const int lane = threadIdx.x & 31;
  constexpr int DPL = (D + 31) / 32;
  const int64_t n_hr = (int64_t)a.total_q * a.num_heads_q;
  // (max, sum) of every split: 32 splits per pass, lane s holds split s
  float M = -INFINITY;
  for (int s0 = 0; s0 < s_eff; s0 += 32) {
    const int s = s0 + lane;
    if (s < s_eff) M = fmaxf(M, __ldcg(&a.ws_ml[s * n_hr + hr]).x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = 0.f;
  float o_acc[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) o_acc[j] = 0.f;
  for (int s0 = 0; s0 < s_eff; s0 += kMergeBatch) {
    float2 ml[kMergeBatch];
    float ov[kMergeBatch][DPL];
#pragma unroll
    for (int q = 0; q < kMergeBatch; ++q) {
      const int s = s0 + q;
      ml[q] = make_float2(-INFINITY, 0.f);
#pragma unroll
      for (int j = 0; j < DPL; ++j) ov[q][j] = 0.f;
      if (s < s_eff) {
        ml[q] = __ldcg(&a.ws_ml[s * n_hr + hr]);
        const float *src = a.ws_o + (s * n_hr + hr) * D;
#pragma unroll
        for (int j = 0; j < DPL; ++j) {
          const int d = lane + 32 * j;
          if (d < D) ov[q][j] = __ldcg(src + d);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kMergeBatch; ++q) {
      const float w = (ml[q].x == -INFINITY) ? 0.f : fast_exp2(ml[q].x - M);
      L += w * ml[q].y;
#pragma unroll
      for (int j = 0; j < DPL; ++j) o_acc[j] = fmaf(w, ov[q][j], o_acc[j]);
    }
  }
  const float inv = 1.0f / L;
  OutT *dst = reinterpret_cast<OutT *>(a.out) + hr * D;
#pragma unroll
  for (int j = 0; j < DPL; ++j) {
    const int d = lane + 32 * j;
    if (d < D) store_out<OutT>(dst + d, o_acc[j] * inv);
  }
  if (lane == 0 && a.lse_out) a.lse_out[hr] = (M + __log2f(L)) * 0.6931471805599453f;
}

}  // namespace d2f
