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
// and writes the normalised output and lse. Lanes cover head_dim.
template <typename OutT, int D>
__device__ void merge_head_row(const AttnArgs &a, int64_t hr, int s_eff) {
  const int lane = threadIdx.x & 31;
  constexpr int DPL = (D + 31) / 32;
  const int64_t n_hr = (int64_t)a.total_q * a.num_heads_q;
  float M = -INFINITY;
  for (int s = 0; s < s_eff; ++s) M = fmaxf(M, __ldcg(&a.ws_ml[s * n_hr + hr]).x);
  float L = 0.f;
  float o[DPL];
#pragma unroll
  for (int j = 0; j < DPL; ++j) o[j] = 0.f;
  for (int s = 0; s < s_eff; ++s) {
    const float2 ml = __ldcg(&a.ws_ml[s * n_hr + hr]);
    const float w = (ml.x == -INFINITY) ? 0.f : fast_exp2(ml.x - M);
    L += w * ml.y;
    const float *src = a.ws_o + (s * n_hr + hr) * D;
#pragma unroll
    for (int j = 0; j < DPL; ++j) {
      const int d = lane + 32 * j;
      if (d < D) o[j] += w * __ldcg(src + d);
    }
  }
  const float inv = 1.0f / L;
  OutT *dst = reinterpret_cast<OutT *>(a.out) + hr * D;
#pragma unroll
  for (int j = 0; j < DPL; ++j) {
    const int d = lane + 32 * j;
    if (d < D) store_out<OutT>(dst + d, o[j] * inv);
  }
  if (lane == 0 && a.lse_out) a.lse_out[hr] = (M + __log2f(L)) * 0.6931471805599453f;
}

}  // namespace d2f
