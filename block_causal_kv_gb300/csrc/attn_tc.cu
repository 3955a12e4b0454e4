// Tensor-core path of d2f_block_attn (bf16, head_dim 64 or 128, B in {8,16,32}).
//
// Source of the computation: "D2F: 확산 언어 모델이 KV 캐시를 얻고 자기회귀
// 모델보다 2.5배 빨라지는 방법", §블록 단위 인과 어텐션 (bidirectional inside a
// block, causal between blocks, finished blocks in a KV cache) and §운영 관점
// (paged cache, one block per page); "D2F 논문 리뷰", §쉽게 이해하기 (a window of
// several active blocks decoded together).
//
// One CTA = (row tile of <= 128 query rows, split, sequence x KV head). The
// G = Hq/Hkv query heads of a KV group are packed into the rows (row r = query
// r / G, head r % G), so every K/V byte is read once per row tile. The CTA's key
// tiles (64 keys: 64/B cache pages, or 64/B window blocks) stream through a
// 4-stage shared-memory ring:
//
//   warp 0 (one lane)  TMA producer: page ids -> cp.async.bulk.tensor loads of
//                      the K and V tiles (128-byte swizzle), completion counted
//                      on the stage's mbarrier; slots past the sequence are skipped.
//   warp 1 (one lane)  MMA issuer: S = Q K^T into TMEM (double-buffered), then
//                      O += P V into TMEM once the softmax has written P.
//   warps 2-5          one thread per query row (= TMEM lane): read S from TMEM,
//                      mask, online softmax in log2 units with lazy rescaling
//                      of O (only when the running max grows by > 2^8), write
//                      bf16 P to shared memory for the second MMA.
//
// Splits of one row tile write unnormalised partials; the last-arriving CTA
// composes them in log space. Every mbarrier wait is bounded; on time-out the
// CTA records D2F_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and
// returns.
#include <string.h>

#include <cstdio>
#include <mutex>

#include "attn_common.cuh"

namespace d2f {
namespace {

constexpr int kThreads = 192;
constexpr int NS = 4;             // K/V ring stages
constexpr int M = kTcRows;        // 128 query rows per tile
constexpr int N = kTcKeys;        // 64 keys per tile
constexpr uint32_t kTmemCols = 256;  // S double buffer (2 x 64) + O (<= 128)
constexpr uint32_t kTmemO = 128;     // first TMEM column of O
constexpr int kEpiThreads = 128;

template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;               // 64-element (128-byte) swizzle columns
  static constexpr int kQHalf = M * 128;               // one 64-wide column block of Q
  static constexpr int kQBytes = kHalves * kQHalf;
  static constexpr int kKVHalf = N * 128;              // 64 key rows x 128 bytes
  static constexpr int kKBytes = kHalves * kKVHalf;
  static constexpr int kStage = 2 * kKBytes;           // K tile then V tile
  static constexpr int kPBytes = M * N * 2;            // bf16 P, 128 rows x 128 bytes
  static constexpr int kQ = 0;
  static constexpr int kRing = kQ + kQBytes;
  static constexpr int kP = kRing + NS * kStage;
  static constexpr int kBars = kP + 2 * kPBytes;
  static constexpr int kBytes = kBars + 256;
  static constexpr int kAlloc = kBytes + 1024;          // slack for 1024-byte alignment
};

struct Bars {
  uint64_t full[NS], empty[NS], s_full[2], p_full[2], pv_done[2], drain;
  uint32_t tmem_base;
  int abort_flag;
  int is_last;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tm_kpool,
                   const __grid_constant__ CUtensorMap tm_vpool,
                   const __grid_constant__ CUtensorMap tm_kwin,
                   const __grid_constant__ CUtensorMap tm_vwin) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  Bars *bars = reinterpret_cast<Bars *>(smem + L::kBars);
  volatile int *abort_flag = &bars->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = blockIdx.x, split = blockIdx.y;
  const int b = blockIdx.z / a.num_heads_kv, g = blockIdx.z % a.num_heads_kv;

  // ---- work of this CTA (uniform across the CTA) ----------------------------
  int q0, n, C;
  if (!load_seq_meta(a, b, q0, n, C)) {
    if (tid == 0 && mt == 0 && split == 0 && g == 0) set_err(a.err, D2F_ERR_INVALID_ARG);
    return;
  }
  const int G = a.group, B = a.block_size, H = a.num_heads_q;
  const int rows_total = G * n;
  const int r_begin = mt * M;
  if (r_begin >= rows_total) return;
  const int nrows = min(M, rows_total - r_begin);
  const int Tc = (C + N - 1) / N, Tw = (n + N - 1) / N;
  int t0, t1, s_eff;
  if (!split_range(Tc + Tw, a.num_splits, split, t0, t1, s_eff)) return;
  const int T = t1 - t0;

  // ---- set-up: barriers, TMEM, Q tile ---------------------------------------
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&bars->full[i]), 1);
      mbar_init(smem_u32(&bars->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->s_full[i]), 1);
      mbar_init(smem_u32(&bars->p_full[i]), kEpiThreads);
      mbar_init(smem_u32(&bars->pv_done[i]), 1);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_kpool);
    tma_prefetch_desc(&tm_vpool);
    tma_prefetch_desc(&tm_kwin);
    tma_prefetch_desc(&tm_vwin);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  {
    // Q rows into the 128-byte-swizzled K-major layout the MMA reads:
    // row rr, 16-byte chunk c of column block h lands at
    //   h*kQHalf + (rr/8)*1024 + (rr%8)*128 + ((c ^ (rr%8)) * 16).
    const uint16_t *Q = reinterpret_cast<const uint16_t *>(a.q);
    constexpr int kChunks = D / 8;
    for (int e = tid; e < M * kChunks; e += kThreads) {
      const int rr = e / kChunks, c = e % kChunks;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (rr < nrows) {
        const int r = r_begin + rr;
        const int64_t off = ((int64_t)(q0 + r / G) * H + g * G + r % G) * D + c * 8;
        v = *reinterpret_cast<const uint4 *>(Q + off);
      }
      const int h = c >> 3, cc = c & 7;
      const uint32_t dst =
          sb + L::kQ + h * L::kQHalf + (rr >> 3) * 1024 + (rr & 7) * 128 + ((cc ^ (rr & 7)) << 4);
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(v.x), "r"(v.y),
                   "r"(v.z), "r"(v.w)
                   : "memory");
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ======================= TMA producer ======================================
    if (lane == 0) {
      int issued = 0;
      const int pages_per_tile = N / B;
      for (int u = 0; u < T; ++u) {
        const int stage = u % NS;
        if (u >= NS &&
            !mbar_wait(smem_u32(&bars->empty[stage]), ((u / NS) - 1) & 1, abort_flag, a.err))
          break;
        const uint32_t full = smem_u32(&bars->full[stage]);
        const uint32_t kdst = sb + L::kRing + stage * L::kStage;
        const uint32_t vdst = kdst + L::kKBytes;
        const int t = t0 + u;
        // Source of each B-row slot of the tile: a physical page (cache tiles) or a
        // window row (window tiles); -1 = nothing to load (past the sequence, or a
        // bad page id). Skipped slots keep stale shared memory: their keys are
        // masked and their V rows are cleared by the softmax warps.
        int src[N / 8];
        uint32_t bytes = 0;
        for (int p = 0; p < pages_per_tile; ++p) {
          src[p] = -1;
          if (t < Tc) {
            const int lp = t * pages_per_tile + p;  // logical page of the sequence
            if (lp * B < C) {
              const int pg = a.page_table[(int64_t)b * a.max_pages_per_seq + lp];
              if (pg >= 0 && pg < a.num_pages)
                src[p] = pg;
              else
                set_err(a.err, D2F_ERR_BAD_INDEX);
            }
          } else {
            const int w0 = (t - Tc) * N + p * B;  // first window row of this block
            if (w0 < n) src[p] = q0 + w0;
          }
          if (src[p] >= 0) bytes += 2u * L::kHalves * B * 128;
        }
        mbar_arrive_expect_tx(full, bytes);
        for (int p = 0; p < pages_per_tile; ++p) {
          if (src[p] < 0) continue;
          const uint32_t row_off = p * B * 128;
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h) {
            if (t < Tc) {
              tma_load_4d(kdst + h * L::kKVHalf + row_off, &tm_kpool, full, h * 64, 0, g, src[p]);
              tma_load_4d(vdst + h * L::kKVHalf + row_off, &tm_vpool, full, h * 64, 0, g, src[p]);
            } else {
              tma_load_3d(kdst + h * L::kKVHalf + row_off, &tm_kwin, full, h * 64, g, src[p]);
              tma_load_3d(vdst + h * L::kKVHalf + row_off, &tm_vwin, full, h * 64, g, src[p]);
            }
          }
        }
        issued = u + 1;
      }
      // Drain: every issued stage must have landed before the CTA may exit.
      for (int u = max(0, issued - NS); u < issued; ++u) {
        volatile int no_abort = 0;
        mbar_wait(smem_u32(&bars->full[u % NS]), (u / NS) & 1, &no_abort, a.err);
      }
    }
  } else if (warp == 1) {
    // ======================= MMA issuer ========================================
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(M, N, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(M, D, 0, 1);
      const uint32_t q_base = sb + L::kQ;
      bool ok = true;
      auto issue_pv = [&](int v) -> bool {
        if (!mbar_wait(smem_u32(&bars->p_full[v & 1]), (v >> 1) & 1, abort_flag, a.err))
          return false;
        tc_fence_after();
        const int stage = v % NS;
        const uint32_t p_base = sb + L::kP + (v & 1) * L::kPBytes;
        const uint32_t v_base = sb + L::kRing + stage * L::kStage + L::kKBytes;
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks) {
          const uint64_t ad = smem_desc_sw128(p_base + ks * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(v_base + ks * 2048, L::kKVHalf, 1024);
          umma_bf16(tmem + kTmemO, ad, bd, idesc_pv, (v > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(smem_u32(&bars->pv_done[v & 1]));
        umma_commit(smem_u32(&bars->empty[stage]));
        return true;
      };
      for (int u = 0; u < T && ok; ++u) {
        const int stage = u % NS;
        if (!mbar_wait(smem_u32(&bars->full[stage]), (u / NS) & 1, abort_flag, a.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k_base = sb + L::kRing + stage * L::kStage;
#pragma unroll
        for (int h = 0; h < L::kHalves; ++h) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc_sw128(q_base + h * L::kQHalf + kk * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(k_base + h * L::kKVHalf + kk * 32, 16, 1024);
            umma_bf16(tmem + (u & 1) * N, ad, bd, idesc_qk, (h | kk) ? 1u : 0u);
          }
        }
        umma_commit(smem_u32(&bars->s_full[u & 1]));
        if (u >= 1) ok = issue_pv(u - 1);
      }
      if (ok) issue_pv(T - 1);
      // Drain: wait until every MMA issued above has completed.
      umma_commit(smem_u32(&bars->drain));
      volatile int no_abort = 0;
      mbar_wait(smem_u32(&bars->drain), 0, &no_abort, a.err);
    }
  } else {
    // ======================= softmax / epilogue (128 threads) ====================
    const int quad = warp & 3;            // TMEM lanes 32*quad .. 32*quad+31
    const int row = quad * 32 + lane;     // row of the tile = TMEM lane
    const bool row_valid = row < nrows;
    const int r = r_begin + row;
    const int win_end = row_valid ? ((r / G) / B + 1) * B : 0;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    const float sl2 = a.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;

    for (int u = 0; u < T; ++u) {
      const int t = t0 + u;
      ok = mbar_wait(smem_u32(&bars->s_full[u & 1]), (u >> 1) & 1, abort_flag, a.err);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      uint32_t s_lo[32], s_hi[32];
      tmem_ld32(lane_addr + (u & 1) * N, s_lo);
      tmem_ld32(lane_addr + (u & 1) * N + 32, s_hi);

      // keys c < lim of this tile are visible to this row
      const int tile_lim = t < Tc ? C - t * N : n - (t - Tc) * N;  // valid keys of the tile
      int lim = t < Tc ? tile_lim : win_end - (t - Tc) * N;
      lim = row_valid ? max(0, min(lim, N)) : 0;
      float tmax = -INFINITY;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        if (c < lim) tmax = fmaxf(tmax, __uint_as_float(s_lo[c]) * sl2);
        if (c + 32 < lim) tmax = fmaxf(tmax, __uint_as_float(s_hi[c]) * sl2);
      }
      // Lazy rescale: keep the reference max unless the tile max exceeds it by 2^8.
      const bool need = tmax > m_ref + 8.0f;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? tmax : m_ref;
        const float alpha = need ? fast_exp2(m_ref - m_new) : 1.0f;
        l *= alpha;
        if (u > 0) {
          ok = mbar_wait(smem_u32(&bars->pv_done[(u - 1) & 1]), ((u - 1) >> 1) & 1, abort_flag,
                         a.err);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t o[32];
            tmem_ld32(lane_addr + kTmemO + ch * 32, o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st32(lane_addr + kTmemO + ch * 32, o);
          }
          tmem_wait_st();
        }
        m_ref = m_new;
      }
      // P = 2^(s - m_ref) for visible keys, 0 otherwise, rounded to bf16.
      uint32_t pk[32];
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int c0 = 2 * j, c1 = 2 * j + 1;
        const float p0 = c0 < lim ? fast_exp2(fmaf(__uint_as_float(s_lo[c0]), sl2, -m_ref)) : 0.f;
        const float p1 = c1 < lim ? fast_exp2(fmaf(__uint_as_float(s_lo[c1]), sl2, -m_ref)) : 0.f;
        pk[j] = pack_bf16x2(p0, p1);
        const float p2 = c0 + 32 < lim ? fast_exp2(fmaf(__uint_as_float(s_hi[c0]), sl2, -m_ref)) : 0.f;
        const float p3 = c1 + 32 < lim ? fast_exp2(fmaf(__uint_as_float(s_hi[c1]), sl2, -m_ref)) : 0.f;
        pk[16 + j] = pack_bf16x2(p2, p3);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j)
        psum += __uint_as_float(pk[j] << 16) + __uint_as_float(pk[j] & 0xffff0000u);
      l += psum;

      // The P buffer is free once the MMA that read it two tiles ago completed.
      if (u >= 2) {
        ok = mbar_wait(smem_u32(&bars->pv_done[u & 1]), ((u - 2) >> 1) & 1, abort_flag, a.err);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
      const uint32_t p_row = sb + L::kP + (u & 1) * L::kPBytes + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(p_row + ((c ^ (row & 7)) << 4)),
                     "r"(pk[4 * c]), "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                     : "memory");
      }
      // A ragged tile (partial last page or short window) may hold stale or
      // non-finite V rows past its valid keys; P is 0 there, but 0 * NaN is not
      // 0, so clear those rows before the P.V product reads them.
      if (row < N && row >= tile_lim) {
        const uint32_t v_row = sb + L::kRing + (u % NS) * L::kStage + L::kKBytes +
                               (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
        for (int h = 0; h < L::kHalves; ++h)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(v_row + h * L::kKVHalf +
                                                                           (c << 4)),
                         "r"(0u)
                         : "memory");
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars->p_full[u & 1]));
    }
    if (ok) {
      ok = mbar_wait(smem_u32(&bars->pv_done[(T - 1) & 1]), ((T - 1) >> 1) & 1, abort_flag, a.err);
      ok = __all_sync(0xffffffffu, ok);
    }
    __syncwarp();
    asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
    const bool aborted = *abort_flag != 0;
    if (!aborted) {
      tc_fence_after();
      const int64_t hr = (int64_t)(q0 + r / G) * H + g * G + r % G;
      const int64_t n_hr = (int64_t)a.total_q * H;
      if (s_eff == 1) {
        const float inv = 1.0f / l;
        uint16_t *dst = reinterpret_cast<uint16_t *>(a.out) + hr * D;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(lane_addr + kTmemO + ch * 32, o);
          if (row_valid) {
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              w[j] = pack_bf16x2(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
            uint4 *d4 = reinterpret_cast<uint4 *>(dst + ch * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) d4[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
          }
        }
        if (row_valid && a.lse_out) a.lse_out[hr] = (m_ref + __log2f(l)) * 0.6931471805599453f;
      } else {
        float *dst = a.ws_o + ((int64_t)split * n_hr + hr) * D;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(lane_addr + kTmemO + ch * 32, o);
          if (row_valid) {
            uint4 *d4 = reinterpret_cast<uint4 *>(dst + ch * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j) d4[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
          }
        }
        if (row_valid) a.ws_ml[split * n_hr + hr] = make_float2(m_ref, l);
        __threadfence();
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
        int32_t *cnt = a.counters + ((int64_t)blockIdx.z * a.m_tiles + mt);
        if (tid == 64) bars->is_last = atomicAdd(cnt, 1) == s_eff - 1;
        asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
        if (bars->is_last) {
          __threadfence();
          for (int rr = warp - 2; rr < nrows; rr += 4) {
            const int r2 = r_begin + rr;
            const int64_t hr2 = (int64_t)(q0 + r2 / G) * H + g * G + r2 % G;
            merge_head_row<uint16_t, D>(a, hr2, s_eff);
          }
          if (tid == 64) *cnt = 0;
        }
      }
    }
  }

  // ---- teardown ---------------------------------------------------------------
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode(EncodeTiledFn fn, CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims,
            const cuuint64_t *strides, const cuuint32_t *box) {
  const cuuint32_t elem_strides[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims,
                        strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const AttnArgs &a, cudaStream_t s, char *why, size_t why_len) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) {
    snprintf(why, why_len, "cuTensorMapEncodeTiled is not available from the driver");
    return cudaErrorNotSupported;
  }
  CUtensorMap kp, vp, kw, vw;
  const cuuint64_t pool_dims[4] = {(cuuint64_t)D, (cuuint64_t)a.block_size,
                                   (cuuint64_t)a.num_heads_kv, (cuuint64_t)a.num_pages};
  const cuuint64_t pool_strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)a.block_size * D * 2,
                                      (cuuint64_t)a.num_heads_kv * a.block_size * D * 2};
  const cuuint32_t pool_box[4] = {64, (cuuint32_t)a.block_size, 1, 1};
  const cuuint64_t win_dims[3] = {(cuuint64_t)D, (cuuint64_t)a.num_heads_kv, (cuuint64_t)a.total_q};
  const cuuint64_t win_strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.num_heads_kv * D * 2};
  const cuuint32_t win_box[3] = {64, 1, (cuuint32_t)a.block_size};
  if (!encode(fn, &kp, a.k_pool, 4, pool_dims, pool_strides, pool_box) ||
      !encode(fn, &vp, a.v_pool, 4, pool_dims, pool_strides, pool_box) ||
      !encode(fn, &kw, a.k_win, 3, win_dims, win_strides, win_box) ||
      !encode(fn, &vw, a.v_win, 3, win_dims, win_strides, win_box)) {
    snprintf(why, why_len, "cuTensorMapEncodeTiled rejected a K/V tensor (alignment or size)");
    return cudaErrorInvalidValue;
  }
  const int smem = Layout<D>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.m_tiles, a.num_splits, a.batch * a.num_heads_kv), block(kThreads);
  attn_tc_kernel<D><<<grid, block, smem, s>>>(a, kp, vp, kw, vw);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_tc(const AttnArgs &a, cudaStream_t s, char *why, size_t why_len) {
  if (a.batch == 0 || a.total_q == 0) return cudaSuccess;
  if (a.head_dim == 128) return launch_d<128>(a, s, why, why_len);
  if (a.head_dim == 64) return launch_d<64>(a, s, why, why_len);
  snprintf(why, why_len, "tensor-core path supports head_dim 64 or 128");
  return cudaErrorInvalidValue;
}

}  // namespace d2f
