// Tensor-core path of d2f_block_attn (bf16, head_dim 64 or 128, B in {8,16,32}).
//
// Source of the computation: "D2F: 확산 언어 모델이 KV 캐시를 얻고 자기회귀
// 모델보다 2.5배 빨라지는 방법", §블록 단위 인과 어텐션 (bidirectional inside a
// block, causal between blocks, finished blocks in a KV cache) and §운영 관점
// (paged cache, one block per page); "D2F 논문 리뷰", §쉽게 이해하기 (a window of
// several active blocks decoded together); "확산 언어 모델(Diffusion LLM)이란
// 무엇인가", §FlashBlock (attention parts recombined in log space).
//
// Work decomposition. A row tile is <= QR query rows of one (sequence, KV
// head): the G = Hq/Hkv query heads of the group are packed into the rows
// (row r = query r / G, head r % G), so every K/V byte is read once per row
// tile. QR is 128, or 64 when every sequence has at most 64 rows (the Q tile
// then takes half the shared memory and the ring gets a third stage). A CTA
// holds MT row tiles (1, or 2 for GQA groups of 129..384 rows) of one
// (sequence, KV head), each with its own softmax warpgroup, so one K/V tile
// read serves both. The key tiles (64 keys = 64/B cache pages or 64/B window
// blocks, cache first) are split among the `cs` CTAs of one thread-block
// cluster. With MT = 1 a CTA needs at most ~113 KB of shared memory and 256 TMEM
// columns, so two CTAs share an SM and hide each other's latencies. Each CTA
// streams its share through an NS-stage shared-memory ring:
//
//   producers    page ids (requested with the sequence metadata, 32 at a time)
//                -> cp.async.bulk.tensor loads of the K and V tiles, one box per
//                page (or window block) and tensor, 128-byte swizzle, completion
//                counted on an mbarrier. Warp 0; with two row tiles a second
//                warp; with 64-row tiles also the two softmax warps whose TMEM
//                lanes hold no rows. A tile's boxes are spread over lanes and
//                warps: one thread issues a copy only every ~170 cycles.
//   warps 1..MT  MMA issuers, one lane per row tile (warp 1 also owns TMEM):
//                S = Q K^T into TMEM (double-buffered), then O += P V with P read
//                from TMEM. One thread issues a tcgen05.mma only every ~100
//                cycles whatever its N, so each row tile has its own issuer.
//   softmax      one warpgroup per row tile, one thread per query row
//                (TMEM lane = row): read the row's 64 scores, apply the
//                block-causal mask as a per-row key limit, online softmax in log2
//                units with lazy rescaling of O (only when the running max grows
//                by more than 2^8), write bf16 P over the scores it came from
//                (TMEM columns 0-31 of the S buffer), where the second MMA reads
//                its A operand.
//
// TMEM columns of warpgroup w: [w*(128+D), +64) and [+64, +128) the two S/P
// buffers, then D columns of O.
//
// The MMA always has M = 128: with a 64-row Q tile, A rows 64-127 read whatever
// shared memory follows the tile. Rows 64-127 of S, P and O are never read back
// (their TMEM lanes belong to warps that load K/V instead).
//
// Composition. With cs > 1 every CTA writes its rows, normalised (O / l, bf16)
// with their (max, sum), into a staging block per owning CTA (row r -> CTA
// r mod cs), in its own shared memory (over its ring: every CTA is done with it).
// One cluster barrier publishes the blocks; each owner reads its block from
// every CTA of the cluster straight from that CTA's shared memory, composes its
// rows in log space and writes the output; a closing cluster barrier keeps the
// blocks alive until every owner has read them. No partial goes to global
// memory.
//
// Set-up that reads no global memory (mbarriers, TMEM) runs before the
// grid-dependency wait, so under programmatic dependent launch it overlaps the
// previous kernel. Every mbarrier wait is bounded; on time-out the CTA records
// D2F_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and returns.
#include <string.h>

#include <cstdio>
#include <mutex>

#include "attn_common.cuh"

namespace d2f {
namespace {

constexpr int kWgThreads = 128;                // one softmax warpgroup: a thread per TMEM lane
constexpr int M = kTcRows;                     // UMMA M: 128 rows
constexpr int N = kTcKeys;                     // 64 keys per tile
constexpr uint32_t kTmemO = 128;               // O within a warpgroup's columns (S / P: 2 x 64 before it)
constexpr int kMaxCluster = 8;
constexpr int kBarSetup = 1;                   // named barrier: MMA warp + softmax warps
constexpr int kBarSk = 2;                      // named barrier: the softmax warps (stream-K form)
constexpr int kSmemTwoPerSm = 115712;          // dynamic bytes that still let 2 CTAs share an SM
static_assert(kMaxLongestFirstBatch * 4 + 4 <= 2 * 64 * 64 * 2, "ordering scratch fits a ring stage");

template <int D, int NS, int QR, int MT>
struct Layout {
  static constexpr int kHalves = D / 64;         // 64-element (128-byte) swizzle columns
  static constexpr int kQHalf = QR * 128;        // one 64-wide column block of one Q tile
  static constexpr int kTileQBytes = kHalves * kQHalf;
  static constexpr int kQBytes = MT * kTileQBytes;  // MT row tiles of Q
  // TMEM: per warpgroup, two S / P buffers of 64 columns, then D columns of O
  static constexpr uint32_t kWgCols = 128 + D;
  static constexpr uint32_t kTmemCols = MT * kWgCols <= 256 ? 256 : 512;
  // A K or V tile of 64 keys: eight 8-key groups, each kHalves blocks of 8 rows x
  // 128 bytes (one 64-column half), group-major. A page (B / 8 groups, both
  // halves) is then contiguous, one TMA box, and the MMA reads half h of all 64
  // keys at a uniform 8-row stride.
  static constexpr int kGroupBytes = kHalves * 1024;
  static constexpr int kKBytes = 8 * kGroupBytes;
  static constexpr int kStage = 2 * kKBytes;     // K tile then V tile
  static constexpr int kQ = 0;
  static constexpr int kRing = kQ + kQBytes;
  static constexpr int kBars = kRing + NS * kStage;
  static constexpr int kBytes = kBars + 256;
  // 1024 bytes of slack to align the base by hand, unless that would cost the
  // second CTA per SM; then the kernel checks the base it was given instead.
  static constexpr int kAlloc =
      (kBytes + 1024 <= kSmemTwoPerSm || kBytes > kSmemTwoPerSm) ? kBytes + 1024 : kBytes;
  static constexpr int kCtasPerSm = kAlloc <= kSmemTwoPerSm ? 2 : 1;
  // Warp roles: warp 0 producer; then the MMA issuers: one per row tile, or,
  // for one row tile at one CTA per SM, one for S and one for P.V (kSplit);
  // with MT = 2 a second producer warp; then MT softmax warpgroups. With
  // QR = 64 the two softmax warps whose TMEM lanes (64-127) hold no rows load
  // K/V as well.
  static constexpr bool kSplit = MT == 1 && kCtasPerSm == 1;
  static constexpr int kIssuers = kSplit ? 2 : MT;
  static constexpr int kFirstSoft = 1 + kIssuers + (MT == 2 ? 1 : 0);
  static constexpr int kThreads = 32 * kFirstSoft + kWgThreads * MT;
  static constexpr int kSoftWarps = 4 * MT;
  static constexpr int kProducers = 1 + (MT == 2 ? 1 : 0) + (QR == 64 ? 2 : 0);
  // Composition blocks (overlay Q and the ring): per owner, LR rows of D bf16
  // then LR (max, sum) pairs.
  static constexpr int kRowBytes = 2 * D;
  __host__ __device__ static constexpr int rows_per_owner(int cs) { return (MT * QR + cs - 1) / cs; }
  __host__ __device__ static constexpr int block_bytes(int cs) {
    return (rows_per_owner(cs) * (kRowBytes + 8) + 15) & ~15;
  }
  __host__ __device__ static constexpr int staging(int) { return 0; }  // over Q and the ring
  static_assert((MT * QR + kMaxCluster - 1) * (kRowBytes + 8) + 16 * kMaxCluster <= kBars,
                "staging blocks must fit in the Q + ring area");
  static_assert(MT == 1 || MT == 2, "one or two softmax warpgroups");
  static_assert(MT * kWgCols <= 512, "S / P buffers and accumulators fit TMEM");
  static_assert(kAlloc <= 232448, "shared memory per CTA");
};

constexpr int kMaxStages = 6;

#ifdef D2F_TRACE
// Development build only: SM clock at points of the first 64 key tiles of CTA
// (0, 0, 0), per actor (0/1: first thread of softmax warpgroup 0/1, 2: MMA).
static __device__ long long g_d2f_pass[3][8][64];
#define D2F_PASS_MARK(actor, point, u)                                                   \
  do {                                                                                   \
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && (u) < 64)               \
      g_d2f_pass[actor][point][u] = clock64();                                           \
  } while (0)
#else
#define D2F_PASS_MARK(actor, point, u) ((void)0)
#endif

struct Bars {
  // s_full / p_full / pv_done: [warpgroup][S/P buffer]
  uint64_t full[kMaxStages], empty[kMaxStages], s_full[2][2], p_full[2][2], pv_done[2][2], q_full,
      drain;
  uint32_t tmem_base;
  int abort_flag;
  int sk[6];  // stream-K form: the share's first (sequence, KV head, tile), length, W (lo, hi)
};
static_assert(sizeof(Bars) <= 256, "barrier block");

template <int D, int NS, int QR, int MT>
__global__ void __launch_bounds__((Layout<D, NS, QR, MT>::kThreads),
                                  (Layout<D, NS, QR, MT>::kCtasPerSm))
    attn_tc_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tm_kpool,
                   const __grid_constant__ CUtensorMap tm_vpool,
                   const __grid_constant__ CUtensorMap tm_kwin,
                   const __grid_constant__ CUtensorMap tm_vwin) {
  using L = Layout<D, NS, QR, MT>;
  static_assert(NS >= 2 && NS <= kMaxStages, "ring depth");
  extern __shared__ uint8_t smem_raw[];
  {
    // The swizzled tiles need a 1024-byte aligned base. Every CTA of the grid
    // sees the same placement, so a misfit returns from all of them together.
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if (pad + L::kBytes > dyn) {
      if (threadIdx.x == 0) set_err(a.err, D2F_ERR_UNSUPPORTED);
      return;
    }
  }
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  Bars *bars = reinterpret_cast<Bars *>(smem + L::kBars);
  volatile int *abort_flag = &bars->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cs = gridDim.x;  // CTAs of the cluster = splits of this row tile
  const int split = blockIdx.x;
  const int mt = blockIdx.y;
  int b = blockIdx.z / a.num_heads_kv;  // sequence (remapped longest-first below)
  const int g = blockIdx.z % a.num_heads_kv;

  if (tid == 0) D2F_TRACE_MARK(0, 0);
  // ---- set-up that reads no global memory --------------------------------------
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&bars->full[i]), L::kProducers);
      mbar_init(smem_u32(&bars->empty[i]), MT);  // one release per MMA issuer
    }
    for (int w = 0; w < MT; ++w)
      for (int i = 0; i < 2; ++i) {
        mbar_init(smem_u32(&bars->s_full[w][i]), 1);
        mbar_init(smem_u32(&bars->p_full[w][i]), QR);  // the threads of rows < QR
        mbar_init(smem_u32(&bars->pv_done[w][i]), 1);
      }
    mbar_init(smem_u32(&bars->q_full), QR * MT);
    mbar_init(smem_u32(&bars->drain), L::kIssuers);
    bars->abort_flag = 0;
    mbar_fence_init();  // the initialised barriers, visible at cluster scope
    tma_prefetch_desc(&tm_kpool);
    tma_prefetch_desc(&tm_vpool);
    tma_prefetch_desc(&tm_kwin);
    tma_prefetch_desc(&tm_vwin);
  }
  __syncthreads();
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), L::kTmemCols);
    tmem_relinquish();
  }

  // L2 prefetch of this split's first cached pages while the previous kernel in
  // the stream finishes. The ids and the context length read here are hints only
  // (L2-only loads, nothing cached in L1; ids clamped to the pool): if the
  // previous kernel changes them, a prefetch is wasted, and every value the
  // attention uses is read again after the dependency wait. L2 is the point of
  // coherence, so a prefetched line never hides a later write. Only where the
  // split's whole key range fits in the ring's first fill: there the prefetch
  // shortens the latency chain (LLaDA layer: 10.4 -> 9.9 us), while over long
  // ranges it only crowds the start (Dream layer 75.6 -> 76.4 us, Long B=16
  // 331.7 -> 334.5 us with it).
  if (warp == 0 && a.page_table != nullptr && !a.longest_first && a.part != 2 &&
      a.tiles_per_split <= NS) {
    const int ppt0 = N / a.block_size;
    const int lp = split * a.tiles_per_split * ppt0 + lane;
    const int hint_c = __ldcg(a.ctx_len + b);
    const int pg = lp < a.max_pages_per_seq
                       ? __ldcg(a.page_table + (int64_t)b * a.max_pages_per_seq + lp) : -1;
    if (lp * a.block_size < hint_c && lp < (split + 1) * a.tiles_per_split * ppt0 && pg >= 0 &&
        pg < a.num_pages) {
      const uint32_t page_bytes = (uint32_t)a.block_size * D * 2;
      const int64_t off = ((int64_t)pg * a.num_heads_kv + g) * page_bytes;
      prefetch_l2(static_cast<const char *>(a.k_pool) + off, page_bytes);
      prefetch_l2(static_cast<const char *>(a.v_pool) + off, page_bytes);
    }
  }

  // producer index of this warp (-1: not a producer)
  const int prod = warp == 0 ? 0
                   : (MT == 2 && warp == 1 + MT) ? 1
                   : (QR == 64 && warp >= L::kFirstSoft && (warp & 3) >= 2) ? 1 + (MT == 2) + ((warp & 3) - 2)
                   : -1;
  // D2F_ATTN_CACHE_READY: the page table, context lengths, window layout and
  // cached pages are final before the previous kernel started, so every thread
  // may read them before waiting for it. The producers load cached tiles early
  // and wait before their first window tile or once the ring is full; the softmax
  // warps wait just before they load Q; the MMA issuers read no global memory.
  // Every other read (Q, window K/V) and every write comes after a wait.
  const bool early = a.cache_ready != 0;
  bool waited = !early;
  if (!early) grid_dependency_wait();  // inputs may come from the previous kernel in the stream
  if (tid == 0) D2F_TRACE_MARK(0, 1);

  if (a.longest_first) {
    // More CTAs than resident slots and sequences of different lengths: take the
    // sequences longest context first (ties by index), so the long CTAs start in
    // the first wave and the short ones fill in after them. Every CTA derives the
    // same permutation from the same ctx_len values. Scratch: ring stage 0, which
    // no copy has touched yet.
    int *scr = reinterpret_cast<int *>(smem + L::kRing);
    for (int j = tid; j < a.batch; j += L::kThreads) scr[j] = __ldg(a.ctx_len + j);
    __syncthreads();
    const int want = b;  // this CTA takes the sequence of rank `want`
    for (int j = tid; j < a.batch; j += L::kThreads) {
      const int cj = scr[j];
      int rank = 0;
      for (int i = 0; i < a.batch; ++i) {
        const int ci = scr[i];
        rank += (ci > cj || (ci == cj && i < j)) ? 1 : 0;
      }
      if (rank == want) scr[kMaxLongestFirstBatch] = j;
    }
    __syncthreads();
    b = scr[kMaxLongestFirstBatch];
    __syncthreads();  // stage 0 is free for the copies again
  }

  // Page ids of this split's first tiles, requested together with the sequence
  // metadata: the split's tile range comes from the host (tiles_per_split), so
  // its first logical page is known up front.
  const int ppt = N / a.block_size;  // pages (or window blocks) per tile
  const int pre_chunk = split * a.tiles_per_split * ppt;
  int pre_ids = -1;
  if (prod >= 0 && pre_chunk + lane < a.max_pages_per_seq)
    pre_ids = __ldg(a.page_table + (int64_t)b * a.max_pages_per_seq + pre_chunk + lane);

  // ---- work of this CTA (uniform across the cluster except has_work) ---------
  int q0 = 0, n = 0, C = 0;
  bool active = load_seq_meta(a, b, q0, n, C);
  if (!active && tid == 0 && mt == 0 && split == 0 && g == 0) set_err(a.err, D2F_ERR_INVALID_ARG);
  const int G = a.group, B = a.block_size, H = a.num_heads_q;
  const int rows_total = G * n;
  const int r_begin = mt * MT * QR;  // first of the MT row tiles of this CTA
  active = active && r_begin < rows_total;
  const int nrows = active ? min(MT * QR, rows_total - r_begin) : 0;  // valid rows, all tiles
  const int mt_live = (nrows + QR - 1) / QR;  // row tiles of this CTA that hold rows
  // key tiles: the cached tokens', then the window's (one part only, if asked)
  const int Tc = a.part == 2 ? 0 : (C + N - 1) / N, Tw = a.part == 1 ? 0 : (n + N - 1) / N;
  // Split s takes tiles [s*tps, (s+1)*tps); tps comes from the host's max_ctx and
  // grows here only if a sequence is longer than that hint promised.
  const int tps = max(a.tiles_per_split, (Tc + Tw + cs - 1) / cs);
  const int t0 = split * tps, t1 = min(Tc + Tw, t0 + tps);
  const bool has_work = active && t0 < t1;
  const int T = has_work ? t1 - t0 : 0;
  grid_launch_dependents();

  uint32_t tmem = 0;
  if (active && warp >= 1) {  // TMEM address, published by warp 1
    tc_fence_before();
    named_sync(kBarSetup, L::kThreads - 32);
    tc_fence_after();
    tmem = bars->tmem_base;
  }
  if (tid == 0) D2F_TRACE_MARK(0, 2);

  // softmax-thread identity (warps 1+MT..): warpgroup wg takes row tile wg of the
  // CTA; row = TMEM lane (a warp reaches lanes 32 * (warp % 4) .. + 31)
  const int wg = warp >= L::kFirstSoft ? (warp - L::kFirstSoft) >> 2 : 0;
  const int quad = warp & 3;
  const int row = quad * 32 + lane;
  const int lrow = wg * QR + row;  // row of the CTA's MT row tiles
  const int r = r_begin + lrow;
  const bool rv = row < QR && lrow < nrows;
  const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16) + wg * L::kWgCols;
  float m_ref = -INFINITY, l = 0.f;

  if (has_work && prod >= 0) {
    // ======================= TMA producers (whole warps) ========================
    // A tile is 2 x ppt boxes, box i = (tensor i / ppt: 0 = K, 1 = V; slot
    // i % ppt: page or window block), B rows x D columns each. Producer `prod`
    // takes boxes prod, prod + kProducers, ..., one per lane. A thread's
    // bulk-tensor copies issue one after another (~170 cycles each, measured on
    // GB300), so the boxes of a tile are spread over lanes and warps.
    constexpr int NP = L::kProducers;
    const int box = prod + NP * lane;
    const bool lane_on = box < 2 * ppt;
    const int tensor = lane_on ? box / ppt : 0, slot = lane_on ? box % ppt : 0;
    const int n_pages = (C + B - 1) / B;          // cached pages of the sequence
    const int p_first = t0 * ppt;                 // first logical page of this CTA
    const int32_t *pt = a.page_table + (int64_t)b * a.max_pages_per_seq;
    auto fetch = [&](int base) -> int {
      const int lp = base + lane;
      return (lp < n_pages && lp < p_first + T * ppt) ? __ldg(pt + lp) : -1;
    };
    int chunk = pre_chunk;                        // logical page held by lane 0 of ids_cur
    int ids_cur = pre_ids;
    if (chunk != p_first) {                       // the host's range hint did not hold
      chunk = p_first;
      ids_cur = fetch(chunk);
    }
    int ids_next = fetch(chunk + 32);
    int issued = 0;
    for (int u = 0; u < T; ++u) {
      const int stage = u % NS;
      const int t = t0 + u;
      if (!waited && (t >= Tc || u >= NS)) {  // warp-uniform
        grid_dependency_wait();
        waited = true;
      }
      if (u >= NS) {
        bool ok = true;
        if (lane == 0)
          ok = mbar_wait(smem_u32(&bars->empty[stage]), ((u / NS) - 1) & 1, abort_flag, a.err, a.wait_cycles);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      }
      // Source of this lane's slot: a physical page or a window row; -1 = nothing
      // to load (past the sequence, or a bad page id). Skipped slots keep stale
      // shared memory: their keys are masked and their V rows cleared.
      int src = -1;
      if (t < Tc) {
        const int lp0 = t * ppt;
        if (lp0 - chunk >= 32) {                  // warp-uniform: move to the next 32 ids
          chunk += 32;
          ids_cur = ids_next;
          ids_next = fetch(chunk + 32);
        }
        const int pg = __shfl_sync(0xffffffffu, ids_cur, (lp0 - chunk + slot) & 31);
        if (lane_on && (lp0 + slot) * B < C) {
          if (pg >= 0 && pg < a.num_pages)
            src = pg;
          else
            set_err(a.err, D2F_ERR_BAD_INDEX);
        }
      } else if (lane_on) {
        const int w0 = (t - Tc) * N + slot * B;   // first window row of this block
        if (w0 < n) src = q0 + w0;
      }
      if (lane == 0 && prod == 0) D2F_PASS_MARK(2, 6, u);
      const unsigned have = __ballot_sync(0xffffffffu, src >= 0);
      const uint32_t full = smem_u32(&bars->full[stage]);
      if (lane == 0) mbar_arrive_expect_tx(full, __popc(have) * (uint32_t)B * D * 2u);
      __syncwarp();
      const uint32_t dst = sb + L::kRing + stage * L::kStage + tensor * L::kKBytes +
                           slot * (B / 8) * L::kGroupBytes;
      if (src >= 0) {
        if (t < Tc)  // page src of KV head g: (page, head) row src * Hkv + g of the pool map
          tma_load_5d(dst, tensor ? &tm_vpool : &tm_kpool, full, 0, 0, 0, 0, src * a.num_heads_kv + g);
        else         // window rows src .. src + B - 1 (src is a multiple of 8)
          tma_load_5d(dst, tensor ? &tm_vwin : &tm_kwin, full, 0, 0, 0, src >> 3, g);
      }
      // Fused append: a window block listed as an append source goes from this
      // stage to its page once the tile has landed (row group 0 only: one CTA per
      // sequence, KV head and window tile stores it). The store has read the
      // stage before this thread can refill it.
      if (a.n_append > 0 && mt == 0 && t >= Tc && src >= 0) {
        bool landed = false;
        // list length: the host's, or (bounded by it) the one in device memory
        const int napp = a.app_n_dev ? min(max(*a.app_n_dev, 0), a.n_append) : a.n_append;
        for (int ap = 0; ap < napp; ++ap) {
          if (__ldg(a.app_src + ap) != src) continue;
          const int dp = __ldg(a.app_dst + ap);
          if (dp < 0 || dp >= a.num_pages) {
            set_err(a.err, D2F_ERR_BAD_INDEX);
            continue;
          }
          if (!landed && !mbar_wait(full, (u / NS) & 1, abort_flag, a.err, a.wait_cycles)) break;
          landed = true;
          tma_store_5d(tensor ? &tm_vpool : &tm_kpool, dst, 0, 0, 0, 0, dp * a.num_heads_kv + g);
        }
        if (landed) {
          bulk_commit_group();
          bulk_wait_group_read0();
        }
      }
      issued = u + 1;
      if (lane == 0 && prod == 0) D2F_PASS_MARK(2, 7, u);
    }
    // Drain: every issued stage must have landed before the CTA moves on, and
    // every fused-append store must be complete.
    bulk_wait_group0();
    if (lane == 0) {
      for (int u = max(0, issued - NS); u < issued; ++u) {
        volatile int no_abort = 0;
        mbar_wait(smem_u32(&bars->full[u % NS]), (u / NS) & 1, &no_abort, a.err, kDrainCycles);
      }
    }
  } else if (has_work && L::kSplit && warp <= 2) {
    // ============ MMA issuers of the one row tile: warp 1 S, warp 2 P.V =========
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(M, N, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(M, D, 0, 1);
      // descriptors of Q and of stage 0's K and V; each MMA advances them by a constant
      const uint64_t q_desc = smem_desc_sw128(sb + L::kQ, 16, 1024);
      const uint64_t k_desc = smem_desc_sw128(sb + L::kRing, 16, L::kGroupBytes);
      const uint64_t v_desc = smem_desc_sw128(sb + L::kRing + L::kKBytes, 1024, L::kGroupBytes);
      bool ok = mbar_wait(smem_u32(&bars->q_full), 0, abort_flag, a.err, a.wait_cycles);
      for (int u = 0; u < T && ok; ++u) {
        const int stage = u % NS;
        ok = mbar_wait(smem_u32(&bars->full[stage]), (u / NS) & 1, abort_flag, a.err, a.wait_cycles);
        if (!ok) break;
        if (warp == 1) {
          // S_u overwrites the S/P buffer of P_{u-2}: its P.V must be complete
          if (u >= 2 && !mbar_wait(smem_u32(&bars->pv_done[0][u & 1]), ((u - 2) >> 1) & 1,
                                   abort_flag, a.err, a.wait_cycles)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kd = smem_desc_advance(k_desc, stage * L::kStage);
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = smem_desc_advance(q_desc, h * L::kQHalf + kk * 32);
              const uint64_t bd = smem_desc_advance(kd, h * 1024 + kk * 32);
              umma_bf16(tmem + (u & 1) * N, ad, bd, idesc_qk, (h | kk) ? 1u : 0u);
            }
          }
          umma_commit(smem_u32(&bars->s_full[0][u & 1]));
        } else {
          if (!mbar_wait(smem_u32(&bars->p_full[0][u & 1]), (u >> 1) & 1, abort_flag, a.err, a.wait_cycles)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t vd = smem_desc_advance(v_desc, stage * L::kStage);
#pragma unroll
          for (int ks = 0; ks < N / 16; ++ks) {
            const uint64_t bd = smem_desc_advance(vd, ks * 2 * L::kGroupBytes);
            umma_bf16_tmem_a(tmem + kTmemO, tmem + (u & 1) * N + ks * 8, bd, idesc_pv,
                             (u > 0 || ks > 0) ? 1u : 0u);
          }
          umma_commit(smem_u32(&bars->pv_done[0][u & 1]));
          umma_commit(smem_u32(&bars->empty[stage]));
        }
      }
      umma_commit(smem_u32(&bars->drain));
      volatile int no_abort = 0;
      mbar_wait(smem_u32(&bars->drain), 0, &no_abort, a.err, kDrainCycles);
    }
  } else if (has_work && !L::kSplit && warp <= MT) {
    // ============ MMA issuer of row tile wi (one lane) ===========================
    // A thread's tcgen05.mma instructions issue one after another, each taking
    // ~100 cycles to issue whatever its N (measured on GB300), so each row tile
    // gets its own issuing warp; the tensor pipe interleaves their MMAs.
    const int wi = warp - 1;
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(M, N, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(M, D, 0, 1);
      // descriptors of this row tile's Q and of stage 0's K and V; each MMA advances
      // them by a constant
      const uint64_t q_desc = smem_desc_sw128(sb + L::kQ + wi * L::kTileQBytes, 16, 1024);
      const uint64_t k_desc = smem_desc_sw128(sb + L::kRing, 16, L::kGroupBytes);
      const uint64_t v_desc = smem_desc_sw128(sb + L::kRing + L::kKBytes, 1024, L::kGroupBytes);
      bool ok = mbar_wait(smem_u32(&bars->q_full), 0, abort_flag, a.err, a.wait_cycles);
      // Key tile u: S goes to S/P buffer u % 2 of warpgroup wi; P.V_u accumulates
      // into warpgroup wi's O.
      auto issue_pv = [&](int u, int i) -> bool {
        if (!mbar_wait(smem_u32(&bars->p_full[i][u & 1]), (u >> 1) & 1, abort_flag, a.err, a.wait_cycles))
          return false;
        tc_fence_after();
        D2F_PASS_MARK(2, 3 + i, u);
        const uint64_t vd = smem_desc_advance(v_desc, (u % NS) * L::kStage);
        const uint32_t tw = tmem + i * L::kWgCols;
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks) {  // 16 keys = 8 TMEM columns of P per step
          const uint64_t bd = smem_desc_advance(vd, ks * 2 * L::kGroupBytes);
          umma_bf16_tmem_a(tw + kTmemO, tw + (u & 1) * N + ks * 8, bd, idesc_pv,
                           (u > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(smem_u32(&bars->pv_done[i][u & 1]));
        return true;
      };
      // P.V of the previous key tile, then release its stage (the stage is free
      // once every issuer has released it)
      auto finish = [&](int u) -> bool {
        if (!issue_pv(u, wi)) return false;
        umma_commit(smem_u32(&bars->empty[u % NS]));
        return true;
      };
      const bool idle = wi >= mt_live;  // a row tile without rows: only release stages
      for (int u = 0; u < T && ok; ++u) {
        const int stage = u % NS;
        if (!mbar_wait(smem_u32(&bars->full[stage]), (u / NS) & 1, abort_flag, a.err, a.wait_cycles)) {
          ok = false;
          break;
        }
        if (idle) {
          mbar_arrive(smem_u32(&bars->empty[stage]));
          continue;
        }
        tc_fence_after();
        if (wi == 0) D2F_PASS_MARK(2, 0, u);
        if (u == 0) D2F_TRACE_MARK(0, 10);
        if (u == T - 1) D2F_TRACE_MARK(0, 3);
        // S_u overwrites the S/P buffer that P_{u-2} occupied: P.V_{u-2} was issued
        // before this (MMAs of one thread execute in order).
        const uint64_t kd = smem_desc_advance(k_desc, stage * L::kStage);
#pragma unroll
        for (int h = 0; h < L::kHalves; ++h) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = smem_desc_advance(q_desc, h * L::kQHalf + kk * 32);
            const uint64_t bd = smem_desc_advance(kd, h * 1024 + kk * 32);
            umma_bf16(tmem + wi * L::kWgCols + (u & 1) * N, ad, bd, idesc_qk, (h | kk) ? 1u : 0u);
          }
        }
        umma_commit(smem_u32(&bars->s_full[wi][u & 1]));
        if (wi == 0) D2F_PASS_MARK(2, 1, u);
        if (u >= 1) ok = finish(u - 1);
        if (u >= 1 && wi == 0) D2F_PASS_MARK(2, 2, u - 1);
      }
      if (ok && !idle) finish(T - 1);
      // Drain: wait until every MMA issued above has completed.
      umma_commit(smem_u32(&bars->drain));
      volatile int no_abort = 0;
      mbar_wait(smem_u32(&bars->drain), 0, &no_abort, a.err, kDrainCycles);
    }
  } else if (has_work) {
    // ============ softmax (a warpgroup per row tile, a thread per TMEM lane) =====
    const bool live = wg < mt_live;  // warpgroup-uniform
    {
      if (!waited) {  // Q may come from the previous kernel
        grid_dependency_wait();
        waited = true;
      }
      // The Q rows into the 128-byte-swizzled K-major layout the MMA reads: in
      // row tile wg, 16-byte chunk c of column block h lands at
      //   wg*kTileQBytes + h*kQHalf + (row/8)*1024 + (row%8)*128 + ((c ^ (row%8)) * 16).
      constexpr int kQc = D / 8;
      if (live && row < QR) {  // warp-uniform
        uint4 qv[kQc];
        const uint4 *src = reinterpret_cast<const uint4 *>(
            reinterpret_cast<const uint16_t *>(a.q) + ((int64_t)(q0 + r / G) * H + g * G + r % G) * D);
#pragma unroll
        for (int c = 0; c < kQc; ++c) qv[c] = rv ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < kQc; ++c) {
          const uint32_t dst = sb + L::kQ + wg * L::kTileQBytes + (c >> 3) * L::kQHalf +
                               (row >> 3) * 1024 + (row & 7) * 128 + (((c & 7) ^ (row & 7)) << 4);
          asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(qv[c].x),
                       "r"(qv[c].y), "r"(qv[c].z), "r"(qv[c].w)
                       : "memory");
        }
        fence_proxy_async_smem();
      }
      mbar_arrive(smem_u32(&bars->q_full));
    }
    const int win_end = rv ? ((r / G) / B + 1) * B : 0;
    const float sl2 = a.scale_log2;
    bool ok = true;
    for (int u = 0; u < T && ok && live; ++u) {
      const int t = t0 + u;
      const int tile_lim = t < Tc ? C - t * N : n - (t - Tc) * N;  // valid keys of the tile
      ok = mbar_wait(smem_u32(&bars->s_full[wg][u & 1]), (u >> 1) & 1, abort_flag, a.err, a.wait_cycles);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      const bool pm = lane == 0 && warp == L::kFirstSoft + 4 * wg;  // first thread of the warpgroup
      if (pm) D2F_PASS_MARK(wg, 0, u);
      if (tid == 128 && u == 0) D2F_TRACE_MARK(0, 4);
      if (tid == 128 && u == 1) D2F_TRACE_MARK(0, 14);
      if (tid == 128 && u == 2) D2F_TRACE_MARK(0, 15);
      if (tid == 128 && u == T - 1) D2F_TRACE_MARK(0, 5);
      uint32_t sv[N];
      const uint32_t s_addr = lane_addr + (u & 1) * N;
      tmem_ld64(s_addr, sv);
      if (pm) D2F_PASS_MARK(wg, 1, u);

      // keys c < lim of this tile are visible to this row
      int lim = t < Tc ? tile_lim : win_end - (t - Tc) * N;
      lim = rv ? max(0, min(lim, N)) : 0;
      float sf[N];
#pragma unroll
      for (int c = 0; c < N; ++c) sf[c] = __uint_as_float(sv[c]);
      if (!__all_sync(0xffffffffu, lim >= N)) {  // ragged tile: hide masked keys
#pragma unroll
        for (int c = 0; c < N; ++c)
          if (c >= lim) sf[c] = -INFINITY;
      }
      // tree maximum of the 64 scores with three-input maxima (scale > 0, so
      // max(s) * scale = max(s * scale)): 64 -> 22 -> 8 -> 3 -> 1
      static_assert(N == 64, "maximum tree shape");
      float t1[22], t2[8];
#pragma unroll
      for (int c = 0; c < 21; ++c) t1[c] = fmax3(sf[3 * c], sf[3 * c + 1], sf[3 * c + 2]);
      t1[21] = sf[63];
#pragma unroll
      for (int c = 0; c < 7; ++c) t2[c] = fmax3(t1[3 * c], t1[3 * c + 1], t1[3 * c + 2]);
      t2[7] = t1[21];
      const float tmax = fmax3(fmax3(t2[0], t2[1], t2[2]), fmax3(t2[3], t2[4], t2[5]),
                               fmaxf(t2[6], t2[7])) * sl2;
      // Lazy rescale: keep the reference max unless the tile max exceeds it by 2^8.
      const bool need = tmax > m_ref + 8.0f;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? tmax : m_ref;
        const float alpha = need ? fast_exp2(m_ref - m_new) : 1.0f;
        l *= alpha;
        if (u > 0) {
          // every earlier P.V (MMAs complete in order) has landed in O
          ok = mbar_wait(smem_u32(&bars->pv_done[wg][(u - 1) & 1]), ((u - 1) >> 1) & 1, abort_flag,
                         a.err, a.wait_cycles);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t o[32];
            const uint32_t oa = lane_addr + kTmemO + ch * 32;
            tmem_ld32(oa, o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st32(oa, o);
          }
          tmem_wait_st();
        }
        m_ref = m_new;
      }
      // P = 2^(s*scale - m_ref) in bf16: the exponent argument is formed in float
      // for a pair of keys at once, rounded to bf16 and exponentiated as a packed
      // pair (P is a bf16 MMA operand, so it carries bf16 precision either way).
      // Masked keys are -inf -> 0. A row with no visible key so far keeps
      // m_ref = -inf: subtract 0 instead.
      if (pm) D2F_PASS_MARK(wg, 2, u);
      const float mb = m_ref == -INFINITY ? 0.f : m_ref;
      uint32_t pk[N / 2];
#pragma unroll
      for (int j = 0; j < N / 2; ++j) {
        float x0, x1;
        fma2_bc(x0, x1, sf[2 * j], sf[2 * j + 1], sl2, -mb);
        pk[j] = ex2_bf16x2(pack_bf16x2(x0, x1));
      }
      // row sum of the P actually used (the rounded values), in float pairs
      float ps0[N / 4], ps1[N / 4];
#pragma unroll
      for (int j = 0; j < N / 4; ++j)
        add2(ps0[j], ps1[j], __uint_as_float(pk[2 * j] << 16),
             __uint_as_float(pk[2 * j] & 0xffff0000u), __uint_as_float(pk[2 * j + 1] << 16),
             __uint_as_float(pk[2 * j + 1] & 0xffff0000u));
#pragma unroll
      for (int w = N / 8; w >= 1; w >>= 1)
#pragma unroll
        for (int c = 0; c < w; ++c)
          add2(ps0[c], ps1[c], ps0[2 * c], ps1[2 * c], ps0[2 * c + 1], ps1[2 * c + 1]);
      l += ps0[0] + ps1[0];
      if (pm) D2F_PASS_MARK(wg, 3, u);
      // P over the scores it came from (this thread's own lane): column c of the
      // S/P buffer now holds keys 2c and 2c+1.
      tmem_st32(s_addr, pk);
      tmem_wait_st();
      if (pm) D2F_PASS_MARK(wg, 4, u);
      // A ragged tile (partial last page or short window) may hold stale or
      // non-finite V rows past its valid keys; P is 0 there, but 0 * NaN is not
      // 0, so clear those rows before the P.V product reads them. Every
      // warpgroup clears them (the same zeros) before its own P.V is issued.
      if (row < N && row >= tile_lim) {
        const uint32_t v_row = sb + L::kRing + (u % NS) * L::kStage + L::kKBytes +
                               (row >> 3) * L::kGroupBytes + (row & 7) * 128;
#pragma unroll
        for (int h = 0; h < L::kHalves; ++h)
#pragma unroll
          for (int c = 0; c < 8; ++c)
            asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(v_row + h * 1024 +
                                                                           (c << 4)),
                         "r"(0u)
                         : "memory");
        fence_proxy_async_smem();
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bars->p_full[wg][u & 1]));
      if (pm) D2F_PASS_MARK(wg, 5, u);
      if (tid == 128 && u == 0) D2F_TRACE_MARK(0, 13);
      if (tid == 128 && u == T - 1) D2F_TRACE_MARK(0, 6);
    }
    if (ok && live) {  // the last P.V product
      const int last = T - 1;
      ok = mbar_wait(smem_u32(&bars->pv_done[wg][last & 1]), (last >> 1) & 1, abort_flag, a.err, a.wait_cycles);
      ok = __all_sync(0xffffffffu, ok);
    }
    tc_fence_after();
  }

  // ---- epilogue ---------------------------------------------------------------
  // A producer that loaded only cached tiles (or had none), an MMA issuer, or a
  // thread without work has not waited yet; the epilogue's writes come after the
  // previous kernel in every thread.
  if (!waited) grid_dependency_wait();
  __syncwarp();
  __syncthreads();  // every role is done; Q and the ring are free
  if (tid == 0) D2F_TRACE_MARK(0, 7);
  const bool aborted = *abort_flag != 0;
  bool tmem_freed = false;
  if (cs == 1) {
    if (warp >= L::kFirstSoft && active && !aborted && __any_sync(0xffffffffu, rv)) {
      const int64_t hr = (int64_t)(q0 + r / G) * H + g * G + r % G;
      // this part's normaliser in log2 units (l = 0: no visible key, e.g. the
      // cached part of a sequence without cached tokens: output 0, lse -inf)
      const bool any = has_work && l > 0.f;
      const float lw = any ? m_ref + __log2f(l) : -INFINITY;
      // composition with a kept cached part: weights 2^(L - M) of the two parts
      float wv = any ? 1.f : 0.f, wp = 0.f, lse2 = lw;
      if (a.prev_lse && rv) {
        const float lp = a.prev_lse[hr] * 1.4426950408889634f;
        const float M = fmaxf(lw, lp);
        if (M > -INFINITY) {
          wv = any ? fast_exp2(lw - M) : 0.f;
          wp = lp > -INFINITY ? fast_exp2(lp - M) : 0.f;
          lse2 = M + __log2f(wv + wp);
          const float rs = 1.0f / (wv + wp);
          wv *= rs;
          wp *= rs;
        }
      }
      const float inv = any ? wv / l : 0.f;
      uint16_t *dst = reinterpret_cast<uint16_t *>(a.out) + hr * D;
      const uint4 *prev = reinterpret_cast<const uint4 *>(
          reinterpret_cast<const uint16_t *>(a.prev_out) + hr * D);
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        if (has_work) {
          tmem_ld32(lane_addr + kTmemO + ch * 32, o);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = 0u;
        }
        if (rv) {
          uint32_t pv[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 q4 = wp > 0.f ? prev[ch * 4 + j] : make_uint4(0, 0, 0, 0);
            pv[4 * j] = q4.x;
            pv[4 * j + 1] = q4.y;
            pv[4 * j + 2] = q4.z;
            pv[4 * j + 3] = q4.w;
          }
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            w[j] = pack_bf16x2(
                fmaf(__uint_as_float(o[2 * j]), inv, wp * bf16_bits_to_float(pv[j] & 0xffffu)),
                fmaf(__uint_as_float(o[2 * j + 1]), inv, wp * bf16_bits_to_float(pv[j] >> 16)));
          uint4 *d4 = reinterpret_cast<uint4 *>(dst + ch * 32);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            d4[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
      }
      if (rv && a.lse_out) a.lse_out[hr] = lse2 * 0.6931471805599453f;
    }
  } else if (active) {
    const int LR = L::rows_per_owner(cs);  // rows a CTA owns (at most)
    const int BS = L::block_bytes(cs);     // one owner's block: LR rows + LR (max, sum)
    const uint32_t stg = sb + L::staging(cs);  // [owner][BS], this CTA's rows
    // 1) stage this CTA's rows: local row lrow (wg*QR + lane row) -> owner
    //    lrow % cs, slot lrow / cs; the 16-byte chunks of a row are XOR-swizzled
    //    by (lrow % 8).
    if (warp >= L::kFirstSoft && __any_sync(0xffffffffu, rv)) {
      const int owner = lrow % cs, lr = lrow / cs, key = lrow & 7;
      const uint32_t blk = stg + owner * BS;
      const bool mine = has_work && !aborted;  // CTA-uniform
      const bool keep = mine && rv && l > 0.f;
      if (mine) {
        const float inv = keep ? 1.0f / l : 0.f;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(lane_addr + kTmemO + ch * 32, o);
          if (keep) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int c = ch * 4 + j;  // 8 bf16 per 16-byte chunk
              const uint32_t dst = blk + lr * L::kRowBytes + ((c ^ key) << 4);
              asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst),
                           "r"(pack_bf16x2(__uint_as_float(o[8 * j]) * inv,
                                           __uint_as_float(o[8 * j + 1]) * inv)),
                           "r"(pack_bf16x2(__uint_as_float(o[8 * j + 2]) * inv,
                                           __uint_as_float(o[8 * j + 3]) * inv)),
                           "r"(pack_bf16x2(__uint_as_float(o[8 * j + 4]) * inv,
                                           __uint_as_float(o[8 * j + 5]) * inv)),
                           "r"(pack_bf16x2(__uint_as_float(o[8 * j + 6]) * inv,
                                           __uint_as_float(o[8 * j + 7]) * inv))
                           : "memory");
            }
          }
        }
      }
      if (rv) {
        const float mx = keep ? m_ref : -INFINITY, sm = keep ? l : 0.f;
        asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(blk + LR * L::kRowBytes + lr * 8),
                     "f"(mx), "f"(sm)
                     : "memory");
      }
    }
    // 2) the cluster barrier publishes every CTA's staged blocks to the cluster
    //    (release / acquire at cluster scope).
    __syncwarp();
    tc_fence_before();
    cluster_sync();
    if (tid == 0) D2F_TRACE_MARK(0, 8);
    if (warp == 1) {  // every O row is staged: TMEM is free for the next grid's CTAs
      tc_fence_after();
      tmem_dealloc(bars->tmem_base, L::kTmemCols);
      tmem_freed = true;
    }
    // 3) compose the rows this CTA owns, reading each source CTA's block for this
    //    owner (block `split` of its staging area) straight from its shared
    //    memory: every warp of the CTA (the producers and issuers are done), LPR
    //    lanes per row, lane c of a row's group holds columns [c * D/LPR,
    //    (c + 1) * D/LPR); every source's chunks of a row are requested before any
    //    is used. Eight lanes per row for 128-row tiles, whose CTAs own many
    //    rows (twice the rows per round, twice the loads per lane: Dream layer
    //    72.3 -> 71.0 us); sixteen for 64-row tiles, whose owners' rows fit one
    //    round either way (LLaDA layer: 9.6 us, 10.5 with eight).
    const uint32_t own_blk = stg + split * BS;  // the same offset in every CTA
    constexpr int kWarps = L::kThreads / 32;
    {
      constexpr int LPR = QR == 128 ? 8 : 16;      // lanes per row
      constexpr int kCols = D / LPR;               // columns per lane
      constexpr int kBytes = 2 * kCols;            // 8, 16 or 32 bytes per lane
      constexpr int kRowsPerWarp = 32 / LPR;
      const int grp = lane / LPR, sub = lane % LPR;
      for (int lr0 = warp * kRowsPerWarp; lr0 * cs + split < nrows; lr0 += kRowsPerWarp * kWarps) {
        const int lr = lr0 + grp;
        const int crow = lr * cs + split;  // CTA row of this lane group
        const bool valid = crow < nrows;
        const int key = crow & 7;
        const int r2 = r_begin + crow;
        const int64_t hr2 = (int64_t)(q0 + r2 / G) * H + g * G + r2 % G;
        // This lane's bytes of the row from every source CTA, requested before
        // the weights are known, so the (max, sum) pairs and the values travel
        // together; a part of weight 0 is skipped below, not loaded on demand.
        uint32_t v[kMaxCluster][kCols / 2];
#pragma unroll
        for (int j = 0; j < kMaxCluster; ++j) {
#pragma unroll
          for (int c = 0; c < kCols / 2; ++c) v[j][c] = 0u;
          if (valid && j < cs) {
            if constexpr (kBytes >= 16) {
#pragma unroll
              for (int h = 0; h < kBytes / 16; ++h) {
                const int chunk = sub * (kBytes / 16) + h;  // 16-byte chunk of the row
                const float4 q =
                    dsmem_ld_f4(dsmem_addr(own_blk + lr * L::kRowBytes + ((chunk ^ key) << 4), j));
                v[j][4 * h] = __float_as_uint(q.x);
                v[j][4 * h + 1] = __float_as_uint(q.y);
                v[j][4 * h + 2] = __float_as_uint(q.z);
                v[j][4 * h + 3] = __float_as_uint(q.w);
              }
            } else {  // half a chunk
              const float2 q = dsmem_ld_f2(
                  dsmem_addr(own_blk + lr * L::kRowBytes + (((sub >> 1) ^ key) << 4) + (sub & 1) * 8, j));
              v[j][0] = __float_as_uint(q.x);
              v[j][1] = __float_as_uint(q.y);
            }
          }
        }
        float2 ml = make_float2(-INFINITY, 0.f);
        if (valid && sub < cs) ml = dsmem_ld_f2(dsmem_addr(own_blk + LR * L::kRowBytes + lr * 8, sub));
        // a kept cached part is one more normalised part: (its lse in log2 units, 1)
        const float lp = (a.prev_lse && valid) ? a.prev_lse[hr2] * 1.4426950408889634f : -INFINITY;
        float mx = fmaxf(ml.x, lp);
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        // weight of a normalised part: 2^(m_j - M) * l_j
        const float w = (sub < cs && ml.y > 0.f) ? fast_exp2(ml.x - mx) * ml.y : 0.f;
        const float wp = lp > -INFINITY ? fast_exp2(lp - mx) : 0.f;
        float ws = w;
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
        ws += wp;
        float acc[kCols];
#pragma unroll
        for (int c = 0; c < kCols; ++c) acc[c] = 0.f;
        if (wp > 0.f) {  // this lane's columns of the kept part
          const uint16_t *pr = reinterpret_cast<const uint16_t *>(a.prev_out) + hr2 * D + sub * kCols;
#pragma unroll
          for (int c = 0; c < kCols; ++c) acc[c] = wp * bf16_bits_to_float(pr[c]);
        }
        float wj[kMaxCluster];
#pragma unroll
        for (int j = 0; j < kMaxCluster; ++j) wj[j] = __shfl_sync(0xffffffffu, w, grp * LPR + j);
#pragma unroll
        for (int j = 0; j < kMaxCluster; ++j) {
          if (!(j < cs && wj[j] > 0.f)) continue;
#pragma unroll
          for (int c = 0; c < kCols / 2; ++c) {
            acc[2 * c] = fmaf(wj[j], bf16_bits_to_float(v[j][c] & 0xffffu), acc[2 * c]);
            acc[2 * c + 1] = fmaf(wj[j], bf16_bits_to_float(v[j][c] >> 16), acc[2 * c + 1]);
          }
        }
        if (valid && !aborted) {
          const float inv = ws > 0.f ? 1.0f / ws : 0.f;
          uint32_t pk[kCols / 2];
#pragma unroll
          for (int c = 0; c < kCols / 2; ++c)
            pk[c] = pack_bf16x2(acc[2 * c] * inv, acc[2 * c + 1] * inv);
          uint16_t *dst = reinterpret_cast<uint16_t *>(a.out) + hr2 * D + sub * kCols;
          if constexpr (kBytes >= 16) {
#pragma unroll
            for (int h = 0; h < kBytes / 16; ++h)
              reinterpret_cast<uint4 *>(dst)[h] = make_uint4(pk[4 * h], pk[4 * h + 1], pk[4 * h + 2], pk[4 * h + 3]);
          } else {
            *reinterpret_cast<uint2 *>(dst) = make_uint2(pk[0], pk[1]);
          }
          if (sub == 0 && a.lse_out) a.lse_out[hr2] = (mx + __log2f(ws)) * 0.6931471805599453f;
        }
      }
    }
    if (tid == 64) D2F_TRACE_MARK(0, 12);
    // 4) this CTA's reads of the other CTAs' staging blocks are done; they may
    //    leave once every CTA has arrived
    __syncwarp();
    cluster_arrive();
    cluster_wait();
  }

  // ---- teardown ---------------------------------------------------------------
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1 && !tmem_freed) tmem_dealloc(bars->tmem_base, L::kTmemCols);
  if (tid == 0) D2F_TRACE_MARK(0, 11);
}

// ---------------------------------------------------------------------------
// Stream-K form (head_dim 128, one 128-row tile per (sequence, KV head), the
// 6-stage ring at one CTA per SM)
//
// With one split per (sequence, KV head) and fewer of them than SMs, the split
// layout above leaves SMs idle (long-context batch 4 x 32 heads: 128 CTAs on
// 152 SMs, each streaming at the ~50 GB/s its MMA / softmax chain allows). Here
// the key tiles of every (sequence, KV head) are laid end to end (pair p =
// b * Hkv + g, tiles cache first then window, the order above) and each of
// `grid` CTAs takes an equal contiguous share: a few whole pairs plus a piece
// of a pair at either end. The roles are those of the one-CTA variant (warp 0
// loads, warp 1 issues Q K^T, warp 2 P V, warps 3-6 softmax); they walk the
// share's segments in the same order with one running tile count, so the ring
// stages and the S / P buffers keep their phases across segments. At the start
// of a segment the softmax warps load its Q rows (the previous segment's last
// Q K^T has completed: they waited for its S) and the Q K^T issuer waits for
// them; the first P V of a segment overwrites O (the softmax warps read the
// previous O before they release the segment's first P).
//
// A segment that is a whole pair writes its output directly. A piece of a
// pair writes its rows normalised (O / l, bf16) with their (max, sum) into one
// of the CTA's two partial slots (0: the share's first segment, 1: its last)
// and arrives on the pair's counter; the last CTA to arrive composes the
// pair's pieces in log space and writes the output (the same composition as
// the cluster path, through global memory). Every wait is bounded as above.
// ---------------------------------------------------------------------------

// The key tiles of sequence b (cache, then window) and its window layout;
// T = 0 for a sequence without window rows or whose metadata contradicts the
// host sizes (recorded as D2F_ERR_INVALID_ARG by warp 0).
struct SkSeq {
  int q0, n, C, Tc, T;
  bool ok;
};
__device__ __forceinline__ SkSeq sk_seq(const AttnArgs &a, int b) {
  SkSeq s;
  s.ok = load_seq_meta(a, b, s.q0, s.n, s.C) && a.group * s.n <= kTcRows;
  s.Tc = s.ok ? (s.C + N - 1) / N : 0;
  s.T = (s.ok && s.n > 0) ? s.Tc + (s.n + N - 1) / N : 0;
  return s;
}

// The CTA whose share holds tile position u of the line of W tiles.
__device__ __forceinline__ int sk_cta_of(long long u, long long W, int grid) {
  return (int)(((u + 1) * grid - 1) / W);
}
__device__ __forceinline__ long long sk_start(int c, long long W, int grid) {
  return (long long)c * W / grid;
}
// The same share boundaries without a 64-bit division per call (compositions
// walk them per row): with W = Wq grid + Wr, c W / grid = c Wq + c Wr / grid,
// and c Wr < grid^2 < 2^32 for grids of at most 65535 CTAs (the planner's bound).
struct SkShares {
  long long Wq;
  unsigned Wr, grid;
  __device__ __forceinline__ long long start(int c) const {
    return (long long)c * Wq + (long long)(((unsigned)c * Wr) / grid);
  }
};
__device__ __forceinline__ SkShares sk_shares(long long W, int grid) {
  return SkShares{W / grid, (unsigned)(W % grid), (unsigned)grid};
}
// The first tile of a pair (line position P, T tiles) at or after line position x.
__device__ __forceinline__ int sk_first_tile(long long x, long long P, int T) {
  if (x <= P) return 0;
  const long long d = x - P;
  return d >= T ? T : (int)d;
}

// The last piece of a pair is in: compose its rows from the pieces of the CTAs
// cf..cl that hold a tile of it, in log space, and write them (bf16) with their
// lse. CTA cc's piece: slot 2 cc + 1 if cc = cf and its share began before the
// pair (the pair is its last segment), else slot 2 cc. The slots were written by
// other CTAs: read from L2. The pieces are gathered once, up to eight at a time
// (the share boundaries take integer divisions).
constexpr int kComposeGroup = 8;
struct SkPieces {
  const uint8_t *p[kComposeGroup];
  int n;
};
// The next pieces from CTA cc on (lo: its share's start), at most eight.
__device__ __forceinline__ SkPieces sk_gather(const uint8_t *slots, int cf, int cl, long long P, int T,
                                              SkShares sh, int &cc, long long &lo) {
  SkPieces g;
  g.n = 0;
#pragma unroll
  for (int i = 0; i < kComposeGroup; ++i) g.p[i] = slots;
  while (cc <= cl && g.n < kComposeGroup) {
    const long long hi = sh.start(cc + 1);
    if (sk_first_tile(lo, P, T) < sk_first_tile(hi, P, T)) {
      const int wc = (cc == cf && lo < P) ? 1 : 0;
      const uint8_t *pp = slots + (size_t)(2 * cc + wc) * kSkSlotBytes;
#pragma unroll
      for (int i = 0; i < kComposeGroup; ++i)
        if (i == g.n) g.p[i] = pp;
      ++g.n;
    }
    lo = hi;
    ++cc;
  }
  return g;
}
// Called by every lane of each warp of the composing warpgroup (lane = row %
// 32 of the warp's 32 rows; rv: the lane's row is a query row, hr its output
// row). Pass 1, lane = row: the pieces' (max, sum) and each piece's weight for
// the row. Pass 2, coalesced: a warp load covers two rows (16 lanes x 16 bytes
// each), the weights come by shuffle; four rows and four pieces in flight.
__device__ __noinline__ void sk_compose(const uint8_t *slots, uint16_t *out, float *lse_out, int64_t hr,
                                        bool rv, int row, int cf, int cl, long long P, int T,
                                        SkShares sh) {
  constexpr int D = 128;
  constexpr size_t kMl = (size_t)kTcRows * D * 2;  // (max, sum) pairs after the rows
  const int lane = threadIdx.x & 31;
  const int row0 = row - lane;  // the warp's first row
  int cc = cf;
  long long lo = sh.start(cf);
  const SkPieces g0 = sk_gather(slots, cf, cl, P, T, sh, cc, lo);
  const bool more = cc <= cl;  // more than eight pieces: the rest below, one by one
  float2 ml[kComposeGroup];
#pragma unroll
  for (int i = 0; i < kComposeGroup; ++i)
    ml[i] = i < g0.n ? __ldcg(reinterpret_cast<const float2 *>(g0.p[i] + kMl) + row) : make_float2(0.f, 0.f);
  float mx = -INFINITY, ws = 0.f;
  auto fold = [&](float2 m) {
    if (!(m.y > 0.f)) return;
    if (m.x > mx) {
      ws = ws * fast_exp2(mx - m.x) + m.y;
      mx = m.x;
    } else {
      ws += fast_exp2(m.x - mx) * m.y;
    }
  };
#pragma unroll
  for (int i = 0; i < kComposeGroup; ++i)
    if (i < g0.n) fold(ml[i]);
  if (more) {
    int c2 = cc;
    long long l2 = lo;
    while (c2 <= cl) {
      const SkPieces g = sk_gather(slots, cf, cl, P, T, sh, c2, l2);
      for (int i = 0; i < g.n; ++i) fold(__ldcg(reinterpret_cast<const float2 *>(g.p[i & 7] + kMl) + row));
    }
  }
  const float invs = ws > 0.f ? 1.0f / ws : 0.f;
  float wt[kComposeGroup];  // this lane's row: weight of each of the first eight pieces
#pragma unroll
  for (int i = 0; i < kComposeGroup; ++i)
    wt[i] = (i < g0.n && ml[i].y > 0.f) ? fast_exp2(ml[i].x - mx) * ml[i].y * invs : 0.f;
  if (rv && lse_out) lse_out[hr] = ws > 0.f ? (mx + __log2f(ws)) * 0.6931471805599453f : -INFINITY;
  const int chunk = lane & 15;  // 16-byte chunk (8 columns) of a row
  for (int k = 0; k < 16; k += 4) {  // rows row0 + 2 (k + u) + lane / 16, u < 4
    float acc[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[u][e] = 0.f;
#pragma unroll
    for (int pb = 0; pb < kComposeGroup; pb += 4) {
      if (pb >= g0.n) break;
      uint4 v[4][4];
      float wv[4][4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = 2 * (k + u) + (lane >> 4);  // row within the warp
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          wv[u][i] = __shfl_sync(0xffffffffu, wt[pb + i], r);
          const bool on = pb + i < g0.n;
          const uint4 *q4 = reinterpret_cast<const uint4 *>(g0.p[pb + i] + (size_t)(row0 + r) * D * 2) + chunk;
          v[u][i] = on ? __ldcg(q4) : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t x[4] = {v[u][i].x, v[u][i].y, v[u][i].z, v[u][i].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[u][2 * e] = fmaf(wv[u][i], bf16_bits_to_float(x[e] & 0xffffu), acc[u][2 * e]);
            acc[u][2 * e + 1] = fmaf(wv[u][i], bf16_bits_to_float(x[e] >> 16), acc[u][2 * e + 1]);
          }
        }
    }
    if (more) {  // pieces past the first eight, one at a time (their weights per row)
      int c2 = cc;
      long long l2 = lo;
      while (c2 <= cl) {
        const SkPieces g = sk_gather(slots, cf, cl, P, T, sh, c2, l2);
        for (int i = 0; i < g.n; ++i) {
          const float2 m = __ldcg(reinterpret_cast<const float2 *>(g.p[i & 7] + kMl) + row);
          const float wrow = m.y > 0.f ? fast_exp2(m.x - mx) * m.y * invs : 0.f;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int r = 2 * (k + u) + (lane >> 4);
            const float wgt = __shfl_sync(0xffffffffu, wrow, r);
            const uint4 vv = __ldcg(reinterpret_cast<const uint4 *>(g.p[i & 7] + (size_t)(row0 + r) * D * 2) + chunk);
            const uint32_t x[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc[u][2 * e] = fmaf(wgt, bf16_bits_to_float(x[e] & 0xffffu), acc[u][2 * e]);
              acc[u][2 * e + 1] = fmaf(wgt, bf16_bits_to_float(x[e] >> 16), acc[u][2 * e + 1]);
            }
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = 2 * (k + u) + (lane >> 4);
      const long long hr_r = __shfl_sync(0xffffffffu, (long long)hr, r);
      const int rv_r = __shfl_sync(0xffffffffu, rv ? 1 : 0, r);
      if (rv_r) {
        uint4 *d = reinterpret_cast<uint4 *>(out + hr_r * D) + chunk;
        *d = make_uint4(pack_bf16x2(acc[u][0], acc[u][1]), pack_bf16x2(acc[u][2], acc[u][3]),
                        pack_bf16x2(acc[u][4], acc[u][5]), pack_bf16x2(acc[u][6], acc[u][7]));
      }
    }
  }
  if (row == 0) D2F_TRACE_MARK(0, 12);
}
// CTAs cf..cl that hold a tile of the pair (the arrivals its last piece waits for)
__device__ __forceinline__ int sk_pieces(int cf, int cl, long long P, int T, SkShares sh) {
  int n = 0;
  long long lo = sh.start(cf);
  for (int cc = cf; cc <= cl; ++cc) {
    const long long hi = sh.start(cc + 1);
    n += sk_first_tile(lo, P, T) < sk_first_tile(hi, P, T);
    lo = hi;
  }
  return n;
}

template <int D>
__global__ void __launch_bounds__((Layout<D, 6, 128, 1>::kThreads), 1)
    attn_sk_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tm_kpool,
                   const __grid_constant__ CUtensorMap tm_vpool,
                   const __grid_constant__ CUtensorMap tm_kwin,
                   const __grid_constant__ CUtensorMap tm_vwin) {
  constexpr int NS = 6, QR = 128;
  using L = Layout<D, NS, QR, 1>;
  static_assert(L::kSplit && L::kProducers == 1 && L::kFirstSoft == 3, "one-CTA roles");
  extern __shared__ uint8_t smem_raw[];
  {
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if (pad + L::kBytes > dyn) {
      if (threadIdx.x == 0) set_err(a.err, D2F_ERR_UNSUPPORTED);
      return;
    }
  }
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  Bars *bars = reinterpret_cast<Bars *>(smem + L::kBars);
  volatile int *abort_flag = &bars->abort_flag;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, grid = gridDim.x;
  const int Hkv = a.num_heads_kv, G = a.group, H = a.num_heads_q, B = a.block_size;
  const int ppt = N / B;  // pages (or window blocks) per tile

  if (tid == 0) D2F_TRACE_MARK(0, 0);
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(smem_u32(&bars->full[i]), 1);
      mbar_init(smem_u32(&bars->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->s_full[0][i]), 1);
      mbar_init(smem_u32(&bars->p_full[0][i]), QR);
      mbar_init(smem_u32(&bars->pv_done[0][i]), 1);
    }
    mbar_init(smem_u32(&bars->q_full), QR);
    mbar_init(smem_u32(&bars->drain), 2);
    bars->abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tm_kpool);
    tma_prefetch_desc(&tm_vpool);
    tma_prefetch_desc(&tm_kwin);
    tma_prefetch_desc(&tm_vwin);
  }
  __syncthreads();
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), L::kTmemCols);
    tmem_relinquish();
  }
  grid_dependency_wait();  // inputs may come from the previous kernel in the stream

  // ---- the share: W tiles in all, this CTA's [s0, s1); warp 0 locates s0 ----
  if (warp == 0) {
    long long tot = 0;
    bool bad = false;
    for (int b = lane; b < a.batch; b += 32) {
      const SkSeq q = sk_seq(a, b);
      tot += (long long)q.T * Hkv;
      bad |= !q.ok;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    if (__any_sync(0xffffffffu, bad) && lane == 0 && c == 0) set_err(a.err, D2F_ERR_INVALID_ARG);
    const long long W = tot;
    const long long s0 = W > 0 ? sk_start(c, W, grid) : 0, s1 = W > 0 ? sk_start(c + 1, W, grid) : 0;
    int b0 = 0, g0 = 0, ta0 = 0;
    long long run = 0;
    for (int base = 0; base < a.batch && s1 > s0; base += 32) {
      const int b = base + lane;
      const SkSeq q = b < a.batch ? sk_seq(a, b) : SkSeq{0, 0, 0, 0, 0, false};
      const long long t = (long long)q.T * Hkv;
      long long incl = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const long long excl = run + incl - t;
      const bool hit = t > 0 && excl <= s0 && s0 < excl + t;
      const unsigned who = __ballot_sync(0xffffffffu, hit);
      if (hit) {
        const long long rel = s0 - excl;
        b0 = b;
        g0 = (int)(rel / q.T);
        ta0 = (int)(rel - (long long)g0 * q.T);
      }
      if (who) {
        const int src = __ffs(who) - 1;
        b0 = __shfl_sync(0xffffffffu, b0, src);
        g0 = __shfl_sync(0xffffffffu, g0, src);
        ta0 = __shfl_sync(0xffffffffu, ta0, src);
        break;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      bars->sk[0] = b0;
      bars->sk[1] = g0;
      bars->sk[2] = ta0;
      bars->sk[3] = (int)(s1 - s0);
      bars->sk[4] = (int)(W & 0xffffffffLL);
      bars->sk[5] = (int)(W >> 32);
    }
  }
  if (warp >= 1) {  // TMEM address, published by warp 1
    tc_fence_before();
    named_sync(kBarSetup, L::kThreads - 32);
    tc_fence_after();
  }
  __syncthreads();
  const uint32_t tmem = bars->tmem_base;
  const int b0 = bars->sk[0], g0 = bars->sk[1], ta0 = bars->sk[2], R = bars->sk[3];
  const long long W = (long long)(uint32_t)bars->sk[4] | ((long long)bars->sk[5] << 32);
  const long long s0 = W > 0 ? sk_start(c, W, grid) : 0;
  const SkShares sh = sk_shares(W > 0 ? W : 1, grid);
  grid_launch_dependents();

  // Every role walks the share's segments in the same order: tiles [ta, tb) of
  // pair (b, g), then the next pair from its first tile, until R tiles are done.
  // `gu` counts the tiles of the whole share (ring stage gu % NS, S / P buffer
  // gu % 2, and their phases).
  if (warp == 0) {
    // ======================= TMA producer ======================================
    const int box = lane;  // box i: tensor i / ppt (0 = K, 1 = V), page or block i % ppt
    const bool lane_on = box < 2 * ppt;
    const int tensor = lane_on ? box / ppt : 0, slot = lane_on ? box % ppt : 0;
    // K/V are read once: evict them first, so the partial slots stay in L2
    const uint64_t kv_policy = l2_policy_evict_first();
    int gu = 0;
    bool ok = true;
    int b = b0, g = g0, ta = ta0, rem = R;
    while (ok && rem > 0 && b < a.batch) {
      const SkSeq q = sk_seq(a, b);
      const int tb = min(q.T, ta + rem);
      const int n_pages = (q.C + B - 1) / B;
      const int32_t *pt = a.page_table + (int64_t)b * a.max_pages_per_seq;
      auto fetch = [&](int base) -> int {
        const int lp = base + lane;
        return (lp < n_pages && lp < tb * ppt) ? __ldg(pt + lp) : -1;
      };
      int chunk = ta * ppt;  // logical page held by lane 0 of ids_cur
      int ids_cur = ta < q.Tc ? fetch(chunk) : -1;
      int ids_next = ta < q.Tc ? fetch(chunk + 32) : -1;
      for (int t = ta; t < tb; ++t, ++gu) {
        const int stage = gu % NS;
        if (gu >= NS) {
          int w = 1;
          if (lane == 0)
            w = mbar_wait(smem_u32(&bars->empty[stage]), ((gu / NS) - 1) & 1, abort_flag, a.err,
                          a.wait_cycles);
          if (!__shfl_sync(0xffffffffu, w, 0)) {
            ok = false;
            break;
          }
        }
        int src = -1;  // a physical page or a window row; -1: nothing to load
        if (t < q.Tc) {
          const int lp0 = t * ppt;
          if (lp0 - chunk >= 32) {  // warp-uniform: move to the next 32 ids
            chunk += 32;
            ids_cur = ids_next;
            ids_next = fetch(chunk + 32);
          }
          const int pg = __shfl_sync(0xffffffffu, ids_cur, (lp0 - chunk + slot) & 31);
          if (lane_on && (lp0 + slot) * B < q.C) {
            if (pg >= 0 && pg < a.num_pages)
              src = pg;
            else
              set_err(a.err, D2F_ERR_BAD_INDEX);
          }
        } else if (lane_on) {
          const int w0 = (t - q.Tc) * N + slot * B;  // first window row of this block
          if (w0 < q.n) src = q.q0 + w0;
        }
        const unsigned have = __ballot_sync(0xffffffffu, src >= 0);
        const uint32_t full = smem_u32(&bars->full[stage]);
        if (lane == 0) mbar_arrive_expect_tx(full, __popc(have) * (uint32_t)B * D * 2u);
        __syncwarp();
        const uint32_t dst = sb + L::kRing + stage * L::kStage + tensor * L::kKBytes +
                             slot * (B / 8) * L::kGroupBytes;
        if (src >= 0) {
          if (t < q.Tc)
            tma_load_5d_hint(dst, tensor ? &tm_vpool : &tm_kpool, full, 0, 0, 0, 0, src * Hkv + g, kv_policy);
          else
            tma_load_5d_hint(dst, tensor ? &tm_vwin : &tm_kwin, full, 0, 0, 0, src >> 3, g, kv_policy);
        }
      }
      rem -= max(0, tb - ta);
      ta = 0;
      if (++g == Hkv) {
        g = 0;
        ++b;
      }
    }
    // Drain: every issued stage has landed before the CTA moves on.
    if (lane == 0) {
      for (int u = max(0, gu - NS); u < gu; ++u) {
        volatile int no_abort = 0;
        mbar_wait(smem_u32(&bars->full[u % NS]), (u / NS) & 1, &no_abort, a.err, kDrainCycles);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ============ MMA issuers: warp 1 S = Q K^T, warp 2 O += P V =============
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(M, N, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(M, D, 0, 1);
      // descriptors of Q and of stage 0's K and V; each MMA advances them by a constant
      const uint64_t q_desc = smem_desc_sw128(sb + L::kQ, 16, 1024);
      const uint64_t k_desc = smem_desc_sw128(sb + L::kRing, 16, L::kGroupBytes);
      const uint64_t v_desc = smem_desc_sw128(sb + L::kRing + L::kKBytes, 1024, L::kGroupBytes);
      int gu = 0, k = 0;  // tiles and segments so far
      bool ok = true;
      int b = b0, g = g0, ta = ta0, rem = R;
      while (ok && rem > 0 && b < a.batch) {
        const SkSeq q = sk_seq(a, b);
        const int tb = min(q.T, ta + rem);
        if (tb > ta && warp == 1)  // this segment's Q rows are in shared memory
          ok = mbar_wait(smem_u32(&bars->q_full), k & 1, abort_flag, a.err, a.wait_cycles);
        for (int t = ta; t < tb && ok; ++t, ++gu) {
          const int stage = gu % NS;
          ok = mbar_wait(smem_u32(&bars->full[stage]), (gu / NS) & 1, abort_flag, a.err, a.wait_cycles);
          if (!ok) break;
          if (warp == 1) {
            // S_gu overwrites the S / P buffer of P_{gu-2}: its P V must be complete
            if (gu >= 2 && !mbar_wait(smem_u32(&bars->pv_done[0][gu & 1]), ((gu - 2) >> 1) & 1,
                                      abort_flag, a.err, a.wait_cycles)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t kd = smem_desc_advance(k_desc, stage * L::kStage);
#pragma unroll
            for (int h = 0; h < L::kHalves; ++h) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = smem_desc_advance(q_desc, h * L::kQHalf + kk * 32);
                const uint64_t bd = smem_desc_advance(kd, h * 1024 + kk * 32);
                umma_bf16(tmem + (gu & 1) * N, ad, bd, idesc_qk, (h | kk) ? 1u : 0u);
              }
            }
            umma_commit(smem_u32(&bars->s_full[0][gu & 1]));
          } else {
            if (!mbar_wait(smem_u32(&bars->p_full[0][gu & 1]), (gu >> 1) & 1, abort_flag, a.err,
                           a.wait_cycles)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t vd = smem_desc_advance(v_desc, stage * L::kStage);
            const bool first = t == ta;  // the segment's first P V overwrites O
#pragma unroll
            for (int ks = 0; ks < N / 16; ++ks) {
              const uint64_t bd = smem_desc_advance(vd, ks * 2 * L::kGroupBytes);
              umma_bf16_tmem_a(tmem + kTmemO, tmem + (gu & 1) * N + ks * 8, bd, idesc_pv,
                               (!first || ks > 0) ? 1u : 0u);
            }
            umma_commit(smem_u32(&bars->pv_done[0][gu & 1]));
            umma_commit(smem_u32(&bars->empty[stage]));
          }
        }
        if (tb > ta) ++k;
        rem -= max(0, tb - ta);
        ta = 0;
        if (++g == Hkv) {
          g = 0;
          ++b;
        }
      }
      umma_commit(smem_u32(&bars->drain));
      volatile int no_abort = 0;
      mbar_wait(smem_u32(&bars->drain), 0, &no_abort, a.err, kDrainCycles);
    }
  } else {
    // ============ softmax: one warpgroup, a thread per query row (TMEM lane) =====
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    const float sl2 = a.scale_log2;
    int gu = 0;
    bool ok = true;
    int b = b0, g = g0, ta = ta0, rem = R;
    long long pre_p = s0 - ta0;  // position of the current pair's first tile on the line
#ifdef D2F_TRACE
    int seg_no = 0;
#endif
    while (ok && rem > 0 && b < a.batch) {
      const SkSeq q = sk_seq(a, b);
      const int tb = min(q.T, ta + rem);
      if (tb > ta) {
        const int rows_total = G * q.n;
        const bool rv = row < rows_total;
        const int64_t hr = (int64_t)(q.q0 + row / G) * H + g * G + row % G;  // valid where rv
        {
          // This segment's Q rows into the 128-byte-swizzled K-major layout (the
          // previous segment's Q K^T have all completed: their S were waited for).
          constexpr int kQc = D / 8;
          uint4 qv[kQc];
          const uint4 *src = reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(a.q) + hr * D);
#pragma unroll
          for (int cq = 0; cq < kQc; ++cq) qv[cq] = rv ? __ldg(src + cq) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int cq = 0; cq < kQc; ++cq) {
            const uint32_t dst = sb + L::kQ + (cq >> 3) * L::kQHalf + (row >> 3) * 1024 + (row & 7) * 128 +
                                 (((cq & 7) ^ (row & 7)) << 4);
            asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(qv[cq].x),
                         "r"(qv[cq].y), "r"(qv[cq].z), "r"(qv[cq].w)
                         : "memory");
          }
          fence_proxy_async_smem();
          mbar_arrive(smem_u32(&bars->q_full));
        }
        const int win_end = rv ? ((row / G) / B + 1) * B : 0;
        float m_ref = -INFINITY, l = 0.f;
        for (int t = ta; t < tb && ok; ++t, ++gu) {
          const int tile_lim = t < q.Tc ? q.C - t * N : q.n - (t - q.Tc) * N;  // valid keys
          ok = mbar_wait(smem_u32(&bars->s_full[0][gu & 1]), (gu >> 1) & 1, abort_flag, a.err,
                         a.wait_cycles);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t sv[N];
          const uint32_t s_addr = lane_addr + (gu & 1) * N;
          tmem_ld64(s_addr, sv);
          int lim = t < q.Tc ? tile_lim : win_end - (t - q.Tc) * N;
          lim = rv ? max(0, min(lim, N)) : 0;
          float sf[N];
#pragma unroll
          for (int cc = 0; cc < N; ++cc) sf[cc] = __uint_as_float(sv[cc]);
          if (!__all_sync(0xffffffffu, lim >= N)) {  // ragged tile: hide masked keys
#pragma unroll
            for (int cc = 0; cc < N; ++cc)
              if (cc >= lim) sf[cc] = -INFINITY;
          }
          float t1[22], t2[8];
#pragma unroll
          for (int cc = 0; cc < 21; ++cc) t1[cc] = fmax3(sf[3 * cc], sf[3 * cc + 1], sf[3 * cc + 2]);
          t1[21] = sf[63];
#pragma unroll
          for (int cc = 0; cc < 7; ++cc) t2[cc] = fmax3(t1[3 * cc], t1[3 * cc + 1], t1[3 * cc + 2]);
          t2[7] = t1[21];
          const float tmax = fmax3(fmax3(t2[0], t2[1], t2[2]), fmax3(t2[3], t2[4], t2[5]),
                                   fmaxf(t2[6], t2[7])) * sl2;
          // lazy rescale: keep the reference max unless the tile max exceeds it by 2^8
          const bool need = tmax > m_ref + 8.0f;
          if (__any_sync(0xffffffffu, need)) {
            const float m_new = need ? tmax : m_ref;
            const float alpha = need ? fast_exp2(m_ref - m_new) : 1.0f;
            l *= alpha;
            if (t > ta) {  // every earlier P V of this segment has landed in O
              ok = mbar_wait(smem_u32(&bars->pv_done[0][(gu - 1) & 1]), ((gu - 1) >> 1) & 1,
                             abort_flag, a.err, a.wait_cycles);
              if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
              }
              tc_fence_after();
#pragma unroll
              for (int ch = 0; ch < D / 32; ++ch) {
                uint32_t o[32];
                const uint32_t oa = lane_addr + kTmemO + ch * 32;
                tmem_ld32(oa, o);
#pragma unroll
                for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                tmem_st32(oa, o);
              }
              tmem_wait_st();
            }
            m_ref = m_new;
          }
          const float mb = m_ref == -INFINITY ? 0.f : m_ref;
          uint32_t pk[N / 2];
#pragma unroll
          for (int j = 0; j < N / 2; ++j) {
            float x0, x1;
            fma2_bc(x0, x1, sf[2 * j], sf[2 * j + 1], sl2, -mb);
            pk[j] = ex2_bf16x2(pack_bf16x2(x0, x1));
          }
          float ps0[N / 4], ps1[N / 4];
#pragma unroll
          for (int j = 0; j < N / 4; ++j)
            add2(ps0[j], ps1[j], __uint_as_float(pk[2 * j] << 16),
                 __uint_as_float(pk[2 * j] & 0xffff0000u), __uint_as_float(pk[2 * j + 1] << 16),
                 __uint_as_float(pk[2 * j + 1] & 0xffff0000u));
#pragma unroll
          for (int w = N / 8; w >= 1; w >>= 1)
#pragma unroll
            for (int cc = 0; cc < w; ++cc)
              add2(ps0[cc], ps1[cc], ps0[2 * cc], ps1[2 * cc], ps0[2 * cc + 1], ps1[2 * cc + 1]);
          l += ps0[0] + ps1[0];
          tmem_st32(s_addr, pk);
          tmem_wait_st();
          // a ragged tile's V rows past its valid keys: cleared before its P V (0 * NaN)
          if (row < N && row >= tile_lim) {
            const uint32_t v_row = sb + L::kRing + (gu % NS) * L::kStage + L::kKBytes +
                                   (row >> 3) * L::kGroupBytes + (row & 7) * 128;
#pragma unroll
            for (int h = 0; h < L::kHalves; ++h)
#pragma unroll
              for (int cc = 0; cc < 8; ++cc)
                asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(v_row + h * 1024 + (cc << 4)),
                             "r"(0u)
                             : "memory");
            fence_proxy_async_smem();
          }
          tc_fence_before();
          mbar_arrive(smem_u32(&bars->p_full[0][gu & 1]));
        }
        // the segment's last P V product (when every tile went through)
        if (ok) {
          ok = mbar_wait(smem_u32(&bars->pv_done[0][(gu - 1) & 1]), ((gu - 1) >> 1) & 1, abort_flag,
                         a.err, a.wait_cycles);
          ok = __all_sync(0xffffffffu, ok);
        }
        // Every softmax thread arrives here for every segment it started, so a
        // give-up in any of the four warps is known to all before the epilogue's
        // barriers (a warp that passed its waits must not wait there for one that
        // left).
        ok = named_sync_and(kBarSk, QR, ok);
        if (row == 0) D2F_TRACE_MARK(0, 4 + min(seg_no++, 3));
        if (!ok) break;
        tc_fence_after();

        // ---- epilogue of the segment ----
        const int cf = sk_cta_of(pre_p, W, grid), cl = sk_cta_of(pre_p + q.T - 1, W, grid);
        const bool any = __any_sync(0xffffffffu, rv);  // warp-uniform TMEM reads
        if (cf == cl) {  // the whole pair: the output directly
          const float inv = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll
          for (int ch = 0; ch < D / 32 && any; ++ch) {
            uint32_t o[32];
            tmem_ld32(lane_addr + kTmemO + ch * 32, o);
            if (rv) {
              uint32_t w[16];
#pragma unroll
              for (int j = 0; j < 16; ++j)
                w[j] = pack_bf16x2(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
              uint4 *d4 = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(a.out) + hr * D + ch * 32);
#pragma unroll
              for (int j = 0; j < 4; ++j) d4[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
            }
          }
          if (rv && a.lse_out)
            a.lse_out[hr] = l > 0.f ? (m_ref + __log2f(l)) * 0.6931471805599453f : -INFINITY;
        } else {
          // A piece: its rows (O / l, bf16) and (max, sum) into this CTA's slot,
          // then one arrival on the pair's counter.
          const int which = (c == cf && s0 < pre_p) ? 1 : 0;  // the share's last segment : first
          uint8_t *slot = a.sk_slots + (size_t)(2 * c + which) * kSkSlotBytes;
          const bool keep = rv && l > 0.f;
          const float inv = keep ? 1.0f / l : 0.f;
#pragma unroll
          for (int ch = 0; ch < D / 32 && any; ++ch) {
            uint32_t o[32];
            tmem_ld32(lane_addr + kTmemO + ch * 32, o);
            if (keep) {
              uint32_t w[16];
#pragma unroll
              for (int j = 0; j < 16; ++j)
                w[j] = pack_bf16x2(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
              uint4 *d4 = reinterpret_cast<uint4 *>(slot + (size_t)row * D * 2 + ch * 64);
              const uint64_t keep_policy = l2_policy_evict_last();  // read back by the last piece
#pragma unroll
              for (int j = 0; j < 4; ++j)
                st_global_v4_hint(d4 + j, make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]),
                                  keep_policy);
            }
          }
          reinterpret_cast<float2 *>(slot + (size_t)QR * D * 2)[row] =
              make_float2(keep ? m_ref : -INFINITY, keep ? l : 0.f);
          __threadfence();  // this row's piece before the arrival
          named_sync(kBarSk, QR);
          if (row == 0) {
            const int target = sk_pieces(cf, cl, pre_p, q.T, sh);  // CTAs holding tiles of the pair
            const int pair = b * Hkv + g;
            const int last = atomic_add_acq_rel(a.sk_cnt + pair, 1) == target - 1;
            if (last) a.sk_cnt[pair] = 0;  // every piece of this launch is in
            bars->sk[0] = last;
          }
          named_sync(kBarSk, QR);
          if (bars->sk[0] && row == 0) D2F_TRACE_MARK(0, 8);
          if (bars->sk[0])  // the last piece in: compose the pair's pieces (every lane)
            sk_compose(a.sk_slots, reinterpret_cast<uint16_t *>(a.out), a.lse_out, hr, rv, row, cf, cl,
                       pre_p, q.T, sh);
          named_sync(kBarSk, QR);  // bars->sk[0] is reused by the next piece
        }
      }
      rem -= max(0, tb - ta);
      pre_p += q.T;
      ta = 0;
      if (++g == Hkv) {
        g = 0;
        ++b;
      }
    }
    tc_fence_before();
  }

  // ---- teardown ---------------------------------------------------------------
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) D2F_TRACE_MARK(0, 3);
  if (warp == 1) tmem_dealloc(bars->tmem_base, L::kTmemCols);
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
  const cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims,
                        strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Function attributes (shared-memory opt-in and carveout) are per device; set
// them once per device and kernel variant.
template <int D, int NS, int QR, int MT>
cudaError_t ensure_attrs() {
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  e = cudaFuncSetAttribute(attn_tc_kernel<D, NS, QR, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Layout<D, NS, QR, MT>::kAlloc);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_tc_kernel<D, NS, QR, MT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

// The four K/V tensor maps of a launch (pool K, pool V, window K, window V).
template <int D>
cudaError_t encode_maps(const AttnArgs &a, CUtensorMap &kp, CUtensorMap &vp, CUtensorMap &kw,
                        CUtensorMap &vw, char *why, size_t why_len) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) {
    snprintf(why, why_len, "cuTensorMapEncodeTiled is not available from the driver");
    return cudaErrorNotSupported;
  }
  // 5-D views whose box is one page (or window block) of one KV head, both
  // column halves, landing group-major in shared memory (see Layout):
  // (64 columns, 8 rows, column half, 8-row group, page x head | token group x head).
  constexpr int H2 = D / 64;
  const cuuint64_t B8 = (cuuint64_t)a.block_size / 8, rowb = (cuuint64_t)D * 2;
  const cuuint64_t pool_dims[5] = {64, 8, (cuuint64_t)H2, B8,
                                   (cuuint64_t)a.num_pages * a.num_heads_kv};
  const cuuint64_t pool_strides[4] = {rowb, 128, 8 * rowb, (cuuint64_t)a.block_size * rowb};
  const cuuint64_t tok = (cuuint64_t)a.num_heads_kv * rowb;  // window row stride
  const cuuint64_t win_dims[5] = {64, 8, (cuuint64_t)H2, (cuuint64_t)a.total_q / 8,
                                  (cuuint64_t)a.num_heads_kv};
  const cuuint64_t win_strides[4] = {tok, 128, 8 * tok, rowb};
  const cuuint32_t box[5] = {64, 8, (cuuint32_t)H2, (cuuint32_t)(a.block_size / 8), 1};
  if (!encode(fn, &kp, a.k_pool, 5, pool_dims, pool_strides, box) ||
      !encode(fn, &vp, a.v_pool, 5, pool_dims, pool_strides, box) ||
      !encode(fn, &kw, a.k_win, 5, win_dims, win_strides, box) ||
      !encode(fn, &vw, a.v_win, 5, win_dims, win_strides, box)) {
    snprintf(why, why_len, "cuTensorMapEncodeTiled rejected a K/V tensor (alignment or size)");
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

template <int D, int NS, int QR, int MT>
cudaError_t launch_d(const AttnArgs &a, cudaStream_t s, char *why, size_t why_len) {
  CUtensorMap kp, vp, kw, vw;
  cudaError_t e = encode_maps<D>(a, kp, vp, kw, vw, why, why_len);
  if (e != cudaSuccess) return e;
  e = ensure_attrs<D, NS, QR, MT>();
  if (e != cudaSuccess) return e;
  const int cs = a.num_splits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, a.m_tiles, a.batch * a.num_heads_kv);
  cfg.blockDim = dim3(Layout<D, NS, QR, MT>::kThreads);
  cfg.dynamicSmemBytes = Layout<D, NS, QR, MT>::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  e = cudaLaunchKernelEx(&cfg, attn_tc_kernel<D, NS, QR, MT>, a, kp, vp, kw, vw);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_sk(const AttnArgs &a, cudaStream_t s, char *why, size_t why_len) {
  CUtensorMap kp, vp, kw, vw;
  cudaError_t e = encode_maps<D>(a, kp, vp, kw, vw, why, why_len);
  if (e != cudaSuccess) return e;
  using L = Layout<D, 6, 128, 1>;
  {
    static std::mutex mu;
    static bool done[64] = {};
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64 || !done[dev]) {
      e = cudaFuncSetAttribute(attn_sk_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_sk_kernel<D>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) done[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.sk);
  cfg.blockDim = dim3(L::kThreads);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, attn_sk_kernel<D>, a, kp, vp, kw, vw);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// CTAs of the one-CTA-per-SM variant (head_dim 128, 128-row tiles, 6 stages) that
// can be resident at once in clusters of cs: clusters are placed within one GPC,
// so this is below the SM count for most cs. 0 when the query fails. Cached per
// device.
int attn_tc_deep_slots(int cs) {
  static std::mutex mu;
  static int cache[64][kMaxCluster + 1] = {};
  if (cs < 1 || cs > kMaxCluster) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev][cs] == 0) {
    if (ensure_attrs<128, 6, 128, 1>() != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs, 1, 1);
    cfg.blockDim = dim3(Layout<128, 6, 128, 1>::kThreads);
    cfg.dynamicSmemBytes = Layout<128, 6, 128, 1>::kAlloc;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attn_tc_kernel<128, 6, 128, 1>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cache[dev][cs] = n * cs;
  }
  return cache[dev][cs];
}

cudaError_t launch_attn_tc(const AttnArgs &a, cudaStream_t s, char *why, size_t why_len) {
  if (a.batch == 0 || a.total_q == 0) return cudaSuccess;
  if (a.num_splits < 1 || a.num_splits > kMaxCluster) {
    snprintf(why, why_len, "tensor-core path takes 1..%d splits", kMaxCluster);
    return cudaErrorInvalidValue;
  }
  // Ring depth by shared-memory budget: two CTAs per SM hold Q + NS stages in
  // ~113 KB (head_dim 64: 6 stages; head_dim 128: 3 stages with 64-row tiles, 2
  // with 128-row tiles); the 6-stage head_dim-128 variant takes a whole SM.
  // The MT = 2 variant holds two 128-row tiles of one (sequence, KV head) with a
  // softmax warpgroup each (GQA groups of 129..384 rows): every K/V tile is
  // loaded once for both, and the CTA takes a whole SM.
  const int rows = a.tc_rows, ns = a.tc_stages, mt = a.tc_mt;
  if (a.sk > 0 && a.head_dim == 128 && rows == 128 && ns == 6 && mt == 1)
    return launch_sk<128>(a, s, why, why_len);
  if (a.head_dim == 128) {
    if (rows == 64 && ns == 3 && mt == 1) return launch_d<128, 3, 64, 1>(a, s, why, why_len);
    if (rows == 128 && ns == 2 && mt == 1) return launch_d<128, 2, 128, 1>(a, s, why, why_len);
    if (rows == 128 && ns == 6 && mt == 1) return launch_d<128, 6, 128, 1>(a, s, why, why_len);
    if (rows == 128 && ns == 5 && mt == 2) return launch_d<128, 5, 128, 2>(a, s, why, why_len);
  } else if (a.head_dim == 64) {
    if (rows == 64 && ns == 6 && mt == 1) return launch_d<64, 6, 64, 1>(a, s, why, why_len);
    if (rows == 128 && ns == 6 && mt == 1) return launch_d<64, 6, 128, 1>(a, s, why, why_len);
  }
  snprintf(why, why_len,
           "no tensor-core variant for head_dim %d, %d-row tiles x %d, %d stages", a.head_dim,
           rows, mt, ns);
  return cudaErrorInvalidValue;
}

#ifdef D2F_TRACE
D2F_TRACE_COPY_FN(d2f_trace_copy_attn)
extern "C" int d2f_trace_copy_pass(void *host, size_t bytes) {
  if (bytes > sizeof(g_d2f_pass)) bytes = sizeof(g_d2f_pass);
  return cudaMemcpyFromSymbol(host, g_d2f_pass, bytes) == cudaSuccess ? 0 : 1;
}
#endif

}  // namespace d2f
