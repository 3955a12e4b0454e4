// Host side of the libd2f C ABI: argument validation, split planning,
// workspace layout and kernel dispatch. No allocation, no host<->device copy,
// no synchronisation happens here.
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "d2f_internal.cuh"

namespace d2f {

static thread_local char g_last_error[512] = "";

void set_last_error(const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
}

bool pdl_enabled() {
  static const bool on = [] {
    const char *e = getenv("D2F_PDL");
    return !(e && strcmp(e, "0") == 0);
  }();
  return on;
}

int num_sms_current_device() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }

int fail(int status, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char *what) {
  return fail(D2F_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------------------
// Attention plan
// ---------------------------------------------------------------------------
struct AttnPlan {
  bool tc;        // tensor-core path
  int m_tiles;
  int rows;       // rows per tile: 64 or 128 on the tensor-core path
  int stages;     // tensor-core K/V ring depth
  int mt;         // tensor-core 128-row tiles per CTA
  bool longest_first;  // more CTAs than one wave: longest sequences first
  int splits;
  int tiles_per_split;
  int n_counters;
  int sk;         // stream-K form: its grid (CTAs), else 0
  size_t off_ml, off_o, off_sk, bytes;
};

// D2F_ATTN_SK=1 / 0 forces / forbids the stream-K form of the one-CTA-per-SM
// variant (tests); unset = planner.
int force_sk() {
  const char *e = getenv("D2F_ATTN_SK");
  if (!e || !e[0]) return -1;
  return e[0] == '1' ? 1 : 0;
}
constexpr int kSkMaxBatch = 4096;

bool force_simt() {
  const char *e = getenv("D2F_ATTN_PATH");
  return e && strcmp(e, "simt") == 0;
}

// D2F_TC_ROWS=128 keeps the tensor-core path on 128-row tiles even where every
// sequence fits a 64-row tile; D2F_TC_ROWS=64 cuts every (sequence, KV head) into
// 64-row tiles (for comparing the two; results agree within rounding).
bool force_full_rows() {
  const char *e = getenv("D2F_TC_ROWS");
  return e && strcmp(e, "128") == 0;
}
bool force_half_rows() {
  const char *e = getenv("D2F_TC_ROWS");
  return e && strcmp(e, "64") == 0;
}

// D2F_TC_DEEP=1 / 0 forces / forbids the one-CTA-per-SM 6-stage variant for
// head_dim 128 with 128-row tiles (for comparisons and tests); unset = planner.
// D2F_TC_MT=1 / 0 forces / forbids CTAs of two 128-row tiles (two softmax
// warpgroups) for head_dim 128 groups of 2 or 3 row tiles (tests); unset = planner.
int force_mt() {
  const char *e = getenv("D2F_TC_MT");
  if (!e || !e[0]) return -1;
  return e[0] == '1' ? 1 : 0;
}

int force_deep() {
  const char *e = getenv("D2F_TC_DEEP");
  if (!e || !e[0]) return -1;
  return e[0] == '1' ? 1 : 0;
}

int plan_attn(int batch, int total_q, int max_q, int max_ctx, int Hq, int Hkv, int D, int B,
              int dtype, int num_splits, AttnPlan *p) {
  if (batch < 0 || total_q < 0 || max_q < 0 || max_ctx < 0)
    return fail(D2F_ERR_INVALID_ARG, "negative size (batch %d, total_q %d, max_q %d, max_ctx %d)",
                batch, total_q, max_q, max_ctx);
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0)
    return fail(D2F_ERR_INVALID_ARG, "num_heads_q (%d) must be a positive multiple of num_heads_kv (%d)",
                Hq, Hkv);
  if (dtype != D2F_BF16 && dtype != D2F_F32)
    return fail(D2F_ERR_INVALID_ARG, "dtype must be D2F_BF16 or D2F_F32");
  if (B < 1 || num_splits < 0 || num_splits > 4096)
    return fail(D2F_ERR_INVALID_ARG, "block_size %d / num_splits %d out of range", B, num_splits);
  if (max_q > total_q)
    return fail(D2F_ERR_INVALID_ARG, "max_q_per_seq %d exceeds total_q %d", max_q, total_q);
  if ((long long)batch * Hkv > 65535)
    return fail(D2F_ERR_UNSUPPORTED, "batch * num_heads_kv must be <= 65535");
  const bool tc = dtype == D2F_BF16 && (D == 64 || D == 128) && (B == 8 || B == 16 || B == 32) &&
                  !force_simt();
  if (!tc) {
    if (!(D == 32 || D == 64 || D == 128))
      return fail(D2F_ERR_UNSUPPORTED, "head_dim %d: supported are 64, 128 (bf16, B in {8,16,32}) "
                  "and 32, 64, 128 (CUDA-core path)", D);
    if (B > 256) return fail(D2F_ERR_UNSUPPORTED, "block_size %d > 256", B);
  }
  const int G = Hq / Hkv;
  // tensor-core tiles hold 64 rows when every sequence's G * max_q rows fit
  const int rows = !tc ? kSimtRows
                       : (((long long)G * max_q <= 64 && !force_full_rows()) || force_half_rows()
                              ? 64 : kTcRows);
  const int keys = tc ? kTcKeys : kSimtKeys;
  p->tc = tc;
  p->rows = rows;
  p->m_tiles = max(1, cdiv((long long)G * max_q, rows));
  const int t_max = max(1, cdiv(max_ctx, keys) + cdiv(max_q, keys));
  int splits = num_splits;
  const long long base = (long long)max(batch, 1) * Hkv * p->m_tiles;
  if (tc) {
    // The splits of one row tile form a thread-block cluster (at most 8 CTAs)
    // and compose their partials in distributed shared memory: no workspace.
    // Split count: as many splits as one wave of resident CTAs holds, then the
    // fewest splits that keep the longest split's tile count. (Several waves of
    // shorter splits measured slower: every wave pays the ramp-up and the
    // composition again.)
    const int sms = max(1, num_sms_current_device());
    auto pick = [&](bool deep_variant) {
      int most = 1;
      for (int cs = 2; cs <= min(kTcMaxSplits, t_max); ++cs) {
        const long long slots = deep_variant ? attn_tc_deep_slots(cs) : 2LL * sms;
        if (base * cs <= slots) most = cs;
      }
      return cdiv(t_max, cdiv(t_max, most));
    };
    p->stages = D == 64 ? 6 : (rows == 64 ? 3 : 2);
    p->mt = 1;
    const int two = splits ? splits : pick(false);  // two CTAs per SM
    splits = two;
    if (D == 128 && rows == 128 && (p->m_tiles == 2 || p->m_tiles == 3)) {
      // GQA groups of 129..384 rows: a CTA with two softmax warpgroups takes two
      // row tiles of a (sequence, KV head) and reads each K/V tile once for both,
      // through a deeper ring, at one CTA per SM (three row tiles: two CTAs, the
      // second with one row tile). It pays only once splits are long.
      const int groups = cdiv(p->m_tiles, 2);
      const long long base_mt = (long long)max(batch, 1) * Hkv * groups;
      int one = splits ? splits : 1;
      if (!num_splits) {
        int most = 1;
        for (int cs = 2; cs <= min(kTcMaxSplits, t_max); ++cs)
          if (attn_tc_deep_slots(cs) > 0 && base_mt * cs <= attn_tc_deep_slots(cs)) most = cs;
        one = cdiv(t_max, cdiv(t_max, most));
      }
      bool use = cdiv(t_max, two) >= 8 && attn_tc_deep_slots(one) > 0;
      if (force_mt() >= 0) use = force_mt() == 1;
      if (use) {
        p->mt = 2;
        p->stages = 5;
        p->m_tiles = groups;
        splits = one;
      }
    }
    if (p->mt == 1 && D == 128 && rows == 128) {
      // 2 ring stages at two CTAs per SM, or 6 stages at one: per streamed tile a
      // CTA takes ~2.2 us in the first (the ring waits on the load latency) and
      // ~0.9 us in the second (measured on GB300); take the deeper ring when its
      // one wave finishes first and the splits are long enough for the steady
      // state to matter.
      const int one = num_splits ? num_splits : pick(true);
      const int tps2 = cdiv(t_max, two), tps1 = cdiv(t_max, one);
      const long long w2 = cdiv(base * two, 2LL * sms);
      const long long slots1 = attn_tc_deep_slots(one);
      const long long w1 = slots1 > 0 ? cdiv(base * one, slots1) : -1;
      bool deep = tps2 >= 8 && w1 > 0 && w1 * tps1 * 9 < w2 * tps2 * 22;
      if (force_deep() >= 0) deep = force_deep() == 1;
      if (deep) {
        p->stages = 6;
        splits = one;
      }
    }
    p->splits = min(splits, kTcMaxSplits);
    // Stream-K: the one-CTA variant with one split per (sequence, KV head) and
    // fewer of them than resident CTAs leaves SMs idle (batch 4 x 32 heads at
    // context 32768: 128 of 152 SMs, each at the ~50 GB/s its MMA / softmax
    // chain streams). Instead one wave of CTAs takes equal shares of all the key
    // tiles. Each CTA owns two partial slots; the pairs count arrivals.
    p->sk = 0;
    if (D == 128 && rows == 128 && p->mt == 1 && p->stages == 6 && batch <= kSkMaxBatch) {
      const int slots1 = attn_tc_deep_slots(1);
      bool sk = num_splits == 0 && p->splits == 1 && slots1 > 0 && base < slots1;
      if (force_sk() >= 0) sk = force_sk() == 1 && slots1 > 0;
      if (sk) p->sk = slots1;
      // D2F_ATTN_SK_GRID moves the share boundaries (a test switch; any grid is
      // correct, the CTAs never wait on one another)
      if (const char *e = getenv("D2F_ATTN_SK_GRID"))
        if (sk && atoi(e) > 0) p->sk = min(atoi(e), 65535);
    }
    {
      const long long ctas = (long long)max(batch, 1) * Hkv * p->m_tiles * p->splits;
      const bool whole_sm = D == 128 && (p->stages == 6 || p->mt > 1);
      const long long slots = whole_sm ? attn_tc_deep_slots(p->splits) : 2LL * sms;
      const char *ev = getenv("D2F_LONGEST_FIRST");  // 1 / 0: force on / off (tests)
      const bool want = (ev && ev[0]) ? ev[0] == '1' : ctas > slots;
      p->longest_first = batch > 1 && batch <= kMaxLongestFirstBatch && want;
    }
    p->tiles_per_split = cdiv(t_max, p->splits);
    p->n_counters = 0;
    p->off_ml = p->off_o = p->off_sk = p->bytes = 0;
    if (p->sk) {  // pair counters, then 2 slots per CTA
      p->off_sk = align_up((size_t)max(batch, 1) * Hkv * sizeof(int32_t));
      p->bytes = p->off_sk + (size_t)2 * p->sk * kSkSlotBytes;
    }
    return D2F_OK;
  }
  p->sk = 0;
  p->off_sk = 0;
  if (splits == 0) {
    const int sms = num_sms_current_device();
    const long long target = sms > 0 ? 4LL * sms : 1;
    splits = (int)max(1LL, target / base);
    splits = min(splits, t_max);
  }
  p->splits = splits;
  p->n_counters = max(batch, 1) * Hkv * max(1, cdiv((long long)G * max_q, kSimtRows));
  const size_t n_hr = (size_t)total_q * Hq;
  p->off_ml = align_up((size_t)p->n_counters * sizeof(int32_t));
  if (splits > 1) {
    p->off_o = p->off_ml + align_up((size_t)splits * n_hr * sizeof(float2));
    p->bytes = p->off_o + align_up((size_t)splits * n_hr * D * sizeof(float));
  } else {
    p->off_o = p->off_ml;
    p->bytes = p->off_ml;
  }
  return D2F_OK;
}

// ---------------------------------------------------------------------------
// Commit plan
// ---------------------------------------------------------------------------
constexpr int kCommitThreads = 256;
constexpr int kCommitMaxSplits = 64;

struct CommitPlan {
  int splits, chunk;
  size_t off_blkcnt, off_seqcnt, off_blkgap, off_rowarg, off_partial, bytes;
};

int plan_commit(int total_q, int vocab, int dtype, int B, int num_splits, CommitPlan *p) {
  if (total_q < 0 || vocab <= 0)
    return fail(D2F_ERR_INVALID_ARG, "total_q %d / vocab %d out of range", total_q, vocab);
  if (dtype != D2F_BF16 && dtype != D2F_F32)
    return fail(D2F_ERR_INVALID_ARG, "dtype must be D2F_BF16 or D2F_F32");
  if (B < 1 || B > 32) return fail(D2F_ERR_UNSUPPORTED, "commit supports block_size 1..32 (got %d)", B);
  if (total_q % B != 0)
    return fail(D2F_ERR_INVALID_ARG, "total_q %d is not a multiple of block_size %d", total_q, B);
  if (total_q > 65535) return fail(D2F_ERR_UNSUPPORTED, "total_q must be <= 65535");
  if (num_splits < 0 || num_splits > kCommitMaxSplits)
    return fail(D2F_ERR_INVALID_ARG, "num_splits must be in [0, %d]", kCommitMaxSplits);
  const int elt = dtype == D2F_BF16 ? 2 : 4;
  const int vec = 16 / elt;
  int splits = num_splits;
  if (splits == 0) {
    // At most four CTAs per SM over the whole grid (one slice per row once the
    // rows alone fill that), and at least 2048 logits per slice: long slices
    // amortise each CTA's fixed chain (decode-state read, reduction, arrival),
    // enough CTAs keep every SM's loads in flight. Measured on GB300 (commit µs,
    // 126,464 or 152,064 bf16 logits per row, every row masked): 48 rows -> 12
    // slices 9.6 (10.2 at 8 or 16, 13.4 at 2); 128 rows -> 4 slices 18.5 (20.5
    // at 2 or 5); 256 -> 2 slices 24.7 (27.4 at 1, 27.6 at 3); 384 -> 1 slice
    // 32.2 (34.7 at 2); 512 -> 1 slice 37.1 (42.1 at 2). Rows that are no
    // longer masked read nothing, so the count over-states the work of a window
    // with many committed rows: 464 rows of which half are masked take 34.3 at
    // one slice, 31.2 at two, 27.3 at three. A caller that knows its masked
    // count passes num_splits.
    const int sms = max(1, num_sms_current_device());
    const long long rows = max(total_q, 1);
    splits = (int)((4LL * sms) / rows);
    splits = max(1, min(splits, kCommitMaxSplits));
    splits = max(1, min(splits, vocab / 2048));
  }
  const int chunk = cdiv(cdiv(vocab, splits), vec) * vec;
  splits = cdiv(vocab, chunk);
  p->splits = splits;
  p->chunk = chunk;
  // Counters first: their place does not depend on the split count, so one
  // zeroed workspace stays valid across calls with different splits.
  const size_t nq = (size_t)total_q;
  p->off_blkcnt = 0;
  p->off_seqcnt = align_up((nq / B + 1) * sizeof(int32_t));
  p->off_blkgap = p->off_seqcnt + align_up((nq / B + 1) * sizeof(int32_t));
  p->off_rowarg = p->off_blkgap + align_up((nq / B + 1) * sizeof(float));
  p->off_partial = p->off_rowarg + align_up((nq + 1) * sizeof(int32_t));
  p->bytes = p->off_partial + align_up(nq * splits * sizeof(float4));
  return D2F_OK;
}

}  // namespace

// The leading bytes of a commit workspace that must be zero before a call (the
// per-block and per-sequence arrival counters; the rest is written before it is
// read).
int commit_zeroed_prefix(int total_q, int vocab, int dtype, int block_size, int num_splits,
                         size_t *bytes) {
  CommitPlan p{};
  const int st = plan_commit(total_q, vocab, dtype, block_size, num_splits, &p);
  if (st != D2F_OK) return st;
  *bytes = p.off_blkgap;
  return D2F_OK;
}

}  // namespace d2f

using namespace d2f;


extern "C" {

int d2f_version(void) { return 100; }

const char *d2f_status_string(int status) {
  switch (status) {
    case D2F_OK: return "ok";
    case D2F_ERR_INVALID_ARG: return "invalid argument";
    case D2F_ERR_UNSUPPORTED: return "unsupported configuration";
    case D2F_ERR_CUDA: return "CUDA error";
    case D2F_ERR_BAD_INDEX: return "index out of range (device)";
    case D2F_ERR_TIMEOUT: return "bounded wait timed out (device)";
    case D2F_ERR_WORKSPACE: return "workspace missing or too small";
    case D2F_ERR_NO_PAGE: return "a finished block got no page (device)";
    default: return "unknown status";
  }
}

const char *d2f_last_error_string(void) { return g_last_error; }

int d2f_block_attn_workspace_size(int batch, int total_q, int max_q_per_seq, int max_ctx,
                                  int num_heads_q, int num_heads_kv, int head_dim, int block_size,
                                  int dtype, int num_splits, size_t *bytes) {
  if (!bytes) return fail(D2F_ERR_INVALID_ARG, "bytes is NULL");
  AttnPlan p{};
  const int st = plan_attn(batch, total_q, max_q_per_seq, max_ctx, num_heads_q, num_heads_kv,
                           head_dim, block_size, dtype, num_splits, &p);
  if (st != D2F_OK) return st;
  *bytes = p.bytes;
  return D2F_OK;
}

namespace {
int attn_entry(const void *q, const void *k_win, const void *v_win, const void *k_pool,
               const void *v_pool, const int32_t *page_table, int max_pages_per_seq,
               const int32_t *ctx_len, const int32_t *q_start, void *out, float *lse_out,
               int batch, int total_q, int max_q_per_seq, int max_ctx, int num_heads_q,
               int num_heads_kv, int head_dim, int block_size, int num_pages, int dtype,
               float softmax_scale, int num_splits, void *workspace, size_t workspace_bytes,
               const int32_t *src_row, const int32_t *dst_page, int n_append,
               const int32_t *n_append_dev, int part, const void *prev_out,
               const float *prev_lse, int32_t *err_word, void *stream, unsigned flags = 0) {
  if (n_append < 0) return fail(D2F_ERR_INVALID_ARG, "n_append %d < 0", n_append);
  if (flags & ~D2F_ATTN_CACHE_READY) return fail(D2F_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
  if (part < D2F_ATTN_ALL || part > D2F_ATTN_WINDOW)
    return fail(D2F_ERR_INVALID_ARG, "part %d is not a D2F_ATTN_* value", part);
  if (part == D2F_ATTN_CACHED && !lse_out)
    return fail(D2F_ERR_INVALID_ARG, "the cached part needs lse_out (its normaliser is kept)");
  if ((prev_out == nullptr) != (prev_lse == nullptr) || (prev_out && part != D2F_ATTN_WINDOW))
    return fail(D2F_ERR_INVALID_ARG, "prev_out / prev_lse go together, with D2F_ATTN_WINDOW");
  if (prev_out && !aligned16(prev_out))
    return fail(D2F_ERR_INVALID_ARG, "device buffers must be 16-byte aligned");
  // the window part reads no cached page: plan it as a window-only attention
  if (part == D2F_ATTN_WINDOW) max_ctx = 0;
  if (n_append > 0 && (!src_row || !dst_page || !k_pool || !v_pool || num_pages <= 0))
    return fail(D2F_ERR_INVALID_ARG, "an append needs src_row, dst_page, k_pool, v_pool and pages");
  AttnPlan p{};
  int st = plan_attn(batch, total_q, max_q_per_seq, max_ctx, num_heads_q, num_heads_kv, head_dim,
                     block_size, dtype, num_splits, &p);
  if (st != D2F_OK) return st;
  if (batch == 0 || total_q == 0) return D2F_OK;
  if (!q || !k_win || !v_win || !out || !ctx_len || !q_start)
    return fail(D2F_ERR_INVALID_ARG, "a required pointer is NULL");
  if (max_pages_per_seq < 0 || num_pages < 0)
    return fail(D2F_ERR_INVALID_ARG, "max_pages_per_seq / num_pages negative");
  if ((long long)max_pages_per_seq * block_size < max_ctx)
    return fail(D2F_ERR_INVALID_ARG, "max_ctx %d exceeds max_pages_per_seq * block_size", max_ctx);
  if (max_ctx > 0 && (!k_pool || !v_pool || !page_table || num_pages <= 0))
    return fail(D2F_ERR_INVALID_ARG, "a cached context needs k_pool, v_pool, page_table and pages");
  if (!(softmax_scale > 0.f)) return fail(D2F_ERR_INVALID_ARG, "softmax_scale must be > 0");
  const void *ptrs[] = {q, k_win, v_win, k_pool, v_pool, out};
  for (const void *x : ptrs)
    if (x && !aligned16(x)) return fail(D2F_ERR_INVALID_ARG, "device buffers must be 16-byte aligned");
  if (p.bytes > 0 && (!workspace || workspace_bytes < p.bytes))
    return fail(D2F_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", p.bytes,
                workspace ? workspace_bytes : (size_t)0);

  AttnArgs a;
  a.q = q;
  a.k_win = k_win;
  a.v_win = v_win;
  // With no pages at all, the pool maps point at the window so they stay encodable;
  // no cached tile is ever read then (every ctx_len must be 0).
  a.k_pool = (num_pages > 0 && k_pool) ? k_pool : k_win;
  a.v_pool = (num_pages > 0 && v_pool) ? v_pool : v_win;
  a.page_table = page_table;
  a.max_pages_per_seq = max_pages_per_seq;
  a.ctx_len = ctx_len;
  a.q_start = q_start;
  a.out = out;
  a.lse_out = lse_out;
  a.batch = batch;
  a.total_q = total_q;
  a.max_q_per_seq = max_q_per_seq;
  a.num_heads_q = num_heads_q;
  a.num_heads_kv = num_heads_kv;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_pages = num_pages > 0 ? num_pages : 1;
  a.group = num_heads_q / num_heads_kv;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.num_splits = p.splits;
  a.tiles_per_split = p.tiles_per_split;
  a.m_tiles = p.m_tiles;
  a.tc_rows = p.rows;
  a.tc_stages = p.stages;
  a.tc_mt = p.mt > 0 ? p.mt : 1;
  a.longest_first = p.longest_first ? 1 : 0;
  // D2F_WAIT_CYCLES shortens the budget of the waits on another role's work (a
  // test switch for the give-up path; copies and MMAs are still drained in full)
  a.wait_cycles = kWaitCycles;
  if (const char *e = getenv("D2F_WAIT_CYCLES")) {
    const long long v = atoll(e);
    if (v > 0 && v < kWaitCycles) a.wait_cycles = v;
  }
  a.cache_ready = (flags & D2F_ATTN_CACHE_READY) ? 1 : 0;
  // the stream-K form computes the whole attention only: no fused append, no part
  a.sk = (p.sk > 0 && part == D2F_ATTN_ALL && n_append == 0 && !prev_out) ? p.sk : 0;
  a.sk_cnt = reinterpret_cast<int32_t *>(workspace);
  a.sk_slots = reinterpret_cast<uint8_t *>(static_cast<char *>(workspace) + p.off_sk);
  a.counters = reinterpret_cast<int32_t *>(workspace);
  a.ws_ml = reinterpret_cast<float2 *>(static_cast<char *>(workspace) + p.off_ml);
  a.ws_o = reinterpret_cast<float *>(static_cast<char *>(workspace) + p.off_o);
  a.err = err_word;
  if (part != D2F_ATTN_ALL && !p.tc)
    return fail(D2F_ERR_UNSUPPORTED, "attention parts run on the tensor-core path (bf16, head_dim "
                "64/128, block 8/16/32)");
  a.part = part;
  a.prev_out = prev_out;
  a.prev_lse = prev_lse;
  // fused append on the tensor-core path; the CUDA-core path appends after
  a.n_append = p.tc ? n_append : 0;
  a.app_n_dev = n_append_dev;
  a.app_src = src_row;
  a.app_dst = dst_page;
  if (num_pages <= 0 && max_ctx > 0) return fail(D2F_ERR_INVALID_ARG, "no pages");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (p.tc) {
    char why[256] = "";
    e = launch_attn_tc(a, s, why, sizeof why);
    if (e != cudaSuccess) {
      if (why[0]) return fail(D2F_ERR_CUDA, "tensor-core attention: %s (%s)", why, cudaGetErrorString(e));
      return cuda_fail(e, "tensor-core attention launch");
    }
  } else {
    e = launch_attn_simt(a, dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "CUDA-core attention launch");
    if (n_append > 0 && n_append_dev)
      return d2f_kv_append_dev(k_win, v_win, src_row, dst_page, n_append_dev, n_append, total_q,
                               const_cast<void *>(k_pool), const_cast<void *>(v_pool),
                               num_heads_kv, head_dim, block_size, num_pages, dtype, err_word,
                               stream);
    if (n_append > 0)
      return d2f_kv_append(k_win, v_win, src_row, dst_page, n_append, total_q, const_cast<void *>(k_pool),
                           const_cast<void *>(v_pool), num_heads_kv, head_dim, block_size, num_pages,
                           dtype, err_word, stream);
  }
  return D2F_OK;
}
}  // namespace

int d2f_block_attn_append(const void *q, const void *k_win, const void *v_win, const void *k_pool,
                          const void *v_pool, const int32_t *page_table, int max_pages_per_seq,
                          const int32_t *ctx_len, const int32_t *q_start, void *out,
                          float *lse_out, int batch, int total_q, int max_q_per_seq, int max_ctx,
                          int num_heads_q, int num_heads_kv, int head_dim, int block_size,
                          int num_pages, int dtype, float softmax_scale, int num_splits,
                          void *workspace, size_t workspace_bytes, const int32_t *src_row,
                          const int32_t *dst_page, int n_append, int32_t *err_word,
                          void *stream) {
  return attn_entry(q, k_win, v_win, k_pool, v_pool, page_table, max_pages_per_seq, ctx_len,
                    q_start, out, lse_out, batch, total_q, max_q_per_seq, max_ctx, num_heads_q,
                    num_heads_kv, head_dim, block_size, num_pages, dtype, softmax_scale, num_splits,
                    workspace, workspace_bytes, src_row, dst_page, n_append, nullptr, D2F_ATTN_ALL,
                    nullptr, nullptr, err_word, stream);
}

int d2f_block_attn_append_dev(const void *q, const void *k_win, const void *v_win,
                              const void *k_pool, const void *v_pool, const int32_t *page_table,
                              int max_pages_per_seq, const int32_t *ctx_len,
                              const int32_t *q_start, void *out, float *lse_out, int batch,
                              int total_q, int max_q_per_seq, int max_ctx, int num_heads_q,
                              int num_heads_kv, int head_dim, int block_size, int num_pages,
                              int dtype, float softmax_scale, int num_splits, void *workspace,
                              size_t workspace_bytes, const int32_t *src_row,
                              const int32_t *dst_page, const int32_t *n_append_dev,
                              int max_append, int32_t *err_word, void *stream) {
  if (!n_append_dev) return fail(D2F_ERR_INVALID_ARG, "n_append_dev is NULL");
  return attn_entry(q, k_win, v_win, k_pool, v_pool, page_table, max_pages_per_seq, ctx_len,
                    q_start, out, lse_out, batch, total_q, max_q_per_seq, max_ctx, num_heads_q,
                    num_heads_kv, head_dim, block_size, num_pages, dtype, softmax_scale, num_splits,
                    workspace, workspace_bytes, src_row, dst_page, max_append, n_append_dev,
                    D2F_ATTN_ALL, nullptr, nullptr, err_word, stream);
}

int d2f_block_attn_part(const void *q, const void *k_win, const void *v_win, const void *k_pool,
                        const void *v_pool, const int32_t *page_table, int max_pages_per_seq,
                        const int32_t *ctx_len, const int32_t *q_start, void *out, float *lse_out,
                        int batch, int total_q, int max_q_per_seq, int max_ctx, int num_heads_q,
                        int num_heads_kv, int head_dim, int block_size, int num_pages, int dtype,
                        float softmax_scale, int num_splits, void *workspace,
                        size_t workspace_bytes, int part, const void *prev_out,
                        const float *prev_lse, int32_t *err_word, void *stream) {
  return attn_entry(q, k_win, v_win, k_pool, v_pool, page_table, max_pages_per_seq, ctx_len,
                    q_start, out, lse_out, batch, total_q, max_q_per_seq, max_ctx, num_heads_q,
                    num_heads_kv, head_dim, block_size, num_pages, dtype, softmax_scale, num_splits,
                    workspace, workspace_bytes, nullptr, nullptr, 0, nullptr, part, prev_out,
                    prev_lse, err_word, stream);
}

int d2f_block_attn(const void *q, const void *k_win, const void *v_win, const void *k_pool,
                   const void *v_pool, const int32_t *page_table, int max_pages_per_seq,
                   const int32_t *ctx_len, const int32_t *q_start, void *out, float *lse_out,
                   int batch, int total_q, int max_q_per_seq, int max_ctx, int num_heads_q,
                   int num_heads_kv, int head_dim, int block_size, int num_pages, int dtype,
                   float softmax_scale, int num_splits, void *workspace, size_t workspace_bytes,
                   int32_t *err_word, void *stream) {
  return attn_entry(q, k_win, v_win, k_pool, v_pool, page_table, max_pages_per_seq, ctx_len,
                    q_start, out, lse_out, batch, total_q, max_q_per_seq, max_ctx, num_heads_q,
                    num_heads_kv, head_dim, block_size, num_pages, dtype, softmax_scale, num_splits,
                    workspace, workspace_bytes, nullptr, nullptr, 0, nullptr, D2F_ATTN_ALL, nullptr,
                    nullptr, err_word, stream);
}

int d2f_block_attn_flags(const void *q, const void *k_win, const void *v_win, const void *k_pool,
                         const void *v_pool, const int32_t *page_table, int max_pages_per_seq,
                         const int32_t *ctx_len, const int32_t *q_start, void *out,
                         float *lse_out, int batch, int total_q, int max_q_per_seq, int max_ctx,
                         int num_heads_q, int num_heads_kv, int head_dim, int block_size,
                         int num_pages, int dtype, float softmax_scale, int num_splits,
                         void *workspace, size_t workspace_bytes, unsigned flags,
                         int32_t *err_word, void *stream) {
  return attn_entry(q, k_win, v_win, k_pool, v_pool, page_table, max_pages_per_seq, ctx_len,
                    q_start, out, lse_out, batch, total_q, max_q_per_seq, max_ctx, num_heads_q,
                    num_heads_kv, head_dim, block_size, num_pages, dtype, softmax_scale, num_splits,
                    workspace, workspace_bytes, nullptr, nullptr, 0, nullptr, D2F_ATTN_ALL, nullptr,
                    nullptr, err_word, stream, flags);
}

int d2f_commit_workspace_size(int total_q, int vocab, int dtype, int block_size, int num_splits,
                              size_t *bytes) {
  if (!bytes) return fail(D2F_ERR_INVALID_ARG, "bytes is NULL");
  CommitPlan p{};
  const int st = plan_commit(total_q, vocab, dtype, block_size, num_splits, &p);
  if (st != D2F_OK) return st;
  *bytes = p.bytes;
  return D2F_OK;
}

int d2f_commit_metric(const void *logits, int64_t row_stride, int dtype, int vocab,
                      int num_logit_rows, const int32_t *logit_row, int32_t *tokens,
                      uint8_t *masked, const int32_t *q_start, const uint8_t *block_phase,
                      const float *tau, int batch, int total_q, int block_size, int32_t mask_id,
                      int metric, const float *early_gap, uint8_t *stopped, float *conf_out,
                      int32_t *argmax_out, int32_t *block_remaining, int num_splits,
                      void *workspace, size_t workspace_bytes, int32_t *err_word, void *stream) {
  if (metric < D2F_CONF_PMAX || metric > D2F_CONF_LOGIT_GAP)
    return fail(D2F_ERR_INVALID_ARG, "metric %d is not a D2F_CONF_* value", metric);
  if (early_gap && metric == D2F_CONF_NEG_ENTROPY)
    return fail(D2F_ERR_UNSUPPORTED, "the early commit combines with D2F_CONF_PMAX, _MARGIN or "
                "_LOGIT_GAP, not with D2F_CONF_NEG_ENTROPY");
  CommitPlan p{};
  int st = plan_commit(total_q, vocab, dtype, block_size, num_splits, &p);
  if (st != D2F_OK) return st;
  if (batch < 1) return fail(D2F_ERR_INVALID_ARG, "batch must be >= 1");
  if (total_q == 0) return D2F_OK;
  if (!logits || !tokens || !masked || !q_start || !block_phase || !tau)
    return fail(D2F_ERR_INVALID_ARG, "a required pointer is NULL");
  if (row_stride < vocab) return fail(D2F_ERR_INVALID_ARG, "row_stride < vocab");
  if (num_logit_rows <= 0) return fail(D2F_ERR_INVALID_ARG, "num_logit_rows must be > 0");
  if (!workspace || workspace_bytes < p.bytes)
    return fail(D2F_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", p.bytes,
                workspace ? workspace_bytes : (size_t)0);
  const int elt = dtype == D2F_BF16 ? 2 : 4;
  const bool vec_ok = aligned16(logits) && ((row_stride * elt) % 16 == 0);
  const int path = vec_ok ? 1 : 0;
  CommitArgs a;
  a.logits = logits;
  a.row_stride = row_stride;
  a.vocab = vocab;
  a.num_logit_rows = num_logit_rows;
  a.logit_row = logit_row;
  a.tokens = tokens;
  a.masked = masked;
  a.q_start = q_start;
  a.block_phase = block_phase;
  a.tau = tau;
  a.batch = batch;
  a.total_q = total_q;
  a.block_size = block_size;
  a.mask_id = mask_id;
  a.conf_out = conf_out;
  a.argmax_out = argmax_out;
  a.block_remaining = block_remaining;
  a.splits = p.splits;
  a.chunk = p.chunk;
  char *ws = static_cast<char *>(workspace);
  a.partial = reinterpret_cast<float4 *>(ws + p.off_partial);
  a.blk_cnt = reinterpret_cast<int32_t *>(ws + p.off_blkcnt);
  a.err = err_word;
  a.metric = metric;
  a.early_gap = early_gap;
  a.stopped = stopped;
  a.seq_cnt = reinterpret_cast<int32_t *>(ws + p.off_seqcnt);
  a.blk_gap = reinterpret_cast<float *>(ws + p.off_blkgap);
  a.row_arg = reinterpret_cast<int32_t *>(ws + p.off_rowarg);
  const cudaError_t e = launch_commit(a, dtype, path, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "commit launch");
  return D2F_OK;
}

int d2f_commit(const void *logits, int64_t row_stride, int dtype, int vocab, int num_logit_rows,
               const int32_t *logit_row, int32_t *tokens, uint8_t *masked,
               const int32_t *q_start, const uint8_t *block_phase, const float *tau, int batch,
               int total_q, int block_size, int32_t mask_id, float *conf_out,
               int32_t *argmax_out, int32_t *block_remaining, int num_splits, void *workspace,
               size_t workspace_bytes, int32_t *err_word, void *stream) {
  return d2f_commit_metric(logits, row_stride, dtype, vocab, num_logit_rows, logit_row, tokens,
                           masked, q_start, block_phase, tau, batch, total_q, block_size, mask_id,
                           D2F_CONF_PMAX, nullptr, nullptr, conf_out, argmax_out, block_remaining,
                           num_splits, workspace, workspace_bytes, err_word, stream);
}

namespace {
int append_entry(const void *k_win, const void *v_win, const int32_t *src_row,
                 const int32_t *dst_page, int n_append, const int32_t *n_append_dev, int total_q,
                 void *k_pool, void *v_pool, int num_heads_kv, int head_dim, int block_size,
                 int num_pages, int dtype, int32_t *err_word, void *stream) {
  if (n_append < 0 || total_q < 0 || num_heads_kv <= 0 || head_dim <= 0 || block_size < 1 ||
      num_pages < 0)
    return fail(D2F_ERR_INVALID_ARG, "size out of range");
  if (dtype != D2F_BF16 && dtype != D2F_F32)
    return fail(D2F_ERR_INVALID_ARG, "dtype must be D2F_BF16 or D2F_F32");
  if ((long long)n_append * num_heads_kv > 0x7fffffffLL)
    return fail(D2F_ERR_UNSUPPORTED, "n_append * num_heads_kv too large");
  if (n_append == 0) return D2F_OK;
  if (!k_win || !v_win || !src_row || !dst_page || !k_pool || !v_pool)
    return fail(D2F_ERR_INVALID_ARG, "a required pointer is NULL");
  const int elt = dtype == D2F_BF16 ? 2 : 4;
  AppendArgs a;
  a.k_win = k_win;
  a.v_win = v_win;
  a.src_row = src_row;
  a.dst_page = dst_page;
  a.n_append = n_append;
  a.n_dev = n_append_dev;
  a.total_q = total_q;
  a.k_pool = k_pool;
  a.v_pool = v_pool;
  a.num_heads_kv = num_heads_kv;
  a.block_size = block_size;
  a.num_pages = num_pages;
  a.row_bytes = head_dim * elt;
  a.err = err_word;
  const bool vec_ok = aligned16(k_win) && aligned16(v_win) && aligned16(k_pool) &&
                      aligned16(v_pool) && (a.row_bytes % 16 == 0);
  const cudaError_t e = launch_append(a, vec_ok, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "kv_append launch");
  return D2F_OK;
}
}  // namespace

int d2f_kv_append(const void *k_win, const void *v_win, const int32_t *src_row,
                  const int32_t *dst_page, int n_append, int total_q, void *k_pool,
                  void *v_pool, int num_heads_kv, int head_dim, int block_size, int num_pages,
                  int dtype, int32_t *err_word, void *stream) {
  return append_entry(k_win, v_win, src_row, dst_page, n_append, nullptr, total_q, k_pool, v_pool,
                      num_heads_kv, head_dim, block_size, num_pages, dtype, err_word, stream);
}

int d2f_kv_append_dev(const void *k_win, const void *v_win, const int32_t *src_row,
                      const int32_t *dst_page, const int32_t *n_append_dev, int max_append,
                      int total_q, void *k_pool, void *v_pool, int num_heads_kv, int head_dim,
                      int block_size, int num_pages, int dtype, int32_t *err_word, void *stream) {
  if (!n_append_dev) return fail(D2F_ERR_INVALID_ARG, "n_append_dev is NULL");
  return append_entry(k_win, v_win, src_row, dst_page, max_append, n_append_dev, total_q, k_pool,
                      v_pool, num_heads_kv, head_dim, block_size, num_pages, dtype, err_word,
                      stream);
}

int d2f_window_step(int batch, int block_size, int max_blocks, int capacity,
                    int max_pages_per_seq, int32_t mask_id, float tau_add, float tau_act,
                    int32_t *q_start, int32_t *tokens, uint8_t *masked, uint8_t *block_phase,
                    int32_t *row_pos, int32_t *ctx_len, int32_t *page_table, int32_t *next_block,
                    const int32_t *gen_blocks, int32_t *n_leaving, const uint8_t *stopped,
                    const int32_t *free_pages, int32_t *free_count, int32_t *app_src,
                    int32_t *app_dst, int32_t *n_append, int32_t *err_word, void *stream) {
  if (batch < 0 || block_size < 1 || max_blocks < 1 || capacity < 0 || max_pages_per_seq < 0)
    return fail(D2F_ERR_INVALID_ARG, "size out of range");
  if (capacity % block_size != 0)
    return fail(D2F_ERR_INVALID_ARG, "capacity %d is not a multiple of block_size %d", capacity,
                block_size);
  if ((long long)batch * max_blocks * block_size > capacity)
    return fail(D2F_ERR_INVALID_ARG, "capacity %d < batch * max_blocks * block_size", capacity);
  if (tau_add != tau_add || tau_act != tau_act)
    return fail(D2F_ERR_INVALID_ARG, "tau_add / tau_act must not be NaN");
  if (block_size > 128) return fail(D2F_ERR_UNSUPPORTED, "block_size > 128");
  const size_t smem = d2f::window_smem_bytes(batch, capacity, block_size);
  if (smem > 227 * 1024)
    return fail(D2F_ERR_UNSUPPORTED, "window state of %zu bytes exceeds one CTA's shared memory",
                smem);
  if (!q_start || !tokens || !masked || !block_phase || !row_pos || !ctx_len || !next_block ||
      !gen_blocks || !n_leaving || !free_pages || !free_count || !app_src || !app_dst ||
      !n_append || (!page_table && max_pages_per_seq > 0))
    return fail(D2F_ERR_INVALID_ARG, "a required pointer is NULL");
  d2f::WindowArgs a;
  a.batch = batch;
  a.block_size = block_size;
  a.max_blocks = max_blocks;
  a.capacity = capacity;
  a.max_pages_per_seq = max_pages_per_seq;
  a.mask_id = mask_id;
  a.tau_add = tau_add;
  a.tau_act = tau_act;
  a.q_start = q_start;
  a.tokens = tokens;
  a.masked = masked;
  a.block_phase = block_phase;
  a.row_pos = row_pos;
  a.ctx_len = ctx_len;
  a.page_table = page_table;
  a.next_block = next_block;
  a.gen_blocks = gen_blocks;
  a.n_leaving = n_leaving;
  a.stopped = stopped;
  a.free_pages = free_pages;
  a.free_count = free_count;
  a.app_src = app_src;
  a.app_dst = app_dst;
  a.n_append = n_append;
  a.err = err_word;
  const cudaError_t e = d2f::launch_window(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "window step launch");
  return D2F_OK;
}

}  // extern "C"
