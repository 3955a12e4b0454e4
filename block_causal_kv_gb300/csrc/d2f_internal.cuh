// Internal declarations shared by the libd2f translation units: launch
// argument structs, status plumbing and thin inline-PTX wrappers for the
// Blackwell (sm_103a) async machinery (mbarrier, TMA, tcgen05 / TMEM).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "d2f.h"

namespace d2f {

// ---------------------------------------------------------------------------
// Host-side plumbing
// ---------------------------------------------------------------------------
void set_last_error(const char *fmt, ...);
int num_sms_current_device();
// Bytes at the start of a commit workspace that must be zero before a call (its
// arrival counters); the plan of d2f_commit_workspace_size.
int commit_zeroed_prefix(int total_q, int vocab, int dtype, int block_size, int num_splits,
                         size_t *bytes);
// Programmatic dependent launch on every kernel launch unless D2F_PDL=0 (a
// switch for comparing launch overlap; results are identical either way).
bool pdl_enabled();

// Bounded waits give up after this many SM clock cycles (about one second at
// the GB300's clocks), set D2F_ERR_TIMEOUT in the error word and unwind.
constexpr long long kWaitCycles = 2000000000LL;
// Waits that only drain work this CTA already issued (copies landing, MMAs
// completing) give up after ~0.1 s: far longer than a copy or an MMA takes, even
// under a profiler's instrumented replay (where a 2e6-cycle budget, ~1 ms, was
// measured to run out and report a false time-out). After another role gave up,
// such a wait may be on a phase that can no longer complete (a stage that one
// producer issued and another abandoned); it then ends here instead of after
// kWaitCycles.
constexpr long long kDrainCycles = 200000000LL;

// ---------------------------------------------------------------------------
// Launch arguments
// ---------------------------------------------------------------------------
struct AttnArgs {
  const void *q, *k_win, *v_win, *k_pool, *v_pool;
  const int32_t *page_table;
  int max_pages_per_seq;
  const int32_t *ctx_len, *q_start;
  void *out;
  float *lse_out;
  int batch, total_q, max_q_per_seq, num_heads_q, num_heads_kv, head_dim, block_size, num_pages;
  int group;             // num_heads_q / num_heads_kv
  float scale_log2;      // softmax_scale * log2(e)
  int num_splits;        // split count requested (each sequence uses <= this many)
  int tiles_per_split;   // tensor-core path: key tiles per split from the host's max_ctx
  int m_tiles;           // grid.x: row tiles per (sequence, KV head)
  int tc_rows;           // tensor-core path: rows a tile holds (64 or 128)
  int tc_stages;         // tensor-core path: K/V ring depth (2 .. 6)
  int tc_mt;             // tensor-core path: row tiles per CTA, a softmax warpgroup each (1, 2)
  int longest_first;     // tensor-core path: map blockIdx.z to sequences longest context first
  const int32_t *app_src;  // tensor-core path, fused append: window rows of finished blocks
  const int32_t *app_dst;  // ... and their pages; n_append = 0: no append
  int n_append;            // entries (with app_n_dev: the most the list can hold)
  const int32_t *app_n_dev;  // non-null: the list's length, read on the device
  int part;                // tensor-core path: keys attended: 0 all, 1 cached only, 2 window only
  const void *prev_out;    // part 2: a kept cached part to compose with ([total_q][Hq][D], as out)
  const float *prev_lse;   // ... its natural-log normaliser [total_q][Hq]; NULL: no composition
  long long wait_cycles; // tensor-core path: budget of each wait on another role's work
                         // (kWaitCycles; less only to test the give-up path)
  int cache_ready;        // D2F_ATTN_CACHE_READY: producers may load cached tiles before
                         // the dependency wait
  int sk;                // tensor-core path: stream-K form (see attn_tc.cu), else 0
  int32_t *sk_cnt;       // stream-K: [batch * Hkv] arrival counters (zero at rest)
  uint8_t *sk_slots;     // stream-K: [2 * grid] partial slots of kSkSlotBytes
  int32_t *counters;     // [batch * Hkv * m_tiles] merge arrival counters (zero at rest)
  float2 *ws_ml;         // [num_splits][total_q * Hq] (max in log2 units, sum)
  float *ws_o;           // [num_splits][total_q * Hq][head_dim] unnormalised partial output
  int32_t *err;
};

struct CommitArgs {
  const void *logits;
  int64_t row_stride;
  int vocab, num_logit_rows;
  const int32_t *logit_row;
  int32_t *tokens;
  uint8_t *masked;
  const int32_t *q_start;
  const uint8_t *block_phase;
  const float *tau;
  int batch, total_q, block_size;
  int32_t mask_id;
  float *conf_out;
  int32_t *argmax_out, *block_remaining;
  int splits;            // CTAs per row
  int chunk;             // vocabulary entries per CTA
  float4 *partial;       // [total_q][splits] (max, argmax bits, sum, metric term)
  int metric;            // D2F_CONF_*: confidence compared with tau
  const float *early_gap;  // [batch] early-commit logit-gap thresholds, or NULL (off)
  uint8_t *stopped;        // [batch] early-commit flags out, or NULL
  int32_t *seq_cnt;        // [total_q / block_size] block arrivals per sequence, at its first block
  float *blk_gap;          // [total_q / block_size] smallest logit gap over a block's masked rows
  int32_t *row_arg;        // [total_q] greedy token of every masked row
  int32_t *blk_cnt;      // [total_q / block_size] arrivals per block (zero at rest)
  int32_t *err;
};

struct AppendArgs {
  const void *k_win, *v_win;
  const int32_t *src_row, *dst_page;
  int n_append, total_q;   // n_append: entries (with n_dev: the most the list can hold)
  const int32_t *n_dev;    // non-null: the list's length, read on the device
  void *k_pool, *v_pool;
  int num_heads_kv, block_size, num_pages;
  int row_bytes;         // head_dim * element size
  int32_t *err;
};

struct WindowArgs {
  int batch, block_size, max_blocks, capacity, max_pages_per_seq;
  int32_t mask_id;
  float tau_add, tau_act;
  int32_t *q_start, *tokens;
  uint8_t *masked, *block_phase;
  int32_t *row_pos, *ctx_len, *page_table, *next_block;
  const int32_t *gen_blocks;
  int32_t *n_leaving;
  const uint8_t *stopped;
  const int32_t *free_pages;
  int32_t *free_count, *app_src, *app_dst, *n_append;
  int32_t *err;
};

// Launchers (one per translation unit). Return cudaSuccess or the launch error.
// path: 0 scalar loads, 1 128-bit loads (see commit.cu)
cudaError_t launch_commit(const CommitArgs &a, int dtype, int path, cudaStream_t s);
cudaError_t launch_append(const AppendArgs &a, bool vec_ok, cudaStream_t s);
cudaError_t launch_window(const WindowArgs &a, cudaStream_t s);
size_t window_smem_bytes(int batch, int capacity, int block_size);
cudaError_t launch_attn_simt(const AttnArgs &a, int dtype, cudaStream_t s);
cudaError_t launch_attn_tc(const AttnArgs &a, cudaStream_t s, char *why, size_t why_len);
int attn_tc_deep_slots(int cs);  // resident CTAs of the 6-stage head_dim-128 variant

// Tile and row sizes of the two attention paths (also used for workspace sizing).
constexpr int kSimtRows = 16;   // query rows per CTA, CUDA-core path
constexpr int kSimtKeys = 32;   // keys per tile, CUDA-core path
constexpr int kTcRows = 128;    // query rows per CTA (UMMA M), tensor-core path
constexpr int kTcKeys = 64;     // keys per tile (UMMA N of Q.K^T), tensor-core path
constexpr int kTcMaxSplits = 8; // CTAs per cluster sharing one row tile, tensor-core path
constexpr int kMaxLongestFirstBatch = 256;  // largest batch the longest-first order covers
// Stream-K form of the tensor-core attention (head_dim 128, one 128-row tile per
// (sequence, KV head)): a partial slot holds 128 rows of 128 bf16 then 128
// (max, sum) float pairs; each CTA owns two.
constexpr int kSkSlotBytes = 128 * 128 * 2 + 128 * 8;

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__
__device__ __forceinline__ void set_err(int32_t *err, int code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Round-to-nearest-even float -> bf16 bits (the cvt.rn.bf16.f32 instruction).
__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
  return r;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Sequence metadata check shared by the attention kernels: returns false (and
// records D2F_ERR_INVALID_ARG) when the window rows of sequence b contradict the
// host sizes.
__device__ __forceinline__ bool load_seq_meta(const AttnArgs &a, int b, int &q0, int &n, int &C) {
  q0 = a.q_start[b];
  const int q1 = a.q_start[b + 1];
  C = a.ctx_len[b];
  n = q1 - q0;
  const bool ok = q0 >= 0 && q1 >= q0 && q1 <= a.total_q && (q0 % a.block_size) == 0 &&
                  (n % a.block_size) == 0 && n <= a.max_q_per_seq && C >= 0 &&
                  (long long)C <= (long long)a.max_pages_per_seq * a.block_size;
  return ok;
}

// ----- mbarrier --------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase with the given parity; gives up after `budget` SM cycles
// (kWaitCycles unless a caller passes less) or when another thread of the CTA
// has already given up (shared abort flag).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          int32_t *err, long long budget = kWaitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > budget) {
      *abort_flag = 1;
      set_err(err, D2F_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// ----- TMA (tensor copies global -> shared, completion on an mbarrier) -------
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}
// L2 eviction policies for cache hints: a read-once stream (evict first) and
// data that is read back soon (evict last).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// tma_load_5d with an L2 cache policy
__device__ __forceinline__ void tma_load_5d_hint(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                                 int c0, int c1, int c2, int c3, int c4,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "l"(policy)
      : "memory");
}
// 16-byte global store with an L2 cache policy
__device__ __forceinline__ void st_global_v4_hint(void *ptr, uint4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Generic-proxy shared-memory writes -> visible to the async proxy (UMMA reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// L2 prefetch hint for [src, src + bytes) (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)),
               "r"(bytes)
               : "memory");
}

// ----- thread-block clusters / distributed shared memory --------------------
// Full cluster barrier (every thread of every CTA of the cluster).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// The two halves of cluster_sync(), for work placed between them.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Tensor copy from shared memory to global (bulk async-group completion).
__device__ __forceinline__ void tma_store_5d(const CUtensorMap *map, uint32_t src, int c0, int c1,
                                             int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5, %6}], [%1];" ::
          "l"(reinterpret_cast<uint64_t>(map)), "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(c4)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until this thread's committed bulk stores have read their shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until this thread's committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_group0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 dsmem_ld_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ float4 dsmem_ld_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ----- phase tracing (compiled in only with -DD2F_TRACE; absent otherwise) ----
// Records %globaltimer (ns) per CTA and phase into a fixed device array so a
// development build can show where a kernel's time goes.
#ifdef D2F_TRACE
constexpr int kTraceSlots = 20;
constexpr int kTraceCtas = 8192;
// One array per translation unit (each kernel file has its own copy-out hook).
static __device__ unsigned long long g_d2f_trace[kTraceCtas * kTraceSlots];
__device__ __forceinline__ void trace_mark(int slot) {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  const unsigned cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  if (cta < kTraceCtas) g_d2f_trace[cta * kTraceSlots + slot] = t;
}
#define D2F_TRACE_MARK(kernel, slot) trace_mark(slot)
#define D2F_TRACE_COPY_FN(name)                                                          \
  extern "C" int name(void *host, size_t bytes, int clear) {                             \
    if (bytes > sizeof(g_d2f_trace)) bytes = sizeof(g_d2f_trace);                         \
    if (host && cudaMemcpyFromSymbol(host, g_d2f_trace, bytes) != cudaSuccess) return 1;  \
    void *p = nullptr;                                                                    \
    if (clear && (cudaGetSymbolAddress(&p, g_d2f_trace) != cudaSuccess ||                 \
                  cudaMemset(p, 0, sizeof(g_d2f_trace)) != cudaSuccess))                  \
      return 2;                                                                           \
    return 0;                                                                             \
  }
#else
#define D2F_TRACE_MARK(kernel, slot) ((void)0)
#endif

// Device-scope atomic add with acquire-release semantics: the caller's earlier
// writes are visible to whoever later acquires the counter, and the caller sees
// the writes every earlier arriver released.
__device__ __forceinline__ int atomic_add_acq_rel(int32_t *p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}
// Named barrier among `count` threads (a multiple of 32) of the CTA that also
// returns whether `v` held in every one of them.
__device__ __forceinline__ bool named_sync_and(int id, int count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}
// Named barrier among `count` threads (a multiple of 32) of the CTA.
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ----- programmatic dependent launch ----------------------------------------
// Block until every grid this one depends on has completed and its writes are
// visible (no-op when the launch has no programmatic dependency).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the next grid in the stream to be scheduled; it still waits for this
// grid's completion before reading anything (grid_dependency_wait).
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----- tcgen05 / TMEM ---------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, f32 accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem], bf16 inputs, f32 accumulate (A read from TMEM:
// row i = lane i, two consecutive K elements per 32-bit column, lower K in the
// low half).
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on an mbarrier once every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 32 consecutive 32-bit TMEM columns of this thread's lane, waited for in the
// same asm block so no use of the registers can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// 64 consecutive 32-bit TMEM columns of this thread's lane, one load and one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
      "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]),
        "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]),
        "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
        "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]),
        "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}
// Packed float pairs (Blackwell f32x2 arithmetic, one instruction per pair).
// (d0, d1) = (a0, a1) * b + c
__device__ __forceinline__ void fma2_bc(float &d0, float &d1, float a0, float a1, float b,
                                        float c) {
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %4};\n\t"
      "mov.b64 rc, {%5, %5};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// (d0, d1) = (a0, a1) + (b0, b1)
__device__ __forceinline__ void add2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// Largest of three floats, one instruction (NaN operands are ignored, as fmaxf).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// 2^x for both bf16 halves of a packed pair (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ uint32_t ex2_bf16x2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.ftz.bf16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma, 128-byte swizzle.
//   start address >> 4 in bits 0-13, leading byte offset >> 4 in 16-29,
//   stride byte offset >> 4 in 32-45, descriptor version 1 in bits 46-47,
//   swizzle mode 2 (128B) in bits 61-63.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// The descriptor of the same layout `bytes` further on in shared memory (bytes a
// multiple of 16). Only the start-address field (bits 0-13: address >> 4) moves,
// and it cannot carry into the fields above while the address stays below
// 256 KB, so an issuing loop can build each descriptor with one add.
__device__ __forceinline__ uint64_t smem_desc_advance(uint64_t d, uint32_t bytes) {
  return d + (uint64_t)(bytes >> 4);
}

// Instruction descriptor, kind::f16 with bf16 A/B and f32 accumulator.
//   D format f32 (bits 4-5 = 1), A and B format bf16 (bits 7-9 = 1, 10-12 = 1),
//   A major (bit 15) and B major (bit 16): 0 = K-major, 1 = MN-major,
//   N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn_major,
                                                      int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn_major << 15) |
         ((uint32_t)b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
#endif  // __CUDACC__

}  // namespace d2f
