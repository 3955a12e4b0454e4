// d2f_window_step kernel: the pipelined window scheduler between two decode
// steps, on the device, so that a whole step (attention, commit, scheduler) runs
// from one CUDA graph with no host readback.
//
// Sources: "D2F 논문 리뷰: 확산 LLM이 자기회귀 모델보다 빠른 추론을 처음으로 달성한
// 방식", §쉽게 이해하기 (an active window of blocks; a block is added behind the
// last one once its progress passes a threshold; a new block is conservative and
// turns aggressive once the block before it has progressed enough) and "D2F: 확산
// 언어 모델이 KV 캐시를 얻고 자기회귀 모델보다 2.5배 빨라지는 방법", §운영 관점 (a
// completed block is persisted to the paged cache).
//
// One CTA does it all: the work is a few integers per sequence and a few bytes
// per window row, and a single CTA can order the whole step with __syncthreads:
//   1. bring the whole state into shared memory in one wave of loads (the top of
//      the free list follows, its latency hidden behind steps 2-4);
//   2. check the state (nothing is written if it is inconsistent) and count each
//      old block's committed positions;
//   3. decide per sequence: blocks leaving, a block entering, blocks to append;
//   4. one block-wide exclusive scan gives the new layout (blocks before each
//      sequence) and the pages before each sequence's appends, so pages come off
//      the free list in (sequence, block) order whatever the thread count;
//   5. write the per-sequence state, the append list and the phases;
//   6. write the repacked rows from shared memory.
#include "d2f_internal.cuh"

namespace d2f {
namespace {

constexpr int kThreads = 512;

struct SeqDecision {
  int ctx;      // context after the blocks that leave
  int first;    // oldest surviving block, old layout (block index)
  int surv;     // surviving blocks
  int add;      // 1: a new block enters
  int want;     // blocks to append (complete prefix, within the page-table row)
  int short_;   // 1: the page-table row cut the list
};

// Block-wide exclusive scan of (x, y) pairs held by each thread; also returns
// the totals. Threads pass their own partial sums (chunks of sequences).
__device__ __forceinline__ void block_scan2(int x, int y, int &ex, int &ey, int &tx, int &ty,
                                            int2 *warp_tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int ix = x, iy = y;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int nx = __shfl_up_sync(0xffffffffu, ix, o), ny = __shfl_up_sync(0xffffffffu, iy, o);
    if (lane >= o) {
      ix += nx;
      iy += ny;
    }
  }
  if (lane == 31) warp_tot[warp] = make_int2(ix, iy);
  __syncthreads();
  if (warp == 0) {
    int2 v = lane < kThreads / 32 ? warp_tot[lane] : make_int2(0, 0);
    int sx = v.x, sy = v.y;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int nx = __shfl_up_sync(0xffffffffu, sx, o), ny = __shfl_up_sync(0xffffffffu, sy, o);
      if (lane >= o) {
        sx += nx;
        sy += ny;
      }
    }
    if (lane < kThreads / 32) warp_tot[lane] = make_int2(sx - v.x, sy - v.y);  // exclusive
    if (lane == kThreads / 32 - 1) warp_tot[kThreads / 32] = make_int2(sx, sy);  // totals
  }
  __syncthreads();
  ex = warp_tot[warp].x + ix - x;
  ey = warp_tot[warp].y + iy - y;
  tx = warp_tot[kThreads / 32].x;
  ty = warp_tot[kThreads / 32].y;
}

__global__ void __launch_bounds__(kThreads, 1) window_kernel(const WindowArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int B = a.block_size, batch = a.batch, cap = a.capacity;
  const int tid = threadIdx.x;
  // shared layout: scan totals, per-sequence arrays, then rows (window_smem_bytes)
  int2 *s_warp = reinterpret_cast<int2 *>(smem);                      // [kThreads / 32 + 1]
  int *s_qold = reinterpret_cast<int *>(s_warp + kThreads / 32 + 1);  // [batch + 1]
  int *s_qnew = s_qold + (batch + 1);                                 // [batch + 1] in blocks
  int *s_abase = s_qnew + (batch + 1);                                // [batch] pages before b
  int *s_nl = s_abase + batch;                                        // [batch] n_leaving
  int *s_ctx = s_nl + batch;                                          // [batch] ctx_len
  int *s_nb = s_ctx + batch;                                          // [batch] next_block
  int *s_gen = s_nb + batch;                                          // [batch] gen_blocks
  int *s_fp = s_gen + batch;                                          // [kThreads] list top
  SeqDecision *s_dec = reinterpret_cast<SeqDecision *>(s_fp + kThreads);
  int32_t *s_tok = reinterpret_cast<int32_t *>(s_dec + batch);        // [cap]
  uint8_t *s_msk = reinterpret_cast<uint8_t *>(s_tok + cap);          // [cap]
  uint8_t *s_cnt = s_msk + cap;                                       // [cap / B]
  uint8_t *s_stop = s_cnt + cap / B;                                  // [batch]
  __shared__ int s_free;

  grid_launch_dependents();
  grid_dependency_wait();  // the commit (or the caller) wrote the state

  // ---- 1. the whole state in one wave of independent loads ----------------------
  if (tid == 0) s_free = a.free_count[0];
  for (int b = tid; b <= batch; b += kThreads) s_qold[b] = a.q_start[b];
  for (int b = tid; b < batch; b += kThreads) {
    s_nl[b] = a.n_leaving[b];
    s_ctx[b] = a.ctx_len[b];
    s_nb[b] = a.next_block[b];
    s_gen[b] = a.gen_blocks[b];
    s_stop[b] = a.stopped != nullptr ? a.stopped[b] : 0;
  }
  for (int r = tid; r < cap; r += kThreads) {
    s_tok[r] = a.tokens[r];
    s_msk[r] = a.masked[r];
  }
  __syncthreads();
  // The top of the free list, loaded now and stored to shared memory only after
  // the checks and decisions below, which hide its latency.
  const int free0 = s_free;
  const int n_pre = min(max(free0, 0), min(kThreads, cap / B));
  const int fp = tid < n_pre ? a.free_pages[free0 - 1 - tid] : 0;

  // ---- 2. consistency of the state (nothing is written if it fails) --------------
  int bad = tid == 0 && (s_qold[0] != 0 || free0 < 0);
  for (int b = tid; b < batch; b += kThreads) {
    const int n = s_qold[b + 1] - s_qold[b];
    bad |= n < 0 || n % B != 0 || n / B > a.max_blocks || s_qold[b + 1] > cap || s_nl[b] < 0 ||
           s_nl[b] > n / B || s_ctx[b] < 0 || s_ctx[b] % B != 0;
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) set_err(a.err, D2F_ERR_INVALID_ARG);
    return;
  }

  // ---- 2b. committed positions of every old block --------------------------------
  const int old_rows = s_qold[batch];
  for (int jb = tid; jb < old_rows / B; jb += kThreads) {
    int c = 0;
    for (int u = 0; u < B; ++u) c += s_msk[jb * B + u] == 0;
    s_cnt[jb] = (uint8_t)c;
  }
  __syncthreads();

  // ---- 3. per-sequence decisions (each thread a contiguous chunk) -----------------
  const int chunk = (batch + kThreads - 1) / kThreads;
  const int b0 = min(batch, tid * chunk), b1 = min(batch, b0 + chunk);
  int my_blocks = 0, my_want = 0;
  for (int b = b0; b < b1; ++b) {
    SeqDecision d;
    const int nblk = (s_qold[b + 1] - s_qold[b]) / B;
    const int nl = s_nl[b];
    d.ctx = s_ctx[b] + nl * B;
    d.first = s_qold[b] / B + nl;
    d.surv = nblk - nl;
    int add = !s_stop[b] && s_nb[b] < s_gen[b] && d.surv < a.max_blocks;
    if (add && d.surv > 0) add = (float)s_cnt[d.first + d.surv - 1] > a.tau_add * (float)B;
    d.add = add;
    int want = 0;
    while (want < d.surv && s_cnt[d.first + want] == B) ++want;
    const int room = max(0, a.max_pages_per_seq - d.ctx / B);
    d.short_ = want > room;
    d.want = min(want, room);
    s_dec[b] = d;
    my_blocks += d.surv + add;
    my_want += d.want;
  }

  // ---- 4. layout and page bases -------------------------------------------------
  int ex_blocks, ex_want, tot_blocks, tot_want;
  block_scan2(my_blocks, my_want, ex_blocks, ex_want, tot_blocks, tot_want, s_warp);
  for (int b = b0; b < b1; ++b) {
    s_qnew[b] = ex_blocks;
    s_abase[b] = ex_want;
    ex_blocks += s_dec[b].surv + s_dec[b].add;
    ex_want += s_dec[b].want;
  }
  if (tid == 0) s_qnew[batch] = tot_blocks;
  if (tid < n_pre) s_fp[tid] = fp;
  __syncthreads();

  // ---- 5. per-sequence state, append list, phases --------------------------------
  for (int b = b0; b < b1; ++b) {
    const SeqDecision d = s_dec[b];
    const int row0 = s_qnew[b] * B;
    // pages off the top of the list, in (sequence, block) order
    const int granted = max(0, min(d.want, free0 - s_abase[b]));
    if (granted < d.want || d.short_) set_err(a.err, D2F_ERR_NO_PAGE);
    for (int i = 0; i < granted; ++i) {
      const int slot = s_abase[b] + i;
      const int page = slot < n_pre ? s_fp[slot] : a.free_pages[free0 - 1 - slot];
      a.page_table[(int64_t)b * a.max_pages_per_seq + d.ctx / B + i] = page;
      a.app_src[slot] = row0 + i * B;
      a.app_dst[slot] = page;
    }
    a.n_leaving[b] = granted;
    a.ctx_len[b] = d.ctx;
    a.next_block[b] = s_nb[b] + d.add;
    a.q_start[b] = row0;
    for (int k = 0; k < d.surv + d.add; ++k) {
      const int pred = k == 0 ? B : (k - 1 < d.surv ? (int)s_cnt[d.first + k - 1] : 0);
      a.block_phase[s_qnew[b] + k] = (float)pred >= a.tau_act * (float)B ? 1 : 0;
    }
  }
  if (tid == 0) {
    const int n_app = min(tot_want, free0);
    a.q_start[batch] = tot_blocks * B;
    a.free_count[0] = free0 - n_app;
    a.n_append[0] = n_app;
  }

  // ---- 6. rows of the new window (and the idle rows past it) ----------------------
  const int new_rows = tot_blocks * B;
  for (int r = tid; r < cap; r += kThreads) {
    int32_t tok = a.mask_id, pos = -1;
    uint8_t m = 0;
    if (r < new_rows) {
      const int jb = r / B, u = r % B;
      int lo = 0, hi = batch - 1;  // the sequence: largest b with s_qnew[b] <= jb
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_qnew[mid] <= jb) lo = mid; else hi = mid - 1;
      }
      const SeqDecision &d = s_dec[lo];
      const int k = jb - s_qnew[lo];
      if (k < d.surv) {
        const int src = (d.first + k) * B + u;
        tok = s_tok[src];
        m = s_msk[src];
      } else {
        m = 1;
      }
      pos = d.ctx + k * B + u;
    } else if (r % B == 0) {
      a.block_phase[r / B] = 0;
    }
    a.tokens[r] = tok;
    a.masked[r] = m;
    a.row_pos[r] = pos;
  }
}

}  // namespace

size_t window_smem_bytes(int batch, int capacity, int block_size) {
  size_t b = (kThreads / 32 + 1) * sizeof(int2) + (size_t)(batch + 1) * 2 * sizeof(int) +
             (size_t)batch * 5 * sizeof(int) + kThreads * sizeof(int) +
             (size_t)batch * sizeof(SeqDecision);
  b += (size_t)capacity * (sizeof(int32_t) + 1) + (size_t)(capacity / block_size) + batch;
  return (b + 15) & ~(size_t)15;
}

cudaError_t launch_window(const WindowArgs &a, cudaStream_t stream) {
  const size_t smem = window_smem_bytes(a.batch, a.capacity, a.block_size);
  // The opt-in above 48 KB is a per-device function attribute: set it when a larger
  // size is first needed, not on every launch.
  static int opted[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (smem > 48 * 1024 && (dev >= 64 || (int)smem > opted[dev])) {
    e = cudaFuncSetAttribute(window_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev < 64) opted[dev] = (int)smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, window_kernel, a);
}

}  // namespace d2f
