// d2f_commit_noalloc: d2f_commit for callers that cannot allocate device
// memory and therefore cannot hand the library a workspace.
//
// Who needs it: code that runs where allocation is forbidden or unavailable --
// a plugin or callback invoked by a host framework that owns all device memory
// and only passes its own buffers in, a runtime that must not allocate once it
// is serving (fixed memory budget, no allocator on the hot path), or a caller
// that has no allocator handle at all. Such a caller still passes its logits,
// decode state and outputs, but the commit's scratch (per-slice partial
// results, per-row results and the arrival counters) comes from a fixed array
// that lives in this library's device image.
//
// The scratch is kNoAllocScratchBytes (2 MiB). A call needs what
// d2f_commit_workspace_size reports for its shape: at block size 16, for
// example, at most 2,032 window rows at 64 vocabulary slices per row, 15,792 at
// 8 slices, 57,056 at 2; larger requests are refused. Every GPU that loads the
// library holds this array until the process exits.
//
// The array's device address belongs to the CUDA context it was looked up in
// (the module is loaded once per context). It is looked up on the first call in
// each context and cached under the context's unique id, which also tells a
// context re-created after a reset from the one it replaced; make that first
// call before any stream capture. All calls share the one array and it keeps
// what the last call left: each call clears the arrival counters at its start
// (the rest is written before it is read). Calls that overlap on the GPU
// (different streams, no ordering) race on the array and give wrong results:
// serialise them.
#include <cuda.h>

#include <mutex>

#include "d2f_internal.cuh"

namespace d2f {
namespace {

constexpr size_t kNoAllocScratchBytes = 2u << 20;
constexpr int kMaxContexts = 64;

static __device__ __align__(256) unsigned char g_commit_scratch[kNoAllocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);

struct Entry {
  unsigned long long ctx_id;
  void *ptr;
};

std::mutex g_mu;
Entry g_cache[kMaxContexts] = {};
int g_n = 0;

template <typename Fn>
Fn driver_fn(const char *name) {
  void *p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(p);
  return nullptr;
}

// Unique id of the current context (0 when it cannot be had).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

int scratch_for_current_context(void **out) {
  void *p = nullptr;
  unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  if (id != 0)
    for (int i = 0; i < g_n; ++i)
      if (g_cache[i].ctx_id == id) {
        *out = g_cache[i].ptr;
        return D2F_OK;
      }
  // First call in this context (or no context id to key on): look the address up.
  cudaError_t e = cudaGetSymbolAddress(&p, g_commit_scratch);
  if (e != cudaSuccess || !p) {
    set_last_error("cudaGetSymbolAddress of the commit scratch: %s", cudaGetErrorString(e));
    return D2F_ERR_CUDA;
  }
  if (id == 0) id = current_context_id();  // the lookup may have made the context current
  if (id != 0) {
    int slot = g_n < kMaxContexts ? g_n++ : (int)(id % kMaxContexts);  // full: replace one
    g_cache[slot] = Entry{id, p};
  }
  *out = p;
  return D2F_OK;
}

}  // namespace
}  // namespace d2f

extern "C" int d2f_commit_noalloc(const void *logits, int64_t row_stride, int dtype, int vocab,
                                  int num_logit_rows, const int32_t *logit_row, int32_t *tokens,
                                  uint8_t *masked, const int32_t *q_start,
                                  const uint8_t *block_phase, const float *tau, int batch,
                                  int total_q, int block_size, int32_t mask_id, float *conf_out,
                                  int32_t *argmax_out, int32_t *block_remaining, int num_splits,
                                  int32_t *err_word, void *stream) {
  size_t need = 0, zeroed = 0;
  int st = d2f_commit_workspace_size(total_q, vocab, dtype, block_size, num_splits, &need);
  if (st != D2F_OK) return st;
  if (need > d2f::kNoAllocScratchBytes) {
    d2f::set_last_error(
        "d2f_commit_noalloc: %d rows x vocab %d (num_splits %d) need %zu bytes of scratch, more "
        "than its fixed %zu; use d2f_commit with a caller workspace",
        total_q, vocab, num_splits, need, d2f::kNoAllocScratchBytes);
    return D2F_ERR_WORKSPACE;
  }
  if (total_q == 0) return D2F_OK;
  st = d2f::commit_zeroed_prefix(total_q, vocab, dtype, block_size, num_splits, &zeroed);
  if (st != D2F_OK) return st;
  void *scratch = nullptr;
  st = d2f::scratch_for_current_context(&scratch);
  if (st != D2F_OK) return st;
  // The arrival counters must start at zero whatever the previous call left
  // there (a call that stopped on a device error leaves them set).
  cudaError_t e = cudaMemsetAsync(scratch, 0, zeroed, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    d2f::set_last_error("cudaMemsetAsync of the commit scratch: %s", cudaGetErrorString(e));
    return D2F_ERR_CUDA;
  }
  return d2f_commit(logits, row_stride, dtype, vocab, num_logit_rows, logit_row, tokens, masked,
                    q_start, block_phase, tau, batch, total_q, block_size, mask_id, conf_out,
                    argmax_out, block_remaining, num_splits, scratch, d2f::kNoAllocScratchBytes,
                    err_word, stream);
}
