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
// The scratch is kNoAllocScratchBytes (2 MiB), enough for e.g. 2048 window rows
// at 64 vocabulary slices each. Every GPU that loads the library holds this
// array until the process exits. Its device address is looked up once per
// device, by the first call on that device (make that first call before any
// stream capture). All calls share the one array and it keeps what the last call
// left; each call clears the counters it relies on before the kernel runs.
// Calls that overlap on the GPU (different streams, no ordering) race on the
// array and give wrong results: serialise them.
#include <mutex>

#include "d2f_internal.cuh"

namespace d2f {
namespace {

constexpr size_t kNoAllocScratchBytes = 2u << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_commit_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

int scratch_for_current_device(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_last_error("cudaGetDevice: %s", cudaGetErrorString(e));
    return D2F_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    set_last_error("device %d outside the %d devices d2f_commit_noalloc tracks", dev, kMaxDevices);
    return D2F_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_commit_scratch);
    if (e != cudaSuccess || !p) {
      set_last_error("cudaGetSymbolAddress of the commit scratch: %s", cudaGetErrorString(e));
      return D2F_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
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
  size_t need = 0;
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
  void *scratch = nullptr;
  st = d2f::scratch_for_current_device(&scratch);
  if (st != D2F_OK) return st;
  // The arrival counters must start at zero; clear the whole region this call
  // uses (whatever the previous call left there) before the kernel runs.
  cudaError_t e = cudaMemsetAsync(scratch, 0, need, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    d2f::set_last_error("cudaMemsetAsync of the commit scratch: %s", cudaGetErrorString(e));
    return D2F_ERR_CUDA;
  }
  return d2f_commit(logits, row_stride, dtype, vocab, num_logit_rows, logit_row, tokens, masked,
                    q_start, block_phase, tau, batch, total_q, block_size, mask_id, conf_out,
                    argmax_out, block_remaining, num_splits, scratch, d2f::kNoAllocScratchBytes,
                    err_word, stream);
}
