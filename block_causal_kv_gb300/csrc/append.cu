// d2f_kv_append kernel: copy finished blocks of the window K/V into their
// cache pages.
//
// Source: "D2F: 확산 언어 모델이 KV 캐시를 얻고 자기회귀 모델보다 2.5배 빨라지는
// 방법", §블록 단위 인과 어텐션 and §운영 관점 (a completed block's K/V are final
// and persisted; a page holds one block).
//
// One CTA per (append, KV head): the block's B rows of that head are B strided
// rows of the window tensor and one contiguous B x D tile of the page. The copy is
// bitwise, 16 bytes per thread per step when the rows allow it.
#include "d2f_internal.cuh"

namespace d2f {
namespace {

constexpr int kThreads = 128;

template <bool VEC>
__global__ void __launch_bounds__(kThreads) append_kernel(const AppendArgs a) {
  const int ap = blockIdx.x / a.num_heads_kv;
  const int g = blockIdx.x % a.num_heads_kv;
  // a list whose length is in device memory: the launch covers its capacity
  if (a.n_dev != nullptr && ap >= min(max(*a.n_dev, 0), a.n_append)) return;
  const int src = a.src_row[ap];
  const int dst = a.dst_page[ap];
  if (src < 0 || src + a.block_size > a.total_q || dst < 0 || dst >= a.num_pages) {
    if (threadIdx.x == 0 && g == 0) set_err(a.err, D2F_ERR_BAD_INDEX);
    return;
  }
  const int64_t rb = a.row_bytes;
  const int64_t win_row_stride = rb * a.num_heads_kv;  // bytes between window rows
  const int64_t tile_bytes = rb * a.block_size;
  const int64_t src_off = (int64_t)src * win_row_stride + g * rb;
  const int64_t dst_off = ((int64_t)dst * a.num_heads_kv + g) * tile_bytes;
  for (int which = 0; which < 2; ++which) {
    const char *in = (const char *)(which ? a.v_win : a.k_win) + src_off;
    char *out = (char *)(which ? a.v_pool : a.k_pool) + dst_off;
    if (VEC) {
      const int per_row = (int)(rb / 16);
      const int total = per_row * a.block_size;
      for (int i = threadIdx.x; i < total; i += kThreads) {
        const int s = i / per_row, c = i % per_row;
        const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(in + s * win_row_stride) + c);
        reinterpret_cast<uint4 *>(out + s * rb)[c] = v;
      }
    } else {
      const int per_row = (int)(rb / 2);  // element sizes are 2 or 4 bytes
      const int total = per_row * a.block_size;
      for (int i = threadIdx.x; i < total; i += kThreads) {
        const int s = i / per_row, c = i % per_row;
        reinterpret_cast<uint16_t *>(out + s * rb)[c] =
            reinterpret_cast<const uint16_t *>(in + s * win_row_stride)[c];
      }
    }
  }
}

}  // namespace

cudaError_t launch_append(const AppendArgs &a, bool vec_ok, cudaStream_t stream) {
  if (a.n_append == 0) return cudaSuccess;
  dim3 grid(a.n_append * a.num_heads_kv), block(kThreads);
  if (vec_ok)
    append_kernel<true><<<grid, block, 0, stream>>>(a);
  else
    append_kernel<false><<<grid, block, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace d2f
