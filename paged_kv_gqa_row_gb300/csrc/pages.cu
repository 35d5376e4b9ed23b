// lnk_paged_copy_pages: copies whole pages of the K and V pools (every kv
// head), for the copy on write of the host page allocator: a row that writes
// into a page it shares with other rows first gets a private page holding the
// shared page's contents.
//
// One CTA per (page pair, kv head): 64 slots x head_dim elements of K and of V
// (bf16, or one-byte codes of an 8-bit pool), moved with 16-byte loads and
// stores (a page of one head is contiguous).
#include "common.cuh"

namespace lnk {
namespace {

__global__ void copy_pages_kernel(uint8_t* __restrict__ k_pool, uint8_t* __restrict__ v_pool,
                                  const int32_t* __restrict__ src, const int32_t* __restrict__ dst, int num_pages,
                                  int row_bytes, int32_t* status) {
  const int i = blockIdx.x, h = blockIdx.y;
  const int s = src[i], d = dst[i];
  if (s < 0 || s >= num_pages || d < 0 || d >= num_pages) {
    if (threadIdx.x == 0 && h == 0 && status != nullptr) atomicOr(status, LNK_DEV_BAD_PAGE);
    return;
  }
  if (s == d) return;
  const size_t page_bytes = static_cast<size_t>(kPage) * row_bytes;
  const size_t head = static_cast<size_t>(h) * num_pages * page_bytes;
  const size_t n16 = page_bytes / 16;  // 16-byte units per page
  const uint4* ks = reinterpret_cast<const uint4*>(k_pool + head + static_cast<size_t>(s) * page_bytes);
  const uint4* vs = reinterpret_cast<const uint4*>(v_pool + head + static_cast<size_t>(s) * page_bytes);
  uint4* kd = reinterpret_cast<uint4*>(k_pool + head + static_cast<size_t>(d) * page_bytes);
  uint4* vd = reinterpret_cast<uint4*>(v_pool + head + static_cast<size_t>(d) * page_bytes);
  for (size_t j = threadIdx.x; j < n16; j += blockDim.x) {
    kd[j] = ks[j];
    vd[j] = vs[j];
  }
}

}  // namespace
}  // namespace lnk

extern "C" lnk_status lnk_paged_copy_pages(const lnk_attn_desc* desc, lnk_bf16* k_pool, lnk_bf16* v_pool,
                                           const int32_t* src_pages, const int32_t* dst_pages, int32_t n,
                                           int32_t* dev_status, lnk_stream stream) {
  if (desc == nullptr || n < 0) return LNK_EINVAL;
  if (n == 0) return LNK_OK;
  if (k_pool == nullptr || v_pool == nullptr || src_pages == nullptr || dst_pages == nullptr) return LNK_EINVAL;
  if (desc->page_size != lnk::kPage) return LNK_EUNSUPPORTED;
  if (desc->head_dim != 64 && desc->head_dim != 96 && desc->head_dim != 128) return LNK_EUNSUPPORTED;
  if (desc->num_kv_heads <= 0 || desc->num_pages <= 0) return LNK_EINVAL;
  if (desc->kv_dtype != LNK_KV_BF16 && desc->kv_dtype != LNK_KV_E4M3) return LNK_EUNSUPPORTED;
  const int row_bytes = desc->head_dim * (desc->kv_dtype == LNK_KV_E4M3 ? 1 : 2);
  if ((reinterpret_cast<uintptr_t>(k_pool) | reinterpret_cast<uintptr_t>(v_pool)) % 16 != 0) return LNK_EINVAL;
  if (n > 65535 * 1024 || desc->num_kv_heads > 65535) return LNK_ERANGE;
  dim3 grid(n, desc->num_kv_heads);
  lnk::copy_pages_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<uint8_t*>(k_pool), reinterpret_cast<uint8_t*>(v_pool), src_pages, dst_pages,
      desc->num_pages, row_bytes, dev_status);
  return cudaGetLastError() == cudaSuccess ? LNK_OK : LNK_ECUDA;
}
