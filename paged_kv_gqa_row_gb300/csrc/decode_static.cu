// lnk_paged_decode_attn_static: paged decode attention that takes no workspace
// argument and allocates nothing.
//
// Some callers cannot hand the library a scratch buffer: a plugin or callback
// run by a host runtime that reserved all device memory up front and forbids
// allocation on its execution path, or a serving loop that must keep its
// memory footprint and per-step latency fixed, has no allocator to call when
// the step runs.  For them the decode kernel's scratch lives in this file's
// static device array, reserved once when the library is loaded (every GPU
// that loads the library keeps it until the process exits).
//
// The array's host-side name is only a stand-in for the device variable, so
// the device address is obtained with cudaGetSymbolAddress, once per device,
// on the first call made while that device is current; that first call makes
// a runtime call of its own and should therefore come before any stream
// capture.  Only a successful lookup is kept: after a failed one the call
// returns LNK_ECUDA and the next call on that device tries again.  Every call
// shares the array and finds the previous call's data in it: the counters the
// decode kernel needs at zero are cleared on the stream once the call's
// arguments have passed every check, right before the launch (a call that
// returns an error enqueues nothing), and calls whose work overlaps on the
// GPU (other streams, other host threads) race on the array and must be
// serialised by the caller.  The call then runs the ordinary decode path on
// the array.
#include <mutex>

#include "common.cuh"

namespace lnk {
namespace {

// Largest scratch the array provides: enough for a few hundred decode rows at
// Hkv = 8, group 4, head_dim 128 on 152 SMs (lnk_paged_workspace_size gives
// the exact need; larger calls are rejected with LNK_ERANGE).
constexpr size_t kStaticScratchBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the array on the current device (looked up on first use;
// a failed lookup is not remembered).
cudaError_t scratch_address(void** ptr) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace lnk

extern "C" lnk_status lnk_paged_decode_attn_static(const lnk_attn_desc* desc, const lnk_bf16* q_roped,
                                                   const int32_t* positions, const int32_t* table,
                                                   const lnk_bf16* k_pool, const lnk_bf16* v_pool, lnk_bf16* out,
                                                   int32_t B, int32_t* dev_status, lnk_stream stream) {
  if (desc == nullptr || B < 0) return LNK_EINVAL;
  if (B == 0) return LNK_OK;
  const size_t need = lnk_paged_workspace_size(desc, B);
  if (need == 0) return LNK_EINVAL;
  if (need > lnk::kStaticScratchBytes) return LNK_ERANGE;
  void* scratch = nullptr;
  if (lnk::scratch_address(&scratch) != cudaSuccess || scratch == nullptr) return LNK_ECUDA;
  // the same checks and launch as lnk_paged_decode_attn, with the workspace's
  // counters (chunk claims, per-pair segments) zeroed just before the launch
  return lnk::decode_entry(desc, q_roped, positions, table, k_pool, v_pool, out, B, scratch,
                           lnk::kStaticScratchBytes, dev_status, stream, true);
}
