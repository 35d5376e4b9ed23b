// Self-test of the bounded pipeline waits shared by the attention kernels:
// one CTA of two warps waits on barriers that nothing ever arrives at.  Warp
// 0 gives up after the caller's limit and raises the CTA's abort flag; warp 1
// waits with the kernels' own two-second limit and must leave through that
// flag.  The kernel then reports LNK_DEV_TIMEOUT the way the attention
// kernels do, and returns: no trap, no fault, the context stays usable.
#include "common.cuh"
#include "ptx.cuh"

namespace lnk {
namespace {

__global__ void wait_timeout_kernel(int32_t* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar[2];
  __shared__ int abort_word;
  volatile int* abort_flag = &abort_word;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar[0]), 1);
    mbar_init(smem_addr(&bar[1]), 1);
    abort_word = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  bool ok;
  if (warp == 0)
    ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&bar[0]), 0, abort_flag, limit_ns));
  else
    ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&bar[1]), 0, abort_flag));
  __syncthreads();
  if (threadIdx.x == 0 && !ok && *abort_flag && status != nullptr) atomicOr(status, LNK_DEV_TIMEOUT);
}

}  // namespace
}  // namespace lnk

extern "C" lnk_status lnk_selftest_wait_timeout(int32_t* dev_status, uint64_t limit_ns, lnk_stream stream) {
  if (dev_status == nullptr || limit_ns == 0 || limit_ns > lnk::kWaitLimitNs) return LNK_EINVAL;
  lnk::wait_timeout_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(
      dev_status, static_cast<unsigned long long>(limit_ns));
  return cudaGetLastError() == cudaSuccess ? LNK_OK : LNK_ECUDA;
}
