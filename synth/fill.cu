// Device copy of the seeded value generator of synth/__init__.py: value i of
// a tensor is SplitMix64 output i (started at the tensor's key), its four
// 16-bit fields summed, centred and scaled by f32(sqrt(3)/65535) with one
// float32 multiply, then rounded to bf16 (nearest even).  Used to fill large
// page pools on the device; the host copy regenerates any slice exactly.
#include <cuda_runtime.h>
#include <cstdint>

namespace {

constexpr unsigned long long kGamma = 0x9E3779B97F4A7C15ull;
constexpr float kScale = static_cast<float>(1.7320508075688772 / 65535.0);

__device__ __forceinline__ unsigned long long mix64(unsigned long long z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__global__ void fill_kernel(uint16_t* out, long long n, unsigned long long key, long long start) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const unsigned long long h = mix64(key + static_cast<unsigned long long>(start + i + 1) * kGamma);
    const int s = static_cast<int>(h & 0xFFFF) + static_cast<int>((h >> 16) & 0xFFFF) +
                  static_cast<int>((h >> 32) & 0xFFFF) + static_cast<int>((h >> 48) & 0xFFFF) - 131070;
    const float x = __fmul_rn(__int2float_rn(s), kScale);
    const uint32_t u = __float_as_uint(x);
    out[i] = static_cast<uint16_t>((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
  }
}

// Bytes of a prefilled 8-bit (E4M3) pool: sign = bit 63, exponent field
// 4 + (bits 8.. mod 6), mantissa = bits 16..18 of SplitMix64 output i.
__global__ void fill_e4m3_kernel(uint8_t* out, long long n, unsigned long long key, long long start) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
    const unsigned long long h = mix64(key + static_cast<unsigned long long>(start + i + 1) * kGamma);
    const unsigned sign = static_cast<unsigned>(h >> 63);
    const unsigned e = 4u + static_cast<unsigned>((h >> 8) % 6ull);
    const unsigned m = static_cast<unsigned>((h >> 16) & 7ull);
    out[i] = static_cast<uint8_t>((sign << 7) | (e << 3) | m);
  }
}

long long grid_for(long long n) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (n + 255) / 256;
  const long long cap = static_cast<long long>(sms > 0 ? sms : 1) * 16;
  return blocks > cap ? cap : blocks;
}

}  // namespace

extern "C" int synth_fill_e4m3(uint8_t* out, long long n, unsigned long long key, long long start, void* stream) {
  if (n <= 0) return 0;
  fill_e4m3_kernel<<<static_cast<unsigned>(grid_for(n)), 256, 0, static_cast<cudaStream_t>(stream)>>>(out, n, key,
                                                                                                   start);
  return static_cast<int>(cudaGetLastError());
}

extern "C" int synth_fill_normal_bf16(uint16_t* out, long long n, unsigned long long key, long long start,
                                      void* stream) {
  if (n <= 0) return 0;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (n + 255) / 256;
  const long long cap = static_cast<long long>(sms > 0 ? sms : 1) * 16;
  if (blocks > cap) blocks = cap;
  fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(out, n, key, start);
  return static_cast<int>(cudaGetLastError());
}
