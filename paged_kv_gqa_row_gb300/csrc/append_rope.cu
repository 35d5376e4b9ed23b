// K1: per-token QK-norm (optional), RoPE and K/V append into the page pool.
//
// A token's rotated heads (its query heads, then its key heads) and value
// heads are split over S CTAs: CTA s of the token takes heads s, s + S, s + 2S,
// ...  Launches with few tokens use many splits of a few heads each (four
// warps per CTA), so that the per-head work spreads over the SMs instead of
// queueing on one SM per token; launches with many tokens use one CTA per
// token (S = 1).  The rotation and the QK-norm are the float-pair arithmetic
// of rope_math.cuh (each rotated element rounded once to bf16); V is copied
// bit for bit into the token's pool slot.
//
// Sources: "Phi-3 Mini 4K Instruct -- files", src/rope.linnet (tables) and
// src/attention.linnet (rope + write_tokens in prefill_packed / step_packed);
// "Qwen3-4B", QK-norm paragraph; "Mistral 7B Instruct v0.3", Entries table
// (prefill_paged: each token written at its place in the pool).
#include <cuda_fp8.h>

#include <algorithm>

#include "common.cuh"
#include "rope_math.cuh"

namespace lnk {
namespace {

constexpr int kMaxRotated = 128;  // rotated heads (Hq + Hkv) per token
// CTA shapes (warps, rotated heads per warp at most):
//  * split: 4 warps of up to 4 heads, S >= 2 CTAs per token (launches with
//    fewer tokens than SMs);
//  * one CTA per token, 16 warps (launches with up to four tokens per SM);
//  * one CTA per token, 8 warps (more tokens per SM resident at once).
constexpr int kWarpsSplit = 4, kHeadsSplit = 4;
constexpr int kWarpsSmall = 16;
constexpr int kWarpsWide = 8;
constexpr int kWideTokensPerSm = 4;  // launches with at least this many tokens per SM use kWarpsWide
constexpr int kSplitCtasPerSm = 2;   // split launches aim at this many CTAs per SM

using namespace rope;

template <int D, int kWarps, int kMaxHeadsPerWarp>
__global__ void __launch_bounds__(kWarps * 32) append_rope_kernel(const AppendParams p) {
  constexpr int H = D / 2;
  constexpr int kLanes = D / 4;  // lanes holding data: two elements of each half
  // coefficient sets: [0] queries, [1] keys
  __shared__ Coefs s_coef[2][H];
  __shared__ DF s_ss[kWarps * kMaxHeadsPerWarp];
  __shared__ DF s_r[kWarps * kMaxHeadsPerWarp];
  __shared__ long long s_slot;

  // Let the next kernel on the stream start its prologue; it waits for this
  // grid's writes before reading them.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int S = p.splits;
  const int t = blockIdx.x / S;
  const int sp = blockIdx.x % S;  // this CTA's heads: sp + S * l (l: local index)
  const int pos = p.positions[t];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int nrot = p.hq + p.hkv;  // rotated heads: queries then keys
  const int nloc = (nrot - sp + S - 1) / S;  // this CTA's rotated heads
  const bool norm_q = p.q_norm_w != nullptr, norm_k = p.k_norm_w != nullptr;

  // The kernel is launched as a programmatic dependent of the previous kernel
  // on the stream.  Before waiting for it, it reads only positions, rows,
  // slots and the table (which that kernel must not write): the token's slot
  // and the sine and cosine of its angles.
  // ---- per-token coefficients (float pairs, once per frequency) ----
  DF sn{0.f, 0.f}, cs{0.f, 0.f};
  if (tid < H && pos >= 0) angle_sincos(pos, p.inv_freq[tid], sn, cs);
  int bad = 0;
  if (tid == kWarps * 32 - 1) {
    long long slot = -1;
    if (pos >= 0) {
      if (p.slots != nullptr) {
        const int s = p.slots[t];
        if (s < 0 || static_cast<long long>(s) >= static_cast<long long>(p.num_pages) * kPage)
          bad = LNK_DEV_BAD_SLOT;
        else
          slot = s;
      } else {
        const int row = p.rows != nullptr ? p.rows[t] : t;
        if (row < 0 || row >= p.num_rows) {
          bad = LNK_DEV_BAD_ROW;
        } else if (pos >= p.pages_per_row * kPage) {
          bad = LNK_DEV_BAD_POSITION;
        } else {
          const int page = p.table[static_cast<long long>(row) * p.pages_per_row + pos / kPage];
          if (page < 0 || page >= p.num_pages)
            bad = LNK_DEV_BAD_PAGE;
          else
            slot = static_cast<long long>(page) * kPage + pos % kPage;
        }
      }
    }
    s_slot = slot;
  }

  // Wait for the previous kernel on the stream: it may write q, k, v, the
  // QK-norm weights or the status, or still read q_out and the pools.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (bad && p.status != nullptr) atomicOr(p.status, bad);
  if (tid < H && pos >= 0) {
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint16_t* w = which == 0 ? p.q_norm_w : p.k_norm_w;
      float g1 = 1.f, g2 = 1.f;
      if (w != nullptr) {
        g1 = __uint_as_float(static_cast<uint32_t>(w[tid]) << 16);
        g2 = __uint_as_float(static_cast<uint32_t>(w[tid + H]) << 16);
      }
      s_coef[which][tid] = coefs_of(sn, cs, g1, g2);
    }
  }
  // ---- load this warp's rotated heads (all loads in flight together) ----
  const bool has = lane < kLanes;
  const int e = 2 * lane;
  uint32_t xlo[kMaxHeadsPerWarp], xhi[kMaxHeadsPerWarp];
#pragma unroll
  for (int j = 0; j < kMaxHeadsPerWarp; ++j) {
    const int l = warp + j * kWarps;
    const int hh = sp + S * l;
    xlo[j] = xhi[j] = 0u;
    if (l < nloc && has && pos >= 0) {
      const uint16_t* src = hh < p.hq ? p.q + (static_cast<size_t>(t) * p.hq + hh) * D
                                      : p.k + (static_cast<size_t>(t) * p.hkv + (hh - p.hq)) * D;
      xlo[j] = *reinterpret_cast<const uint32_t*>(src + e);
      xhi[j] = *reinterpret_cast<const uint32_t*>(src + H + e);
    }
  }
  // QK-norm: sum of squares per head (squares of bf16 values are exact in float)
  if (norm_q || norm_k) {
#pragma unroll
    for (int j = 0; j < kMaxHeadsPerWarp; ++j) {
      const int l = warp + j * kWarps;
      const int hh = sp + S * l;
      if (l >= nloc) break;
      if (!(hh < p.hq ? norm_q : norm_k)) continue;
      const DF acc = head_sumsq(xlo[j], xhi[j]);
      if (lane == 0) s_ss[l] = acc;
    }
  }
  __syncthreads();
  // one lane per head computes the RMS factor in double precision
  if ((norm_q || norm_k) && tid < nloc && pos >= 0 && (sp + S * tid < p.hq ? norm_q : norm_k)) {
    s_r[tid] = rms_factor(s_ss[tid], D, p.norm_eps);
  }
  __syncthreads();

  const long long slot = s_slot;
  const size_t pool_head_stride = static_cast<size_t>(p.num_pages) * kPage * D;
#pragma unroll
  for (int j = 0; j < kMaxHeadsPerWarp; ++j) {
    const int l = warp + j * kWarps;
    const int hh = sp + S * l;
    if (l >= nloc) break;
    const bool is_q = hh < p.hq;
    uint16_t* dst = nullptr;
    uint8_t* dst8 = nullptr;  // 8-bit pools: the key row's codes
    if (is_q) {
      dst = p.q_out + (static_cast<size_t>(t) * p.hq + hh) * D;
    } else {
      if (slot < 0) continue;
      const size_t off = (hh - p.hq) * pool_head_stride + static_cast<size_t>(slot) * D;
      if (p.kv8) dst8 = reinterpret_cast<uint8_t*>(p.k_pool) + off;
      else dst = p.k_pool + off;
    }
    if (!has) continue;
    if (pos < 0) {  // inactive token: zero query output
      *reinterpret_cast<uint32_t*>(dst + e) = 0u;
      *reinterpret_cast<uint32_t*>(dst + H + e) = 0u;
      continue;
    }
    const int set = is_q ? 0 : 1;
    const bool normed = is_q ? norm_q : norm_k;
    const DF r = normed ? s_r[l] : DF{1.f, 0.f};
    uint32_t lo_bits, hi_bits;
    rotate_pairs(xlo[j], xhi[j], s_coef[set], e, normed, r, lo_bits, hi_bits);
    if (dst8 != nullptr) {
      *reinterpret_cast<uint16_t*>(dst8 + e) = e4m3_pair(lo_bits, p.k_scale);
      *reinterpret_cast<uint16_t*>(dst8 + H + e) = e4m3_pair(hi_bits, p.k_scale);
    } else {
      *reinterpret_cast<uint32_t*>(dst + e) = lo_bits;
      *reinterpret_cast<uint32_t*>(dst + H + e) = hi_bits;
    }
  }
  // value heads: bit copy into the slot (8-bit pools: their codes)
  if (slot >= 0) {
    for (int vh = sp + S * warp; vh < p.hkv; vh += S * kWarps) {
      const uint4* src = reinterpret_cast<const uint4*>(p.v + (static_cast<size_t>(t) * p.hkv + vh) * D);
      const size_t off = vh * pool_head_stride + static_cast<size_t>(slot) * D;
      if (lane < D / 8) {
        const uint4 x = src[lane];
        if (p.kv8) {
          uint2 codes;
          codes.x = e4m3_pair(x.x, p.v_scale) | (static_cast<uint32_t>(e4m3_pair(x.y, p.v_scale)) << 16);
          codes.y = e4m3_pair(x.z, p.v_scale) | (static_cast<uint32_t>(e4m3_pair(x.w, p.v_scale)) << 16);
          reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(p.v_pool) + off)[lane] = codes;
        } else {
          reinterpret_cast<uint4*>(p.v_pool + off)[lane] = x;
        }
      }
    }
  }
}

template <int D, int kWarps, int kHeads>
cudaError_t launch_append_w(const AppendParams& p, cudaStream_t stream) {
  // Prefer the largest shared-memory carveout, like the attention kernels that
  // follow: their CTAs can then start on an SM next to this kernel's (the
  // attention kernel is launched as a programmatic dependent) without the SM
  // first switching its L1 / shared-memory split.
  const cudaError_t carve = prefer_max_shared(reinterpret_cast<const void*>(append_rope_kernel<D, kWarps, kHeads>));
  if (carve != cudaSuccess) return carve;
  const long long ctas = static_cast<long long>(p.T) * p.splits;
  if (ctas > 0x7fffffffll) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, append_rope_kernel<D, kWarps, kHeads>, p);
}

template <int D>
cudaError_t launch_append_t(const AppendParams& p_in, cudaStream_t stream) {
  AppendParams p = p_in;
  const long long sms = device_sm_count();
  const int nrot = p.hq + p.hkv;
  if (static_cast<long long>(p.T) < sms) {
    // few tokens: at least enough splits for kHeadsSplit heads per warp, and
    // up to kSplitCtasPerSm CTAs per SM (one rotated head per CTA at most)
    const int need = (nrot + kWarpsSplit * kHeadsSplit - 1) / (kWarpsSplit * kHeadsSplit);
    const long long want = (kSplitCtasPerSm * sms + p.T - 1) / p.T;
    p.splits = static_cast<int>(std::max<long long>(need, std::min<long long>(nrot, want)));
    return launch_append_w<D, kWarpsSplit, kHeadsSplit>(p, stream);
  }
  p.splits = 1;
  if (static_cast<long long>(p.T) >= kWideTokensPerSm * sms)
    return launch_append_w<D, kWarpsWide, kMaxRotated / kWarpsWide>(p, stream);
  return launch_append_w<D, kWarpsSmall, kMaxRotated / kWarpsSmall>(p, stream);
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, int head_dim, cudaStream_t stream) {
  if (p.T == 0) return cudaSuccess;
  if (p.hq + p.hkv > kMaxRotated) return cudaErrorInvalidValue;
  switch (head_dim) {
    case 64: return launch_append_t<64>(p, stream);
    case 96: return launch_append_t<96>(p, stream);
    case 128: return launch_append_t<128>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lnk
