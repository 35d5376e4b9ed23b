// K1: per-token QK-norm (optional), RoPE and K/V append into the page pool.
//
// One CTA per token.  The token's cos/sin are computed once (double precision,
// from the float32 angle f32(position) * inv_freq[i]) into shared memory; then
// each warp takes whole heads: lane l holds elements (2l, 2l+1) of the first
// half and (D/2 + 2l, D/2 + 2l + 1) of the second half, so the rotate-half
// partner of every element sits in the same lane.  QK-norm and the rotation
// run in double precision and are rounded once to bf16; V is copied bit for
// bit into the token's pool slot.
//
// Sources: "Phi-3 Mini 4K Instruct -- files", src/rope.linnet (tables) and
// src/attention.linnet (rope + write_tokens in prefill_packed / step_packed);
// "Qwen3-4B", QK-norm paragraph; "Mistral 7B Instruct v0.3", Entries table
// (prefill_paged: each token written at its place in the pool).
#include "common.cuh"

namespace lnk {
namespace {

__device__ __forceinline__ double bf16_to_double(uint16_t b) {
  return static_cast<double>(__uint_as_float(static_cast<uint32_t>(b) << 16));
}

// double -> bf16 bits, round to nearest even, directly (one rounding).
__device__ __forceinline__ uint16_t double_to_bf16(double x) {
  const uint64_t u = static_cast<uint64_t>(__double_as_longlong(x));
  const uint64_t sign = (u >> 63) << 15;
  const uint64_t mag = u & 0x7FFFFFFFFFFFFFFFull;
  if (mag == 0) return static_cast<uint16_t>(sign);
  const int e = static_cast<int>(mag >> 52) - 1023 + 127;  // bf16 biased exponent
  if (e <= 0 || e >= 255) {
    // Outside bf16's normal range (never met at unit-scale data): go through
    // float32, which handles subnormals and overflow.
    const uint32_t f = __float_as_uint(__double2float_rn(x));
    const uint32_t r = f + 0x7FFFu + ((f >> 16) & 1u);
    return static_cast<uint16_t>(r >> 16);
  }
  uint64_t kept = mag >> 45;                      // exponent + 7 fraction bits
  const uint64_t rem = mag & ((1ull << 45) - 1);
  const uint64_t half = 1ull << 44;
  if (rem > half || (rem == half && (kept & 1))) kept += 1;  // carries into the exponent
  const uint64_t e_d = kept >> 7;
  const uint64_t frac = kept & 0x7F;
  const int e_b = static_cast<int>(e_d) - 1023 + 127;
  if (e_b >= 255) return static_cast<uint16_t>(sign | 0x7F80u);
  return static_cast<uint16_t>(sign | (static_cast<uint64_t>(e_b) << 7) | frac);
}

__device__ __forceinline__ uint32_t ld_u32(const uint16_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}
__device__ __forceinline__ void st_u32(uint16_t* p, uint32_t v) {
  *reinterpret_cast<uint32_t*>(p) = v;
}

template <int D>
__global__ void __launch_bounds__(256) append_rope_kernel(const AppendParams p) {
  constexpr int H = D / 2;
  constexpr int kLanes = D / 4;  // lanes that hold data
  __shared__ double s_cos[H];
  __shared__ double s_sin[H];
  __shared__ long long s_slot;

  const int t = blockIdx.x;
  const int pos = p.positions[t];
  const int tid = threadIdx.x;

  if (tid < H && pos >= 0) {
    const float a = __fmul_rn(static_cast<float>(pos), p.inv_freq[tid]);
    double s, c;
    sincos(static_cast<double>(a), &s, &c);
    s_cos[tid] = c;
    s_sin[tid] = s;
  }
  if (tid == 0) {
    long long slot = -1;
    int bad = 0;
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
    if (bad && p.status != nullptr) atomicOr(p.status, bad);
    s_slot = slot;
  }
  __syncthreads();

  const long long slot = s_slot;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const bool has = lane < kLanes;
  const int e = 2 * lane;
  const int nheads = p.hq + 2 * p.hkv;
  const size_t pool_head_stride = static_cast<size_t>(p.num_pages) * kPage * D;

  for (int hh = warp; hh < nheads; hh += 8) {
    if (hh >= p.hq + p.hkv) {
      // value head: bit copy into the slot
      if (slot < 0) continue;
      const int vh = hh - p.hq - p.hkv;
      const uint4* src = reinterpret_cast<const uint4*>(p.v + (static_cast<size_t>(t) * p.hkv + vh) * D);
      uint4* dst = reinterpret_cast<uint4*>(p.v_pool + vh * pool_head_stride + static_cast<size_t>(slot) * D);
      if (lane < D / 8) dst[lane] = src[lane];
      continue;
    }
    const bool is_q = hh < p.hq;
    const int head = is_q ? hh : hh - p.hq;
    uint16_t* dst;
    if (is_q) {
      dst = p.q_out + (static_cast<size_t>(t) * p.hq + head) * D;
    } else {
      if (slot < 0) continue;
      dst = p.k_pool + head * pool_head_stride + static_cast<size_t>(slot) * D;
    }
    if (pos < 0) {  // inactive token: zero query output
      if (has) {
        st_u32(dst + e, 0u);
        st_u32(dst + H + e, 0u);
      }
      continue;
    }
    const uint16_t* src =
        is_q ? p.q + (static_cast<size_t>(t) * p.hq + head) * D : p.k + (static_cast<size_t>(t) * p.hkv + head) * D;
    double x1a = 0.0, x1b = 0.0, x2a = 0.0, x2b = 0.0;
    if (has) {
      const uint32_t lo = ld_u32(src + e);
      const uint32_t hi = ld_u32(src + H + e);
      x1a = bf16_to_double(static_cast<uint16_t>(lo & 0xFFFFu));
      x1b = bf16_to_double(static_cast<uint16_t>(lo >> 16));
      x2a = bf16_to_double(static_cast<uint16_t>(hi & 0xFFFFu));
      x2b = bf16_to_double(static_cast<uint16_t>(hi >> 16));
    }
    const uint16_t* w = is_q ? p.q_norm_w : p.k_norm_w;
    if (w != nullptr) {
      double ss = __dadd_rn(__dadd_rn(__dmul_rn(x1a, x1a), __dmul_rn(x1b, x1b)),
                            __dadd_rn(__dmul_rn(x2a, x2a), __dmul_rn(x2b, x2b)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss = __dadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
      const double r = 1.0 / sqrt(__dadd_rn(ss / static_cast<double>(D), p.norm_eps));
      if (has) {
        const uint32_t wlo = ld_u32(w + e);
        const uint32_t whi = ld_u32(w + H + e);
        x1a = __dmul_rn(__dmul_rn(x1a, r), bf16_to_double(static_cast<uint16_t>(wlo & 0xFFFFu)));
        x1b = __dmul_rn(__dmul_rn(x1b, r), bf16_to_double(static_cast<uint16_t>(wlo >> 16)));
        x2a = __dmul_rn(__dmul_rn(x2a, r), bf16_to_double(static_cast<uint16_t>(whi & 0xFFFFu)));
        x2b = __dmul_rn(__dmul_rn(x2b, r), bf16_to_double(static_cast<uint16_t>(whi >> 16)));
      }
    }
    if (!has) continue;
    const double ca = s_cos[e], sa = s_sin[e], cb = s_cos[e + 1], sb = s_sin[e + 1];
    const double o1a = __dsub_rn(__dmul_rn(x1a, ca), __dmul_rn(x2a, sa));
    const double o2a = __dadd_rn(__dmul_rn(x2a, ca), __dmul_rn(x1a, sa));
    const double o1b = __dsub_rn(__dmul_rn(x1b, cb), __dmul_rn(x2b, sb));
    const double o2b = __dadd_rn(__dmul_rn(x2b, cb), __dmul_rn(x1b, sb));
    st_u32(dst + e, static_cast<uint32_t>(double_to_bf16(o1a)) |
                        (static_cast<uint32_t>(double_to_bf16(o1b)) << 16));
    st_u32(dst + H + e, static_cast<uint32_t>(double_to_bf16(o2a)) |
                            (static_cast<uint32_t>(double_to_bf16(o2b)) << 16));
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, int head_dim, cudaStream_t stream) {
  if (p.T == 0) return cudaSuccess;
  switch (head_dim) {
    case 64: append_rope_kernel<64><<<p.T, 256, 0, stream>>>(p); break;
    case 96: append_rope_kernel<96><<<p.T, 256, 0, stream>>>(p); break;
    case 128: append_rope_kernel<128><<<p.T, 256, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace lnk
