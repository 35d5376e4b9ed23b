// K1: per-token QK-norm (optional), RoPE and K/V append into the page pool.
//
// One CTA per token, 16 warps.  The rotated value of element i (paired with
// i + D/2) is
//     o_i       = r (x_i (g_i c_i)       - x_{i+D/2} (g_{i+D/2} s_i))
//     o_{i+D/2} = r (x_{i+D/2} (g_{i+D/2} c_i) + x_i (g_i s_i))
// where c_i, s_i are the cosine and sine of the float32 angle
// f32(position) * inv_freq[i], g the QK-norm weights and r the head's RMS
// factor 1 / sqrt(mean(x^2) + eps) (g = r = 1 without QK-norm).  The four
// per-frequency coefficients are evaluated once per token in double precision
// and kept as pairs of floats (hi + lo); each element is then computed with
// error-free float products and sums (about 2^-46 relative error) and rounded
// once to bf16, looking at the low part only to break an exact tie of the high
// part.  The result is the correctly rounded value of the exact expression
// except in cases far rarer than one in 10^10, without per-element
// double-precision arithmetic (which is slow on this GPU).  V is copied bit
// for bit into the token's pool slot.
//
// Sources: "Phi-3 Mini 4K Instruct -- files", src/rope.linnet (tables) and
// src/attention.linnet (rope + write_tokens in prefill_packed / step_packed);
// "Qwen3-4B", QK-norm paragraph; "Mistral 7B Instruct v0.3", Entries table
// (prefill_paged: each token written at its place in the pool).
#include "common.cuh"

namespace lnk {
namespace {

constexpr int kWarps = 16;
constexpr int kMaxHeadsPerWarp = 8;  // rotated heads (Hq + Hkv) <= 128

struct DF {
  float hi, lo;
};

__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}

__device__ __forceinline__ DF two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ DF split(double v) {
  const float hi = __double2float_rn(v);
  return {hi, __double2float_rn(v - static_cast<double>(hi))};
}

// x * a - y * b for bf16-exact x, y and pair-of-float a, b.
__device__ __forceinline__ DF dot2(float x, DF a, float y, DF b) {
  const DF p = two_prod(x, a.hi);
  const DF q = two_prod(y, b.hi);
  const DF s = two_sum(p.hi, -q.hi);
  const float l = __fadd_rn(__fadd_rn(s.lo, __fsub_rn(p.lo, q.lo)),
                            __fsub_rn(__fmul_rn(x, a.lo), __fmul_rn(y, b.lo)));
  return two_sum(s.hi, l);
}

__device__ __forceinline__ DF mul_df(DF a, DF r) {
  const DF m = two_prod(a.hi, r.hi);
  const float l = __fadd_rn(m.lo, __fadd_rn(__fmul_rn(a.hi, r.lo), __fmul_rn(a.lo, r.hi)));
  return two_sum(m.hi, l);
}

// Round hi + lo (|lo| <= half an ulp of hi, hi = RN(hi + lo)) to bf16, nearest even.
__device__ __forceinline__ uint32_t df_to_bf16(DF v) {
  const uint32_t u = __float_as_uint(v.hi);
  if ((u & 0xFFFFu) == 0x8000u && v.lo != 0.f) {
    // hi sits exactly between two bf16 values: the low part decides
    const bool away = (v.lo > 0.f) == (v.hi > 0.f);
    return (u >> 16) + (away ? 1u : 0u);
  }
  return (u + 0x7FFFu + ((u >> 16) & 1u)) >> 16;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int D>
__global__ void __launch_bounds__(kWarps * 32) append_rope_kernel(const AppendParams p) {
  constexpr int H = D / 2;
  constexpr int kLanes = D / 4;  // lanes holding data: two elements of each half
  // coefficient sets: [0] queries, [1] keys; [.][0] g_i c_i, [1] g_{i+H} s_i,
  // [2] g_{i+H} c_i, [3] g_i s_i
  __shared__ DF s_coef[2][4][H];
  __shared__ DF s_ss[kWarps * kMaxHeadsPerWarp];
  __shared__ DF s_r[kWarps * kMaxHeadsPerWarp];
  __shared__ long long s_slot;

  // Let the next kernel on the stream start its prologue; it waits for this
  // grid's writes before reading them.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int t = blockIdx.x;
  const int pos = p.positions[t];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int nrot = p.hq + p.hkv;  // rotated heads: queries then keys
  const bool norm_q = p.q_norm_w != nullptr, norm_k = p.k_norm_w != nullptr;

  // ---- per-token coefficients (double precision, once per frequency) ----
  if (tid < H && pos >= 0) {
    const float a = __fmul_rn(static_cast<float>(pos), p.inv_freq[tid]);
    double s, c;
    sincos(static_cast<double>(a), &s, &c);
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint16_t* w = which == 0 ? p.q_norm_w : p.k_norm_w;
      double g1 = 1.0, g2 = 1.0;
      if (w != nullptr) {
        g1 = static_cast<double>(__uint_as_float(static_cast<uint32_t>(w[tid]) << 16));
        g2 = static_cast<double>(__uint_as_float(static_cast<uint32_t>(w[tid + H]) << 16));
      }
      s_coef[which][0][tid] = split(g1 * c);
      s_coef[which][1][tid] = split(g2 * s);
      s_coef[which][2][tid] = split(g2 * c);
      s_coef[which][3][tid] = split(g1 * s);
    }
  }
  if (tid == kWarps * 32 - 1) {
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

  // ---- load this warp's rotated heads (all loads in flight together) ----
  const bool has = lane < kLanes;
  const int e = 2 * lane;
  uint32_t xlo[kMaxHeadsPerWarp], xhi[kMaxHeadsPerWarp];
#pragma unroll
  for (int j = 0; j < kMaxHeadsPerWarp; ++j) {
    const int hh = warp + j * kWarps;
    xlo[j] = xhi[j] = 0u;
    if (hh < nrot && has && pos >= 0) {
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
      const int hh = warp + j * kWarps;
      if (hh >= nrot) break;
      if (!(hh < p.hq ? norm_q : norm_k)) continue;
      const float a0 = bf16_lo(xlo[j]), a1 = bf16_hi(xlo[j]), b0 = bf16_lo(xhi[j]), b1 = bf16_hi(xhi[j]);
      DF acc = two_sum(__fmul_rn(a0, a0), __fmul_rn(a1, a1));
      DF u = two_sum(__fmul_rn(b0, b0), __fmul_rn(b1, b1));
      DF v = two_sum(acc.hi, u.hi);
      acc = two_sum(v.hi, __fadd_rn(v.lo, __fadd_rn(acc.lo, u.lo)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float oh = __shfl_xor_sync(0xffffffffu, acc.hi, o);
        const float ol = __shfl_xor_sync(0xffffffffu, acc.lo, o);
        const DF w = two_sum(acc.hi, oh);
        acc = two_sum(w.hi, __fadd_rn(w.lo, __fadd_rn(acc.lo, ol)));
      }
      if (lane == 0) s_ss[hh] = acc;
    }
  }
  __syncthreads();
  // one lane per head computes the RMS factor in double precision
  if ((norm_q || norm_k) && tid < nrot && pos >= 0 && (tid < p.hq ? norm_q : norm_k)) {
    const DF ss = s_ss[tid];
    const double v = (static_cast<double>(ss.hi) + static_cast<double>(ss.lo)) / static_cast<double>(D);
    s_r[tid] = split(1.0 / sqrt(v + p.norm_eps));
  }
  __syncthreads();

  const long long slot = s_slot;
  const size_t pool_head_stride = static_cast<size_t>(p.num_pages) * kPage * D;
#pragma unroll
  for (int j = 0; j < kMaxHeadsPerWarp; ++j) {
    const int hh = warp + j * kWarps;
    if (hh >= nrot) break;
    const bool is_q = hh < p.hq;
    uint16_t* dst;
    if (is_q) {
      dst = p.q_out + (static_cast<size_t>(t) * p.hq + hh) * D;
    } else {
      if (slot < 0) continue;
      dst = p.k_pool + (hh - p.hq) * pool_head_stride + static_cast<size_t>(slot) * D;
    }
    if (!has) continue;
    if (pos < 0) {  // inactive token: zero query output
      *reinterpret_cast<uint32_t*>(dst + e) = 0u;
      *reinterpret_cast<uint32_t*>(dst + H + e) = 0u;
      continue;
    }
    const int set = is_q ? 0 : 1;
    const bool normed = is_q ? norm_q : norm_k;
    const DF r = normed ? s_r[hh] : DF{1.f, 0.f};
    uint32_t lo_bits = 0, hi_bits = 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = e + k;
      const float x1 = k ? bf16_hi(xlo[j]) : bf16_lo(xlo[j]);
      const float x2 = k ? bf16_hi(xhi[j]) : bf16_lo(xhi[j]);
      DF o1 = dot2(x1, s_coef[set][0][i], x2, s_coef[set][1][i]);
      const DF nd = {-s_coef[set][3][i].hi, -s_coef[set][3][i].lo};
      DF o2 = dot2(x2, s_coef[set][2][i], x1, nd);
      if (normed) {
        o1 = mul_df(o1, r);
        o2 = mul_df(o2, r);
      }
      lo_bits |= df_to_bf16(o1) << (16 * k);
      hi_bits |= df_to_bf16(o2) << (16 * k);
    }
    *reinterpret_cast<uint32_t*>(dst + e) = lo_bits;
    *reinterpret_cast<uint32_t*>(dst + H + e) = hi_bits;
  }
  // value heads: bit copy into the slot
  if (slot >= 0) {
    for (int vh = warp; vh < p.hkv; vh += kWarps) {
      const uint4* src = reinterpret_cast<const uint4*>(p.v + (static_cast<size_t>(t) * p.hkv + vh) * D);
      uint4* dst = reinterpret_cast<uint4*>(p.v_pool + vh * pool_head_stride + static_cast<size_t>(slot) * D);
      if (lane < D / 8) dst[lane] = src[lane];
    }
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, int head_dim, cudaStream_t stream) {
  if (p.T == 0) return cudaSuccess;
  if (p.hq + p.hkv > kWarps * kMaxHeadsPerWarp) return cudaErrorInvalidValue;
  switch (head_dim) {
    case 64: append_rope_kernel<64><<<p.T, kWarps * 32, 0, stream>>>(p); break;
    case 96: append_rope_kernel<96><<<p.T, kWarps * 32, 0, stream>>>(p); break;
    case 128: append_rope_kernel<128><<<p.T, kWarps * 32, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace lnk
