// K1: per-token QK-norm (optional), RoPE and K/V append into the page pool.
//
// One CTA per token, 16 warps.  The rotated value of element i (paired with
// i + D/2) is
//     o_i       = r (x_i (g_i c_i)       - x_{i+D/2} (g_{i+D/2} s_i))
//     o_{i+D/2} = r (x_{i+D/2} (g_{i+D/2} c_i) + x_i (g_i s_i))
// where c_i, s_i are the cosine and sine of the float32 angle
// f32(position) * inv_freq[i], g the QK-norm weights and r the head's RMS
// factor 1 / sqrt(mean(x^2) + eps) (g = r = 1 without QK-norm).  The four
// per-frequency coefficients are evaluated once per token as pairs of floats
// (hi + lo; sine and cosine by a float-pair Taylor series after an exact
// reduction by pi/2); each element is then computed with
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
#include <cuda_fp8.h>

#include "common.cuh"

namespace lnk {
namespace {

constexpr int kMaxRotated = 128;  // rotated heads (Hq + Hkv) per token
// Warps per token: 16 for small launches (a short per-token chain), WIDE_WARPS
// when the launch has many tokens per SM (more tokens resident at once).
constexpr int kWarpsSmall = 16;
constexpr int kWarpsWide = 8;
constexpr int kWideTokensPerSm = 4;  // launches with at least this many tokens per SM use kWarpsWide

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

// |a| >= |b| (or a == 0): s + e == a + b exactly.
__device__ __forceinline__ DF fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ DF df_add(DF a, DF b) {
  const DF s = two_sum(a.hi, b.hi);
  const DF t = two_sum(a.lo, b.lo);
  const DF u = fast_two_sum(s.hi, __fadd_rn(s.lo, t.hi));
  return fast_two_sum(u.hi, __fadd_rn(u.lo, t.lo));
}

__device__ __forceinline__ DF df_mul(DF a, DF b) {
  const DF p = two_prod(a.hi, b.hi);
  return fast_two_sum(p.hi, __fadd_rn(p.lo, __fmaf_rn(a.hi, b.lo, __fmul_rn(a.lo, b.hi))));
}

// a (bf16-exact) times a pair of floats
__device__ __forceinline__ DF df_scale(float a, DF b) {
  const DF p = two_prod(a, b.hi);
  return fast_two_sum(p.hi, __fmaf_rn(a, b.lo, p.lo));
}

// 1 / n! as a pair of floats (evaluated in double, exact factorials up to 18!)
struct Coef {
  float hi, lo;
};
constexpr double inv_factorial(int n) {
  double f = 1.0;
  for (int i = 2; i <= n; ++i) f *= i;
  return 1.0 / f;
}
constexpr Coef coef(int n, bool negative) {
  const double v = negative ? -inv_factorial(n) : inv_factorial(n);
  return {static_cast<float>(v), static_cast<float>(v - static_cast<double>(static_cast<float>(v)))};
}

// pi / 2 as the sum of three floats (to about 2^-76), from the digits of pi
constexpr float kPio2a = 0x1.921fb6p+0f;
constexpr float kPio2b = -0x1.777a5cp-25f;
constexpr float kPio2c = -0x1.ee59dap-50f;
constexpr float kTwoOverPi = 0x1.45f306p-1f;

// sin and cos of a float angle (|a| < 2^20) as pairs of floats, to about
// 2^-48 absolute: Cody-Waite reduction by pi/2 with error-free products
// (k < 2^20 * 2/pi is an exact float integer), then the Taylor series of
// sin and cos on |r| <= pi/4 (terms to r^17 and r^18) by Horner's rule, the
// small high-order part in float and the rest in float pairs.
__device__ __forceinline__ void sincos_df(float a, DF& sn, DF& cs) {
  const float k = rintf(__fmul_rn(a, kTwoOverPi));
  const DF p1 = two_prod(k, kPio2a);
  DF r = two_sum(__fsub_rn(a, p1.hi), -p1.lo);  // a - p1.hi is exact
  const DF p2 = two_prod(k, kPio2b);
  r = df_add(r, DF{-p2.hi, -p2.lo});
  r = df_add(r, DF{-__fmul_rn(k, kPio2c), 0.f});
  const DF x = df_mul(r, r);
  // sin(r) / r = sum_n (-1)^n x^n / (2n+1)!,  cos(r) = sum_n (-1)^n x^n / (2n)!
  float fs = coef(17, false).hi;
  fs = __fmaf_rn(fs, x.hi, coef(15, true).hi);
  fs = __fmaf_rn(fs, x.hi, coef(13, false).hi);
  fs = __fmaf_rn(fs, x.hi, coef(11, true).hi);
  DF ps{fs, 0.f};
  {
    constexpr Coef c9 = coef(9, false), c7 = coef(7, true), c5 = coef(5, false), c3 = coef(3, true);
    ps = df_add(df_mul(ps, x), DF{c9.hi, c9.lo});
    ps = df_add(df_mul(ps, x), DF{c7.hi, c7.lo});
    ps = df_add(df_mul(ps, x), DF{c5.hi, c5.lo});
    ps = df_add(df_mul(ps, x), DF{c3.hi, c3.lo});
    ps = df_add(df_mul(ps, x), DF{1.f, 0.f});
  }
  const DF s_r = df_mul(ps, r);
  float fc = coef(18, true).hi;
  fc = __fmaf_rn(fc, x.hi, coef(16, false).hi);
  fc = __fmaf_rn(fc, x.hi, coef(14, true).hi);
  fc = __fmaf_rn(fc, x.hi, coef(12, false).hi);
  DF pc{fc, 0.f};
  {
    constexpr Coef c10 = coef(10, true), c8 = coef(8, false), c6 = coef(6, true), c4 = coef(4, false),
                   c2 = coef(2, true);
    pc = df_add(df_mul(pc, x), DF{c10.hi, c10.lo});
    pc = df_add(df_mul(pc, x), DF{c8.hi, c8.lo});
    pc = df_add(df_mul(pc, x), DF{c6.hi, c6.lo});
    pc = df_add(df_mul(pc, x), DF{c4.hi, c4.lo});
    pc = df_add(df_mul(pc, x), DF{c2.hi, c2.lo});
    pc = df_add(df_mul(pc, x), DF{1.f, 0.f});
  }
  const DF c_r = pc;
  const DF ns_r{-s_r.hi, -s_r.lo}, nc_r{-c_r.hi, -c_r.lo};
  switch (static_cast<int>(k) & 3) {  // a = r + k pi/2
    case 0: sn = s_r; cs = c_r; break;
    case 1: sn = c_r; cs = ns_r; break;
    case 2: sn = ns_r; cs = nc_r; break;
    default: sn = nc_r; cs = s_r; break;
  }
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

// E4M3 codes of two bf16 values (low half first) for a pool with `scale`: one
// IEEE float32 division each, then round to nearest even with saturation to
// +-448; the low value's code in the low byte.
__device__ __forceinline__ uint16_t e4m3_pair(uint32_t bits, float scale) {
  const float2 f = make_float2(__fdiv_rn(__uint_as_float(bits << 16), scale),
                               __fdiv_rn(__uint_as_float(bits & 0xFFFF0000u), scale));
  return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, __NV_E4M3));
}

template <int D, int kWarps>
__global__ void __launch_bounds__(kWarps * 32) append_rope_kernel(const AppendParams p) {
  constexpr int kMaxHeadsPerWarp = kMaxRotated / kWarps;
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

  // ---- per-token coefficients (float pairs, once per frequency) ----
  if (tid < H && pos >= 0) {
    const float a = __fmul_rn(static_cast<float>(pos), p.inv_freq[tid]);
    DF sn, cs;
    if (fabsf(a) < 1048576.f) {
      sincos_df(a, sn, cs);
    } else {  // very large angles (positions beyond 2^20): double precision
      double s, c;
      sincos(static_cast<double>(a), &s, &c);
      sn = split(s);
      cs = split(c);
    }
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint16_t* w = which == 0 ? p.q_norm_w : p.k_norm_w;
      float g1 = 1.f, g2 = 1.f;
      if (w != nullptr) {
        g1 = __uint_as_float(static_cast<uint32_t>(w[tid]) << 16);
        g2 = __uint_as_float(static_cast<uint32_t>(w[tid + H]) << 16);
      }
      s_coef[which][0][tid] = df_scale(g1, cs);
      s_coef[which][1][tid] = df_scale(g2, sn);
      s_coef[which][2][tid] = df_scale(g2, cs);
      s_coef[which][3][tid] = df_scale(g1, sn);
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
    for (int vh = warp; vh < p.hkv; vh += kWarps) {
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

template <int D, int kWarps>
cudaError_t launch_append_w(const AppendParams& p, cudaStream_t stream) {
  // Prefer the largest shared-memory carveout, like the attention kernels that
  // follow: their CTAs can then start on an SM next to this kernel's (the
  // attention kernel is launched as a programmatic dependent) without the SM
  // first switching its L1 / shared-memory split.
  const cudaError_t attr = prefer_max_shared(reinterpret_cast<const void*>(append_rope_kernel<D, kWarps>));
  if (attr != cudaSuccess) return attr;
  append_rope_kernel<D, kWarps><<<p.T, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_append_t(const AppendParams& p, cudaStream_t stream) {
  if (static_cast<long long>(p.T) >= static_cast<long long>(kWideTokensPerSm) * device_sm_count())
    return launch_append_w<D, kWarpsWide>(p, stream);
  return launch_append_w<D, kWarpsSmall>(p, stream);
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
