// Float-pair arithmetic for the rotary embedding and the QK-norm, shared by
// the append kernel and the fused decode step, so that both round every
// rotated element identically.
//
// The rotated value of element i (paired with i + D/2) is
//     o_i       = r (x_i (g_i c_i)       - x_{i+D/2} (g_{i+D/2} s_i))
//     o_{i+D/2} = r (x_{i+D/2} (g_{i+D/2} c_i) + x_i (g_i s_i))
// where c_i, s_i are the cosine and sine of the float32 angle
// f32(position) * inv_freq[i], g the QK-norm weights and r the head's RMS
// factor 1 / sqrt(mean(x^2) + eps) (g = r = 1 without QK-norm).  The four
// per-frequency coefficients are evaluated once per token as pairs of floats
// (hi + lo; sine and cosine by a float-pair Taylor series after an exact
// reduction by pi/2); each element is then computed with error-free float
// products and sums (about 2^-46 relative error) and rounded once to bf16,
// looking at the low part only to break an exact tie of the high part.  The
// result is the correctly rounded value of the exact expression except in
// cases far rarer than one in 10^10, without per-element double-precision
// arithmetic (which is slow on this GPU).
//
// Sources: "Phi-3 Mini 4K Instruct -- files", src/rope.linnet (tables);
// "Qwen3-4B", QK-norm paragraph.
#pragma once

#include <cuda_fp8.h>

#include <cstdint>

namespace lnk {
namespace rope {

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

// Sine and cosine (float pairs) of the float32 angle f32(pos) * inv_freq.
__device__ __forceinline__ void angle_sincos(int pos, float inv_freq, DF& sn, DF& cs) {
  const float a = __fmul_rn(static_cast<float>(pos), inv_freq);
  if (fabsf(a) < 1048576.f) {
    sincos_df(a, sn, cs);
  } else {  // very large angles (positions beyond 2^20): double precision
    double s, c;
    sincos(static_cast<double>(a), &s, &c);
    sn = split(s);
    cs = split(c);
  }
}

// The four coefficients of frequency i for one kind of head (queries or
// keys): g_i c_i, g_{i+D/2} s_i, g_{i+D/2} c_i, g_i s_i, with g1 = g_i and
// g2 = g_{i+D/2} (1 without QK-norm).
struct Coefs {
  DF gc1, gs2, gc2, gs1;
};
__device__ __forceinline__ Coefs coefs_of(DF sn, DF cs, float g1, float g2) {
  return Coefs{df_scale(g1, cs), df_scale(g2, sn), df_scale(g2, cs), df_scale(g1, sn)};
}

// A head's sum of squares when each lane of the warp holds elements
// (e, e + 1) in xlo and (e + D/2, e + D/2 + 1) in xhi (zero on lanes without
// data): squares of bf16 values are exact in float, the sums are float pairs,
// and every lane ends with the same total.
__device__ __forceinline__ DF head_sumsq(uint32_t xlo, uint32_t xhi) {
  const float a0 = bf16_lo(xlo), a1 = bf16_hi(xlo), b0 = bf16_lo(xhi), b1 = bf16_hi(xhi);
  DF acc = two_sum(__fmul_rn(a0, a0), __fmul_rn(a1, a1));
  const DF u = two_sum(__fmul_rn(b0, b0), __fmul_rn(b1, b1));
  const DF v = two_sum(acc.hi, u.hi);
  acc = two_sum(v.hi, __fadd_rn(v.lo, __fadd_rn(acc.lo, u.lo)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, acc.hi, o);
    const float ol = __shfl_xor_sync(0xffffffffu, acc.lo, o);
    const DF w = two_sum(acc.hi, oh);
    acc = two_sum(w.hi, __fadd_rn(w.lo, __fadd_rn(acc.lo, ol)));
  }
  return acc;
}

// The QK-norm factor 1 / sqrt(ss / D + eps), in double precision, as a float pair.
__device__ __forceinline__ DF rms_factor(DF ss, int d, double eps) {
  const double v = (static_cast<double>(ss.hi) + static_cast<double>(ss.lo)) / static_cast<double>(d);
  return split(1.0 / sqrt(v + eps));
}

// The rotated bf16 values of elements (e, e + 1) (low half, packed in lo_bits)
// and (e + D/2, e + D/2 + 1) (high half, in hi_bits) of one head, from its
// values in xlo / xhi and the coefficients c[e], c[e + 1]; r is the QK-norm
// factor when normed.
__device__ __forceinline__ void rotate_pairs(uint32_t xlo, uint32_t xhi, const Coefs* c, int e, bool normed, DF r,
                                             uint32_t& lo_bits, uint32_t& hi_bits) {
  lo_bits = hi_bits = 0u;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const Coefs ci = c[e + k];
    const float x1 = k ? bf16_hi(xlo) : bf16_lo(xlo);
    const float x2 = k ? bf16_hi(xhi) : bf16_lo(xhi);
    DF o1 = dot2(x1, ci.gc1, x2, ci.gs2);
    DF o2 = dot2(x2, ci.gc2, x1, DF{-ci.gs1.hi, -ci.gs1.lo});
    if (normed) {
      o1 = mul_df(o1, r);
      o2 = mul_df(o2, r);
    }
    lo_bits |= df_to_bf16(o1) << (16 * k);
    hi_bits |= df_to_bf16(o2) << (16 * k);
  }
}

}  // namespace rope
}  // namespace lnk
