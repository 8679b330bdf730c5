// swiglu_math.cuh - exactly rounded SwiGLU numerics shared by the fused
// forward and backward kernels (page "Add MXFP8 fused-MLP overrides in
// torchtitan", Numerics and tests):
//   sigma  = fp32 correctly rounded 1/(1+e^-g)
//   a      = RN_bf16(RN_f32(g * sigma))          (bf16 SiLU)
//   y      = RN_bf16(RN_f32(a * u))
//   du     = RN_bf16(RN_f32(dy * a))
//   dg     = RN_bf16(dy * u * sigma * (1 + g(1 - sigma)))  (one rounding)
#pragma once

#include "common.cuh"

namespace mx {
namespace swiglu_math {
namespace {

// ------------------------------------------------------------------ numerics
//
// Three tiers, all giving the exactly defined result:
//   1. fp32 fast path: t = expf(-g) (at most 2 ulp), s = rcp.approx(1 + t)
//      (at most 1 ulp); the bf16 result is kept when it lies farther from a
//      bf16 rounding midpoint than the error bound of the fp32 chain.
//   2. float-float (pairs of fp32 carrying ~46 bits) for the few elements
//      near a midpoint: an own exp (Cody-Waite reduction by ln 2 split in
//      three parts, then the Taylor series of e^r, |r| <= ln2/2, evaluated
//      by Horner's rule with double-float arithmetic in the style of Dekker
//      1971 / Knuth TAOCP 4.2.2 error-free transforms) and a Newton-corrected
//      reciprocal.  Runs on the fp32 pipe.
//   3. fp64 for |g| > 64, for extreme magnitudes of dy*u and for the
//      float-float results that are still within their error of a midpoint.

MX_DEVINL double bf16_bits_to_f64(uint32_t b) { return (double)__uint_as_float(b << 16); }

// RN to bf16 from an fp64 value (ties to even, subnormals, overflow to Inf).
MX_DEVINL uint32_t bf16_from_f64_rn(double x) {
  const unsigned long long b = (unsigned long long)__double_as_longlong(x);
  const uint32_t sign = (uint32_t)(b >> 63) << 15;
  const unsigned long long mag = b & 0x7FFFFFFFFFFFFFFFull;
  if (mag > 0x7FF0000000000000ull) return 0x7FC0u;
  if (mag == 0x7FF0000000000000ull) return sign | 0x7F80u;
  if (mag < 0x0010000000000000ull) return sign;  // zero or fp64 subnormal (far below bf16)
  const int e = (int)(mag >> 52) - 1023;
  const unsigned long long mant = (mag & 0x000FFFFFFFFFFFFFull) | 0x0010000000000000ull;
  const int qexp = e < -126 ? -133 : e - 7;
  const int sh = qexp - e + 52;  // >= 45
  if (sh >= 55) return sign;     // below half the smallest bf16 subnormal
  unsigned long long n = mant >> sh;
  const unsigned long long rem = mant & ((1ull << sh) - 1);
  const unsigned long long half = 1ull << (sh - 1);
  if (rem > half || (rem == half && (n & 1))) ++n;
  if (e < -126) return sign | (uint32_t)n;  // n == 128 encodes 2^-126
  int ee = e;
  if (n == 256) { n = 128; ++ee; }
  if (ee > 127) return sign | 0x7F80u;
  return sign | ((uint32_t)(ee + 127) << 7) | (uint32_t)(n - 128);
}

// The bf16 rounding midpoint nearest to x (x finite, non-zero): halfway
// between RN_bf16(x) and its neighbour on x's side.
MX_DEVINL double nearest_bf16_midpoint(double x) {
  const uint32_t b = bf16_from_f64_rn(x);
  const double v = bf16_bits_to_f64(b);
  const uint32_t mag = b & 0x7FFFu;
  uint32_t nmag;
  if (fabs(x) >= fabs(v)) nmag = mag + 1;
  else nmag = mag == 0 ? 0 : mag - 1;
  const double w = bf16_bits_to_f64((b & 0x8000u) | nmag);
  return 0.5 * (v + w);
}

// |low 16 bits of p - 0x8000| > margin: p's bf16 rounding is decided with
// room to spare (the bf16 midpoints are the fp32 values whose low half is
// exactly 0x8000).
MX_DEVINL bool clear_of_midpoint(float p, uint32_t margin) {
  const uint32_t low = __float_as_uint(p) & 0xFFFFu;
  return (low - (0x8000u - margin)) > 2u * margin;
}

MX_DEVINL float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// ---- float-float
struct ff {
  float hi, lo;
};
MX_DEVINL ff fast_two_sum(float a, float b) {  // |a| >= |b|
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
MX_DEVINL ff two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}
MX_DEVINL ff ff_add(ff x, ff y) {
  ff s = two_sum(x.hi, y.hi);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, y.lo)));
}
MX_DEVINL ff ff_add_f(ff x, float b) {
  ff s = two_sum(x.hi, b);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, x.lo));
}
MX_DEVINL ff ff_mul(ff x, ff y) {
  const float p = __fmul_rn(x.hi, y.hi);
  float e = __fmaf_rn(x.hi, y.hi, -p);
  e = __fmaf_rn(x.hi, y.lo, e);
  e = __fmaf_rn(x.lo, y.hi, e);
  return fast_two_sum(p, e);
}
MX_DEVINL ff ff_mul_f(ff x, float b) {
  const float p = __fmul_rn(x.hi, b);
  float e = __fmaf_rn(x.hi, b, -p);
  e = __fmaf_rn(x.lo, b, e);
  return fast_two_sum(p, e);
}
MX_DEVINL ff ff_rcp(ff x) {  // one Newton step on a correctly rounded quotient
  const float q = __fdiv_rn(1.0f, x.hi);
  float e = __fmaf_rn(-x.hi, q, 1.0f);
  e = __fmaf_rn(-x.lo, q, e);
  return fast_two_sum(q, __fmul_rn(q, e));
}

// e^x as float-float for |x| <= 64 (relative error well below 2^-44).
MX_DEVINL ff ff_exp(float x) {
  // ln 2 = L1 + L2 + L3, L1 with 15 significant bits so that n*L1 is exact
  constexpr float L1 = 0x1.62e4p-1f, L2 = 0x1.7f7d1cp-20f, L3 = 0x1.ef357ap-45f;
  const float n = rintf(__fmul_rn(x, 0x1.715476p+0f));
  ff r = two_sum(x, -__fmul_rn(n, L1));  // exact
  const float p2 = __fmul_rn(n, L2);
  r = ff_add(r, ff{-p2, -__fmaf_rn(n, L2, -p2)});
  r = ff_add_f(r, -__fmul_rn(n, L3));
  // Taylor coefficients 1/k! (k = 7..11 in fp32, k = 0..6 as float-float)
  float tail = 0x1.ae6456p-26f;
  tail = __fmaf_rn(tail, r.hi, 0x1.27e4fcp-22f);
  tail = __fmaf_rn(tail, r.hi, 0x1.71de3ap-19f);
  tail = __fmaf_rn(tail, r.hi, 0x1.a01a02p-16f);
  tail = __fmaf_rn(tail, r.hi, 0x1.a01a02p-13f);
  const ff c[7] = {{1.0f, 0.0f},
                   {1.0f, 0.0f},
                   {0.5f, 0.0f},
                   {0x1.555556p-3f, -0x1.555556p-28f},
                   {0x1.555556p-5f, -0x1.555556p-30f},
                   {0x1.111112p-7f, -0x1.dddddep-32f},
                   {0x1.6c16c2p-10f, -0x1.27d27ep-35f}};
  ff acc{tail, 0.0f};
#pragma unroll
  for (int k = 6; k >= 0; --k) acc = ff_add(ff_mul(acc, r), c[k]);
  const float two_n = __uint_as_float((uint32_t)((int)n + 127) << 23);
  return {__fmul_rn(acc.hi, two_n), __fmul_rn(acc.lo, two_n)};
}

// fp32 ulp of a positive normal float
MX_DEVINL float ulp_of(float x) { return __uint_as_float(__float_as_uint(x) & 0x7F800000u) * 0x1p-23f; }

__device__ __noinline__ float sigmoid_f32_fp64(float g) {
  const double s = 1.0 / (1.0 + exp(-(double)g));
  return __double2float_rn(s);
}

// Correctly rounded fp32 sigma for |g| <= 64 via float-float; falls back to
// fp64 if the float-float value is within its error of an fp32 midpoint.
MX_DEVINL float sigmoid_f32_ff(float g, ff* t_out, ff* s_out) {
  const ff t = ff_exp(-g);
  const ff s = ff_rcp(ff_add_f(t, 1.0f));
  *t_out = t;
  *s_out = s;
  const float half_ulp = 0.5f * ulp_of(s.hi);
  if (fabsf(fabsf(s.lo) - half_ulp) <= s.hi * 0x1p-40f) return sigmoid_f32_fp64(g);
  return s.hi;
}

// bf16 SiLU from a correctly rounded fp32 sigma
MX_DEVINL uint32_t silu_from_sigma(float g, float sig) { return f32_to_bf16_bits(__fmul_rn(g, sig)); }

// Result of the shared fast path for one element.
struct SigFast {
  float t, s;   // expf(-g), approx 1/(1+t)
  bool ok;      // |g| <= 64 (fast path usable at all)
};
MX_DEVINL SigFast sig_fast(float g) {
  SigFast r;
  r.ok = fabsf(g) <= 64.0f;  // false for NaN / Inf too
  r.t = expf(-g);
  r.s = rcp_approx(__fadd_rn(1.0f, r.t));
  return r;
}

// Tiers 2 and 3 of a(g), kept out of line: they run for well under 0.1%
// of the elements and would otherwise bloat every unrolled copy of the fast
// path (instruction-cache misses).
__device__ __noinline__ uint32_t silu_bits_slow(float g) {
  if (fabsf(g) <= 64.0f) {
    ff t, s;
    return silu_from_sigma(g, sigmoid_f32_ff(g, &t, &s));
  }
  return silu_from_sigma(g, sigmoid_f32_fp64(g));
}

// a(g): RN_bf16(RN_f32(g * sigma_c)).  Fast-path error of g*s against
// g*sigma_c is at most 9 fp32 ulps; 16 leaves room.
MX_DEVINL uint32_t silu_bits_from(float g, const SigFast& f) {
  const float p = __fmul_rn(g, f.s);
  if (f.ok && clear_of_midpoint(p, 16)) return f32_to_bf16_bits(p);
  return silu_bits_slow(g);
}


// dg by fp64 with exact-tie handling (see the comment inside).
__device__ __noinline__ uint32_t dg_bits_fp64(float dyf, float g, float u) {
  const double gd = (double)g;
  const double t = exp(-gd);
  const double dyu64 = (double)dyf * (double)u;  // exact
  if (t > 1e300) return bf16_from_f64_rn(dyu64 * -0.0);  // sigma underflows: f is a tiny negative
  const double s = 1.0 / (1.0 + t);
  const double oms = t * s;
  double pd = dyu64 * (s * (1.0 + gd * oms));
  // Exact ties: dy*u (16 significant bits) can sit exactly on a bf16 rounding
  // midpoint while f is 1 (large g) or 1/2 (tiny |g|) to fp64 precision.
  // The exact product then lies just off the midpoint on the side given by
  // the sign of f - 1 (positive for large g) or f - 1/2 (sign of g).
  if (pd != 0.0 && isfinite(pd)) {
    const double m = nearest_bf16_midpoint(pd);
    if (fabs(pd - m) <= fabs(pd) * 0x1p-40) {
      double dir = 0.0;
      if (m == dyu64) dir = 1.0;
      else if (m == 0.5 * dyu64) dir = (gd > 0.0) ? 1.0 : ((gd < 0.0) ? -1.0 : 0.0);
      if (dir != 0.0) pd = m + copysign(fabs(m) * 0x1p-20, dyu64 * dir);
      else if (m == 0.5 * dyu64) pd = m;  // g == 0: an exact tie, ties to even
    }
  }
  return bf16_from_f64_rn(pd);
}

// Tiers 2 and 3 of dg (out of line, see silu_bits_slow).
__device__ __noinline__ uint32_t dg_bits_slow(float dyf, float g, float u) {
  if (!isfinite(g)) return 0x7FC0u;
  const float dyu = __fmul_rn(dyf, u);  // exact in the normal range
  const float adyu = fabsf(dyu);
  if (fabsf(g) <= 64.0f && adyu >= 0x1p-100f && adyu <= 0x1p100f) {
    // tier 2: float-float
    const ff t = ff_exp(-g);
    const ff s = ff_rcp(ff_add_f(t, 1.0f));
    const ff omsf = ff_mul(t, s);
    const ff gof = ff_mul_f(omsf, g);
    const ff in = ff_add_f(gof, 1.0f);
    const ff pf = ff_mul_f(ff_mul(s, in), dyu);
    const float rat2 = fabsf(gof.hi) / fabsf(in.hi);
    const uint32_t low = __float_as_uint(pf.hi) & 0xFFFFu;
    if (low != 0x8000u && fabsf(pf.hi) >= 0x1p-100f) return f32_to_bf16_bits(pf.hi);
    if (low == 0x8000u && fabsf(pf.lo) > fabsf(pf.hi) * 0x1p-40f * (1.0f + rat2)) {
      // pf.hi is a bf16 midpoint; the exact value lies on pf.lo's side
      const uint32_t b = __float_as_uint(pf.hi);
      const bool up = (pf.lo > 0.0f) == (pf.hi > 0.0f);  // away from zero
      return ((up ? (b + 0x8000u) : (b - 0x8000u)) >> 16) & 0xFFFFu;
    }
  }
  return dg_bits_fp64(dyf, g, u);
}

// dg = RN_bf16(dy * u * sigma * (1 + g (1 - sigma))), one rounding.
// Tier 1 relative error of p <= (10 + 12 * ratio) * 2^-24.
MX_DEVINL uint32_t dg_bits_from(float dyf, float g, float u, const SigFast& f) {
  const float dyu = __fmul_rn(dyf, u);  // exact in the normal range
  const float oms = __fmul_rn(f.t, f.s);
  const float go = __fmul_rn(g, oms);
  const float inner = __fadd_rn(1.0f, go);
  const float p = __fmul_rn(dyu, __fmul_rn(f.s, inner));
  const float ratio = fabsf(go) * rcp_approx(fabsf(inner));
  const float margin = __fmaf_rn(26.0f, ratio, 24.0f);
  const float ap = fabsf(p), adyu = fabsf(dyu);
  if (f.ok && margin < 16384.0f && adyu >= 0x1p-100f && adyu <= 0x1p100f && ap >= 0x1p-100f &&
      clear_of_midpoint(p, (uint32_t)margin))
    return f32_to_bf16_bits(p);
  return dg_bits_slow(dyf, g, u);
}


// ---- packed fast path (both lanes of an f32x2 pair)

MX_DEVINL float ex2_approx(float y) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
  return r;
}

// e^-g on both lanes, |g| <= 64.  2^Y with Y = RN(-g L), L = RN_f32(log2 e),
// from the hardware ex2 approximation (at most 2.06 ulp on [-92.5, 92.5]),
// corrected by the factor 1 - c ln2 where c = g log2 e + Y is recovered in
// two pieces: g L + Y exactly by one FMA (Y is the rounded -g L), and
// g (log2 e - L) from the low part of log2 e (Cody-Waite splitting).  The
// first-order correction leaves a relative error below 2^-36, so the result
// is within ex2's error plus one rounding (at most 2.6 ulp, checked on
// every bf16 g).
MX_DEVINL f2 f2_exp_neg(f2 G) {
  const f2 L = f2_splat(__uint_as_float(0x3FB8AA3Bu));     // RN_f32(log2 e)
  const f2 NL = f2_splat(__uint_as_float(0xBFB8AA3Bu));
  const f2 LC = f2_splat(__uint_as_float(0x32A57060u));    // RN_f32(log2 e - L)
  const f2 NLN2 = f2_splat(__uint_as_float(0xBF317218u));  // -RN_f32(ln 2)
  const f2 Y = f2_mul(G, NL);
  const f2 R = f2_fma(G, L, Y);
  const f2 C = f2_fma(G, LC, R);
  const f2 K = f2_mul(C, NLN2);
  float y0, y1;
  f2_unpack(Y, y0, y1);
  const f2 E = f2_pack(ex2_approx(y0), ex2_approx(y1));
  return f2_fma(E, K, E);
}

// t = e^-g and s = rcp.approx(1 + t) (at most 0.98 ulp) on both lanes.
struct SigFast2 {
  f2 T, S;
};
MX_DEVINL SigFast2 sig_fast2(f2 G) {
  SigFast2 r;
  r.T = f2_exp_neg(G);
  float d0, d1;
  f2_unpack(f2_add(r.T, f2_splat(1.0f)), d0, d1);
  r.S = f2_pack(rcp_approx(d0), rcp_approx(d1));
  return r;
}

// ---- packed certificates (both lanes of a pair at once)
//
// Each returns the candidate bf16 pair and a mismatch word that is zero in
// the 16-bit half of every lane whose rounding is certain: the exact value
// lies in an interval around the fp32 fast value that covers the fast
// chain's error, and both ends of the interval round to the same bf16
// (rounding is monotone, so everything between them does too).  A failing
// lane leaves a nonzero half, so the per-lane decisions need no recomputation.

// RN_f32 of the products of the bf16 halves of a and b (lane 0 from the low
// halves): exact in fp32's range (8 x 8 significant bits), computed by the
// mixed-precision FMA with -0 as the addend so that a zero product keeps its
// sign.
MX_DEVINL f2 f2_mul_bf16x2(uint32_t a, uint32_t b) {
  float lo, hi;
  asm("{\n .reg .b16 al, ah, bl, bh;\n"
      " mov.b32 {al, ah}, %2;\n mov.b32 {bl, bh}, %3;\n"
      " fma.rn.f32.bf16 %0, al, bl, 0f80000000;\n fma.rn.f32.bf16 %1, ah, bh, 0f80000000;\n}"
      : "=f"(lo), "=f"(hi)
      : "r"(a), "r"(b));
  return make_float2(lo, hi);
}

MX_DEVINL f2 f2_abs(f2 v) { return make_float2(fabsf(v.x), fabsf(v.y)); }
MX_DEVINL f2 f2_neg(f2 v) { return make_float2(-v.x, -v.y); }

// a = RN_bf16(g s): p = g s is within 9 fp32 ulps of g * sigma_c (sigma_c the
// correctly rounded sigma); the interval [p(1 - 2^-19), p(1 + 2^-19)] is at
// least 15.5 ulps wide on each side.
MX_DEVINL uint32_t silu2_cert(f2 G, f2 S, uint32_t& miss) {
  const f2 P = f2_mul(G, S);
  const uint32_t lo = f2_to_bf16x2(f2_mul(P, f2_splat(__uint_as_float(0x3F7FFFE0u))));  // 1 - 2^-19
  const uint32_t hi = f2_to_bf16x2(f2_mul(P, f2_splat(__uint_as_float(0x3F800010u))));  // 1 + 2^-19
  miss = lo ^ hi;
  return lo;
}

// Margin constants of dg, in units of 2^-24: the fast value PG = dyu (s (1 +
// g t s)) is within |dyu| s (DG_C0 |1 + go| + DG_C1 |go|) 2^-24 of the exact
// dyu F(g) (go = g t s; the cancellation in 1 + go amplifies go's error),
// including the rounding of PG and of the interval ends, while PG is a
// normal fp32 value.
constexpr float DG_C0 = 24.0f * 0x1p-24f;
constexpr float DG_C1 = 26.0f * 0x1p-24f;

// the half-width factor W = s (C0 |in| + C1 |go|) of the dg interval
MX_DEVINL f2 dg2_width(f2 S, f2 GO, f2 IN) {
  return f2_mul(S, f2_fma(f2_abs(GO), f2_splat(DG_C1), f2_mul(f2_abs(IN), f2_splat(DG_C0))));
}

// dg = RN_bf16(dyu F), returned as RN_bf16(PG): the interval
// PG -+ (|dyu| W + 2^-149) also covers the absolute rounding error (at most
// 2^-150) of a PG or an interval end in fp32's subnormal range.  The ends
// are compared without their signs: when both round to a zero, the exact
// value rounds to the zero of its own sign, which is PG's (the sign of the
// fast factor is exact, see the probe), so PG's own rounding is the result.
MX_DEVINL uint32_t dg2_cert(f2 DYU, f2 PG, f2 W, uint32_t& miss) {
  const f2 AD = f2_abs(DYU);
  const uint32_t lo = f2_to_bf16x2(f2_fma(AD, f2_neg(W), f2_add(PG, f2_splat(-0x1p-149f))));
  const uint32_t hi = f2_to_bf16x2(f2_fma(AD, W, f2_add(PG, f2_splat(0x1p-149f))));
  miss = (lo ^ hi) & 0x7FFF7FFFu;
  return f2_to_bf16x2(PG);
}

// bit 15 / bit 31 set for a lane whose bf16 g has |g| > 64 or is not finite
// (magnitude bits above 0x4280 carry into the top bit of their half)
MX_DEVINL uint32_t g_out_of_range2(uint32_t gp) { return ((gp & 0x7FFF7FFFu) + 0x3D7F3D7Fu) & 0x80008000u; }

// the lanes (bit 0: low, bit 1: high) a mismatch word marks
MX_DEVINL uint32_t miss_lanes(uint32_t miss) { return ((miss & 0xFFFFu) ? 1u : 0u) | ((miss >> 16) ? 2u : 0u); }

}  // namespace
}  // namespace swiglu_math
}  // namespace mx
