// swiglu.cu - fused SwiGLU forward / backward with dual MXFP8 quantization.
//
// Forward: h13 = [g | u] tiles stream through a TMA ring; each consumer
// thread computes y = RN_bf16(a * u) for 8 consecutive elements, quantizes
// them rowwise straight from registers and parks the bf16 y tile in shared
// memory, where the columnwise quantization reads it.  y never reaches
// global memory.
//
// Backward: dy and h13 tiles in, dh13 = [dg | du] out, quantized rowwise and
// columnwise the same way (or, for the bf16 weight-gradient recipe, written
// transposed in bf16 together with the recomputed y).
//
// Numerics (page "Add MXFP8 fused-MLP overrides in torchtitan", Numerics and
// tests: bitwise forward parity with standalone-cast quantization and a
// correctly-rounded sigmoid):
//   sigma  = fp32 correctly rounded 1/(1+e^-g)
//   a      = RN_bf16(RN_f32(g * sigma))          (bf16 SiLU)
//   y      = RN_bf16(RN_f32(a * u))
//   du     = RN_bf16(RN_f32(dy * a))
//   dg     = RN_bf16(dy * u * sigma * (1 + g(1 - sigma)))  (one rounding)
// Fast path: fp32 with expf (at most 2 ulp) and correctly rounded reciprocal
// and products; the result is accepted only if it lies farther from a bf16
// rounding midpoint than the accumulated error bound.  Otherwise (about 0.2%
// of elements, plus |g| > 64 and non-normal ranges) the value is recomputed in
// fp64 and rounded once.
#include "tile_quant.cuh"
#include "kernels.h"

namespace mx {

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

MX_DEVINL uint32_t silu_bits(float g) { return silu_bits_from(g, sig_fast(g)); }

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

// ------------------------------------------------------------------ kernels
//
// Both kernels stream tiles through a 2-stage TMA ring and run three roles:
//   producer warp  TMA loads of the input tiles
//   8 consumer     phase A: every element through the fp32 fast path into a
//   warps          shared-memory result tile; elements whose rounding the
//                  fast path cannot certify are queued.  Phase C: MX
//                  quantization of the previous (complete) tile, rows on
//                  warps 4-7 and columns on warps 0-3
//   fixer warp     phase B: recomputes the queued elements of a tile with
//                  the exact tiers (32 at a time) and patches the result
//                  tile, then releases the input stage
// Per tile, one barrier of consumers + fixer (A done) and one of consumers
// only (C done).  The long dependency chains of the exact tiers run on the
// fixer while the consumers quantize the previous tile and start the next,
// so they stay off the critical path.  Result tiles and queues are double-
// buffered; a queue that overflows (adversarial inputs) is resolved in
// place by the consumer that found the element.

constexpr int CW = 8;                    // consumer warps
constexpr int CT = CW * 32;              // consumer threads
constexpr int PRODUCER = CW;             // warp index
constexpr int FIXER = CW + 1;            // warp index
constexpr int THREADS = (CW + 2) * 32;
constexpr int QCAP = 1024;               // queued elements per tile buffer

MX_DEVINL void bar_ab() { named_bar_sync(1, CT + 32); }  // consumers + fixer
MX_DEVINL void bar_c() { named_bar_sync(2, CT); }        // consumers

// ---- forward: tile = 128 rows x 64 y-columns
constexpr int SF_R = 128, SF_C = 64;
constexpr int SF_STAGES = 2;
constexpr int SF_BOX = SF_R * SF_C * 2;       // 16 KB
constexpr int SF_STAGE_BYTES = 2 * SF_BOX;    // g, u
constexpr size_t SF_SMEM = SF_STAGES * SF_STAGE_BYTES + 2 * SF_BOX + 2 * QCAP * 2 + 1024 + 128;

struct SwiFwdParams {
  int64_t M, h;
  int64_t row_tiles, col_tiles;
  uint8_t* q_row; ScaleDst s_row;
  uint8_t* q_col; ScaleDst s_col;
  int32_t* err;
};

template <bool COL>
__global__ void __launch_bounds__(THREADS, 2)
    swiglu_fwd_kernel(const __grid_constant__ CUtensorMap tmh, SwiFwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ytile = smem + SF_STAGES * SF_STAGE_BYTES;            // 2 x 16 KB
  uint16_t* queue = reinterpret_cast<uint16_t*>(ytile + 2 * SF_BOX);   // 2 x QCAP
  uint64_t* full = reinterpret_cast<uint64_t*>(queue + 2 * QCAP);
  uint64_t* empty = full + SF_STAGES;
  __shared__ int s_qn[2];
  __shared__ long long s_abort;  // first tile index whose wait timed out
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int64_t n_tiles = p.row_tiles * p.col_tiles;

  if (tid == 0) {
    for (int s = 0; s < SF_STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    fence_mbar_init();
    s_qn[0] = s_qn[1] = 0;
    s_abort = 0x7FFFFFFFFFFFFFFFll;
  }
  __syncthreads();

  if (warp == PRODUCER) {
    if (lane == 0) {
      prefetch_tmap(&tmh);
      int stage = 0; uint32_t phase = 0;
      for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const int64_t rt = t / p.col_tiles, ct = t - rt * p.col_tiles;
        if (!mbar_wait(&empty[stage], phase ^ 1, p.err)) break;
        mbar_arrive_expect_tx(&full[stage], SF_STAGE_BYTES);
        uint8_t* dst = smem + stage * SF_STAGE_BYTES;
        tma_load_2d(dst, &tmh, (int32_t)(ct * SF_C), (int32_t)(rt * SF_R), &full[stage]);
        tma_load_2d(dst + SF_BOX, &tmh, (int32_t)(p.h + ct * SF_C), (int32_t)(rt * SF_R), &full[stage]);
        if (++stage == SF_STAGES) { stage = 0; phase ^= 1; }
      }
    }
    return;
  }

  if (warp == FIXER) {
    // ---- phase B for tile t, between its A barrier and the next one
    int stage = 0, buf = 0;
    for (int64_t t = blockIdx.x;; t += gridDim.x, buf ^= 1) {
      const bool have = t < n_tiles;
      bar_ab();
      if (!have || s_abort <= t) break;
      const uint8_t* gt = smem + stage * SF_STAGE_BYTES;
      const uint8_t* ut = gt + SF_BOX;
      uint8_t* yt = ytile + buf * SF_BOX;
      const uint16_t* q = queue + buf * QCAP;
      const int n = min(s_qn[buf], QCAP);
      for (int i = lane; i < n; i += 32) {
        const int idx = q[i];
        const int off = (idx / SF_C) * 128 + (idx % SF_C) * 2;
        const float g = bf16_lo(*reinterpret_cast<const uint16_t*>(gt + off));
        const float u = bf16_lo(*reinterpret_cast<const uint16_t*>(ut + off));
        const float a = bf16_lo(silu_bits_slow(g));
        *reinterpret_cast<uint16_t*>(yt + off) = (uint16_t)f32_to_bf16_bits(__fmul_rn(a, u));
      }
      __syncwarp();
      if (lane == 0) {
        s_qn[buf] = 0;
        mbar_arrive(&empty[stage]);   // inputs of tile t no longer needed
      }
      if (++stage == SF_STAGES) stage = 0;
    }
    return;
  }

  // ---- consumers
  int stage = 0; uint32_t phase = 0; int buf = 0;
  const int seg = lane & 7;
  int64_t t_prev = -1;
  for (int64_t t = blockIdx.x;; t += gridDim.x, buf ^= 1) {
    const bool have = t < n_tiles;
    if (have) {
      const bool ok = mbar_wait(&full[stage], phase, p.err);
      if (!ok) atomicMin(&s_abort, (long long)t);
      const uint8_t* gt = smem + stage * SF_STAGE_BYTES;
      const uint8_t* ut = gt + SF_BOX;
      uint8_t* yt = ytile + buf * SF_BOX;
      uint16_t* q = queue + buf * QCAP;
      // ---- phase A
      if (ok) {
#pragma unroll 1
        for (int it = 0; it < SF_R / (4 * CW); ++it) {
          const int rr = it * (4 * CW) + warp * 4 + (lane >> 3);
          const uint4 gv = *reinterpret_cast<const uint4*>(gt + rr * 128 + seg * 16);
          const uint4 uv = *reinterpret_cast<const uint4*>(ut + rr * 128 + seg * 16);
          const uint32_t gp[4] = {gv.x, gv.y, gv.z, gv.w};
          const uint32_t up[4] = {uv.x, uv.y, uv.z, uv.w};
          uint32_t yp[4];
          uint32_t slow = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float g0 = bf16_lo(gp[i]), g1 = bf16_hi(gp[i]);
            const SigFast f0 = sig_fast(g0), f1 = sig_fast(g1);
            const float p0 = __fmul_rn(g0, f0.s), p1 = __fmul_rn(g1, f1.s);
            slow |= (f0.ok && clear_of_midpoint(p0, 16) ? 0u : 1u) << (2 * i);
            slow |= (f1.ok && clear_of_midpoint(p1, 16) ? 0u : 1u) << (2 * i + 1);
            const __nv_bfloat162 a2 = __floats2bfloat162_rn(p0, p1);
            const float2 af = __bfloat1622float2(a2);
            const __nv_bfloat162 y2 = __floats2bfloat162_rn(__fmul_rn(af.x, bf16_lo(up[i])),
                                                            __fmul_rn(af.y, bf16_hi(up[i])));
            yp[i] = *reinterpret_cast<const uint32_t*>(&y2);
          }
          while (slow) {
            const int j = __ffs(slow) - 1;
            slow &= slow - 1;
            const int slot = atomicAdd(&s_qn[buf], 1);
            if (slot < QCAP) {
              q[slot] = (uint16_t)(rr * SF_C + seg * 8 + j);
            } else {  // queue full: resolve here
              const uint32_t gw = gp[j >> 1], uw = up[j >> 1];
              const float g = (j & 1) ? bf16_hi(gw) : bf16_lo(gw);
              const float u = (j & 1) ? bf16_hi(uw) : bf16_lo(uw);
              const uint32_t y = f32_to_bf16_bits(__fmul_rn(bf16_lo(silu_bits_slow(g)), u));
              uint32_t& w = yp[j >> 1];
              w = (j & 1) ? ((w & 0xFFFFu) | (y << 16)) : ((w & 0xFFFF0000u) | y);
            }
          }
          *reinterpret_cast<uint4*>(yt + rr * 128 + seg * 16) = make_uint4(yp[0], yp[1], yp[2], yp[3]);
        }
      }
      if (++stage == SF_STAGES) { stage = 0; phase ^= 1; }
    }
    bar_ab();
    if (s_abort <= (have ? t : t_prev)) break;
    // ---- phase C of the previous tile (complete: the fixer patched it
    // before this barrier)
    if (t_prev >= 0) {
      const int pb = buf ^ 1;
      const uint8_t* yt = ytile + pb * SF_BOX;
      const int64_t rt = t_prev / p.col_tiles, ct = t_prev - rt * p.col_tiles;
      const int64_t r0 = rt * SF_R, c0 = ct * SF_C;
      if (warp >= 4 || !COL) {
        const int w = COL ? warp - 4 : warp;
        const int nw = COL ? 4 : CW;
        for (int rr = w * 4 + (lane >> 3); rr < SF_R; rr += nw * 4) {
          const uint4 v = *reinterpret_cast<const uint4*>(yt + rr * 128 + seg * 16);
          const uint32_t pk[4] = {v.x, v.y, v.z, v.w};
          uint32_t sc;
          const uint2 codes = quant_row8(pk, sc);
          const int64_t r = r0 + rr;
          const int64_t c = c0 + seg * 8;
          if (r < p.M) {
            *reinterpret_cast<uint2*>(p.q_row + r * p.h + c) = codes;
            if ((seg & 3) == 0) p.s_row.put(r, c >> 5, sc);
          }
        }
      } else {
        const int item = warp * 32 + lane;
        const int pc = item & 31, rb = item >> 5;
        uint32_t v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = *reinterpret_cast<const uint32_t*>(yt + (rb * 32 + i) * 128 + pc * 4);
        uint32_t ca[8], cb[8], sa, sb;
        quant_col32x2(v, ca, cb, sa, sb);
        const int64_t rg = r0 + rb * 32;
        if (rg < p.M) {
          const int64_t col = c0 + 2 * pc;
          uint8_t* dst = p.q_col + col * p.M + rg;
          store16(dst, ca[0], ca[1], ca[2], ca[3]);
          store16(dst + 16, ca[4], ca[5], ca[6], ca[7]);
          store16(dst + p.M, cb[0], cb[1], cb[2], cb[3]);
          store16(dst + p.M + 16, cb[4], cb[5], cb[6], cb[7]);
          p.s_col.put(col, rg >> 5, sa);
          p.s_col.put(col + 1, rg >> 5, sb);
        }
      }
    }
    if (!have) break;
    bar_c();   // the previous tile's buffers are free for the next phase A
    t_prev = t;
  }
}

// ---- backward: tile = 64 rows x 64 y-columns
constexpr int SB_R = 64, SB_C = 64;
constexpr int SB_STAGES = 2;
constexpr int SB_BOX = SB_R * SB_C * 2;       // 8 KB
constexpr int SB_STAGE_BYTES = 3 * SB_BOX;    // dy, g, u
constexpr size_t SB_SMEM = SB_STAGES * SB_STAGE_BYTES + 2 * 3 * SB_BOX + 2 * QCAP * 2 + 1024 + 128;

struct SwiBwdParams {
  int64_t M, h;
  int64_t row_tiles, col_tiles;
  uint8_t* q_row; ScaleDst s_row;   // [M, 2h]
  uint8_t* q_col; ScaleDst s_col;   // [2h, M]
  uint16_t* dh13_t;                 // [2h, M]
  uint16_t* y_t;                    // [h, M]
  int32_t* err;
};

// exact dg, du (and y) of one element, written into the result tile
template <int MODE>
MX_DEVINL void bwd_exact(float dyf, float g, float u, uint8_t* ot, int off) {
  const SigFast sf = sig_fast(g);
  const float a = bf16_lo(silu_bits_from(g, sf));
  *reinterpret_cast<uint16_t*>(ot + off) = (uint16_t)dg_bits_from(dyf, g, u, sf);
  *reinterpret_cast<uint16_t*>(ot + SB_BOX + off) = (uint16_t)f32_to_bf16_bits(__fmul_rn(dyf, a));
  if (MODE == 2) *reinterpret_cast<uint16_t*>(ot + 2 * SB_BOX + off) = (uint16_t)f32_to_bf16_bits(__fmul_rn(a, u));
}

// MODE 0: rowwise only; 1: rowwise + columnwise MX; 2: rowwise + bf16 transposed
// dh13 and y.
template <int MODE>
__global__ void __launch_bounds__(THREADS, 2)
    swiglu_bwd_kernel(const __grid_constant__ CUtensorMap tmdy, const __grid_constant__ CUtensorMap tmh,
                      SwiBwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* otile = smem + SB_STAGES * SB_STAGE_BYTES;  // 2 buffers x {dg, du, y}
  uint16_t* queue = reinterpret_cast<uint16_t*>(otile + 2 * 3 * SB_BOX);
  uint64_t* full = reinterpret_cast<uint64_t*>(queue + 2 * QCAP);
  uint64_t* empty = full + SB_STAGES;
  __shared__ int s_qn[2];
  __shared__ long long s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int64_t n_tiles = p.row_tiles * p.col_tiles;

  if (tid == 0) {
    for (int s = 0; s < SB_STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    fence_mbar_init();
    s_qn[0] = s_qn[1] = 0;
    s_abort = 0x7FFFFFFFFFFFFFFFll;
  }
  __syncthreads();

  if (warp == PRODUCER) {
    if (lane == 0) {
      prefetch_tmap(&tmdy);
      prefetch_tmap(&tmh);
      int stage = 0; uint32_t phase = 0;
      for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const int64_t rt = t / p.col_tiles, ct = t - rt * p.col_tiles;
        if (!mbar_wait(&empty[stage], phase ^ 1, p.err)) break;
        mbar_arrive_expect_tx(&full[stage], SB_STAGE_BYTES);
        uint8_t* dst = smem + stage * SB_STAGE_BYTES;
        const int32_t x = (int32_t)(ct * SB_C), y = (int32_t)(rt * SB_R);
        tma_load_2d(dst, &tmdy, x, y, &full[stage]);
        tma_load_2d(dst + SB_BOX, &tmh, x, y, &full[stage]);
        tma_load_2d(dst + 2 * SB_BOX, &tmh, (int32_t)(p.h + x), y, &full[stage]);
        if (++stage == SB_STAGES) { stage = 0; phase ^= 1; }
      }
    }
    return;
  }

  if (warp == FIXER) {
    int stage = 0, buf = 0;
    for (int64_t t = blockIdx.x;; t += gridDim.x, buf ^= 1) {
      const bool have = t < n_tiles;
      bar_ab();
      if (!have || s_abort <= t) break;
      const uint8_t* dyt = smem + stage * SB_STAGE_BYTES;
      uint8_t* ot = otile + buf * 3 * SB_BOX;
      const uint16_t* q = queue + buf * QCAP;
      const int n = min(s_qn[buf], QCAP);
      for (int i = lane; i < n; i += 32) {
        const int idx = q[i];
        const int off = (idx / SB_C) * 128 + (idx % SB_C) * 2;
        const float dyf = bf16_lo(*reinterpret_cast<const uint16_t*>(dyt + off));
        const float g = bf16_lo(*reinterpret_cast<const uint16_t*>(dyt + SB_BOX + off));
        const float u = bf16_lo(*reinterpret_cast<const uint16_t*>(dyt + 2 * SB_BOX + off));
        bwd_exact<MODE>(dyf, g, u, ot, off);
      }
      __syncwarp();
      if (lane == 0) {
        s_qn[buf] = 0;
        mbar_arrive(&empty[stage]);
      }
      if (++stage == SB_STAGES) stage = 0;
    }
    return;
  }

  int stage = 0; uint32_t phase = 0; int buf = 0;
  const int seg = lane & 7;
  int64_t t_prev = -1;
  for (int64_t t = blockIdx.x;; t += gridDim.x, buf ^= 1) {
    const bool have = t < n_tiles;
    if (have) {
      const bool ok = mbar_wait(&full[stage], phase, p.err);
      if (!ok) atomicMin(&s_abort, (long long)t);
      const uint8_t* dyt = smem + stage * SB_STAGE_BYTES;
      const uint8_t* gt = dyt + SB_BOX;
      const uint8_t* ut = dyt + 2 * SB_BOX;
      uint8_t* ot = otile + buf * 3 * SB_BOX;   // dg | du | y
      uint16_t* q = queue + buf * QCAP;
      // ---- phase A
      if (ok) {
#pragma unroll 1
        for (int it = 0; it < SB_R / (4 * CW); ++it) {
          const int rr = it * (4 * CW) + warp * 4 + (lane >> 3);
          const uint4 dv = *reinterpret_cast<const uint4*>(dyt + rr * 128 + seg * 16);
          const uint4 gv = *reinterpret_cast<const uint4*>(gt + rr * 128 + seg * 16);
          const uint4 uv = *reinterpret_cast<const uint4*>(ut + rr * 128 + seg * 16);
          const uint32_t dp[4] = {dv.x, dv.y, dv.z, dv.w};
          const uint32_t gp[4] = {gv.x, gv.y, gv.z, gv.w};
          const uint32_t up[4] = {uv.x, uv.y, uv.z, uv.w};
          uint32_t dgp[4], dup[4], yp[4];
          uint32_t slow = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t dgw = 0;
            float pa[2], dyv[2], uvv[2];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const float dyf = hh ? bf16_hi(dp[i]) : bf16_lo(dp[i]);
              const float g = hh ? bf16_hi(gp[i]) : bf16_lo(gp[i]);
              const float u = hh ? bf16_hi(up[i]) : bf16_lo(up[i]);
              const SigFast sf = sig_fast(g);
              pa[hh] = __fmul_rn(g, sf.s);
              dyv[hh] = dyf;
              uvv[hh] = u;
              bool ok_e = sf.ok && clear_of_midpoint(pa[hh], 16);
              // dg tier 1 (see dg_bits_from)
              const float dyu = __fmul_rn(dyf, u);
              const float oms = __fmul_rn(sf.t, sf.s);
              const float go = __fmul_rn(g, oms);
              const float inner = __fadd_rn(1.0f, go);
              const float pg = __fmul_rn(dyu, __fmul_rn(sf.s, inner));
              const float ratio = fabsf(go) * rcp_approx(fabsf(inner));
              const float margin = __fmaf_rn(26.0f, ratio, 24.0f);
              const float adyu = fabsf(dyu), apg = fabsf(pg);
              ok_e = ok_e && margin < 16384.0f && adyu >= 0x1p-100f && adyu <= 0x1p100f && apg >= 0x1p-100f &&
                     clear_of_midpoint(pg, (uint32_t)margin);
              slow |= (ok_e ? 0u : 1u) << (2 * i + hh);
              dgw |= f32_to_bf16_bits(pg) << (16 * hh);
            }
            const __nv_bfloat162 a2 = __floats2bfloat162_rn(pa[0], pa[1]);
            const float2 af = __bfloat1622float2(a2);
            const __nv_bfloat162 du2 = __floats2bfloat162_rn(__fmul_rn(dyv[0], af.x), __fmul_rn(dyv[1], af.y));
            dup[i] = *reinterpret_cast<const uint32_t*>(&du2);
            dgp[i] = dgw;
            if (MODE == 2) {
              const __nv_bfloat162 y2 = __floats2bfloat162_rn(__fmul_rn(af.x, uvv[0]), __fmul_rn(af.y, uvv[1]));
              yp[i] = *reinterpret_cast<const uint32_t*>(&y2);
            }
          }
          *reinterpret_cast<uint4*>(ot + rr * 128 + seg * 16) = make_uint4(dgp[0], dgp[1], dgp[2], dgp[3]);
          *reinterpret_cast<uint4*>(ot + SB_BOX + rr * 128 + seg * 16) = make_uint4(dup[0], dup[1], dup[2], dup[3]);
          if (MODE == 2)
            *reinterpret_cast<uint4*>(ot + 2 * SB_BOX + rr * 128 + seg * 16) = make_uint4(yp[0], yp[1], yp[2], yp[3]);
          while (slow) {
            const int j = __ffs(slow) - 1;
            slow &= slow - 1;
            const int slot = atomicAdd(&s_qn[buf], 1);
            const int idx = rr * SB_C + seg * 8 + j;
            if (slot < QCAP) {
              q[slot] = (uint16_t)idx;
            } else {  // queue full: resolve here (after this thread's own stores above)
              const int off = rr * 128 + (seg * 8 + j) * 2;
              bwd_exact<MODE>(bf16_lo(*reinterpret_cast<const uint16_t*>(dyt + off)),
                              bf16_lo(*reinterpret_cast<const uint16_t*>(gt + off)),
                              bf16_lo(*reinterpret_cast<const uint16_t*>(ut + off)), ot, off);
            }
          }
        }
      }
      if (++stage == SB_STAGES) { stage = 0; phase ^= 1; }
    }
    bar_ab();
    if (s_abort <= (have ? t : t_prev)) break;
    // ---- phase C of the previous tile
    if (t_prev >= 0) {
      const int pb = buf ^ 1;
      const uint8_t* ot = otile + pb * 3 * SB_BOX;
      const int64_t rt = t_prev / p.col_tiles, ct = t_prev - rt * p.col_tiles;
      const int64_t r0 = rt * SB_R, c0 = ct * SB_C;
      if (warp >= 4 || MODE == 0) {
        // rows of dg and du: 8 lanes per 64-column row; 4 rows per warp step
        const int w = MODE == 0 ? warp : warp - 4;
        const int nw = MODE == 0 ? CW : 4;
        for (int k = w * 4 + (lane >> 3); k < 2 * SB_R; k += nw * 4) {
          const int which = k / SB_R, rr = k % SB_R;
          const uint4 v = *reinterpret_cast<const uint4*>(ot + which * SB_BOX + rr * 128 + seg * 16);
          const uint32_t pk[4] = {v.x, v.y, v.z, v.w};
          uint32_t sc;
          const uint2 codes = quant_row8(pk, sc);
          const int64_t r = r0 + rr;
          const int64_t c = (which ? p.h : 0) + c0 + seg * 8;
          if (r < p.M) {
            *reinterpret_cast<uint2*>(p.q_row + r * 2 * p.h + c) = codes;
            if ((seg & 3) == 0) p.s_row.put(r, c >> 5, sc);
          }
        }
      } else if (MODE == 1) {
        // columns of dg, du: 64 column pairs x 2 row blocks = 128 items on warps 0-3
        const int item = warp * 32 + lane;
        const int pcx = item & 63, rb = item >> 6;
        const int which = pcx >> 5, pc = pcx & 31;
        const uint8_t* src = ot + which * SB_BOX;
        uint32_t v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = *reinterpret_cast<const uint32_t*>(src + (rb * 32 + i) * 128 + pc * 4);
        uint32_t ca[8], cb[8], sa, sb;
        quant_col32x2(v, ca, cb, sa, sb);
        const int64_t rg = r0 + rb * 32;
        if (rg < p.M) {
          const int64_t orow = (which ? p.h : 0) + c0 + 2 * pc;
          uint8_t* dst = p.q_col + orow * p.M + rg;
          store16(dst, ca[0], ca[1], ca[2], ca[3]);
          store16(dst + 16, ca[4], ca[5], ca[6], ca[7]);
          store16(dst + p.M, cb[0], cb[1], cb[2], cb[3]);
          store16(dst + p.M + 16, cb[4], cb[5], cb[6], cb[7]);
          p.s_col.put(orow, rg >> 5, sa);
          p.s_col.put(orow + 1, rg >> 5, sb);
        }
      } else {
        // bf16 transposed dg, du (into dh13_t) and y (into y_t): 96 column
        // pairs x 2 blocks of 32 rows = 192 items on warps 0-3
        for (int item = warp * 32 + lane; item < 192; item += 128) {
          const int pcx = item % 96, rb = item / 96;
          const int which = pcx / 32, pc = pcx % 32;
          const uint8_t* src = ot + which * SB_BOX;
          uint32_t wa[16], wb[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint32_t r0v = *reinterpret_cast<const uint32_t*>(src + (rb * 32 + 2 * i) * 128 + pc * 4);
            const uint32_t r1v = *reinterpret_cast<const uint32_t*>(src + (rb * 32 + 2 * i + 1) * 128 + pc * 4);
            wa[i] = (r0v & 0xFFFFu) | (r1v << 16);
            wb[i] = (r0v >> 16) | (r1v & 0xFFFF0000u);
          }
          const int64_t rg = r0 + rb * 32;
          if (rg < p.M) {
            const int64_t col = c0 + 2 * pc;
            uint16_t* base = which == 2 ? p.y_t : p.dh13_t;
            if (base) {
              const int64_t orow = (which == 1 ? p.h : 0) + col;
              uint16_t* da = base + orow * p.M + rg;
              uint16_t* db = da + p.M;
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                store16(da + q4 * 8, wa[4 * q4], wa[4 * q4 + 1], wa[4 * q4 + 2], wa[4 * q4 + 3]);
                store16(db + q4 * 8, wb[4 * q4], wb[4 * q4 + 1], wb[4 * q4 + 2], wb[4 * q4 + 3]);
              }
            }
          }
        }
      }
    }
    if (!have) break;
    bar_c();
    t_prev = t;
  }
}

}  // namespace

int launch_swiglu_fwd(const SwigluLaunch& s, cudaStream_t stream) {
  CUtensorMap tm;
  uint64_t dims[2] = {(uint64_t)(2 * s.h), (uint64_t)s.M};
  uint64_t strides[1] = {(uint64_t)(2 * s.h * 2)};
  uint32_t box[2] = {SF_C, SF_R};
  int rc = make_tmap(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(s.h13), dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
  if (rc) return rc;
  SwiFwdParams p{};
  p.M = s.M; p.h = s.h;
  p.row_tiles = (s.M + SF_R - 1) / SF_R;
  p.col_tiles = s.h / SF_C;
  const bool mma = s.layout == MX_SCALE_MMA;
  const int64_t Sr = s.h / 32, Sc = s.M / 32;
  p.q_row = (uint8_t*)s.q_row; p.s_row = ScaleDst{(uint8_t*)s.s_row, (Sr + 3) / 4, Sr, mma};
  p.q_col = (uint8_t*)s.q_col; p.s_col = ScaleDst{(uint8_t*)s.s_col, (Sc + 3) / 4, Sc, mma};
  p.err = s.err;
  const int64_t n_tiles = p.row_tiles * p.col_tiles;
  if (n_tiles == 0) return MX_OK;
  const int grid = (int)std::min<int64_t>(n_tiles, (int64_t)num_sms() * 2);
  cudaError_t e;
  if (s.q_col) {
    auto k = swiglu_fwd_kernel<true>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SF_SMEM);
    if (e == cudaSuccess) { k<<<grid, THREADS, SF_SMEM, stream>>>(tm, p); e = cudaGetLastError(); }
  } else {
    auto k = swiglu_fwd_kernel<false>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SF_SMEM);
    if (e == cudaSuccess) { k<<<grid, THREADS, SF_SMEM, stream>>>(tm, p); e = cudaGetLastError(); }
  }
  return cuda_status(e, "swiglu_fwd_kernel launch");
}

int launch_swiglu_bwd(const SwigluLaunch& s, cudaStream_t stream) {
  CUtensorMap tdy, th;
  {
    uint64_t dims[2] = {(uint64_t)s.h, (uint64_t)s.M};
    uint64_t strides[1] = {(uint64_t)(s.h * 2)};
    uint32_t box[2] = {SB_C, SB_R};
    int rc = make_tmap(&tdy, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(s.dy), dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
  }
  {
    uint64_t dims[2] = {(uint64_t)(2 * s.h), (uint64_t)s.M};
    uint64_t strides[1] = {(uint64_t)(2 * s.h * 2)};
    uint32_t box[2] = {SB_C, SB_R};
    int rc = make_tmap(&th, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(s.h13), dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
  }
  SwiBwdParams p{};
  p.M = s.M; p.h = s.h;
  p.row_tiles = (s.M + SB_R - 1) / SB_R;
  p.col_tiles = s.h / SB_C;
  const bool mma = s.layout == MX_SCALE_MMA;
  const int64_t Sr = 2 * s.h / 32, Sc = s.M / 32;
  p.q_row = (uint8_t*)s.q_row; p.s_row = ScaleDst{(uint8_t*)s.s_row, (Sr + 3) / 4, Sr, mma};
  p.q_col = (uint8_t*)s.q_col; p.s_col = ScaleDst{(uint8_t*)s.s_col, (Sc + 3) / 4, Sc, mma};
  p.dh13_t = (uint16_t*)s.dh13_t; p.y_t = (uint16_t*)s.y_t;
  p.err = s.err;
  const int64_t n_tiles = p.row_tiles * p.col_tiles;
  if (n_tiles == 0) return MX_OK;
  const int grid = (int)std::min<int64_t>(n_tiles, (int64_t)num_sms() * 2);
  const int mode = s.q_col ? 1 : ((s.dh13_t || s.y_t) ? 2 : 0);
  cudaError_t e;
#define MX_LAUNCH_B(MODE)                                                                       \
  do {                                                                                          \
    auto k = swiglu_bwd_kernel<MODE>;                                                           \
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SB_SMEM);     \
    if (e == cudaSuccess) { k<<<grid, THREADS, SB_SMEM, stream>>>(tdy, th, p); e = cudaGetLastError(); } \
  } while (0)
  if (mode == 0) MX_LAUNCH_B(0);
  else if (mode == 1) MX_LAUNCH_B(1);
  else MX_LAUNCH_B(2);
#undef MX_LAUNCH_B
  return cuda_status(e, "swiglu_bwd_kernel launch");
}

}  // namespace mx
