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

MX_DEVINL double bf16_bits_to_f64(uint32_t b) { return (double)__uint_as_float(b << 16); }

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

MX_DEVINL float sigmoid_f32_slow(float g) {
  const double s = 1.0 / (1.0 + exp(-(double)g));
  return __double2float_rn(s);
}

// bf16 SiLU a(g) as bit pattern.
MX_DEVINL uint32_t silu_bits(float g) {
  float p = 0.f;
  bool slow = !(fabsf(g) <= 64.0f);
  if (!slow) {
    const float t = expf(-g);
    const float s = __frcp_rn(__fadd_rn(1.0f, t));
    p = __fmul_rn(g, s);
    const int low = (int)(__float_as_uint(p) & 0xFFFFu);
    slow = (abs(low - 0x8000) <= 64) || (fabsf(p) < 1e-30f);
  }
  if (slow) p = __fmul_rn(g, sigmoid_f32_slow(g));
  return f32_to_bf16_bits(p);
}

MX_DEVINL uint32_t dg_bits(float dyf, float g, float u) {
  if (!isfinite(g)) return 0x7FC0u;
  const float dyu = __fmul_rn(dyf, u);  // exact when in the normal range
  const float adyu = fabsf(dyu);
  if (fabsf(g) <= 64.0f && adyu >= 1e-30f && adyu <= 1e30f) {
    const float t = expf(-g);
    const float s = __frcp_rn(__fadd_rn(1.0f, t));
    const float oms = __fmul_rn(t, s);
    const float go = __fmul_rn(g, oms);
    const float inner = __fadd_rn(1.0f, go);
    const float f = __fmul_rn(s, inner);
    const float p = __fmul_rn(dyu, f);
    const float ratio = fabsf(go) / fabsf(inner);
    const int low = (int)(__float_as_uint(p) & 0xFFFFu);
    const float dist = (float)abs(low - 0x8000);
    if (dist > 32.0f + 32.0f * ratio && fabsf(p) >= 1e-30f && fabsf(p) <= 1e30f)
      return f32_to_bf16_bits(p);
  }
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

// ------------------------------------------------------------------ forward

constexpr int SF_R = 128;            // tile rows
constexpr int SF_C = 64;             // tile y-columns
constexpr int SF_STAGES = 2;
constexpr int SF_BOX = SF_R * SF_C * 2;  // 16 KB
constexpr int SF_STAGE_BYTES = 2 * SF_BOX;
constexpr int SF_CW = 8;
constexpr int SF_THREADS = (SF_CW + 1) * 32;
constexpr size_t SF_SMEM = SF_STAGES * SF_STAGE_BYTES + 2 * SF_BOX + 1024 + 64;

struct SwiFwdParams {
  int64_t M, h;
  int64_t row_tiles, col_tiles;
  uint8_t* q_row; ScaleDst s_row;
  uint8_t* q_col; ScaleDst s_col;
  int32_t* err;
};

template <bool COL>
__global__ void __launch_bounds__(SF_THREADS, 2)
    swiglu_fwd_kernel(const __grid_constant__ CUtensorMap tmh, SwiFwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ytile = smem + SF_STAGES * SF_STAGE_BYTES;           // 2 x 16 KB
  uint64_t* full = reinterpret_cast<uint64_t*>(ytile + 2 * SF_BOX);
  uint64_t* empty = full + SF_STAGES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n_tiles = p.row_tiles * p.col_tiles;

  __shared__ long long s_abort;  // first tile index whose wait timed out
  if (threadIdx.x == 0) {
    for (int s = 0; s < SF_STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], SF_CW); }
    fence_mbar_init();
    s_abort = 0x7FFFFFFFFFFFFFFFll;
  }
  __syncthreads();

  if (warp == SF_CW) {
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

  int stage = 0; uint32_t phase = 0; int buf = 0;
  for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const int64_t rt = t / p.col_tiles, ct = t - rt * p.col_tiles;
    const int64_t r0 = rt * SF_R, c0 = ct * SF_C;
    // On a timed-out wait the warp still takes part in this tile's named
    // barrier (so no other warp is left waiting there), then all leave.
    const bool ok = mbar_wait(&full[stage], phase, p.err);
    if (!ok) atomicMin(&s_abort, (long long)t);
    const uint8_t* gt = smem + stage * SF_STAGE_BYTES;
    const uint8_t* ut = gt + SF_BOX;
    uint8_t* yt = ytile + buf * SF_BOX;
    const int seg = lane & 7;
#pragma unroll 1
    for (int it = 0; ok && it < SF_R / (4 * SF_CW); ++it) {
      const int rr = it * (4 * SF_CW) + warp * 4 + (lane >> 3);
      const uint4 gv = *reinterpret_cast<const uint4*>(gt + rr * 128 + seg * 16);
      const uint4 uv = *reinterpret_cast<const uint4*>(ut + rr * 128 + seg * 16);
      const uint32_t gp[4] = {gv.x, gv.y, gv.z, gv.w};
      const uint32_t up[4] = {uv.x, uv.y, uv.z, uv.w};
      uint32_t yp[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float a0 = bf16_lo(silu_bits(bf16_lo(gp[i])));
        const float a1 = bf16_lo(silu_bits(bf16_hi(gp[i])));
        const uint32_t y0 = f32_to_bf16_bits(__fmul_rn(a0, bf16_lo(up[i])));
        const uint32_t y1 = f32_to_bf16_bits(__fmul_rn(a1, bf16_hi(up[i])));
        yp[i] = y0 | (y1 << 16);
      }
      uint32_t s;
      const uint2 codes = quant_row8(yp, s);
      const int64_t r = r0 + rr;
      const int64_t c = c0 + seg * 8;
      if (r < p.M) {
        *reinterpret_cast<uint2*>(p.q_row + r * p.h + c) = codes;
        if ((seg & 3) == 0) p.s_row.put(r, c >> 5, s);
      }
      if (COL) *reinterpret_cast<uint4*>(yt + rr * 128 + seg * 16) = make_uint4(yp[0], yp[1], yp[2], yp[3]);
    }
    __syncwarp();
    if (ok && lane == 0) mbar_arrive(&empty[stage]);
    if (++stage == SF_STAGES) { stage = 0; phase ^= 1; }

    if (COL) {
      named_bar_sync(1, SF_CW * 32);
      if (s_abort <= t) break;
      const int rb = warp & 3;
      const int col = (warp >> 2) * 32 + lane;  // 0..63
      uint32_t v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = *reinterpret_cast<const uint16_t*>(yt + (rb * 32 + i) * 128 + col * 2);
      uint32_t codes[8];
      const uint32_t s = quant_col32(v, codes);
      const int64_t rg = r0 + rb * 32;
      if (rg < p.M) {
        uint8_t* dst = p.q_col + (c0 + col) * p.M + rg;
        store16(dst, codes[0], codes[1], codes[2], codes[3]);
        store16(dst + 16, codes[4], codes[5], codes[6], codes[7]);
        p.s_col.put(c0 + col, rg >> 5, s);
      }
      buf ^= 1;
    } else if (!ok) {
      break;
    }
  }
}

// ------------------------------------------------------------------ backward

constexpr int SB_R = 64;
constexpr int SB_C = 64;
constexpr int SB_STAGES = 2;
constexpr int SB_BOX = SB_R * SB_C * 2;      // 8 KB
constexpr int SB_STAGE_BYTES = 3 * SB_BOX;   // dy, g, u
constexpr int SB_CW = 8;
constexpr int SB_THREADS = (SB_CW + 1) * 32;
constexpr size_t SB_SMEM = SB_STAGES * SB_STAGE_BYTES + 2 * 3 * SB_BOX + 1024 + 64;

struct SwiBwdParams {
  int64_t M, h;
  int64_t row_tiles, col_tiles;
  uint8_t* q_row; ScaleDst s_row;   // [M, 2h]
  uint8_t* q_col; ScaleDst s_col;   // [2h, M]
  uint16_t* dh13_t;                 // [2h, M]
  uint16_t* y_t;                    // [h, M]
  int32_t* err;
};

// MODE 0: rowwise only; 1: rowwise + columnwise MX; 2: rowwise + bf16 transposed
// dh13 and y.
template <int MODE>
__global__ void __launch_bounds__(SB_THREADS, 2)
    swiglu_bwd_kernel(const __grid_constant__ CUtensorMap tmdy, const __grid_constant__ CUtensorMap tmh,
                      SwiBwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* otile = smem + SB_STAGES * SB_STAGE_BYTES;  // 2 buffers x {dg, du, y}
  uint64_t* full = reinterpret_cast<uint64_t*>(otile + 2 * 3 * SB_BOX);
  uint64_t* empty = full + SB_STAGES;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n_tiles = p.row_tiles * p.col_tiles;

  __shared__ long long s_abort;  // first tile index whose wait timed out
  if (threadIdx.x == 0) {
    for (int s = 0; s < SB_STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], SB_CW); }
    fence_mbar_init();
    s_abort = 0x7FFFFFFFFFFFFFFFll;
  }
  __syncthreads();

  if (warp == SB_CW) {
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

  int stage = 0; uint32_t phase = 0; int buf = 0;
  for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const int64_t rt = t / p.col_tiles, ct = t - rt * p.col_tiles;
    const int64_t r0 = rt * SB_R, c0 = ct * SB_C;
    const bool ok = mbar_wait(&full[stage], phase, p.err);
    if (!ok) atomicMin(&s_abort, (long long)t);
    const uint8_t* dyt = smem + stage * SB_STAGE_BYTES;
    const uint8_t* gt = dyt + SB_BOX;
    const uint8_t* ut = dyt + 2 * SB_BOX;
    uint8_t* ot = otile + buf * 3 * SB_BOX;   // dg | du | y
    const int seg = lane & 7;
#pragma unroll 1
    for (int it = 0; ok && it < SB_R / (4 * SB_CW); ++it) {
      const int rr = it * (4 * SB_CW) + warp * 4 + (lane >> 3);
      const uint4 dv = *reinterpret_cast<const uint4*>(dyt + rr * 128 + seg * 16);
      const uint4 gv = *reinterpret_cast<const uint4*>(gt + rr * 128 + seg * 16);
      const uint4 uv = *reinterpret_cast<const uint4*>(ut + rr * 128 + seg * 16);
      const uint32_t dp[4] = {dv.x, dv.y, dv.z, dv.w};
      const uint32_t gp[4] = {gv.x, gv.y, gv.z, gv.w};
      const uint32_t up[4] = {uv.x, uv.y, uv.z, uv.w};
      uint32_t dgp[4], dup[4], yp[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t dgw = 0, duw = 0, yw = 0;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const float dyf = hh ? bf16_hi(dp[i]) : bf16_lo(dp[i]);
          const float g = hh ? bf16_hi(gp[i]) : bf16_lo(gp[i]);
          const float u = hh ? bf16_hi(up[i]) : bf16_lo(up[i]);
          const float a = bf16_lo(silu_bits(g));
          const uint32_t du = f32_to_bf16_bits(__fmul_rn(dyf, a));
          const uint32_t dg = dg_bits(dyf, g, u);
          dgw |= dg << (16 * hh);
          duw |= du << (16 * hh);
          if (MODE == 2) yw |= f32_to_bf16_bits(__fmul_rn(a, u)) << (16 * hh);
        }
        dgp[i] = dgw; dup[i] = duw; yp[i] = yw;
      }
      uint32_t sg, su;
      const uint2 cg = quant_row8(dgp, sg);
      const uint2 cu = quant_row8(dup, su);
      const int64_t r = r0 + rr;
      const int64_t c = c0 + seg * 8;
      if (r < p.M) {
        *reinterpret_cast<uint2*>(p.q_row + r * 2 * p.h + c) = cg;
        *reinterpret_cast<uint2*>(p.q_row + r * 2 * p.h + p.h + c) = cu;
        if ((seg & 3) == 0) {
          p.s_row.put(r, c >> 5, sg);
          p.s_row.put(r, (p.h + c) >> 5, su);
        }
      }
      if (MODE != 0) {
        *reinterpret_cast<uint4*>(ot + rr * 128 + seg * 16) = make_uint4(dgp[0], dgp[1], dgp[2], dgp[3]);
        *reinterpret_cast<uint4*>(ot + SB_BOX + rr * 128 + seg * 16) = make_uint4(dup[0], dup[1], dup[2], dup[3]);
        if (MODE == 2)
          *reinterpret_cast<uint4*>(ot + 2 * SB_BOX + rr * 128 + seg * 16) = make_uint4(yp[0], yp[1], yp[2], yp[3]);
      }
    }
    __syncwarp();
    if (ok && lane == 0) mbar_arrive(&empty[stage]);
    if (++stage == SB_STAGES) { stage = 0; phase ^= 1; }

    if (MODE != 0) {
      named_bar_sync(1, SB_CW * 32);
      if (s_abort <= t) break;
      if (MODE == 1) {
        // 128 columns (dg 0..63, du 64..127) x 2 row blocks = 256 items
        const int item = warp * 32 + lane;
        const int colx = item & 127, rb = item >> 7;
        const int which = colx >> 6, col = colx & 63;
        const uint8_t* src = ot + which * SB_BOX;
        uint32_t v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = *reinterpret_cast<const uint16_t*>(src + (rb * 32 + i) * 128 + col * 2);
        uint32_t codes[8];
        const uint32_t s = quant_col32(v, codes);
        const int64_t rg = r0 + rb * 32;
        const int64_t orow = (which ? p.h : 0) + c0 + col;
        if (rg < p.M) {
          uint8_t* dst = p.q_col + orow * p.M + rg;
          store16(dst, codes[0], codes[1], codes[2], codes[3]);
          store16(dst + 16, codes[4], codes[5], codes[6], codes[7]);
          p.s_col.put(orow, rg >> 5, s);
        }
      } else {
        // bf16 transposed dg, du (into dh13_t) and y (into y_t): 192 columns x
        // 2 half-tiles of 32 rows = 384 items
        for (int item = warp * 32 + lane; item < 384; item += SB_CW * 32) {
          const int colx = item % 192, rb = item / 192;
          const int which = colx / 64, col = colx % 64;
          const uint8_t* src = ot + which * SB_BOX;
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint32_t a0 = *reinterpret_cast<const uint16_t*>(src + (rb * 32 + 2 * i) * 128 + col * 2);
            const uint32_t a1 = *reinterpret_cast<const uint16_t*>(src + (rb * 32 + 2 * i + 1) * 128 + col * 2);
            w[i] = a0 | (a1 << 16);
          }
          const int64_t rg = r0 + rb * 32;
          if (rg < p.M) {
            uint16_t* dst;
            if (which == 2) dst = p.y_t ? p.y_t + (c0 + col) * p.M + rg : nullptr;
            else dst = p.dh13_t ? p.dh13_t + ((which ? p.h : 0) + c0 + col) * p.M + rg : nullptr;
            if (dst) {
#pragma unroll
              for (int q = 0; q < 4; ++q) store16(dst + q * 8, w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
            }
          }
        }
      }
      buf ^= 1;
    } else if (!ok) {
      break;
    }
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
    if (e == cudaSuccess) { k<<<grid, SF_THREADS, SF_SMEM, stream>>>(tm, p); e = cudaGetLastError(); }
  } else {
    auto k = swiglu_fwd_kernel<false>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SF_SMEM);
    if (e == cudaSuccess) { k<<<grid, SF_THREADS, SF_SMEM, stream>>>(tm, p); e = cudaGetLastError(); }
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
    if (e == cudaSuccess) { k<<<grid, SB_THREADS, SB_SMEM, stream>>>(tdy, th, p); e = cudaGetLastError(); } \
  } while (0)
  if (mode == 0) MX_LAUNCH_B(0);
  else if (mode == 1) MX_LAUNCH_B(1);
  else MX_LAUNCH_B(2);
#undef MX_LAUNCH_B
  return cuda_status(e, "swiglu_bwd_kernel launch");
}

}  // namespace mx
