// tile_quant.cuh - MXFP8 block quantization of bf16 values held in registers,
// used by the standalone cast kernel and by the fused SwiGLU kernels.
//
// Row blocks: one thread holds a whole 32-element block (quant_row32).
// Column blocks: one thread holds the 32 elements of two adjacent columns as
// packed pairs (quant_col32x2), or lanes l and l ^ 16 hold 16 rows each
// (quant_col16x2).  Scaling by the power-of-two inverse scale is exact; the E4M3
// conversion rounds to nearest even and saturates.
#pragma once

#include "common.cuh"

namespace mx {

// Scale bytes of a [R, S] scale matrix, linear or MMA-tiled.
struct ScaleDst {
  uint8_t* base;        // NULL = not written
  int64_t tiles_per_row;  // MMA layout: ceil(S/4)
  int64_t ld;           // linear layout: S
  int mma;              // 1 = MMA layout
  MX_DEVINL void put(int64_t r, int64_t c, uint32_t s) const {
    if (mma) base[mma_scale_offset(r, c, tiles_per_row)] = (uint8_t)s;
    else base[r * ld + c] = (uint8_t)s;
  }
};

// |x| of a packed bf16 pair, and the pairwise maximum propagating NaN:
// on magnitudes the float order equals the order of the bit patterns, and a
// NaN or an infinity lands at or above 0x7F80, which the scale rule maps to
// 0xFF.
MX_DEVINL uint32_t abs2(uint32_t p) { return p & 0x7FFF7FFFu; }
MX_DEVINL uint32_t max2(uint32_t a, uint32_t b) {
  const __nv_bfloat162 r =
      __hmax2_nan(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}
// max(|a|, |b|) per half in one instruction (the sign of the result is the
// xor of the signs: callers use the magnitude bits only); NaN propagates as
// the canonical NaN
MX_DEVINL uint32_t maxabs2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// larger magnitude of the two halves, as a 16-bit pattern (NaN -> >= 0x7F80)
MX_DEVINL uint32_t max_halves(uint32_t m2) {
  const uint32_t lo = m2 & 0xFFFFu, hi = m2 >> 16;
  const uint32_t isnan = (lo > 0x7F80u) | (hi > 0x7F80u);
  return isnan ? 0x7FC0u : max(lo, hi);
}

// Both elements of a packed bf16 pair times a power-of-two inverse scale
// given as a bf16 (exact: a power of two in the normal range), each product
// formed by the mixed-precision FMA straight from the bf16 halves (RN_f32 of
// the product, -0 added so that zeros keep their sign), then RNE saturating
// E4M3: the pair's two codes in the low 16 bits.
MX_DEVINL void scale2_pow2(uint32_t p, uint16_t inv_lo, uint16_t inv_hi, float& lo, float& hi) {
  asm("{\n .reg .b16 pl, ph;\n mov.b32 {pl, ph}, %2;\n"
      " fma.rn.f32.bf16 %0, pl, %3, 0f80000000;\n fma.rn.f32.bf16 %1, ph, %4, 0f80000000;\n}"
      : "=f"(lo), "=f"(hi)
      : "r"(p), "h"(inv_lo), "h"(inv_hi));
}
MX_DEVINL uint32_t e4m3x2_pow2(uint32_t p, uint16_t inv_bf16) {
  float lo, hi;
  scale2_pow2(p, inv_bf16, inv_bf16, lo, hi);
  return cvt_e4m3x2(lo, hi);
}

// 2^-(s-127) as a bf16 bit pattern (s <= 247 for finite blocks: normal)
MX_DEVINL uint16_t inv_scale_bf16_from_e8m0(uint32_t s) { return (uint16_t)((254u - s) << 7); }

// Both elements of a packed bf16 pair times an fp32 scale (inv2 holds it in
// both lanes), one packed fp32 multiply (RN, no flush), then RNE saturating
// E4M3: the pair's two codes in the low 16 bits.
MX_DEVINL uint32_t e4m3x2_scaled(uint32_t p, f2 inv2) {
  const f2 r = f2_mul(f2_from_bf16x2(p), inv2);
  return cvt_e4m3x2(r.x, r.y);
}

MX_DEVINL f2 splat_f32x2(float f) { return f2_splat(f); }

// Quantize one whole 32-element block held by one thread as 16 packed bf16
// pairs (element 2i in the low half of p[i]).  Writes the 32 codes as 8
// words (element 0 in the lowest byte) and returns the scale byte.
MX_DEVINL uint32_t quant_row32(const uint32_t (&p)[16], uint32_t (&codes)[8], uint32_t rceil = 1u) {
  uint32_t m2 = maxabs2(p[0], p[1]);
#pragma unroll
  for (int i = 2; i < 16; ++i) m2 = maxabs2(m2, p[i]);
  const uint32_t s = e8m0_from_amax_bits(max_halves(m2 & 0x7FFF7FFFu), rceil);
  if (s == 0xFF) {
#pragma unroll
    for (int i = 0; i < 8; ++i) codes[i] = 0x7F7F7F7Fu;
    return s;
  }
  const uint16_t inv = inv_scale_bf16_from_e8m0(s);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    codes[i] = e4m3x2_pow2(p[2 * i], inv) | (e4m3x2_pow2(p[2 * i + 1], inv) << 16);
  return s;
}

// After quant_col16x2, lanes l (rh = 0: rows 0-15) and l ^ 16 (rh = 1:
// rows 16-31) swap halves: lane rh = 0 ends with column A's 32 codes and
// lane rh = 1 with column B's (rows in order), ready for one 32-byte store
// each.  All 32 lanes take part.
MX_DEVINL void col16x2_gather(const uint32_t (&ca)[4], const uint32_t (&cb)[4], int rh, uint32_t (&out)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t r = __shfl_xor_sync(0xFFFFFFFFu, rh ? ca[i] : cb[i], 16);
    out[i] = rh ? r : ca[i];
    out[4 + i] = rh ? cb[i] : r;
  }
}

// Quantize two 32-element column blocks held by one thread as 32 packed
// words (row i of column A in the low half of v[i], column B in the high
// half).  Writes 8 words of codes per column and returns both scales.
MX_DEVINL void quant_col32x2(const uint32_t (&v)[32], uint32_t (&ca)[8], uint32_t (&cb)[8], uint32_t& sa,
                             uint32_t& sb, uint32_t rceil = 1u) {
  uint32_t m2 = maxabs2(v[0], v[1]);
#pragma unroll
  for (int i = 2; i < 32; ++i) m2 = maxabs2(m2, v[i]);
  m2 &= 0x7FFF7FFFu;
  const uint32_t la = m2 & 0xFFFFu, lb = m2 >> 16;
  sa = e8m0_from_amax_bits(la > 0x7F80u ? 0x7FC0u : la, rceil);
  sb = e8m0_from_amax_bits(lb > 0x7F80u ? 0x7FC0u : lb, rceil);
  // column A in the low halves, column B in the high halves: each half is
  // scaled by its own column's power of two straight from the bf16 bits
  const uint16_t ia = inv_scale_bf16_from_e8m0(sa == 0xFF ? 127u : sa);
  const uint16_t ib = inv_scale_bf16_from_e8m0(sb == 0xFF ? 127u : sb);
  float lo[32], hi[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) scale2_pow2(v[i], ia, ib, lo[i], hi[i]);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t a01 = cvt_e4m3x2(lo[4 * i], lo[4 * i + 1]);
    const uint32_t a23 = cvt_e4m3x2(lo[4 * i + 2], lo[4 * i + 3]);
    const uint32_t b01 = cvt_e4m3x2(hi[4 * i], hi[4 * i + 1]);
    const uint32_t b23 = cvt_e4m3x2(hi[4 * i + 2], hi[4 * i + 3]);
    ca[i] = a01 | (a23 << 16);
    cb[i] = b01 | (b23 << 16);
  }
  if (sa == 0xFF)
#pragma unroll
    for (int i = 0; i < 8; ++i) ca[i] = 0x7F7F7F7Fu;
  if (sb == 0xFF)
#pragma unroll
    for (int i = 0; i < 8; ++i) cb[i] = 0x7F7F7F7Fu;
}

// Two 32-element column blocks split over lanes l and l ^ 16: each lane
// reads 16 rows of both columns as packed words through ld(i) (column A in
// the low halves, twice: once for the block maximum, which is combined
// across the lane pair, once to convert, so that few registers stay live
// inside a GEMM epilogue).  Writes this lane's 16 codes per column as 4
// words and returns both scales (the same in both lanes of the pair).
template <class Ld>
MX_DEVINL void quant_col16x2(const Ld& ld, uint32_t (&ca)[4], uint32_t (&cb)[4], uint32_t& sa, uint32_t& sb,
                             uint32_t rceil = 1u) {
  uint32_t m2 = maxabs2(ld(0), ld(1));
#pragma unroll
  for (int i = 2; i < 16; ++i) m2 = maxabs2(m2, ld(i));
  m2 = maxabs2(m2, __shfl_xor_sync(0xFFFFFFFFu, m2, 16)) & 0x7FFF7FFFu;
  const uint32_t la = m2 & 0xFFFFu, lb = m2 >> 16;
  sa = e8m0_from_amax_bits(la > 0x7F80u ? 0x7FC0u : la, rceil);
  sb = e8m0_from_amax_bits(lb > 0x7F80u ? 0x7FC0u : lb, rceil);
  const uint16_t ia = inv_scale_bf16_from_e8m0(sa == 0xFF ? 127u : sa);
  const uint16_t ib = inv_scale_bf16_from_e8m0(sb == 0xFF ? 127u : sb);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float lo[4], hi[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) scale2_pow2(ld(4 * i + k), ia, ib, lo[k], hi[k]);
    const uint32_t a01 = cvt_e4m3x2(lo[0], lo[1]);
    const uint32_t a23 = cvt_e4m3x2(lo[2], lo[3]);
    const uint32_t b01 = cvt_e4m3x2(hi[0], hi[1]);
    const uint32_t b23 = cvt_e4m3x2(hi[2], hi[3]);
    ca[i] = sa == 0xFF ? 0x7F7F7F7Fu : (a01 | (a23 << 16));
    cb[i] = sb == 0xFF ? 0x7F7F7F7Fu : (b01 | (b23 << 16));
  }
}

// ---- FP8 per-tensor ("tensorwise") scaling: one fp32 scale s per tensor,
// s = RN_f32(448 / max(amax, 2^-40)); code = E4M3 (RNE, saturating) of
// RN_f32(x * s).  s is not a power of two, so the product rounds once in
// fp32 before the E4M3 conversion rounds again.
MX_DEVINL float tw_scale(float amax) { return __fdiv_rn(448.0f, fmaxf(amax, 0x1p-40f)); }

// 32 row elements held as 16 packed bf16 pairs -> 8 words of codes.
MX_DEVINL void tw_row32(const uint32_t (&p)[16], uint32_t (&codes)[8], f2 s2) {
#pragma unroll
  for (int i = 0; i < 8; ++i) codes[i] = e4m3x2_scaled(p[2 * i], s2) | (e4m3x2_scaled(p[2 * i + 1], s2) << 16);
}

// Two columns of 32 rows held as 32 packed words (column A in the low
// halves) -> 8 words of codes per column.
MX_DEVINL void tw_col32x2(const uint32_t (&v)[32], uint32_t (&ca)[8], uint32_t (&cb)[8], f2 s2) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    f2 r[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) r[k] = f2_mul(f2_from_bf16x2(v[4 * i + k]), s2);
    ca[i] = cvt_e4m3x2(r[0].x, r[1].x) | (cvt_e4m3x2(r[2].x, r[3].x) << 16);
    cb[i] = cvt_e4m3x2(r[0].y, r[1].y) | (cvt_e4m3x2(r[2].y, r[3].y) << 16);
  }
}

MX_DEVINL void store16(void* dst, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4*>(dst) = make_uint4(a, b, c, d);
}

// 32 bytes to global memory: one 256-bit store when v8 (dst 32-byte aligned),
// else two 16-byte stores (dst 16-byte aligned)
MX_DEVINL void store32_codes(uint8_t* dst, const uint32_t (&c)[8], bool v8) {
  if (v8) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(c[0]), "r"(c[1]),
                 "r"(c[2]), "r"(c[3]), "r"(c[4]), "r"(c[5]), "r"(c[6]), "r"(c[7])
                 : "memory");
  } else {
    store16(dst, c[0], c[1], c[2], c[3]);
    store16(dst + 16, c[4], c[5], c[6], c[7]);
  }
}

}  // namespace mx
