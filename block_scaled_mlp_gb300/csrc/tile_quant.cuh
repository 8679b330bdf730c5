// tile_quant.cuh - MXFP8 block quantization of bf16 values held in registers,
// used by the standalone cast kernel and by the fused SwiGLU kernels.
//
// Row blocks: four consecutive lanes each hold 8 consecutive elements of one
// 32-element block.  Column blocks: one thread holds all 32 elements.
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

// max |x| over 8 bf16 values given as 4 packed pairs -> bf16 bit pattern of
// the maximum magnitude (integer compare of |bits| orders finite values and
// puts Inf/NaN above every finite value).
MX_DEVINL uint32_t absmax_bits8(const uint32_t (&p)[4]) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = max(m, p[i] & 0x7FFFu);
    m = max(m, (p[i] >> 16) & 0x7FFFu);
  }
  return m;
}

// Quantize 8 elements (4 packed bf16 pairs, element 2i in the low half) of a
// row block spread over 4 consecutive lanes.  Returns the 8 codes as two
// 32-bit words (element 0 in the lowest byte) and the block scale byte.
MX_DEVINL uint2 quant_row8(const uint32_t (&p)[4], uint32_t& scale_out) {
  uint32_t m = absmax_bits8(p);
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
  const uint32_t s = e8m0_from_amax_bits(m);
  scale_out = s;
  uint2 out;
  if (s == 0xFF) {
    out.x = out.y = 0x7F7F7F7Fu;
    return out;
  }
  const float inv = inv_scale_from_e8m0(s);
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    c[i] = cvt_e4m3x2(bf16_lo(p[i]) * inv, bf16_hi(p[i]) * inv);
  out.x = c[0] | (c[1] << 16);
  out.y = c[2] | (c[3] << 16);
  return out;
}

// Quantize one 32-element column block held by one thread as 32 bf16 bit
// patterns (low 16 bits of each word).  Writes 8 words of codes.
MX_DEVINL uint32_t quant_col32(const uint32_t (&v)[32], uint32_t (&codes)[8]) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 32; ++i) m = max(m, v[i] & 0x7FFFu);
  const uint32_t s = e8m0_from_amax_bits(m);
  if (s == 0xFF) {
#pragma unroll
    for (int i = 0; i < 8; ++i) codes[i] = 0x7F7F7F7Fu;
    return s;
  }
  const float inv = inv_scale_from_e8m0(s);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t lo = cvt_e4m3x2(bf16_lo(v[4 * i]) * inv, bf16_lo(v[4 * i + 1]) * inv);
    const uint32_t hi = cvt_e4m3x2(bf16_lo(v[4 * i + 2]) * inv, bf16_lo(v[4 * i + 3]) * inv);
    codes[i] = lo | (hi << 16);
  }
  return s;
}

MX_DEVINL void store16(void* dst, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  *reinterpret_cast<uint4*>(dst) = make_uint4(a, b, c, d);
}

}  // namespace mx
