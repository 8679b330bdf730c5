// quant.cu - standalone MXFP8 cast of bf16 matrices (rowwise, columnwise or
// both from one read), plus a bf16 transposed copy used by the bf16
// weight-gradient recipe.
//
// Design: a persistent kernel streams 128x128 bf16 tiles through a 2-stage
// TMA ring in shared memory (one producer warp, eight consumer warps), each
// tile as two 64-column boxes stored with the 128-byte swizzle (16-byte
// chunk c of row r at chunk position c ^ (r & 7)).  The rowwise path gives
// each thread one whole 32-element block (four 16-byte reads); the
// columnwise path reads 4-byte column pairs down 32 rows (one thread per two
// column blocks) - the transpose happens in shared memory, so every global
// load and store stays coalesced, and the swizzle keeps both read patterns
// free of bank conflicts.
#include "tile_quant.cuh"
#include "kernels.h"

namespace mx {

namespace {

constexpr int QT_R = 128;          // tile rows
constexpr int QT_C = 128;          // tile cols (two 64-column TMA boxes)
// Two stages, two CTAs per SM: the quantize sweep (N x N, row / col /
// both, fraction of measured HBM bandwidth) at 8192: 0.77 / 0.67 / 0.72 and
// at 16384: 0.91 / 0.81 / 0.84, against 0.71-0.72 / 0.62-0.64 / 0.70 and
// 0.84 / 0.78 / 0.82 with three stages; three CTAs of two stages, or one
// CTA of four, measured lower still.
constexpr int QT_STAGES = 2;
constexpr int QT_BOX_BYTES = QT_R * 64 * 2;        // 16 KB
constexpr int QT_TILE_BYTES = 2 * QT_BOX_BYTES;    // 32 KB
constexpr int QT_CONSUMER_WARPS = 8;
constexpr int QT_THREADS = (QT_CONSUMER_WARPS + 1) * 32;
constexpr int QT_SCALE_BYTES = 2 * 512;             // one MMA scale tile per axis
constexpr size_t QT_SMEM = QT_STAGES * QT_TILE_BYTES + 2 * QT_SCALE_BYTES + 1024 + 64;

struct QuantKParams {
  int64_t rows, cols;
  int32_t batch;
  int64_t row_tiles, col_tiles;
  // rowwise MX
  uint8_t* q_row; int64_t qr_ld; int64_t qr_bs;
  ScaleDst s_row; int64_t sr_bs;
  // columnwise MX: dest [cols, *] codes, row c at q_col + c*qc_ld + qc_off
  uint8_t* q_col; int64_t qc_ld; int64_t qc_off; int64_t qc_bs;
  ScaleDst s_col; int64_t sc_off; int64_t sc_bs;
  // columnwise bf16 transpose: dest [cols, *] bf16
  uint16_t* t_col; int64_t tc_ld; int64_t tc_off; int64_t tc_bs;
  uint32_t rceil;  // 1: RCEIL scales, 0: FLOOR
  const float* amax;  // FP8 per-tensor mode: amax of each batch item
  int32_t tile_scales;  // MMA layout, tile-aligned: a tile's scales are one 512-byte tile per axis
  int32_t v8_row, v8_col;  // code destinations 32-byte aligned: one 256-bit store per 32 codes
  int32_t* err;
};

// COLK: 0 no columnwise output, 1 MXFP8 columnwise, 2 bf16 transpose.
//
// Scales in the MMA layout: a 128x128 tile's row scales are exactly one
// 512-byte scale tile, and so are its column scales.  The consumers put
// their scale bytes into a shared-memory copy of those tiles (double-
// buffered by tile parity; bytes of rows or columns past the matrix are 0,
// the layout's padding), meet at a named barrier, and warp 0 writes each
// tile with one 16-byte store per lane, instead of 1024 single-byte stores
// scattered over the tile.
//
// TW: FP8 per-tensor codes instead of MX blocks (no scale bytes written):
// every element of batch item b is scaled by s = 448 / amax[b].
template <bool ROW, int COLK, bool TW = false>
__global__ void __launch_bounds__(QT_THREADS, 2)
    quant_kernel(const __grid_constant__ CUtensorMap tmx, QuantKParams p) {
  static_assert(!TW || COLK != 2, "per-tensor FP8 writes codes only");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sscale = smem + QT_STAGES * QT_TILE_BYTES;  // [2 tile parities][row 512 | col 512]
  uint64_t* full = reinterpret_cast<uint64_t*>(sscale + 2 * QT_SCALE_BYTES);
  uint64_t* empty = full + QT_STAGES;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t tiles_per_b = p.row_tiles * p.col_tiles;
  const int64_t n_tiles = tiles_per_b * p.batch;

  __shared__ int s_dead;
  if (threadIdx.x == 0) {
    for (int s = 0; s < QT_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], QT_CONSUMER_WARPS);
    }
    fence_mbar_init();
    s_dead = 0;
  }
  __syncthreads();

  if (warp == QT_CONSUMER_WARPS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmx);
      int stage = 0;
      uint32_t phase = 0;
      for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
        const int64_t b = t / tiles_per_b;
        const int64_t rem = t - b * tiles_per_b;
        const int64_t rt = rem / p.col_tiles, ct = rem - rt * p.col_tiles;
        if (!mbar_wait(&empty[stage], phase ^ 1, p.err)) break;
        mbar_arrive_expect_tx(&full[stage], QT_TILE_BYTES);
        uint8_t* dst = smem + stage * QT_TILE_BYTES;
        tma_load_3d(dst, &tmx, (int32_t)(ct * QT_C), (int32_t)(rt * QT_R), (int32_t)b, &full[stage]);
        tma_load_3d(dst + QT_BOX_BYTES, &tmx, (int32_t)(ct * QT_C + 64), (int32_t)(rt * QT_R),
                    (int32_t)b, &full[stage]);
        if (++stage == QT_STAGES) { stage = 0; phase ^= 1; }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  int stage = 0;
  uint32_t phase = 0;
  int par = 0;
  for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, par ^= 1) {
    const int64_t b = t / tiles_per_b;
    const int64_t rem = t - b * tiles_per_b;
    const int64_t rt = rem / p.col_tiles, ct = rem - rt * p.col_tiles;
    const int64_t r0 = rt * QT_R, c0 = ct * QT_C;
    // a wait that runs out marks the CTA dead: the remaining tiles are
    // skipped, but every consumer warp still meets the per-tile barrier
    bool live = __all_sync(0xFFFFFFFFu, *reinterpret_cast<volatile int*>(&s_dead) == 0);
    if (live && !warp_wait(&full[stage], phase, p.err)) {
      if (lane == 0) atomicExch(&s_dead, 1);
      live = false;
    }
    if (!live && !p.tile_scales) break;
    uint8_t* srow_t = sscale + par * QT_SCALE_BYTES;
    uint8_t* scol_t = srow_t + 512;
    if (live) {
    const uint8_t* tile = smem + stage * QT_TILE_BYTES;

    if (ROW) {
      // one thread per 32-element row block.  A quarter-warp covers rows
      // 4g..4g+3 of one box, two blocks per row, so its eight 16-byte reads
      // land on eight distinct swizzled chunk positions; quarter-warps 2k and
      // 2k+1 write the two halves of the same 128-byte row segments.
      const int qw = lane >> 3, e = lane & 7;
      const int box = qw & 1, jj = e & 1;
      uint8_t* qrow = p.q_row + b * p.qr_bs;
      ScaleDst sd = p.s_row;
      sd.base += b * p.sr_bs;
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int rr = it * 64 + warp * 8 + (qw >> 1) * 4 + (e >> 1);
        const uint8_t* rowp = tile + box * QT_BOX_BYTES + rr * 128;
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = *reinterpret_cast<const uint4*>(rowp + (((jj * 4 + k) ^ (rr & 7)) << 4));
          pk[4 * k] = v.x; pk[4 * k + 1] = v.y; pk[4 * k + 2] = v.z; pk[4 * k + 3] = v.w;
        }
        uint32_t codes[8];
        uint32_t s = 0;
        if constexpr (TW) tw_row32(pk, codes, splat_f32x2(tw_scale(p.amax[b])));
        else s = quant_row32(pk, codes, p.rceil);
        const int64_t r = r0 + rr;
        const int64_t c = c0 + box * 64 + jj * 32;
        const bool in = r < p.rows && c < p.cols;
        if (in) {
          uint8_t* dst = qrow + r * p.qr_ld + c;
          store32_codes(dst, codes, p.v8_row);
          if (!TW && !p.tile_scales) sd.put(r, c >> 5, s);
        }
        if (p.tile_scales) srow_t[(rr & 31) * 16 + (rr >> 5) * 4 + box * 2 + jj] = in ? (uint8_t)s : 0;
      }
    }

    if (COLK != 0) {
      // one thread per (column pair, 32-row block)
      const int rb = warp & 3;
      const int pair = (warp >> 2) * 32 + lane;     // 0..63
      const int box = pair >> 5, pc = pair & 31;
      uint32_t v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)  // row rb*32+i: chunk pc/4 sits at (pc/4) ^ (i & 7)
        v[i] = *reinterpret_cast<const uint32_t*>(tile + box * QT_BOX_BYTES + (rb * 32 + i) * 128 +
                                                  ((((pc >> 2) ^ (i & 7)) << 4) | ((pc & 3) << 2)));
      const int64_t rg = r0 + rb * 32;
      const int64_t cg = c0 + box * 64 + pc * 2;
      const int cl = box * 64 + pc * 2;  // column within the tile
      if (COLK == 1 && p.tile_scales && !(rg < p.rows && cg < p.cols)) {
        scol_t[(cl & 31) * 16 + (cl >> 5) * 4 + rb] = 0;
        scol_t[((cl + 1) & 31) * 16 + ((cl + 1) >> 5) * 4 + rb] = 0;
      }
      if (rg < p.rows && cg < p.cols) {
        if (COLK == 1) {
          uint8_t* qcol = p.q_col + b * p.qc_bs;
          ScaleDst sd = p.s_col;
          sd.base += b * p.sc_bs;
          uint32_t ca[8], cb[8], sa = 0, sb = 0;
          if constexpr (TW) tw_col32x2(v, ca, cb, splat_f32x2(tw_scale(p.amax[b])));
          else quant_col32x2(v, ca, cb, sa, sb, p.rceil);
          uint8_t* dst = qcol + cg * p.qc_ld + p.qc_off + rg;
          store32_codes(dst, ca, p.v8_col);
          store32_codes(dst + p.qc_ld, cb, p.v8_col);
          if (TW) {
          } else if (p.tile_scales) {
            scol_t[(cl & 31) * 16 + (cl >> 5) * 4 + rb] = (uint8_t)sa;
            scol_t[((cl + 1) & 31) * 16 + ((cl + 1) >> 5) * 4 + rb] = (uint8_t)sb;
          } else {
            sd.put(cg, p.sc_off + (rg >> 5), sa);
            sd.put(cg + 1, p.sc_off + (rg >> 5), sb);
          }
        } else {
          uint16_t* tcol = p.t_col + b * p.tc_bs;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint32_t a0 = half ? (v[2 * i] >> 16) : (v[2 * i] & 0xFFFFu);
              const uint32_t a1 = half ? (v[2 * i + 1] >> 16) : (v[2 * i + 1] & 0xFFFFu);
              w[i] = a0 | (a1 << 16);
            }
            uint16_t* dst = tcol + (cg + half) * p.tc_ld + p.tc_off + rg;
#pragma unroll
            for (int q = 0; q < 4; ++q) store16(dst + q * 8, w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
        }
      }
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    }  // live
    if (++stage == QT_STAGES) { stage = 0; phase ^= 1; }
    if (p.tile_scales && (ROW || COLK == 1)) {
      // all of this tile's scale bytes are in shared memory: warp 0 writes
      // the row tile (lanes 0-31) and warp 1 the column tile, 16 bytes a lane
      named_bar_sync(1, QT_CONSUMER_WARPS * 32);
      if (ROW && warp == 0 && live) {
        const uint4 v = *reinterpret_cast<const uint4*>(srow_t + lane * 16);
        uint8_t* dst = p.s_row.base + b * p.sr_bs + (rt * p.s_row.tiles_per_row + ct) * 512;
        *reinterpret_cast<uint4*>(dst + lane * 16) = v;
      }
      if (COLK == 1 && warp == 1 && live) {
        const uint4 v = *reinterpret_cast<const uint4*>(scol_t + lane * 16);
        uint8_t* dst = p.s_col.base + b * p.sc_bs + (ct * p.s_col.tiles_per_row + (p.sc_off >> 2) + rt) * 512;
        *reinterpret_cast<uint4*>(dst + lane * 16) = v;
      }
    }
  }
}

// amax of each batch item (FP8 per-tensor recipe): blockIdx.y is the item;
// each thread keeps the packed bf16 maximum of |x| over 16-byte vectors
// (four independent loads in flight), the block reduces it and one atomicMax
// on the fp32 bit pattern merges the blocks of an item (non-negative floats
// order like their bit patterns; a NaN, 0x7FC00000, beats every number).
constexpr int AMAX_THREADS = 256;

__global__ void __launch_bounds__(AMAX_THREADS)
    fp8_amax_kernel(const uint4* __restrict__ x, int64_t vec_per_item, float* amax) {
  const uint4* xb = x + (int64_t)blockIdx.y * vec_per_item;
  const int64_t stride = (int64_t)gridDim.x * AMAX_THREADS;
  uint32_t m[4] = {0, 0, 0, 0};
  int64_t i = (int64_t)blockIdx.x * AMAX_THREADS + threadIdx.x;
  for (; i + 3 * stride < vec_per_item; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = __ldcs(xb + i + k * stride);
#pragma unroll
    for (int k = 0; k < 4; ++k) m[k] = max2(m[k], max2(max2(abs2(v[k].x), abs2(v[k].y)), max2(abs2(v[k].z), abs2(v[k].w))));
  }
  for (; i < vec_per_item; i += stride) {
    const uint4 v = __ldcs(xb + i);
    m[0] = max2(m[0], max2(max2(abs2(v.x), abs2(v.y)), max2(abs2(v.z), abs2(v.w))));
  }
  uint32_t r = max2(max2(m[0], m[1]), max2(m[2], m[3]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) r = max2(r, __shfl_xor_sync(0xFFFFFFFFu, r, o));
  __shared__ uint32_t s_m[AMAX_THREADS / 32];
  if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = r;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = s_m[0];
    for (int w = 1; w < AMAX_THREADS / 32; ++w) t = max2(t, s_m[w]);
    atomicMax(reinterpret_cast<unsigned int*>(amax) + blockIdx.y, max_halves(t) << 16);
  }
}

}  // namespace

int launch_fp8_amax(const void* x, int64_t batch, int64_t n, float* amax, cudaStream_t stream) {
  if (batch <= 0 || n <= 0) return MX_OK;
  count_launch(MX_KERNEL_MEMSET);
  cudaError_t e = cudaMemsetAsync(amax, 0, (size_t)batch * 4, stream);
  if (e != cudaSuccess) return cuda_status(e, "cudaMemsetAsync");
  const int64_t vec = n / 8;
  const int64_t want = ((int64_t)num_sms() * 8 + batch - 1) / batch;   // ~8 blocks per SM in all
  const int64_t need = (vec + AMAX_THREADS * 4 - 1) / (AMAX_THREADS * 4);
  const int gx = (int)std::max<int64_t>(1, std::min<int64_t>(want, need));
  count_launch(MX_KERNEL_QUANT);
  fp8_amax_kernel<<<dim3(gx, (unsigned)batch), AMAX_THREADS, 0, stream>>>(reinterpret_cast<const uint4*>(x), vec,
                                                                          amax);
  return cuda_status(cudaGetLastError(), "fp8_amax_kernel launch");
}

int launch_quant(const QuantLaunch& q, cudaStream_t stream) {
  const bool row = q.q_row != nullptr;
  const int colk = q.q_col ? 1 : (q.t_col ? 2 : 0);
  CUtensorMap tm;
  {
    uint64_t dims[3] = {(uint64_t)q.cols, (uint64_t)q.rows, (uint64_t)q.batch};
    uint64_t strides[2] = {(uint64_t)q.cols * 2, (uint64_t)q.cols * q.rows * 2};
    uint32_t box[3] = {64, QT_R, 1};
    int rc = make_tmap(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q.x), dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  QuantKParams p{};
  p.rows = q.rows; p.cols = q.cols; p.batch = q.batch;
  p.row_tiles = (q.rows + QT_R - 1) / QT_R;
  p.col_tiles = (q.cols + QT_C - 1) / QT_C;
  p.q_row = (uint8_t*)q.q_row; p.qr_ld = q.cols; p.qr_bs = q.qr_bs ? q.qr_bs : q.rows * q.cols;
  const int64_t S_row = q.cols / 32;
  p.s_row = ScaleDst{(uint8_t*)q.s_row, (S_row + 3) / 4, S_row, q.layout == MX_SCALE_MMA};
  p.sr_bs = q.sr_bs ? q.sr_bs
                    : (q.layout == MX_SCALE_MMA ? ((q.rows + 127) / 128) * ((S_row + 3) / 4) * 512 : q.rows * S_row);
  p.q_col = (uint8_t*)q.q_col; p.qc_ld = q.qc_ld; p.qc_off = q.qc_off; p.qc_bs = q.qc_bs;
  const int64_t S_col = q.qc_ld / 32;
  p.s_col = ScaleDst{(uint8_t*)q.s_col, (S_col + 3) / 4, S_col, q.layout == MX_SCALE_MMA};
  p.sc_off = q.qc_off / 32; p.sc_bs = q.sc_bs;
  p.t_col = (uint16_t*)q.t_col; p.tc_ld = q.tc_ld; p.tc_off = q.tc_off; p.tc_bs = q.tc_bs;
  p.rceil = q.floor_scale ? 0u : 1u;
  p.amax = q.amax;
  // whole scale tiles per 128x128 tile: MMA layout, columnwise MXFP8 output
  // (rowwise alone measured ~3% slower with the per-tile barrier than with
  // byte stores), the columnwise scale columns starting on a tile boundary
  p.tile_scales = (!q.tw && q.layout == MX_SCALE_MMA && colk == 1 && (p.sc_off & 3) == 0) ? 1 : 0;
  p.err = q.err;
#ifndef MX_QT_V8
#define MX_QT_V8 1
#endif
  auto a32 = [](const void* ptr, int64_t a, int64_t b, int64_t c) {
    return ((reinterpret_cast<uintptr_t>(ptr) | (uintptr_t)a | (uintptr_t)b | (uintptr_t)c) & 31) == 0;
  };
  p.v8_row = MX_QT_V8 && q.q_row && a32(q.q_row, p.qr_ld, p.qr_bs, 0);
  p.v8_col = MX_QT_V8 && q.q_col && a32(q.q_col, p.qc_ld, p.qc_off, p.qc_bs);

  const int64_t n_tiles = p.row_tiles * p.col_tiles * q.batch;
  if (n_tiles == 0) return MX_OK;
  int grid = (int)std::min<int64_t>(n_tiles, (int64_t)num_sms() * 2);
  cudaError_t e;
#define MX_LAUNCH_Q(R, C, TW)                                                                  \
  do {                                                                                         \
    auto k = quant_kernel<R, C, TW>;                                                           \
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)QT_SMEM);    \
    if (e == cudaSuccess) {                                                                    \
      count_launch(MX_KERNEL_QUANT);                                                           \
      k<<<grid, QT_THREADS, QT_SMEM, stream>>>(tm, p);                                         \
      e = cudaGetLastError();                                                                  \
    }                                                                                          \
  } while (0)
  if (q.tw) {
    if (!q.amax || colk == 2) return fail(MX_ERR_INVALID_ARG, "per-tensor FP8 cast: amax required, codes only");
    if (row && colk == 0) MX_LAUNCH_Q(true, 0, true);
    else if (row && colk == 1) MX_LAUNCH_Q(true, 1, true);
    else if (!row && colk == 1) MX_LAUNCH_Q(false, 1, true);
    else return MX_ERR_INVALID_ARG;
  }
  else if (row && colk == 0) MX_LAUNCH_Q(true, 0, false);
  else if (row && colk == 1) MX_LAUNCH_Q(true, 1, false);
  else if (row && colk == 2) MX_LAUNCH_Q(true, 2, false);
  else if (!row && colk == 1) MX_LAUNCH_Q(false, 1, false);
  else if (!row && colk == 2) MX_LAUNCH_Q(false, 2, false);
  else return MX_ERR_INVALID_ARG;
#undef MX_LAUNCH_Q
  return cuda_status(e, "quant_kernel launch");
}

}  // namespace mx
