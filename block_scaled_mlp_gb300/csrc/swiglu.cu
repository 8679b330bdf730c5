// swiglu.cu - fused SwiGLU forward / backward with dual MXFP8 quantization.
//
// Forward: h13 = [g | u] tiles stream through a TMA ring; each consumer
// thread computes y = RN_bf16(a(g) u) for the 32-element row block or the
// 32-row column blocks it quantizes, straight from the g and u tiles into
// registers (a(g) from a table of exact values over every bf16 g).  y never
// reaches global memory.
//
// Backward: dy and h13 tiles in, dh13 = [dg | du] out, quantized rowwise and
// columnwise (or, for the bf16 weight-gradient recipe, written transposed in
// bf16 together with the recomputed y), through a shared-memory result tile.
//
// Numerics: swiglu_math.cuh (exactly rounded a, y, du, dg).  The backward's
// fast path runs on packed fp32 pairs (own exp from ex2.approx, rcp.approx);
// a result is accepted only if its rounding interval (the value plus or
// minus the error bound of its chain) rounds to one bf16 value, otherwise the
// exact tiers decide.
#include "tile_quant.cuh"
#include "swiglu_math.cuh"
#include "kernels.h"

namespace mx {

namespace {

using namespace swiglu_math;

// ------------------------------------------------------------------ kernels
//
// The backward kernel streams tiles through a 2-stage TMA ring and runs
// three roles (the forward, which needs no exact tiers, is simpler and is
// described at its own section below):
//   producer warp  TMA loads of the input tiles
//   8 consumer     phase A: every element through the fp32 fast path into a
//   warps          shared-memory result tile; elements whose rounding it
//                  cannot certify are queued.  Phase C: MX quantization of
//                  the previous (complete) tile, rows on warps 4-7 and
//                  columns on warps 0-3
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

// Result tiles: 128-byte rows (64 bf16), 16-byte chunk c of row r stored at
// chunk position c ^ (r & 7), so that row-block reads (one thread per
// 32-element block) and column reads (one thread per column pair) are both
// free of bank conflicts.
MX_DEVINL int tile_off(int r, int col) { return r * 128 + ((((col >> 3) ^ (r & 7)) << 4) | ((col & 7) << 1)); }
MX_DEVINL int tile_chunk(int r, int c16) { return r * 128 + ((c16 ^ (r & 7)) << 4); }
// word pc (columns 2pc, 2pc+1) of row r
MX_DEVINL int tile_word(int r, int pc) { return r * 128 + ((((pc >> 2) ^ (r & 7)) << 4) | ((pc & 3) << 2)); }

// Row quantization of one 32-element block of a result tile: the 64-byte
// half jj of row rr.
MX_DEVINL uint32_t quant_tile_block(const uint8_t* tile, int rr, int jj, uint32_t (&codes)[8], uint32_t rceil) {
  uint32_t pk[16];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint4 v = *reinterpret_cast<const uint4*>(tile + tile_chunk(rr, jj * 4 + k));
    pk[4 * k] = v.x; pk[4 * k + 1] = v.y; pk[4 * k + 2] = v.z; pk[4 * k + 3] = v.w;
  }
  return quant_row32(pk, codes, rceil);
}


// ---- forward: tile = 128 rows x 64 y-columns
//
// The forward needs no exact tiers (a(g) comes from the table of exact values
// over every bf16 g), so it streams like the quantize kernel: one producer
// warp keeps a 2-stage ring of g and u tiles (two 16 KB boxes with the
// 128-byte swizzle: 16-byte chunk c of row r at chunk position c ^ (r & 7)),
// and each consumer thread computes the y values it quantizes straight from
// those tiles into registers, with no result tile and no block barrier.
// Every thread quantizes one 32-element row block; with columns, warps 2k
// and 2k+1 then stage their y rows in a small shared buffer, meet at a pair
// barrier, and each thread quantizes 16 rows of one column pair from it
// (lanes l and l ^ 16 share the pair's 32-row block).
constexpr int SF_R = 128, SF_C = 64;
constexpr int SF_STAGES = 2;
constexpr int SF_BOX = SF_R * SF_C * 2;       // 16 KB
constexpr int SF_STAGE_BYTES = 2 * SF_BOX;    // g, u
constexpr int SF_WARPS = 8;                   // consumer warps
constexpr int SF_THREADS = (SF_WARPS + 1) * 32;
// Shared memory per mode: the stages, plus 16 KB of y staging in dual mode,
// plus 64 bytes of barriers and flags; no static shared memory and no
// alignment slack (the dynamic region is declared 1024-aligned, which the
// kernel checks).  The rest of the SM's 256 KB stays L1, where the a(g)
// table lookups hit: two CTAs need 130.1 KB (rows) and 162.1 KB (dual)
// with the 1 KB each reserves, inside the 132 KB and 164 KB shared-memory
// configurations.  At 8192 x 8192 the rowwise kernel ran 0.067 ms with 1
// KB of slack and 1 KB of static flags per CTA against 0.076 ms with 32 KB
// more, and the dual one 0.104 ms with one staging buffer (and a second
// pair barrier per tile) against 0.111 ms with two.
constexpr size_t sf_smem(bool col) { return SF_STAGES * SF_STAGE_BYTES + (col ? 4 * 32 * 128 : 0) + 64; }
// Preferred shared-memory carveout (percent of the SM's maximum), which
// picks the shared-memory configuration and so the L1 left for the table.
// Swept at 8192 x 8192: rows 58.0-58.6 us at 50-70% (60.2 at the driver's
// default and at 72-85%, 66.9 at 100%, 70.9 below 50% where one CTA per SM
// fits); dual 84.5-84.7 us at 58-70% (87 at 72-85%, 102 below 58%).  The
// middle of each range:
constexpr int sf_carveout(bool col) { return col ? 64 : 55; }

struct SwiFwdParams {
  int64_t M, h;
  int64_t row_tiles, col_tiles;
  uint8_t* q_row; ScaleDst s_row;
  uint8_t* q_col; ScaleDst s_col;
  uint32_t rceil;  // 1: RCEIL scales, 0: FLOOR
  const uint16_t* silu_a;  // a(g) = RN_bf16(g sigma(g)) indexed by the bits of bf16 g
  int32_t v8_row, v8_col;  // codes 32-byte aligned: one 256-bit store per 32 codes
  int32_t* err;
};

// y = RN_bf16(a(g) u) for a packed pair: a(g) from the table, the product of
// two bf16 values exact in fp32
MX_DEVINL uint32_t swiglu2(uint32_t gp, uint32_t up, const uint16_t* tab) {
  const uint32_t a = (uint32_t)__ldg(tab + (gp & 0xFFFFu)) | ((uint32_t)__ldg(tab + (gp >> 16)) << 16);
  return f2_to_bf16x2(f2_mul_bf16x2(a, up));
}

// Result staging for the columns (dual mode): warps 2k and 2k+1 cover rows
// 32k..32k+31 of the tile; their y values go to the pair's 4 KB buffer, row
// q at q * 128, its 16-byte chunk c at c ^ (q & 7) ^ ((q >> 4) << 2): the
// row writes (a quarter-warp: four rows, eight chunks) and the column reads
// (rows q and q + 16 in the two half-warps) both stay free of bank
// conflicts.  The pair meets twice per tile: buffer written, buffer read.
constexpr int SF_PAIR_BYTES = 32 * 128;
MX_DEVINL int sf_pair_chunk(int q, int c) { return q * 128 + ((c ^ (q & 7) ^ ((q >> 4) << 2)) << 4); }
// barrier 1 + pr of the two warps of pair pr (literal barrier ids, so that
// the kernel reserves five barriers, not all sixteen)
template <int ID>
MX_DEVINL void pair_bar_id() { asm volatile("bar.sync %0, 64;" ::"n"(ID) : "memory"); }
MX_DEVINL void pair_bar(int pr) {
  switch (pr) {
    case 0: pair_bar_id<1>(); break;
    case 1: pair_bar_id<2>(); break;
    case 2: pair_bar_id<3>(); break;
    default: pair_bar_id<4>(); break;
  }
}

template <bool COL>
__global__ void __launch_bounds__(SF_THREADS, 2)
    swiglu_fwd_kernel(const __grid_constant__ CUtensorMap tmh, SwiFwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the 128-byte-swizzled TMA boxes need a 1024-byte aligned base; the
  // launch sizes no slack for rounding up, so a misaligned base is reported
  // and the CTA does nothing
  if (smem_u32(smem_raw) & 1023u) {
    if (threadIdx.x == 0) record_error(p.err, MX_ERR_ALIGNMENT);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* ybuf = smem + SF_STAGES * SF_STAGE_BYTES;   // dual: [4 warp pairs][4 KB]
  uint64_t* full = reinterpret_cast<uint64_t*>(ybuf + (COL ? 4 * SF_PAIR_BYTES : 0));
  uint64_t* empty = full + SF_STAGES;
  int& s_dead = *reinterpret_cast<int*>(empty + SF_STAGES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n_tiles = p.row_tiles * p.col_tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SF_STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], SF_WARPS); }
    fence_mbar_init();
    s_dead = 0;
  }
  __syncthreads();

  if (warp == SF_WARPS) {
    // ------------------------------------------------------------ producer
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

  // -------------------------------------------------------------- consumers
  // A wait that runs out marks the CTA dead.  Rowwise only, the consumers
  // then stop; in dual mode every consumer warp still runs every tile and
  // meets its pair barrier (so that no partner waits for it), skipping the
  // waits and the work.
  const uint16_t* tab = p.silu_a;
  const int pr = warp >> 1;   // warp pair
  int stage = 0; uint32_t phase = 0;
  for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
    const int64_t rt = t / p.col_tiles, ct = t - rt * p.col_tiles;
    const int64_t r0 = rt * SF_R, c0 = ct * SF_C;
    bool live = *reinterpret_cast<volatile int*>(&s_dead) == 0;
    live = __all_sync(0xFFFFFFFFu, live);
    if (live && !warp_wait(&full[stage], phase, p.err)) {
      if (lane == 0) atomicExch(&s_dead, 1);
      live = false;
    }
    if (!COL && !live) break;
    uint8_t* yb = ybuf + pr * SF_PAIR_BYTES;

    if (live) {
      const uint8_t* gt = smem + stage * SF_STAGE_BYTES;
      const uint8_t* ut = gt + SF_BOX;
      // rows: a quarter-warp covers rows 4q..4q+3 of the warp's 16-row band,
      // two blocks per row, so its eight 16-byte reads land on eight
      // distinct swizzled chunk positions
      const int e = lane & 7, jj = e & 1;
      const int rr = warp * 16 + (lane >> 3) * 4 + (e >> 1);
      uint32_t y[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int off = rr * 128 + (((jj * 4 + k) ^ (rr & 7)) << 4);
        const uint4 g4 = *reinterpret_cast<const uint4*>(gt + off);
        const uint4 u4 = *reinterpret_cast<const uint4*>(ut + off);
        y[4 * k] = swiglu2(g4.x, u4.x, tab);
        y[4 * k + 1] = swiglu2(g4.y, u4.y, tab);
        y[4 * k + 2] = swiglu2(g4.z, u4.z, tab);
        y[4 * k + 3] = swiglu2(g4.w, u4.w, tab);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);   // this warp is done with the stage
      if (COL) {
        const int q = rr & 31;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          *reinterpret_cast<uint4*>(yb + sf_pair_chunk(q, jj * 4 + k)) =
              make_uint4(y[4 * k], y[4 * k + 1], y[4 * k + 2], y[4 * k + 3]);
      }
      uint32_t codes[8];
      const uint32_t sc = quant_row32(y, codes, p.rceil);
      const int64_t r = r0 + rr;
      if (r < p.M) {
        const int64_t c = c0 + jj * 32;
        uint8_t* dst = p.q_row + r * p.h + c;
        store32_codes(dst, codes, p.v8_row);
        p.s_row.put(r, c >> 5, sc);
      }
    }
    if (++stage == SF_STAGES) { stage = 0; phase ^= 1; }
    if (COL) {
      pair_bar(pr);   // both warps' y rows are in the pair buffer
      if (live) {
        // columns: warp 2k + j takes column pairs 16j..16j+15 of the pair's
        // 32-row block; lanes l and l ^ 16 share a pair, 16 rows each
        const int rh = lane >> 4;
        const int pc = (warp & 1) * 16 + (lane & 15);
        uint32_t ca[4], cb[4], sa, sb;
        quant_col16x2(
            [&](int i) {
              return *reinterpret_cast<const uint32_t*>(yb + sf_pair_chunk(rh * 16 + i, pc >> 2) + ((pc & 3) << 2));
            },
            ca, cb, sa, sb, p.rceil);
        const int64_t rg = r0 + pr * 32;
        uint32_t col[8];
        col16x2_gather(ca, cb, rh, col);   // lane rh: column 2 pc + rh, all 32 rows
        if (rg < p.M) {
          const int64_t cg = c0 + 2 * pc;
          store32_codes(p.q_col + (cg + rh) * p.M + rg, col, p.v8_col);
          if (rh == 0) {
            p.s_col.put(cg, rg >> 5, sa);
            p.s_col.put(cg + 1, rg >> 5, sb);
          }
        }
      }
      pair_bar(pr);   // both warps have read the buffer
    }
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
  uint32_t rceil;                   // 1: RCEIL scales, 0: FLOOR
  int32_t v8_row, v8_col, v8_t;     // destinations 32-byte aligned: 256-bit stores
  int32_t* err;
};

// exact dg, du (and y) of one element, written into the result tiles at off
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
        const int row = idx / SB_C, col = idx % SB_C;
        const int off = row * 128 + col * 2;
        const float dyf = bf16_lo(*reinterpret_cast<const uint16_t*>(dyt + off));
        const float g = bf16_lo(*reinterpret_cast<const uint16_t*>(dyt + SB_BOX + off));
        const float u = bf16_lo(*reinterpret_cast<const uint16_t*>(dyt + 2 * SB_BOX + off));
        bwd_exact<MODE>(dyf, g, u, ot, tile_off(row, col));
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
          uint32_t dgp[4], dup[4], yp[4], miss[4], any = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const f2 G = f2_from_bf16x2(gp[i]);
            const SigFast2 f = sig_fast2(G);
            // a = RN_bf16(g s), certified; du = RN_bf16(dy a), y = RN_bf16(a u)
            // from exact products of bf16 halves
            uint32_t ma, mg;
            const uint32_t A = silu2_cert(G, f.S, ma);
            dup[i] = f2_to_bf16x2(f2_mul_bf16x2(dp[i], A));
            if (MODE == 2) yp[i] = f2_to_bf16x2(f2_mul_bf16x2(A, up[i]));
            // dg tier 1: (dy u) * (s * (1 + g (t s))), dy u exact, certified by
            // its interval
            const f2 DYU = f2_mul_bf16x2(dp[i], up[i]);
            const f2 GO = f2_mul(G, f2_mul(f.T, f.S));
            const f2 IN = f2_add(GO, f2_splat(1.0f));
            const f2 PG = f2_mul(DYU, f2_mul(f.S, IN));
            dgp[i] = dg2_cert(DYU, PG, dg2_width(f.S, GO, IN), mg);
            miss[i] = ma | mg | g_out_of_range2(gp[i]);
            any |= miss[i];
          }
          uint32_t slow = 0;
          if (any) {  // rare: which elements failed
#pragma unroll
            for (int i = 0; i < 4; ++i) slow |= miss_lanes(miss[i]) << (2 * i);
          }
          *reinterpret_cast<uint4*>(ot + tile_chunk(rr, seg)) = make_uint4(dgp[0], dgp[1], dgp[2], dgp[3]);
          *reinterpret_cast<uint4*>(ot + SB_BOX + tile_chunk(rr, seg)) = make_uint4(dup[0], dup[1], dup[2], dup[3]);
          if (MODE == 2)
            *reinterpret_cast<uint4*>(ot + 2 * SB_BOX + tile_chunk(rr, seg)) = make_uint4(yp[0], yp[1], yp[2], yp[3]);
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
                              bf16_lo(*reinterpret_cast<const uint16_t*>(ut + off)), ot, tile_off(rr, seg * 8 + j));
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
        // rows of dg and du: one thread per 32-element block; a warp covers
        // 16 rows x 2 blocks of one tile per pass
        const int w = MODE == 0 ? warp : warp - 4;
        const int nw = MODE == 0 ? CW : 4;
        const int jj = lane & 1;
        for (int base = w * 16; base < 2 * SB_R; base += nw * 16) {
          const int kk = base + (lane >> 3) * 4 + ((lane & 7) >> 1);
          const int which = kk / SB_R, rr = kk % SB_R;
          uint32_t codes[8];
          const uint32_t sc = quant_tile_block(ot + which * SB_BOX, rr, jj, codes, p.rceil);
          const int64_t r = r0 + rr;
          const int64_t c = (which ? p.h : 0) + c0 + jj * 32;
          if (r < p.M) {
            store32_codes(p.q_row + r * 2 * p.h + c, codes, p.v8_row);
            p.s_row.put(r, c >> 5, sc);
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
        for (int i = 0; i < 32; ++i) v[i] = *reinterpret_cast<const uint32_t*>(src + tile_word(rb * 32 + i, pc));
        uint32_t ca[8], cb[8], sa, sb;
        quant_col32x2(v, ca, cb, sa, sb, p.rceil);
        const int64_t rg = r0 + rb * 32;
        if (rg < p.M) {
          const int64_t orow = (which ? p.h : 0) + c0 + 2 * pc;
          uint8_t* dst = p.q_col + orow * p.M + rg;
          store32_codes(dst, ca, p.v8_col);
          store32_codes(dst + p.M, cb, p.v8_col);
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
            const uint32_t r0v = *reinterpret_cast<const uint32_t*>(src + tile_word(rb * 32 + 2 * i, pc));
            const uint32_t r1v = *reinterpret_cast<const uint32_t*>(src + tile_word(rb * 32 + 2 * i + 1, pc));
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
              for (int h2 = 0; h2 < 2; ++h2) {
                const uint32_t ua[8] = {wa[8 * h2], wa[8 * h2 + 1], wa[8 * h2 + 2], wa[8 * h2 + 3],
                                        wa[8 * h2 + 4], wa[8 * h2 + 5], wa[8 * h2 + 6], wa[8 * h2 + 7]};
                const uint32_t ub[8] = {wb[8 * h2], wb[8 * h2 + 1], wb[8 * h2 + 2], wb[8 * h2 + 3],
                                        wb[8 * h2 + 4], wb[8 * h2 + 5], wb[8 * h2 + 6], wb[8 * h2 + 7]};
                store32_codes(reinterpret_cast<uint8_t*>(da + h2 * 16), ua, p.v8_t);
                store32_codes(reinterpret_cast<uint8_t*>(db + h2 * 16), ub, p.v8_t);
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

// a(g) for every bf16 bit pattern, by the exact tiers (the same function
// the kernels fall back to for the elements their certificates leave open).
__global__ void silu_table_kernel(uint16_t* table) {
  const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < 65536u) table[b] = (uint16_t)swiglu_math::silu_bits_slow(__uint_as_float(b << 16));
}

// a device pointer and a row stride (bytes) that keep every 32-byte block 32-byte aligned
bool aligned32(const void* ptr, int64_t stride) {
  return ((reinterpret_cast<uintptr_t>(ptr) | (uintptr_t)stride) & 31) == 0;
}

}  // namespace

int launch_silu_table_init(uint16_t* table, cudaStream_t stream) {
  if (!table) return fail(MX_ERR_INVALID_ARG, "silu table: null destination");
  silu_table_kernel<<<256, 256, 0, stream>>>(table);
  return cuda_status(cudaGetLastError(), "silu_table_kernel launch");
}

int launch_swiglu_fwd(const SwigluLaunch& s, cudaStream_t stream) {
  CUtensorMap tm;
  uint64_t dims[2] = {(uint64_t)(2 * s.h), (uint64_t)s.M};
  uint64_t strides[1] = {(uint64_t)(2 * s.h * 2)};
  uint32_t box[2] = {SF_C, SF_R};
  int rc = make_tmap(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(s.h13), dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc) return rc;
  SwiFwdParams p{};
  p.M = s.M; p.h = s.h;
  p.row_tiles = (s.M + SF_R - 1) / SF_R;
  p.col_tiles = s.h / SF_C;
  const bool mma = s.layout == MX_SCALE_MMA;
  const int64_t Sr = s.h / 32, Sc = s.M / 32;
  p.q_row = (uint8_t*)s.q_row; p.s_row = ScaleDst{(uint8_t*)s.s_row, (Sr + 3) / 4, Sr, mma};
  p.q_col = (uint8_t*)s.q_col; p.s_col = ScaleDst{(uint8_t*)s.s_col, (Sc + 3) / 4, Sc, mma};
  p.rceil = s.floor_scale ? 0u : 1u;
  p.silu_a = s.silu_a;
  p.err = s.err;
  if (!p.silu_a) return fail(MX_ERR_INVALID_ARG, "swiglu forward: the a(g) table is required");
  p.v8_row = aligned32(s.q_row, s.h);
  p.v8_col = s.q_col && aligned32(s.q_col, s.M);
  const int64_t n_tiles = p.row_tiles * p.col_tiles;
  if (n_tiles == 0) return MX_OK;
  const int grid = (int)std::min<int64_t>(n_tiles, (int64_t)num_sms() * 2);
  cudaError_t e;
  if (s.q_col) {
    auto k = swiglu_fwd_kernel<true>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sf_smem(true));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, sf_carveout(true));
    if (e == cudaSuccess) {
      count_launch(MX_KERNEL_SWIGLU_FWD);
      k<<<grid, SF_THREADS, sf_smem(true), stream>>>(tm, p);
      e = cudaGetLastError();
    }
  } else {
    auto k = swiglu_fwd_kernel<false>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sf_smem(false));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, sf_carveout(false));
    if (e == cudaSuccess) {
      count_launch(MX_KERNEL_SWIGLU_FWD);
      k<<<grid, SF_THREADS, sf_smem(false), stream>>>(tm, p);
      e = cudaGetLastError();
    }
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
  p.rceil = s.floor_scale ? 0u : 1u;
  p.err = s.err;
  p.v8_row = aligned32(s.q_row, 2 * s.h);
  p.v8_col = s.q_col && aligned32(s.q_col, s.M);
  p.v8_t = (!s.dh13_t || aligned32(s.dh13_t, 2 * s.M)) && (!s.y_t || aligned32(s.y_t, 2 * s.M));
  const int64_t n_tiles = p.row_tiles * p.col_tiles;
  if (n_tiles == 0) return MX_OK;
  const int grid = (int)std::min<int64_t>(n_tiles, (int64_t)num_sms() * 2);
  const int mode = s.q_col ? 1 : ((s.dh13_t || s.y_t) ? 2 : 0);
  cudaError_t e;
#define MX_LAUNCH_B(MODE)                                                                       \
  do {                                                                                          \
    auto k = swiglu_bwd_kernel<MODE>;                                                           \
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SB_SMEM);     \
    if (e == cudaSuccess) { count_launch(MX_KERNEL_SWIGLU_BWD); k<<<grid, THREADS, SB_SMEM, stream>>>(tdy, th, p); e = cudaGetLastError(); } \
  } while (0)
  if (mode == 0) MX_LAUNCH_B(0);
  else if (mode == 1) MX_LAUNCH_B(1);
  else MX_LAUNCH_B(2);
#undef MX_LAUNCH_B
  return cuda_status(e, "swiglu_bwd_kernel launch");
}

}  // namespace mx
