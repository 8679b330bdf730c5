// gemm.cu - block-scaled MXFP8 and bf16 GEMMs on the tcgen05 tensor cores.
//
//   C[m, n] = sum_k A[m, k] * B[n, k]     (both operands K-major, fp32
//                                         accumulation in TMEM, bf16 output)
//
// One persistent CTA per SM, warp-specialised:
//   warp 0      TMA producer: A/B tiles (128-byte swizzle) and, for MXFP8,
//               the 512-byte scale tiles (already in the MMA layout in
//               global memory, so a plain bulk copy moves them)
//   warp 1      TMEM allocation + single-thread MMA issue: per 128-element
//               K step it copies the scale tiles into TMEM (tcgen05.cp) and
//               issues 4 x tcgen05.mma (K = 32 for E4M3, 16 x 4 for bf16)
//   warps 2-9   epilogue (two warps per TMEM lane quarter, half of the
//               columns each): tcgen05.ld of the fp32 accumulator, RN to
//               bf16, 64-byte-swizzled staging in shared memory, TMA store
// Modes: dense; M-grouped (forward / input gradient: token rows of group e
// use expert e's weights, rows past the last group are zero); K-grouped
// (weight gradient: expert e contracts over its own token range; an empty
// group writes zeros).  Group offsets are read on the device.
#include "common.cuh"
#include "kernels.h"
#include "swiglu_math.cuh"
#include "tile_quant.cuh"

namespace mx {

namespace {

constexpr int BM = 128;
constexpr int EPI_WARPS = 8;  // two per TMEM lane quarter, each draining half of the columns
constexpr int GEMM_THREADS = 64 + EPI_WARPS * 32;
constexpr int MAX_GROUPS = 1024;

// SUB: 128-row sub-tiles per tile sharing each B stage (2 only for bf16, whose
// two 128x256 fp32 accumulators then fill TMEM; MXFP8 needs TMEM columns for
// its scales).  CL = 2: CTA pairs, each CTA holding its 128 rows of A and
// half of the B rows, the MMA (M = 256) issued by the even CTA.
// KA: 128-byte K atoms per stage (2 only for MXFP8 on one CTA: eight MMAs
// per stage instead of four, because a stage's fixed latency is what limits
// the four-MMA pipeline; two stages of 99 KB then fill shared memory).
// TW: E4M3 operands without block scales (FP8 per-tensor recipe): no scale
// tiles, kind::f8f6f4 MMAs, and the TMEM the scales would take holds a
// second accumulator, so a tile's epilogue overlaps the next tile's MMAs.
template <bool MX, int BN, int SUB = 1, int CL = 1, int KA = 1, bool TW = false>
struct Cfg {
  static_assert(SUB == 1 || (!MX && BN == 256), "two sub-tiles only for the bf16 kernel");
  static_assert(CL == 1 || SUB == 1, "CTA pairs only with single sub-tiles");
  static_assert(KA == 1 || (MX && CL == 1 && SUB == 1 && BN == 256), "two K atoms only for the MXFP8 1-CTA tile");
  static constexpr int TM = SUB * BM;                      // tile rows
  static constexpr int BK = KA * (MX ? 128 : 64);          // elements per stage (KA x 128 bytes of K)
  static constexpr int ATOM_A = TM * 128;                  // one 128-byte K atom of the A tile
  static constexpr int ATOM_B = (BN / CL) * 128;
  static constexpr int A_BYTES = KA * ATOM_A;
  static constexpr int B_BYTES = KA * ATOM_B;               // this CTA's rows of the B tile
  static_assert(!TW || (MX && KA == 1 && SUB == 1), "FP8 per-tensor: E4M3 operands, one K atom");
  static constexpr bool BS = MX && !TW;                     // block-scaled MXFP8
  static constexpr int SFA_BYTES = BS ? KA * 512 : 0;      // one scale tile of A per atom
  static constexpr int SFB_BYTES = BS ? KA * (BN / 128) * 512 : 0;  // all of the tile's B scales
  static constexpr int STAGES = KA == 2 ? 2 : CL == 2 ? 6 : SUB == 2 ? 3 : (BN == 256 ? 4 : 6);
  static constexpr int STAGE_TX = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;  // bytes one CTA loads
  static constexpr int NUM_ACC = (TW || !(BN == 256 || SUB == 2)) ? 2 : 1;
  static constexpr int EPI_BYTES = EPI_WARPS * 32 * 64;    // one 32x32 bf16 buffer per warp
  static constexpr int TMEM_COLS = 512;
  static constexpr int SF_COL = NUM_ACC * BN;               // per-stage scale slots from here
  static constexpr int SF_ATOM = 4 + 4 * (BN / 128);       // TMEM columns of one atom's scales
  static constexpr int SF_SLOT = KA * SF_ATOM;               // TMEM columns of one stage's scales
  static constexpr size_t SMEM = (size_t)STAGES * (A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES) + EPI_BYTES +
                                 MAX_GROUPS * 4 * (CL == 1 ? 2 : 1) + 1024 /*align*/ + 256 /*barriers*/;
  // instruction descriptors: block-scaled (E8M0 scales, fp32 D implied);
  // kind::f8f6f4 with fp32 D (bits 4-5 = 1) and E4M3 A and B (type 0);
  // kind::f16 with fp32 D and bf16 A and B (type 1)
  static constexpr uint32_t IDESC =
      BS ? ((1u << 23) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((CL * BM) >> 4) << 24))
         : TW ? ((1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)((CL * BM) >> 4) << 24))
              : ((1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                 ((uint32_t)((CL * BM) >> 4) << 24));
};

struct GemmParams {
  int mode;
  int64_t M, N, K;            // K: contraction length of A (GROUP_K: total tokens)
  int64_t m_tiles, n_tiles, tiles;  // tiles: work units (tiles, or tile pairs with clusters)
  int64_t m_pairs;            // ceil(m_tiles / 2)
  int32_t E;
  const int32_t* offs;
  const uint8_t* sfa;         // MMA-layout scales of A ([M, K/32])
  const uint8_t* sfb;         // MMA-layout scales of B ([N, K/32] or per expert)
  int64_t sfb_expert_stride;  // bytes between experts (GROUP_M)
  int64_t split;              // row split of C between tmC0 / tmC1 (0: none)
  int64_t msub;               // GROUP_K: rows per expert in the output maps
  int64_t band;               // DENSE: tile rows per band of the tile order
  int32_t cols_fast;          // DENSE: columns fastest (B re-read from L2, A streamed once)
  // fused SwiGLU epilogue (the w13 GEMM of the MLP forward): tile n covers
  // hidden units [128n, 128n+128) of g (accumulator columns 0-127) and of u
  // (128-255); C (h13) is stored and y = SwiGLU(h13) quantized by rows
  // and, when yqc is set, by columns (32-row blocks of the tile)
  uint8_t* yq;                // [M, hy] codes
  ScaleDst ys;                // [M, hy/32] scales
  uint8_t* yqc;               // [hy, M] columnwise codes, or NULL
  ScaleDst ysc;               // [hy, M/32] columnwise scales
  int64_t hy;                 // h
  uint32_t rceil;             // 1: RCEIL scales, 0: FLOOR
  int32_t v8_y;               // yq rows 32-byte aligned: one 256-bit store per 32 codes
  const uint16_t* silu_a;     // a(g) = RN_bf16(g sigma(g)) indexed by the bits of bf16 g
  // FP8 per-tensor recipe: amax of A (one) and of B (one, or one per expert
  // when amax_b_per_expert); C = acc * (1/s_a) * (1/s_b), s = 448 / amax
  const float* amax_a;
  const float* amax_b;
  int32_t amax_b_per_expert;
  int32_t starve;             // self-test only: the producer issues nothing, so waits expire
  int32_t* err;
};

MX_DEVINL void store32g(uint8_t* dst, const uint32_t (&c)[8]) {
  store16(dst, c[0], c[1], c[2], c[3]);
  store16(dst + 16, c[4], c[5], c[6], c[7]);
}

struct TileInfo {
  int64_t m_blk, n_blk;
  int32_t e;       // expert (GROUP_M / GROUP_K), 0 for dense
  int64_t k0;      // first contraction element
  int32_t num_kb;  // number of BK steps (0: write zeros)
  bool store;      // false: a pair's filler tile (computed, never stored)
};

// Group data in shared memory; ok == false if the offsets break the contract.
//   ends[e]     cumulative group ends (CL == 1, and GROUP_K with clusters)
//   pair_end[e] cumulative work units (tile pairs x tile columns) of groups
//               0..e (GROUP_M with clusters; the offsets themselves are then
//               read from global)
struct Groups {
  const int32_t* ends;
  const int32_t* pair_end;
  const int32_t* unit_end;  // GROUP_M without clusters: work units of groups 0..e
  int32_t E;
  int64_t tail_pairs;   // GROUP_M with clusters: tile pairs past the last group
  bool ok;
};

// Work unit -> the tile this CTA (cluster rank `rank`) computes.  Without
// clusters a unit is one tile.  With 2-CTA clusters a unit is a pair of
// vertically adjacent tiles that one pair MMA (M = 256) computes together:
// each CTA loads its own 128 rows of A and half of the B tile's rows, both
// with the same expert and the same K range; a group with an odd number of 128-row tiles pads its
// last pair with a filler tile that is computed but not stored.
template <int BK, int CL>
MX_DEVINL TileInfo tile_info(const GemmParams& p, const Groups& g, int64_t u, int rank) {
  TileInfo ti{};
  ti.store = true;
  if (p.mode == GEMM_GROUP_K) {
    const int64_t mt = CL == 2 ? p.m_pairs : p.m_tiles;
    const int64_t per_e = mt * p.n_tiles;
    const int64_t e = u / per_e;
    const int64_t rem = u - e * per_e;
    ti.e = (int32_t)e;
    if (CL == 1 && p.M > p.N) {
      // columns fastest: the smaller operand (B, N x tokens) is the one
      // re-read for every row of tiles and stays in L2; A streams once
      ti.m_blk = rem / p.n_tiles;
      ti.n_blk = rem % p.n_tiles;
    } else {
      ti.m_blk = CL == 2 ? 2 * (rem % mt) + rank : rem % mt;
      ti.n_blk = rem / mt;
    }
    ti.store = ti.m_blk < p.m_tiles;
    const int64_t s = e == 0 ? 0 : g.ends[e - 1];
    const int64_t en = g.ends[e];
    ti.k0 = s;
    ti.num_kb = g.ok ? (int32_t)((en - s) / BK) : 0;
    return ti;
  }
  ti.k0 = 0;
  ti.num_kb = (int32_t)(p.K / BK);
  ti.e = 0;
  if (CL == 1) {
    if (p.mode == GEMM_GROUP_M) {
      // Expert-major: every tile of group e (its 128-row tiles x all tile
      // columns, rows fastest) before group e+1, so that each group's rows and
      // its expert's weights come from DRAM once; the rows past the last
      // group follow as zero tiles.
      if (!g.ok || g.E == 0) {  // invalid offsets: zeros everywhere
        ti.m_blk = u % p.m_tiles;
        ti.n_blk = u / p.m_tiles;
        ti.num_kb = 0;
        return ti;
      }
      const int64_t grouped = g.unit_end[g.E - 1];
      if (u >= grouped) {
        const int64_t first = g.ends[g.E - 1] / BM;
        const int64_t tt = p.m_tiles - first;
        const int64_t r = u - grouped;
        ti.n_blk = r / tt;
        ti.m_blk = first + r % tt;
        ti.num_kb = 0;
        return ti;
      }
      int lo = 0, hi = g.E - 1;  // first group whose unit_end is > u
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (g.unit_end[mid] > u) hi = mid; else lo = mid + 1;
      }
      const int64_t start = lo == 0 ? 0 : g.ends[lo - 1];
      const int64_t tiles_e = (g.ends[lo] - start) / BM;
      const int64_t r = u - (lo == 0 ? 0 : g.unit_end[lo - 1]);
      ti.e = lo;
      if (tiles_e * BM <= p.N) {  // the group's rows are the smaller operand: re-read them
        ti.n_blk = r / tiles_e;
        ti.m_blk = start / BM + r % tiles_e;
      } else {                    // the expert's weights are smaller: columns fastest
        ti.m_blk = start / BM + r / p.n_tiles;
        ti.n_blk = r % p.n_tiles;
      }
      return ti;
    }
    if (p.cols_fast) {  // dense, B the smaller operand: columns fastest
      ti.m_blk = u / p.n_tiles;
      ti.n_blk = u % p.n_tiles;
      return ti;
    }
    // dense: bands of p.band tile rows (sized so that a band of A stays in
    // L2), rows fastest within a band
    const int64_t per_band = p.band * p.n_tiles;
    const int64_t b = u / per_band, r = u - b * per_band;
    const int64_t bm = p.m_tiles - b * p.band < p.band ? p.m_tiles - b * p.band : p.band;
    ti.n_blk = r / bm;
    ti.m_blk = b * p.band + r % bm;
    return ti;
  }
  if (p.mode == GEMM_DENSE) {
    // as for single CTAs, in units of tile-row pairs: columns fastest when B
    // is the smaller operand and stays in L2, otherwise bands of pair rows
    int64_t mp;
    if (p.cols_fast) {
      mp = u / p.n_tiles;
      ti.n_blk = u % p.n_tiles;
    } else {
      const int64_t pb = p.band >= p.m_tiles ? p.m_pairs : (p.band / 2 > 0 ? p.band / 2 : 1);
      const int64_t per_band = pb * p.n_tiles;
      const int64_t b = u / per_band, r = u - b * per_band;
      const int64_t bm = p.m_pairs - b * pb < pb ? p.m_pairs - b * pb : pb;
      ti.n_blk = r / bm;
      mp = b * pb + r % bm;
    }
    ti.m_blk = 2 * mp + rank;
    ti.store = ti.m_blk < p.m_tiles;
    return ti;
  }
  // GROUP_M with clusters, expert-major like the single-CTA form: all tile
  // pairs of group e (rows fastest if its rows are the smaller operand, else
  // columns fastest) before group e+1, then the tail pairs as zero tiles
  const int64_t grouped = g.ok ? g.pair_end[g.E - 1] : 0;
  if (u >= grouped) {
    const int64_t first = g.ok ? (int64_t)p.offs[g.E - 1] / BM : 0;
    const int64_t r = u - grouped;
    ti.n_blk = r / g.tail_pairs;
    ti.m_blk = first + 2 * (r % g.tail_pairs) + rank;
    ti.num_kb = 0;
    ti.store = ti.m_blk < p.m_tiles;
    return ti;
  }
  int lo = 0, hi = g.E - 1;  // first group whose pair_end is > u
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (g.pair_end[mid] > u) hi = mid; else lo = mid + 1;
  }
  const int64_t r = u - (lo == 0 ? 0 : g.pair_end[lo - 1]);
  const int64_t start = lo == 0 ? 0 : (int64_t)p.offs[lo - 1];
  const int64_t mb = ((int64_t)p.offs[lo] - start) / BM;  // tiles of the group
  const int64_t pe = (mb + 1) / 2;                         // tile pairs of the group
  int64_t pi;
  if (mb * BM <= p.N) {
    ti.n_blk = r / pe;
    pi = r % pe;
  } else {
    pi = r / p.n_tiles;
    ti.n_blk = r % p.n_tiles;
  }
  ti.e = lo;
  ti.m_blk = start / BM + 2 * pi + rank;
  ti.store = 2 * pi + rank < mb;
  return ti;
}

// Dequantization factor of an FP8 per-tensor operand: 1 / s with
// s = RN_f32(448 / max(amax, 2^-40)).
MX_DEVINL float tw_inv_scale(float amax) {
  return __frcp_rn(__fdiv_rn(448.0f, fmaxf(amax, 0x1p-40f)));
}

template <bool MX, int BN, int CL, int SUB, bool FUSE, int KA, bool TW>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC0, const __grid_constant__ CUtensorMap tmC1,
                const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                GemmParams p) {
  using C = Cfg<MX, BN, SUB, CL, KA, TW>;
  static_assert(!FUSE || (MX && !TW && SUB == 1 && BN == 256), "fused SwiGLU: MXFP8, 128x256 tiles per CTA");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + C::STAGES * C::A_BYTES;
  uint8_t* sEpi = sB + C::STAGES * C::B_BYTES;
  uint8_t* sSFA = sEpi + C::EPI_BYTES;                       // [STAGES][512]
  uint8_t* sSFB = sSFA + C::STAGES * C::SFA_BYTES;            // [STAGES][BN/128][512]
  int32_t* sGroups = reinterpret_cast<int32_t*>(sSFB + C::STAGES * C::SFB_BYTES);
  int32_t* sUnitEnd = sGroups + MAX_GROUPS;  // CL == 1 only
  uint64_t* full = reinterpret_cast<uint64_t*>(sGroups + MAX_GROUPS * (CL == 1 ? 2 : 1));
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + C::NUM_ACC;
  uint64_t* done_bar = acc_empty + C::NUM_ACC;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done_bar + 1);
  __shared__ int s_groups_ok;
  __shared__ long long s_tail_pairs, s_pair_units;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = CL == 2 ? (int)cluster_ctarank() : 0;
  const int64_t unit0 = CL == 2 ? blockIdx.x / 2 : blockIdx.x;
  const int64_t ustep = CL == 2 ? gridDim.x / 2 : gridDim.x;
  const bool pairs_m = CL == 2 && p.mode == GEMM_GROUP_M;

  // ---- setup: barriers, group data, TMEM
  if (threadIdx.x == 0) {
    // with CTA pairs the even CTA's full and acc_empty barriers serve both
    for (int s = 0; s < C::STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < C::NUM_ACC; ++a) { mbar_init(&acc_full[a], 1); mbar_init(&acc_empty[a], CL * EPI_WARPS); }
    mbar_init(done_bar, 1);
    fence_mbar_init();
    s_groups_ok = 1;
  }
  __syncthreads();
  if (p.mode != GEMM_DENSE) {
    const int64_t limit = p.mode == GEMM_GROUP_M ? p.M : p.K;
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
      const int32_t v = p.offs[e];
      const int32_t prev = e == 0 ? 0 : p.offs[e - 1];
      if (!pairs_m) sGroups[e] = v;
      if (v < prev || (v & 127) != 0 || (int64_t)v > limit) s_groups_ok = 0;
    }
  }
  __syncthreads();
  if (CL == 1 && p.mode == GEMM_GROUP_M && threadIdx.x == 0 && s_groups_ok) {
    int64_t acc = 0;
    int32_t prev = 0;
    for (int e = 0; e < p.E; ++e) {
      const int32_t v = sGroups[e];
      acc += (int64_t)((v - prev) / BM) * p.n_tiles;
      sUnitEnd[e] = (int32_t)acc;
      prev = v;
    }
  }
  if (pairs_m && threadIdx.x == 0) {
    int64_t acc = 0;
    int32_t prev = 0;
    if (s_groups_ok) {
      for (int e = 0; e < p.E; ++e) {
        const int32_t v = p.offs[e];
        acc += ((v - prev) / BM + 1) / 2 * p.n_tiles;
        sGroups[e] = (int32_t)acc;
        prev = v;
      }
    }
    const int64_t tail = p.m_tiles - prev / BM;  // every tile, for invalid offsets
    s_tail_pairs = (tail + 1) / 2;
    s_pair_units = acc + s_tail_pairs * p.n_tiles;
  }
  if (warp == 1) {
    if (CL == 2) { tmem_alloc_pair(tmem_holder, C::TMEM_COLS); tmem_relinquish_pair(); }
    else { tmem_alloc(tmem_holder, C::TMEM_COLS); tmem_relinquish(); }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (CL == 2) cluster_sync();  // the peer's barriers exist before any remote arrive or pair copy
  const uint32_t tmem = *tmem_holder;
  Groups grp{sGroups, sGroups, sUnitEnd, p.E, pairs_m ? s_tail_pairs : 0, s_groups_ok != 0};
  if (!grp.ok && threadIdx.x == 0 && blockIdx.x == 0) record_error(p.err, MX_ERR_BAD_OFFSETS);
  const int64_t n_units = pairs_m ? s_pair_units : p.tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // as the MMA issuer: the warp runs the loop, one elected lane issues
    if (!p.starve) {
      const bool leader = elect_one();
      if (leader) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (C::BS) prefetch_tmap(&tmSFB);
        if (C::BS && CL == 2) prefetch_tmap(&tmSFA);
      }
      int stage = 0; uint32_t phase = 0;
      const int64_t sfa_row_tiles = p.K / 128;  // scale tiles per 128-row block of A
      for (int64_t u = unit0; u < n_units; u += ustep) {
        const TileInfo ti = tile_info<C::BK, CL>(p, grp, u, rank);
        bool ok = true;
        for (int kb = 0; kb < ti.num_kb; ++kb) {
          if (!warp_wait(&empty[stage], phase ^ 1, p.err)) { ok = false; break; }
          const int64_t k = ti.k0 + (int64_t)kb * C::BK;
          const int64_t kt = k / 128;
          if (CL == 2 && leader) {
            // both CTAs' copies complete on the even CTA's barrier, which
            // expects the bytes of the pair; a filler tile's rows and scales
            // past the end read as zeros
            const uint32_t bar = cluster_map(smem_u32(&full[stage]), 0);
            if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_TX);
            tma_load_2d_pair(sA + stage * C::A_BYTES, &tmA, (int32_t)k, (int32_t)(ti.m_blk * BM), bar);
            const int32_t nrow = (int32_t)(ti.n_blk * BN + rank * (BN / 2));
            if (FUSE) {
              // the even CTA loads rows 128n.. of w1 (g, accumulator columns
              // 0-127), the odd CTA the same rows of w3 (u, columns 128-255)
              if (p.mode == GEMM_GROUP_M)
                tma_load_4d_pair(sB + stage * C::B_BYTES, &tmB, (int32_t)k, (int32_t)(ti.n_blk * 128), rank, ti.e,
                                 bar);
              else
                tma_load_3d_pair(sB + stage * C::B_BYTES, &tmB, (int32_t)k, (int32_t)(ti.n_blk * 128), rank, bar);
            } else if (p.mode == GEMM_GROUP_M)
              tma_load_3d_pair(sB + stage * C::B_BYTES, &tmB, (int32_t)k, nrow, ti.e, bar);
            else
              tma_load_2d_pair(sB + stage * C::B_BYTES, &tmB, (int32_t)k, nrow, bar);
            if (C::BS) {
              tma_load_2d_pair(sSFA + stage * C::SFA_BYTES, &tmSFA, 0, (int32_t)(ti.m_blk * sfa_row_tiles + kt),
                               bar);
              if (FUSE && p.mode == GEMM_GROUP_M)  // both halves' scale tiles: a full copy per CTA
                tma_load_5d_pair(sSFB + stage * C::SFB_BYTES, &tmSFB, 0, (int32_t)kt, (int32_t)ti.n_blk, 0, ti.e,
                                 bar);
              else if (FUSE)
                tma_load_4d_pair(sSFB + stage * C::SFB_BYTES, &tmSFB, 0, (int32_t)kt, (int32_t)ti.n_blk, 0, bar);
              else if (p.mode == GEMM_GROUP_M)
                tma_load_4d_pair(sSFB + stage * C::SFB_BYTES, &tmSFB, 0, (int32_t)kt, (int32_t)(ti.n_blk * (BN / 128)),
                                 ti.e, bar);
              else
                tma_load_3d_pair(sSFB + stage * C::SFB_BYTES, &tmSFB, 0, (int32_t)kt, (int32_t)(ti.n_blk * (BN / 128)),
                                 bar);
            }
          } else if (CL == 1 && leader) {
            const uint32_t bytes =
                C::A_BYTES + C::B_BYTES + (C::BS ? (ti.store ? C::SFA_BYTES : 0) + C::SFB_BYTES : 0);
            mbar_arrive_expect_tx(&full[stage], bytes);
#pragma unroll
            for (int at = 0; at < KA; ++at) {
              const int32_t ka = (int32_t)(k + at * 128);
              uint8_t* dA = sA + stage * C::A_BYTES + at * C::ATOM_A;
              uint8_t* dB = sB + stage * C::B_BYTES + at * C::ATOM_B;
              tma_load_2d(dA, &tmA, ka, (int32_t)(ti.m_blk * C::TM), &full[stage]);
              if (FUSE) {  // rows 128n.. of w1 and of w3 in one copy ([2][128] rows)
                if (p.mode == GEMM_GROUP_M)
                  tma_load_4d(dB, &tmB, ka, (int32_t)(ti.n_blk * 128), 0, ti.e, &full[stage]);
                else
                  tma_load_3d(dB, &tmB, ka, (int32_t)(ti.n_blk * 128), 0, &full[stage]);
              } else if (p.mode == GEMM_GROUP_M)
                tma_load_3d(dB, &tmB, ka, (int32_t)(ti.n_blk * BN), ti.e, &full[stage]);
              else
                tma_load_2d(dB, &tmB, ka, (int32_t)(ti.n_blk * BN), &full[stage]);
            }
            if (C::BS) {
              // the KA scale tiles of A are adjacent; B's come in one box of
              // [tile rows][KA atoms][512 B]
              if (ti.store)
                bulk_load(sSFA + stage * C::SFA_BYTES, p.sfa + (ti.m_blk * sfa_row_tiles + kt) * 512, C::SFA_BYTES,
                          &full[stage]);
              // all of the tile's B scale tiles (BN/128 tile rows) in one copy;
              // rows past N are zero-filled and counted
              if (FUSE && p.mode == GEMM_GROUP_M)
                tma_load_5d(sSFB + stage * C::SFB_BYTES, &tmSFB, 0, (int32_t)kt, (int32_t)ti.n_blk, 0, ti.e,
                            &full[stage]);
              else if (FUSE)
                tma_load_4d(sSFB + stage * C::SFB_BYTES, &tmSFB, 0, (int32_t)kt, (int32_t)ti.n_blk, 0, &full[stage]);
              else if (p.mode == GEMM_GROUP_M)
                tma_load_4d(sSFB + stage * C::SFB_BYTES, &tmSFB, 0, (int32_t)kt, (int32_t)(ti.n_blk * (BN / 128)), ti.e,
                            &full[stage]);
              else
                tma_load_3d(sSFB + stage * C::SFB_BYTES, &tmSFB, 0, (int32_t)kt, (int32_t)(ti.n_blk * (BN / 128)),
                            &full[stage]);
            }
          }  // elected lane
          __syncwarp();
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (warp-uniform control flow, so the
    // descriptors and TMEM addresses stay in uniform registers) and one
    // elected lane issues the tcgen05 instructions; a lane-0-only loop costs
    // about 70 cycles per tcgen05 instruction, which starves the tensor pipe.
    // Descriptors are formed once and advanced by adding the byte offset
    // (>> 4) to their start-address field.  With CTA pairs only the even CTA
    // issues; its MMAs and scale copies act on both CTAs.
    if (rank == 0) {
      const bool leader = elect_one();
      const uint64_t a_desc0 = smem_desc(smem_u32(sA), 16, 1024, 2);
      const uint64_t b_desc0 = smem_desc(smem_u32(sB), 16, 1024, 2);
      const uint64_t sfa_desc0 = smem_desc(smem_u32(sSFA), 128, 128, 0);
      const uint64_t sfb_desc0 = smem_desc(smem_u32(sSFB), 128, 128, 0);
      int stage = 0; uint32_t phase = 0;
      int acc = 0; uint32_t acc_phase = 0;
      bool ok = true;
      for (int64_t u = unit0; u < n_units && ok; u += ustep) {
        const TileInfo ti = tile_info<C::BK, CL>(p, grp, u, rank);
        if (ti.num_kb == 0) continue;
        if (!warp_wait(&acc_empty[acc], acc_phase ^ 1, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
        for (int kb = 0; kb < ti.num_kb; ++kb) {
          if (!warp_wait(&full[stage], phase, p.err)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int at = 0; at < KA; ++at) {
            const uint32_t sf_col = tmem + C::SF_COL + stage * C::SF_SLOT + at * C::SF_ATOM;
            if (C::BS && leader) {
              const uint64_t sfa = sfa_desc0 + (uint64_t)((stage * C::SFA_BYTES + at * 512) >> 4);
              if (CL == 2) tmem_cp_32x128b_x4_pair(sf_col, sfa);
              else tmem_cp_32x128b_x4(sf_col, sfa);
#pragma unroll
              for (int j = 0; j < BN / 128; ++j) {
                const uint64_t sfb = sfb_desc0 + (uint64_t)((stage * C::SFB_BYTES + (j * KA + at) * 512) >> 4);
                if (CL == 2) tmem_cp_32x128b_x4_pair(sf_col + 4 + 4 * j, sfb);
                else tmem_cp_32x128b_x4(sf_col + 4 + 4 * j, sfb);
              }
            }
            const uint64_t ad = a_desc0 + (uint64_t)((stage * C::A_BYTES + at * C::ATOM_A) >> 4);
            const uint64_t bd = b_desc0 + (uint64_t)((stage * C::B_BYTES + at * C::ATOM_B) >> 4);
#pragma unroll
            for (int sub = 0; sub < SUB; ++sub) {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint32_t accum = (kb > 0 || at > 0 || k > 0) ? 1u : 0u;
                const uint64_t a = ad + (uint64_t)((sub * BM * 128) >> 4) + 2 * k;
                const uint32_t sf_ids = ((uint32_t)k << 4) | ((uint32_t)k << 29);
                if (!leader) continue;
                if (TW && CL == 2)
                  mma_f8_pair(d_tmem, a, bd + 2 * k, C::IDESC, accum);
                else if (TW)
                  mma_f8(d_tmem, a, bd + 2 * k, C::IDESC, accum);
                else if (MX && CL == 2)
                  mma_mxf8_pair(d_tmem, a, bd + 2 * k, C::IDESC | sf_ids, sf_col, sf_col + 4, accum);
                else if (MX)
                  mma_mxf8(d_tmem, a, bd + 2 * k, C::IDESC | sf_ids, sf_col, sf_col + 4, accum);
                else if (CL == 2)
                  mma_bf16_pair(d_tmem, a, bd + 2 * k, C::IDESC, accum);
                else
                  mma_bf16(d_tmem + (uint32_t)(sub * BN), a, bd + 2 * k, C::IDESC, accum);
              }
            }
          }  // K atoms of the stage
          // the stage is free (in both CTAs of a pair) once these MMAs are done
          if (leader) {
            if (CL == 2) tc_commit_pair_mc(&empty[stage], (uint16_t)0x3);
            else tc_commit(&empty[stage]);
          }
          __syncwarp();
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if (leader) {
          if (CL == 2) tc_commit_pair_mc(&acc_full[acc], (uint16_t)0x3);
          else tc_commit(&acc_full[acc]);
        }
        __syncwarp();
        if (++acc == C::NUM_ACC) { acc = 0; acc_phase ^= 1; }
      }
      // all issued MMAs complete before TMEM is released
      if (leader) {
        if (CL == 2) tc_commit_pair_mc(done_bar, (uint16_t)0x1);
        else tc_commit(done_bar);
      }
      __syncwarp();
      mbar_wait(done_bar, 0, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // warp -> TMEM lane quarter q (rows 32q..32q+31 of the tile) and column
    // half; 32-column chunks staged with the 64-byte swizzle and TMA-stored
    const int ew = warp - 2;
    const int q = warp & 3;
    const int half = ew >> 2;
    uint8_t* stg = sEpi + ew * (32 * 64);
    int acc = 0; uint32_t acc_phase = 0;
    // accumulator drained: arrive on the barrier of the CTA whose thread issues the MMAs
    auto release_acc = [&](int a) {
      if (CL == 2 && rank != 0) mbar_arrive_cluster(cluster_map(smem_u32(&acc_empty[a]), 0));
      else mbar_arrive(&acc_empty[a]);
    };
    for (int64_t u = unit0; u < n_units; u += ustep) {
      const TileInfo ti = tile_info<C::BK, CL>(p, grp, u, rank);
      const int64_t ncol0 = ti.n_blk * BN + half * (BN / 2);
      const int64_t cleft = (p.N - ncol0 + 31) / 32;
      const int nchunks = (int)(cleft < BN / 64 ? (cleft > 0 ? cleft : 0) : BN / 64);
      // output rows of this warp in sub-tile `sub`, and the map they go to
      auto out_rows = [&](int sub, const CUtensorMap*& tmC) {
        int64_t mrow = ti.m_blk * C::TM + sub * BM + q * 32;
        tmC = &tmC0;
        if (p.split > 0 && mrow >= p.split) { tmC = &tmC1; mrow -= p.split; }
        if (p.mode == GEMM_GROUP_K) mrow += (int64_t)ti.e * p.msub;
        return mrow;
      };
      // stage one 32x32 chunk of bf16 words (one row per lane) with the 64-byte
      // swizzle and TMA-store it
      auto store_chunk = [&](const uint32_t (&w)[16], const CUtensorMap* tmC, int64_t col, int64_t mrow) {
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        uint8_t* row = stg + lane * 64;
        const int sw = (lane >> 1) & 3;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(row + ((j ^ sw) * 16)) =
              make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(tmC, stg, (int32_t)col, (int32_t)mrow);
          bulk_commit();
        }
      };
      // FP8 per-tensor: the fp32 accumulator times (1/s_a)(1/s_b), then RN bf16
      float tfac = 1.0f;
      if constexpr (TW)
        tfac = __fmul_rn(tw_inv_scale(p.amax_a[0]), tw_inv_scale(p.amax_b[p.amax_b_per_expert ? ti.e : 0]));
      auto pack = [tfac](const uint32_t (&r)[32], uint32_t (&w)[16]) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if constexpr (TW) {
            w[i] = f2_to_bf16x2(f2_mul(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])),
                                       f2_splat(tfac)));
          } else {
            const __nv_bfloat162 b2 =
                __floats2bfloat162_rn(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
            w[i] = *reinterpret_cast<const uint32_t*>(&b2);
          }
        }
      };
      if (ti.num_kb == 0) {
        if (!ti.store) continue;
        if (FUSE) {  // rows with no group: y codes and scales are zero too
          const int64_t ycol = ti.n_blk * 128 + half * 64;
          const int64_t row = ti.m_blk * BM + q * 32 + lane;
          const uint32_t z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
          store32g(p.yq + row * p.hy + ycol, z);
          store32g(p.yq + row * p.hy + ycol + 32, z);
          p.ys.put(row, ycol >> 5, 0);
          p.ys.put(row, (ycol >> 5) + 1, 0);
          if (p.yqc) {  // columns ycol + 2 lane, +1: one 32-row block each
            const int64_t r0 = ti.m_blk * BM + q * 32;
            const int64_t c = ycol + 2 * lane;
            store32g(p.yqc + c * p.M + r0, z);
            store32g(p.yqc + (c + 1) * p.M + r0, z);
            p.ysc.put(c, r0 >> 5, 0);
            p.ysc.put(c + 1, r0 >> 5, 0);
          }
        }
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        uint4* row = reinterpret_cast<uint4*>(stg + lane * 64);
#pragma unroll
        for (int j = 0; j < 4; ++j) row[j] = make_uint4(0, 0, 0, 0);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (int sub = 0; sub < SUB; ++sub) {
            if (ti.m_blk * C::TM + sub * BM >= p.M) break;  // sub-tile past the last row
            const CUtensorMap* tmC;
            const int64_t mrow = out_rows(sub, tmC);
            for (int c = 0; c < nchunks; ++c) tma_store_2d(tmC, stg, (int32_t)(ncol0 + 32 * c), (int32_t)mrow);
          }
          bulk_commit();
        }
        continue;
      }
      if (!mbar_wait(&acc_full[acc], acc_phase, p.err)) break;
      tc_fence_after();
      if (!ti.store) {  // filler tile: release the accumulator unread
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release_acc(acc);
        if (++acc == C::NUM_ACC) { acc = 0; acc_phase ^= 1; }
        continue;
      }
      if constexpr (FUSE) {
        // this warp: rows 32q.. of the tile, hidden units ycol..ycol+63;
        // g in accumulator columns 64*half.., u in 128 + 64*half..
        const int64_t ycol = ti.n_blk * 128 + half * 64;
        const int64_t mrow = ti.m_blk * BM + q * 32;
        const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * 64);
        uint32_t gw[2][16], uw[2][16];   // RN bf16 pairs: the stored h13 values
        {
          uint32_t r0[32], r1[32];
          tmem_ld_32cols(tb, r0);
          tmem_ld_32cols(tb + 32, r1);
          tmem_ld_wait();
          pack(r0, gw[0]);
          pack(r1, gw[1]);
          tmem_ld_32cols(tb + 128, r0);
          tmem_ld_32cols(tb + 160, r1);
          tmem_ld_wait();
          pack(r0, uw[0]);
          pack(r1, uw[1]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release_acc(acc);
        store_chunk(gw[0], &tmC0, ycol, mrow);
        store_chunk(gw[1], &tmC0, ycol + 32, mrow);
        store_chunk(uw[0], &tmC0, p.hy + ycol, mrow);
        store_chunk(uw[1], &tmC0, p.hy + ycol + 32, mrow);
        // y = SwiGLU(g, u) of this thread's row: a(g) = RN_bf16(g sigma(g))
        // from the table of exact values over every bf16 g, then y =
        // RN_bf16(a u) (the product of two bf16 values is exact in fp32),
        // and the rows quantized
        const int64_t row = mrow + lane;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          uint32_t yw[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint32_t gp = gw[b][i];
            const uint32_t a =
                (uint32_t)__ldg(p.silu_a + (gp & 0xFFFFu)) | ((uint32_t)__ldg(p.silu_a + (gp >> 16)) << 16);
            yw[i] = f2_to_bf16x2(swiglu_math::f2_mul_bf16x2(a, uw[b][i]));
          }
          uint32_t codes[8];
          const uint32_t sc = quant_row32(yw, codes, p.rceil);
          store32_codes(p.yq + row * p.hy + ycol + 32 * b, codes, p.v8_y);
          p.ys.put(row, (ycol >> 5) + b, sc);
          if (p.yqc) {
            // columns: the warp's 32 rows are one 32-row block of each of
            // the 32 columns.  Transpose through the staging buffer: row r
            // in slot r ^ (r >> 4 & 1), its 16-byte chunk j at j ^ (r >> 1 & 3)
            // (no bank conflicts on the row writes or the column reads);
            // lanes l and l ^ 16 take column pair l & 15, 16 rows each.
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
            {
              uint8_t* dst = stg + (lane ^ ((lane >> 4) & 1)) * 64;
              const int sw = (lane >> 1) & 3;
#pragma unroll
              for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4*>(dst + ((j ^ sw) * 16)) =
                    make_uint4(yw[4 * j], yw[4 * j + 1], yw[4 * j + 2], yw[4 * j + 3]);
            }
            __syncwarp();
            const int pc = lane & 15, rh = lane >> 4;
            auto col_word = [&](int r) {
              const int rr = rh * 16 + r;
              return *reinterpret_cast<const volatile uint32_t*>(stg + (rr ^ rh) * 64 +
                                                                 (((pc >> 2) ^ ((rr >> 1) & 3)) << 4) + ((pc & 3) << 2));
            };
            uint32_t ca[4], cb[4], sa, sb;
            quant_col16x2(col_word, ca, cb, sa, sb, p.rceil);
            __syncwarp();  // the staging buffer is free for the next store
            const int64_t c = ycol + 32 * b + 2 * pc;
            uint8_t* dst = p.yqc + c * p.M + mrow + 16 * rh;
            store16(dst, ca[0], ca[1], ca[2], ca[3]);
            store16(dst + p.M, cb[0], cb[1], cb[2], cb[3]);
            if (rh == 0) {
              p.ysc.put(c, mrow >> 5, sa);
              p.ysc.put(c + 1, mrow >> 5, sb);
            }
          }
        }
        if (++acc == C::NUM_ACC) { acc = 0; acc_phase ^= 1; }
        continue;
      }
      if (SUB == 1) {
        // drain this warp's whole share of the accumulator into registers
        // (all loads in flight, one wait), hand the accumulator back, and only
        // then round and store: the MMA warp waits for one TMEM round trip,
        // and the next tile's MMAs overlap the conversion and the stores
        const CUtensorMap* tmC;
        const int64_t mrow = out_rows(0, tmC);
        const int live = ti.m_blk * C::TM < p.M ? nchunks : 0;
        const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN + half * (BN / 2));
        if constexpr (C::NUM_ACC == 1) {
          uint32_t r[BN / 64][32];
#pragma unroll
          for (int c = 0; c < BN / 64; ++c) tmem_ld_32cols(tbase + c * 32, r[c]);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) release_acc(acc);
#pragma unroll
          for (int c = 0; c < BN / 64; ++c) {
            uint32_t w[16];
            pack(r[c], w);
            if (c < live) store_chunk(w, tmC, ncol0 + 32 * c, mrow);
          }
        } else {
          // two accumulators: the MMA warp is already filling the other one,
          // so the drain is not on its critical path (two chunks at a time
          // keeps fewer registers live)
          uint32_t w[BN / 64][16];
#pragma unroll
          for (int c = 0; c < BN / 64; c += 2) {
            uint32_t r0[32], r1[32];
            tmem_ld_32cols(tbase + c * 32, r0);
            tmem_ld_32cols(tbase + (c + 1) * 32, r1);
            tmem_ld_wait();
            pack(r0, w[c]);
            pack(r1, w[c + 1]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) release_acc(acc);
#pragma unroll
          for (int c = 0; c < BN / 64; ++c)
            if (c < live) store_chunk(w[c], tmC, ncol0 + 32 * c, mrow);
        }
      } else {
#pragma unroll 1
        for (int sub = 0; sub < SUB; ++sub) {
          const CUtensorMap* tmC;
          const int64_t mrow = out_rows(sub, tmC);
          // a sub-tile past the last row is drained but not stored
          const int live = ti.m_blk * C::TM + sub * BM < p.M ? nchunks : 0;
          const uint32_t tbase =
              tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)((acc + sub) * BN + half * (BN / 2));
#pragma unroll 1
          for (int c = 0; c < BN / 64; ++c) {
            uint32_t r[32];
            tmem_ld_32cols(tbase + c * 32, r);
            tmem_ld_wait();
            if (sub == SUB - 1 && c == BN / 64 - 1) {
              // accumulator fully read: hand it back to the MMA warp
              tc_fence_before();
              __syncwarp();
              if (lane == 0) release_acc(acc);
            }
            if (c >= live) continue;
            uint32_t w[16];
            pack(r, w);
            store_chunk(w, tmC, ncol0 + 32 * c, mrow);
          }
        }
      }
      if (++acc == C::NUM_ACC) { acc = 0; acc_phase ^= 1; }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (CL == 2) cluster_sync();  // no pair MMA, copy or remote arrive targets an exited CTA
  tc_fence_after();
  if (warp == 1) {
    if (CL == 2) tmem_dealloc_pair(tmem, C::TMEM_COLS);
    else tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <bool MX, int BN, int CL, int SUB, bool FUSE = false, int KA = 1, bool TW = false>
int launch_cfg(const GemmLaunch& g, const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tC0,
               const CUtensorMap& tC1, const CUtensorMap& tSFA, const CUtensorMap& tSFB, GemmParams& p,
               cudaStream_t stream) {
  using C = Cfg<MX, BN, SUB, CL, KA, TW>;
  p.m_tiles = (p.M + C::TM - 1) / C::TM;
  p.n_tiles = (p.N + BN - 1) / BN;
  {
    // dense tile order: one band (rows fastest over all of M) while the whole
    // of A stays in L2; otherwise bands of tile rows whose A slice takes
    // ~48 MB, so that A is read from DRAM once and B once per band
    const int64_t row_bytes = (int64_t)C::TM * p.K * (MX ? 1 : 2);
    int64_t band = (int64_t)(48ll << 20) / (row_bytes > 0 ? row_bytes : 1);
    if (row_bytes * p.m_tiles <= (96ll << 20)) band = p.m_tiles;
    p.band = band < 1 ? 1 : (band > p.m_tiles ? p.m_tiles : band);
    // B smaller than A and resident in L2: re-read B, stream A once
    const int64_t a_bytes = row_bytes * p.m_tiles, b_bytes = p.N * p.K * (MX ? 1 : 2);
    p.cols_fast = b_bytes < a_bytes && b_bytes <= (96ll << 20);
  }
  p.m_pairs = (p.m_tiles + 1) / 2;
  const int64_t experts = g.mode == GEMM_GROUP_K ? g.E : 1;
  int64_t units;
  if (CL == 1) units = p.m_tiles * p.n_tiles * experts;
  else if (g.mode == GEMM_GROUP_M) units = (p.m_pairs + g.E) * p.n_tiles;  // upper bound; exact count on device
  else units = p.m_pairs * p.n_tiles * experts;
  p.tiles = units;
  if (units == 0) return MX_OK;
  if (units > INT32_MAX) return fail(MX_ERR_UNSUPPORTED, "gemm: too many tiles");
  auto k = gemm_kernel<MX, BN, CL, SUB, FUSE, KA, TW>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute");
  if (CL == 1) {
    const int grid = (int)std::min<int64_t>(units, num_sms());
    count_launch(FUSE ? MX_KERNEL_GEMM_SWIGLU : MX_KERNEL_GEMM);
    k<<<grid, GEMM_THREADS, C::SMEM, stream>>>(tA, tB, tC0, tC1, tSFA, tSFB, p);
    return cuda_status(cudaGetLastError(), "gemm_kernel launch");
  }
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(GEMM_THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent grid: as many pairs as can be resident at once (SMs that
  // cannot be paired within their GPC stay idle rather than forming a tail)
  static int resident[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int& nres = resident[dev & 63];
  if (nres == 0) {
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, k, &cfg);
    if (e != cudaSuccess || n <= 0) return cuda_status(e != cudaSuccess ? e : cudaErrorInvalidConfiguration,
                                                       "cudaOccupancyMaxActiveClusters");
    nres = n;
  }
  const int clusters = (int)std::min<int64_t>(units, nres);
  cfg.gridDim = dim3(2 * clusters);
  count_launch(FUSE ? MX_KERNEL_GEMM_SWIGLU : MX_KERNEL_GEMM);
  e = cudaLaunchKernelEx(&cfg, k, tA, tB, tC0, tC1, tSFA, tSFB, p);
  return cuda_status(e, "gemm_kernel cluster launch");
}

}  // namespace

#ifndef MX_GEMM_BN
#define MX_GEMM_BN 256
#endif
// Dense and M-grouped MXFP8 GEMMs on CTA pairs (cta_group::2, 256x256
// tiles, six stages): 3.23-3.51 against 3.17-3.46 PFLOP/s on single CTAs at
// the MLP's dense shapes, 2-3% less GEMM time in the MoE steps.  The
// K-grouped weight gradients and the fused w13 GEMM stay on single CTAs.
// Build with -DMX_GEMM_PAIR=0 for single CTAs everywhere.
#ifndef MX_GEMM_KA2
#define MX_GEMM_KA2 0  // MXFP8: stages of two 128-byte K atoms (eight MMAs)
#endif
#ifndef MX_GEMM_PAIR
#define MX_GEMM_PAIR 1
#endif
// K-grouped MXFP8 weight gradients on CTA pairs too (1) or on single CTAs
// (0): pairs measured 7-9% faster on the MoE 64E weight gradients once the
// epilogue drains the accumulator with one wait
#ifndef MX_GEMM_PAIR_K
#define MX_GEMM_PAIR_K 1
#endif
// the w13 GEMM with the fused SwiGLU epilogue on CTA pairs (1) or single CTAs (0)
#ifndef MX_GEMM_PAIR_FUSE
#define MX_GEMM_PAIR_FUSE 1
#endif

int launch_gemm(const GemmLaunch& g, cudaStream_t stream) {
  constexpr int BN0 = MX_GEMM_BN;
  const bool mx = g.mx != 0;
  const bool bs = mx && !g.tw;   // block-scaled MXFP8
  // MXFP8: 128x256 tiles, 256x256 on CTA pairs for the dense and M-grouped
  // forms.  bf16:
  // 256x256 tiles on one CTA as two 128-row sub-tiles (128-row tiles for the
  // grouped forward form).
  constexpr int BN = BN0;
  const bool pair = mx && MX_GEMM_PAIR && BN0 == 256 && (g.mode != GEMM_GROUP_K || (bs && MX_GEMM_PAIR_K)) &&
                    (!g.fuse_swiglu || MX_GEMM_PAIR_FUSE);
  const bool two_sub = !mx && BN == 256 && g.mode != GEMM_GROUP_M;
  // MXFP8 on one CTA: two K atoms per stage where K allows it
  const int ka = (mx && !pair && BN == 256 && g.mode != GEMM_GROUP_K && g.K % 256 == 0 && MX_GEMM_KA2) ? 2 : 1;
  const uint32_t BROWS = pair ? BN / 2 : BN;  // rows of one B load
  const int esz = mx ? 1 : 2;
  const CUtensorMapDataType dt = mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t bk = mx ? 128 : 64;
  const CUtensorMapSwizzle opswz = CU_TENSOR_MAP_SWIZZLE_128B;
  CUtensorMap tA, tB, tC0, tC1;
  int rc;
  {
    uint64_t dims[2] = {(uint64_t)g.K, (uint64_t)g.M};
    uint64_t strides[1] = {(uint64_t)g.K * esz};
    uint32_t box[2] = {bk, (uint32_t)(two_sub ? 2 * BM : BM)};
    rc = make_tmap(&tA, dt, 2, const_cast<void*>(g.a), dims, strides, box, opswz);
    if (rc) return rc;
  }
  const bool fuse = g.fuse_swiglu != 0;
  if (fuse) {
    // w13 [(E,) 2h, K] viewed as [(E,) 2, h, K]: one box = rows 128n.. of w1
    // and the same rows of w3
    const uint64_t hh = (uint64_t)(g.N / 2);
    uint64_t dims[4] = {(uint64_t)g.K, hh, 2, (uint64_t)g.E};
    uint64_t strides[3] = {(uint64_t)g.K, (uint64_t)g.K * hh, (uint64_t)g.K * g.N};
    uint32_t box[4] = {bk, 128, pair ? 1u : 2u, 1};   // pairs: one half (w1 or w3) per CTA
    rc = make_tmap(&tB, dt, g.mode == GEMM_GROUP_M ? 4 : 3, const_cast<void*>(g.b), dims, strides, box, opswz);
  } else if (g.mode == GEMM_GROUP_M) {
    uint64_t dims[3] = {(uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.E};
    uint64_t strides[2] = {(uint64_t)g.K * esz, (uint64_t)g.K * g.N * esz};
    uint32_t box[3] = {bk, BROWS, 1};
    rc = make_tmap(&tB, dt, 3, const_cast<void*>(g.b), dims, strides, box, opswz);
  } else {
    uint64_t dims[2] = {(uint64_t)g.K, (uint64_t)g.N};
    uint64_t strides[1] = {(uint64_t)g.K * esz};
    uint32_t box[2] = {bk, BROWS};
    rc = make_tmap(&tB, dt, 2, const_cast<void*>(g.b), dims, strides, box, opswz);
  }
  if (rc) return rc;
  // output maps
  const int64_t experts = g.mode == GEMM_GROUP_K ? g.E : 1;
  const int64_t rows0 = g.split > 0 ? g.split : g.M;
  const int64_t rows1 = g.split > 0 ? g.M - g.split : g.M;
  {
    uint64_t dims[2] = {(uint64_t)g.N, (uint64_t)(rows0 * experts)};
    uint64_t strides[1] = {(uint64_t)g.N * 2};
    uint32_t box[2] = {32, 32};
    rc = make_tmap(&tC0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.c0, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
    if (rc) return rc;
  }
  if (g.split > 0) {
    uint64_t dims[2] = {(uint64_t)g.N, (uint64_t)(rows1 * experts)};
    uint64_t strides[1] = {(uint64_t)g.N * 2};
    uint32_t box[2] = {32, 32};
    rc = make_tmap(&tC1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.c1, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
    if (rc) return rc;
  } else {
    tC1 = tC0;
  }
  GemmParams p{};
  p.mode = g.mode;
  p.M = g.M; p.N = g.N; p.K = g.K;
  p.E = g.mode == GEMM_DENSE ? 1 : g.E;
  p.offs = g.offs;
  p.sfa = (const uint8_t*)g.sfa;
  p.sfb = (const uint8_t*)g.sfb;
  p.sfb_expert_stride = (g.N / 128) * (g.K / 128) * 512;
  p.split = g.split;
  p.msub = g.split > 0 ? g.split : g.M;
  p.yq = (uint8_t*)g.yq;
  p.hy = g.N / 2;
  {
    const int64_t S = p.hy / 32;
    p.ys = ScaleDst{(uint8_t*)g.ys, (S + 3) / 4, S, 1};
    const int64_t Sc = g.M / 32;
    p.yqc = (uint8_t*)g.yq_col;
    p.ysc = ScaleDst{(uint8_t*)g.ys_col, (Sc + 3) / 4, Sc, 1};
  }
  p.rceil = g.floor_scale ? 0u : 1u;
  p.v8_y = ((reinterpret_cast<uintptr_t>(g.yq) | (uintptr_t)(g.N / 2)) & 31) == 0;
  p.silu_a = g.silu_a;
  p.amax_a = g.amax_a;
  p.amax_b = g.amax_b;
  p.amax_b_per_expert = g.amax_b_per_expert;
  p.starve = g.starve;
  p.err = g.err;
  // B scales viewed as 32-bit words: one 512-byte tile = 128 words; tile
  // (row rb, column cb) of a [R, S] scale matrix at word (rb*ceil(S/4) + cb)*128.
  // Box: one column tile of each of the BN/128 tile rows.
  CUtensorMap tSFB = tB;
  if (mx && fuse) {
    // the scale tile rows of w1 block n and w3 block n: [(E,) 2, h/128, K/128, 128 words]
    const uint64_t col_tiles = (uint64_t)(g.K / 128);
    const uint64_t hrows = (uint64_t)(g.N / 256);
    uint64_t dims[5] = {128, col_tiles, hrows, 2, (uint64_t)g.E};
    uint64_t strides[4] = {512, col_tiles * 512, col_tiles * 512 * hrows, col_tiles * 512 * hrows * 2};
    uint32_t box[5] = {128, (uint32_t)ka, 1, 2, 1};
    rc = make_tmap(&tSFB, CU_TENSOR_MAP_DATA_TYPE_UINT32, g.mode == GEMM_GROUP_M ? 5 : 4, const_cast<void*>(g.sfb),
                   dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
  } else if (mx && !g.tw) {
    const uint64_t col_tiles = (uint64_t)(g.K / 128);
    const uint64_t tile_rows = (uint64_t)(g.N / 128);
    if (g.mode == GEMM_GROUP_M) {
      uint64_t dims[4] = {128, col_tiles, tile_rows, (uint64_t)g.E};
      uint64_t strides[3] = {512, col_tiles * 512, col_tiles * 512 * tile_rows};
      uint32_t box[4] = {128, (uint32_t)ka, (uint32_t)(BN / 128), 1};
      rc = make_tmap(&tSFB, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<void*>(g.sfb), dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {
      uint64_t dims[3] = {128, col_tiles, tile_rows};
      uint64_t strides[2] = {512, col_tiles * 512};
      uint32_t box[3] = {128, (uint32_t)ka, (uint32_t)(BN / 128)};
      rc = make_tmap(&tSFB, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(g.sfb), dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (rc) return rc;
  }
  // A scales viewed as 32-bit words, one 512-byte tile per row: tile
  // (row block rb, column cb) at row rb*(K/128) + cb.
  CUtensorMap tSFA = tB;
  if (pair && !g.tw) {
    uint64_t dims[2] = {128, (uint64_t)(g.M / 128) * (uint64_t)(g.K / 128)};
    uint64_t strides[1] = {512};
    uint32_t box[2] = {128, 1};
    rc = make_tmap(&tSFA, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(g.sfa), dims, strides, box,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
  }
  if (fuse) {
    if (!mx || BN != 256 || g.mode == GEMM_GROUP_K || g.N % 256 || !g.yq || !g.ys)
      return fail(MX_ERR_UNSUPPORTED, "fused SwiGLU GEMM: MXFP8 forward form, 2h a multiple of 256");
    if (!g.silu_a) return fail(MX_ERR_INVALID_ARG, "fused SwiGLU GEMM: the a(g) table is required");
    if (!g.yq_col != !g.ys_col || (g.yq_col && g.M % 128))
      return fail(MX_ERR_UNSUPPORTED, "fused SwiGLU GEMM: columnwise y needs both buffers and M a multiple of 128");
    if (pair) return launch_cfg<true, 256, 2, 1, true, 1>(g, tA, tB, tC0, tC1, tSFA, tSFB, p, stream);
    if (ka == 2) return launch_cfg<true, 256, 1, 1, true, 2>(g, tA, tB, tC0, tC1, tSFA, tSFB, p, stream);
    return launch_cfg<true, 256, 1, 1, true, 1>(g, tA, tB, tC0, tC1, tSFA, tSFB, p, stream);
  }
  if (g.tw) {
    if (!mx || BN != 256 || !g.amax_a || !g.amax_b)
      return fail(MX_ERR_INVALID_ARG, "FP8 per-tensor GEMM: E4M3 operands and both amax pointers");
    if (pair) return launch_cfg<true, 256, 2, 1, false, 1, true>(g, tA, tB, tC0, tC1, tSFA, tSFB, p, stream);
    return launch_cfg<true, 256, 1, 1, false, 1, true>(g, tA, tB, tC0, tC1, tSFA, tSFB, p, stream);
  }
  if (mx) {
    if (pair) return launch_cfg<true, BN0, 2, 1>(g, tA, tB, tC0, tC1, tSFA, tSFB, p, stream);
    if (ka == 2) return launch_cfg<true, 256, 1, 1, false, 2>(g, tA, tB, tC0, tC1, tSFA, tSFB, p, stream);
    return launch_cfg<true, BN0, 1, 1>(g, tA, tB, tC0, tC1, tSFA, tSFB, p, stream);
  }
  if (two_sub) return launch_cfg<false, BN0, 1, 2>(g, tA, tB, tC0, tC1, tSFA, tSFB, p, stream);
  return launch_cfg<false, BN0, 1, 1>(g, tA, tB, tC0, tC1, tSFA, tSFB, p, stream);
}

}  // namespace mx
