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
//   warps 2-5   epilogue: tcgen05.ld of the fp32 accumulator, RN to bf16,
//               128-byte-swizzled staging in shared memory, TMA store
// Modes: dense; M-grouped (forward / input gradient: token rows of group e
// use expert e's weights, rows past the last group are zero); K-grouped
// (weight gradient: expert e contracts over its own token range; an empty
// group writes zeros).  Group offsets are read on the device.
#include "common.cuh"
#include "kernels.h"

namespace mx {

namespace {

constexpr int BM = 128;
constexpr int EPI_WARPS = 4;
constexpr int GEMM_THREADS = 64 + EPI_WARPS * 32;
constexpr int MAX_GROUPS = 1024;

template <bool MX, int BN>
struct Cfg {
  static constexpr int BK = MX ? 128 : 64;                 // elements per stage (128 bytes)
  static constexpr int UK = MX ? 32 : 16;                  // elements per MMA
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int SFA_BYTES = MX ? 512 : 0;
  static constexpr int SFB_BYTES = MX ? (BN / 128) * 512 : 0;
  static constexpr int STAGES = BN == 256 ? 4 : 6;
  static constexpr int NUM_ACC = BN == 256 ? 1 : 2;
  static constexpr int EPI_BYTES = EPI_WARPS * 32 * 128;   // one 32x64 bf16 buffer per warp
  static constexpr int TMEM_COLS = 512;
  static constexpr int SF_COL = NUM_ACC * BN;
  static constexpr size_t SMEM = (size_t)STAGES * (A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES) + EPI_BYTES +
                                 MAX_GROUPS * 4 + 1024 /*align*/ + 256 /*barriers*/;
  static constexpr uint32_t IDESC =
      MX ? ((1u << 23) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24))
         : ((1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24));
};

struct GemmParams {
  int mode;
  int64_t M, N, K;            // K: contraction length of A (GROUP_K: total tokens)
  int64_t m_tiles, n_tiles, tiles;
  int32_t E;
  const int32_t* offs;
  const uint8_t* sfa;         // MMA-layout scales of A ([M, K/32])
  const uint8_t* sfb;         // MMA-layout scales of B ([N, K/32] or per expert)
  int64_t sfb_expert_stride;  // bytes between experts (GROUP_M)
  int64_t split;              // row split of C between tmC0 / tmC1 (0: none)
  int64_t msub;               // GROUP_K: rows per expert in the output maps
  int32_t* err;
};

struct TileInfo {
  int64_t m_blk, n_blk;
  int32_t e;       // expert (GROUP_M / GROUP_K), 0 for dense
  int64_t k0;      // first contraction element
  int32_t num_kb;  // number of BK steps (0: write zeros)
};

// Group ends in shared memory; ok == false if they break the contract.
struct Groups {
  const int32_t* ends;
  int32_t E;
  bool ok;
};

template <int BK>
MX_DEVINL TileInfo tile_info(const GemmParams& p, const Groups& g, int64_t t) {
  TileInfo ti{};
  if (p.mode == GEMM_GROUP_K) {
    const int64_t per_e = p.m_tiles * p.n_tiles;
    const int64_t e = t / per_e;
    const int64_t rem = t - e * per_e;
    ti.e = (int32_t)e;
    ti.m_blk = rem % p.m_tiles;
    ti.n_blk = rem / p.m_tiles;
    const int64_t s = e == 0 ? 0 : g.ends[e - 1];
    const int64_t en = g.ends[e];
    ti.k0 = s;
    ti.num_kb = g.ok ? (int32_t)((en - s) / BK) : 0;
    return ti;
  }
  ti.m_blk = t % p.m_tiles;
  ti.n_blk = t / p.m_tiles;
  ti.k0 = 0;
  ti.num_kb = (int32_t)(p.K / BK);
  ti.e = 0;
  if (p.mode == GEMM_GROUP_M) {
    const int64_t row = ti.m_blk * BM;
    if (!g.ok || g.E == 0 || row >= g.ends[g.E - 1]) {
      ti.num_kb = 0;  // tail rows (or invalid offsets): zeros
    } else {
      int lo = 0, hi = g.E - 1;  // first group whose end is > row
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (g.ends[mid] > row) hi = mid; else lo = mid + 1;
      }
      ti.e = lo;
    }
  }
  return ti;
}

template <bool MX, int BN>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC0, const __grid_constant__ CUtensorMap tmC1,
                GemmParams p) {
  using C = Cfg<MX, BN>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + C::STAGES * C::A_BYTES;
  uint8_t* sEpi = sB + C::STAGES * C::B_BYTES;
  uint8_t* sSFA = sEpi + C::EPI_BYTES;
  uint8_t* sSFB = sSFA + C::STAGES * C::SFA_BYTES;
  int32_t* sEnds = reinterpret_cast<int32_t*>(sSFB + C::STAGES * C::SFB_BYTES);
  uint64_t* full = reinterpret_cast<uint64_t*>(sEnds + MAX_GROUPS);
  uint64_t* empty = full + C::STAGES;
  uint64_t* acc_full = empty + C::STAGES;
  uint64_t* acc_empty = acc_full + C::NUM_ACC;
  uint64_t* done_bar = acc_empty + C::NUM_ACC;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(done_bar + 1);
  __shared__ int s_groups_ok;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- setup: barriers, group ends, TMEM
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < C::NUM_ACC; ++a) { mbar_init(&acc_full[a], 1); mbar_init(&acc_empty[a], EPI_WARPS); }
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
      sEnds[e] = v;
      if (v < prev || (v & 127) != 0 || (int64_t)v > limit) s_groups_ok = 0;
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  Groups grp{sEnds, p.E, s_groups_ok != 0};
  if (!grp.ok && threadIdx.x == 0 && blockIdx.x == 0) record_error(p.err, MX_ERR_BAD_OFFSETS);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      int stage = 0; uint32_t phase = 0;
      const int64_t sfa_row_tiles = p.K / 128;  // scale tiles per 128-row block of A
      for (int64_t t = blockIdx.x; t < p.tiles; t += gridDim.x) {
        const TileInfo ti = tile_info<C::BK>(p, grp, t);
        bool ok = true;
        for (int kb = 0; kb < ti.num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, p.err)) { ok = false; break; }
          const int64_t k = ti.k0 + (int64_t)kb * C::BK;
          uint32_t bytes = C::A_BYTES + C::B_BYTES;
          int nsfb = 0;
          if (MX) {
            const int64_t n_sub_total = p.N / 128;
            const int64_t left = n_sub_total - ti.n_blk * (BN / 128);
            nsfb = (int)(left < BN / 128 ? left : BN / 128);
            bytes += 512 + 512 * nsfb;
          }
          mbar_arrive_expect_tx(&full[stage], bytes);
          tma_load_2d(sA + stage * C::A_BYTES, &tmA, (int32_t)k, (int32_t)(ti.m_blk * BM), &full[stage]);
          if (p.mode == GEMM_GROUP_M)
            tma_load_3d(sB + stage * C::B_BYTES, &tmB, (int32_t)k, (int32_t)(ti.n_blk * BN), ti.e, &full[stage]);
          else
            tma_load_2d(sB + stage * C::B_BYTES, &tmB, (int32_t)k, (int32_t)(ti.n_blk * BN), &full[stage]);
          if (MX) {
            const int64_t kt = k / 128;
            bulk_load(sSFA + stage * C::SFA_BYTES, p.sfa + (ti.m_blk * sfa_row_tiles + kt) * 512, 512, &full[stage]);
            const uint8_t* sfb = p.sfb + (p.mode == GEMM_GROUP_M ? (int64_t)ti.e * p.sfb_expert_stride : 0);
            for (int j = 0; j < nsfb; ++j) {
              const int64_t nsub = ti.n_blk * (BN / 128) + j;
              bulk_load(sSFB + stage * C::SFB_BYTES + j * 512, sfb + (nsub * sfa_row_tiles + kt) * 512, 512,
                        &full[stage]);
            }
          }
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0; uint32_t phase = 0;
      int acc = 0; uint32_t acc_phase = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < p.tiles && ok; t += gridDim.x) {
        const TileInfo ti = tile_info<C::BK>(p, grp, t);
        if (ti.num_kb == 0) continue;
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
        for (int kb = 0; kb < ti.num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b_base = smem_u32(sB + stage * C::B_BYTES);
          if (MX) {
            tmem_cp_32x128b_x4(tmem + C::SF_COL, smem_desc(smem_u32(sSFA + stage * C::SFA_BYTES), 128, 128, 0));
#pragma unroll
            for (int j = 0; j < BN / 128; ++j)
              tmem_cp_32x128b_x4(tmem + C::SF_COL + 4 + 4 * j,
                                 smem_desc(smem_u32(sSFB + stage * C::SFB_BYTES + j * 512), 128, 128, 0));
          }
#pragma unroll
          for (int k = 0; k < 128 / 32; ++k) {
            const uint64_t ad = smem_desc(a_base + k * 32, 16, 1024, 2);
            const uint64_t bd = smem_desc(b_base + k * 32, 16, 1024, 2);
            const uint32_t accum = (kb > 0 || k > 0) ? 1u : 0u;
            if (MX) {
              const uint32_t idesc = C::IDESC | ((uint32_t)k << 4) | ((uint32_t)k << 29);
              mma_mxf8(d_tmem, ad, bd, idesc, tmem + C::SF_COL, tmem + C::SF_COL + 4, accum);
            } else {
              mma_bf16(d_tmem, ad, bd, C::IDESC, accum);
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        tc_commit(&acc_full[acc]);
        if (++acc == C::NUM_ACC) { acc = 0; acc_phase ^= 1; }
      }
      // all issued MMAs complete before TMEM is released
      tc_commit(done_bar);
      mbar_wait(done_bar, 0, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint8_t* stg = sEpi + (warp - 2) * (32 * 128);
    int acc = 0; uint32_t acc_phase = 0;
    for (int64_t t = blockIdx.x; t < p.tiles; t += gridDim.x) {
      const TileInfo ti = tile_info<C::BK>(p, grp, t);
      // output row of this warp's 32 rows
      int64_t mrow = ti.m_blk * BM + q * 32;
      const CUtensorMap* tmC = &tmC0;
      if (p.split > 0 && mrow >= p.split) { tmC = &tmC1; mrow -= p.split; }
      if (p.mode == GEMM_GROUP_K) mrow += (int64_t)ti.e * p.msub;
      const int64_t ncol0 = ti.n_blk * BN;
      const int64_t cleft = (p.N - ncol0 + 63) / 64;
      const int nchunks = (int)(cleft < BN / 64 ? cleft : BN / 64);
      if (ti.num_kb == 0) {
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        uint4* row = reinterpret_cast<uint4*>(stg + lane * 128);
#pragma unroll
        for (int j = 0; j < 8; ++j) row[j] = make_uint4(0, 0, 0, 0);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          for (int c = 0; c < nchunks; ++c) tma_store_2d(tmC, stg, (int32_t)(ncol0 + 64 * c), (int32_t)mrow);
          bulk_commit();
        }
        continue;
      }
      if (!mbar_wait(&acc_full[acc], acc_phase, p.err)) break;
      tc_fence_after();
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      for (int c = 0; c < BN / 64; ++c) {
        uint32_t r0[32], r1[32];
        tmem_ld_32cols(tbase + c * 64, r0);
        tmem_ld_32cols(tbase + c * 64 + 32, r1);
        tmem_ld_wait();
        if (c == BN / 64 - 1) {
          // accumulator fully read: hand it back to the MMA warp
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[acc]);
        }
        if (c >= nchunks) continue;
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          w[i] = f32_to_bf16_bits(__uint_as_float(r0[2 * i])) | (f32_to_bf16_bits(__uint_as_float(r0[2 * i + 1])) << 16);
          w[16 + i] = f32_to_bf16_bits(__uint_as_float(r1[2 * i])) | (f32_to_bf16_bits(__uint_as_float(r1[2 * i + 1])) << 16);
        }
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
        uint8_t* row = stg + lane * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) * 16)) = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(tmC, stg, (int32_t)(ncol0 + 64 * c), (int32_t)mrow);
          bulk_commit();
        }
      }
      if (++acc == C::NUM_ACC) { acc = 0; acc_phase ^= 1; }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <bool MX, int BN>
int launch_cfg(const GemmLaunch& g, const CUtensorMap& tA, const CUtensorMap& tB, const CUtensorMap& tC0,
               const CUtensorMap& tC1, GemmParams& p, cudaStream_t stream) {
  using C = Cfg<MX, BN>;
  p.n_tiles = (p.N + BN - 1) / BN;
  p.tiles = p.m_tiles * p.n_tiles * (g.mode == GEMM_GROUP_K ? g.E : 1);
  if (p.tiles == 0) return MX_OK;
  const int grid = (int)std::min<int64_t>(p.tiles, num_sms());
  auto k = gemm_kernel<MX, BN>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e == cudaSuccess) {
    k<<<grid, GEMM_THREADS, C::SMEM, stream>>>(tA, tB, tC0, tC1, p);
    e = cudaGetLastError();
  }
  return cuda_status(e, "gemm_kernel launch");
}

}  // namespace

int launch_gemm(const GemmLaunch& g, cudaStream_t stream) {
  constexpr int BN = 256;
  const bool mx = g.mx != 0;
  const int esz = mx ? 1 : 2;
  const CUtensorMapDataType dt = mx ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint32_t bk = mx ? 128 : 64;
  CUtensorMap tA, tB, tC0, tC1;
  int rc;
  {
    uint64_t dims[2] = {(uint64_t)g.K, (uint64_t)g.M};
    uint64_t strides[1] = {(uint64_t)g.K * esz};
    uint32_t box[2] = {bk, (uint32_t)BM};
    rc = make_tmap(&tA, dt, 2, const_cast<void*>(g.a), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  if (g.mode == GEMM_GROUP_M) {
    uint64_t dims[3] = {(uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.E};
    uint64_t strides[2] = {(uint64_t)g.K * esz, (uint64_t)g.K * g.N * esz};
    uint32_t box[3] = {bk, (uint32_t)BN, 1};
    rc = make_tmap(&tB, dt, 3, const_cast<void*>(g.b), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    uint64_t dims[2] = {(uint64_t)g.K, (uint64_t)g.N};
    uint64_t strides[1] = {(uint64_t)g.K * esz};
    uint32_t box[2] = {bk, (uint32_t)BN};
    rc = make_tmap(&tB, dt, 2, const_cast<void*>(g.b), dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (rc) return rc;
  // output maps
  const int64_t experts = g.mode == GEMM_GROUP_K ? g.E : 1;
  const int64_t rows0 = g.split > 0 ? g.split : g.M;
  const int64_t rows1 = g.split > 0 ? g.M - g.split : g.M;
  {
    uint64_t dims[2] = {(uint64_t)g.N, (uint64_t)(rows0 * experts)};
    uint64_t strides[1] = {(uint64_t)g.N * 2};
    uint32_t box[2] = {64, 32};
    rc = make_tmap(&tC0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.c0, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  }
  if (g.split > 0) {
    uint64_t dims[2] = {(uint64_t)g.N, (uint64_t)(rows1 * experts)};
    uint64_t strides[1] = {(uint64_t)g.N * 2};
    uint32_t box[2] = {64, 32};
    rc = make_tmap(&tC1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.c1, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc) return rc;
  } else {
    tC1 = tC0;
  }
  GemmParams p{};
  p.mode = g.mode;
  p.M = g.M; p.N = g.N; p.K = g.K;
  p.m_tiles = g.M / BM;
  p.E = g.mode == GEMM_DENSE ? 1 : g.E;
  p.offs = g.offs;
  p.sfa = (const uint8_t*)g.sfa;
  p.sfb = (const uint8_t*)g.sfb;
  p.sfb_expert_stride = (g.N / 128) * (g.K / 128) * 512;
  p.split = g.split;
  p.msub = g.split > 0 ? g.split : g.M;
  p.err = g.err;
  if (mx) return launch_cfg<true, BN>(g, tA, tB, tC0, tC1, p, stream);
  return launch_cfg<false, BN>(g, tA, tB, tC0, tC1, p, stream);
}

}  // namespace mx
