// kernels.h - internal host interface between the C-ABI layer (api.cu) and
// the kernel launchers (quant.cu, swiglu.cu, gemm.cu).  Not installed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/mxmlp.h"

namespace mx {

// ---------------------------------------------------------------- host utils
int num_sms();
// Records a thread-local message; returns `code`.
int fail(int code, const char* fmt, ...);
int cuda_status(cudaError_t e, const char* what);
// Adds one to the launch counter of a kernel family (mx_kernel_family).
void count_launch(int family);
int make_tmap(CUtensorMap* m, CUtensorMapDataType dt, int rank, void* base, const uint64_t* dims,
              const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz);

// ---------------------------------------------------------------- quantize
struct QuantLaunch {
  const void* x;
  int64_t rows, cols;
  int32_t batch;
  int layout;
  // rowwise MX: codes [rows, cols] per batch item; batch strides qr_bs
  // (codes) and sr_bs (scale bytes), 0 = densely packed
  void* q_row;
  void* s_row;
  int64_t qr_bs, sr_bs;
  // columnwise MX: codes of column c at q_col + c*qc_ld + qc_off (+ b*qc_bs)
  void* q_col;
  void* s_col;
  int64_t qc_ld, qc_off, qc_bs, sc_bs;
  // columnwise bf16 transpose (instead of q_col): element (r, c) at
  // t_col[c*tc_ld + tc_off + r] (+ b*tc_bs)
  void* t_col;
  int64_t tc_ld, tc_off, tc_bs;
  int floor_scale;   // 1: FLOOR E8M0 scales; 0 (default): RCEIL
  // FP8 per-tensor codes instead of MX blocks: item b scaled by
  // 448 / amax[b] (device fp32); no scale bytes are written
  int tw;
  const float* amax;
  int32_t* err;
};
int launch_quant(const QuantLaunch& q, cudaStream_t stream);
// amax[b] = max |x| over item b of x [batch, n] (bf16, n % 8 == 0, 16-byte
// aligned); clears amax first.
int launch_fp8_amax(const void* x, int64_t batch, int64_t n, float* amax, cudaStream_t stream);

// ---------------------------------------------------------------- SwiGLU
struct SwigluLaunch {
  const void* h13;   // [M, 2h]
  const void* dy;    // [M, h] (backward only)
  int64_t M, h;
  int layout;
  void* q_row; void* s_row;   // fwd: y rows [M,h]; bwd: dh13 rows [M,2h]
  void* q_col; void* s_col;   // fwd: y cols [h,M]; bwd: dh13 cols [2h,M]
  void* dh13_t;               // bwd, optional: [2h, M] bf16
  void* y_t;                  // bwd, optional: [h, M] bf16
  int floor_scale;            // 1: FLOOR E8M0 scales; 0 (default): RCEIL
  const uint16_t* silu_a;     // fwd: a(g) for every bf16 g (see launch_silu_table_init)
  int32_t* err;
};
int launch_swiglu_fwd(const SwigluLaunch& s, cudaStream_t stream);
int launch_swiglu_bwd(const SwigluLaunch& s, cudaStream_t stream);

// ---------------------------------------------------------------- GEMM
enum GemmMode { GEMM_DENSE = 0, GEMM_GROUP_M = 1, GEMM_GROUP_K = 2 };

struct GemmLaunch {
  int mx;                 // 1: MXFP8 block-scaled, 0: bf16
  int mode;               // GemmMode
  // C[m, n] = sum_k A[m, k] B[n, k]
  const void* a;          // [M, K] (DENSE/GROUP_M) or [M, Ktot] (GROUP_K)
  const void* sfa;        // MMA-layout scales of A
  const void* b;          // [N, K], [E, N, K] (GROUP_M) or [N, Ktot] (GROUP_K)
  const void* sfb;
  int64_t M, N, K;        // GROUP_K: K = total tokens
  const int32_t* offs;    // group ends (GROUP_M: over M, GROUP_K: over K)
  int32_t E;
  // output: row m of C goes to c0 (m < split) or c1 (m - split) when split>0;
  // GROUP_K: output [E, M, N], expert e row m at (e*Msub + m) of c0/c1 where
  // Msub = split ? split : M.
  void* c0;
  void* c1;
  int64_t split;
  // fused SwiGLU epilogue (MXFP8, DENSE or GROUP_M): B = w13 [(E,) 2h, K]
  // with w1 rows first; c0 receives h13 [M, 2h] and yq/ys the rowwise MXFP8
  // y = SwiGLU(h13) [M, h] (scales in the MMA layout)
  int fuse_swiglu;
  void* yq;
  void* ys;
  void* yq_col;      // optional columnwise y: codes [h, M] and MMA-layout scales [h, M/32]
  void* ys_col;
  int floor_scale;   // 1: FLOOR E8M0 scales for y
  const uint16_t* silu_a;  // a(g) = RN_bf16(g sigma(g)) for every bf16 g (65536 entries, device)
  // FP8 per-tensor recipe (mx = 1, E4M3 codes without block scales): amax
  // of A ([1]) and of B ([1], or [E] when amax_b_per_expert), device fp32
  int tw;
  const float* amax_a;
  const float* amax_b;
  int amax_b_per_expert;
  int starve;        // self-test of the bounded waits: the producer issues nothing
  int32_t* err;
};
int launch_gemm(const GemmLaunch& g, cudaStream_t stream);

// Fills table[b] = a(g) = RN_bf16(RN_f32(g sigma(g))) for every bf16 bit
// pattern b = bits(g), by the exact tiers of swiglu_math.cuh (swiglu.cu).
int launch_silu_table_init(uint16_t* table, cudaStream_t stream);

// token-group padding (dispatch.cu)
size_t token_group_pad_workspace(int64_t R, int32_t E);
int launch_token_group_pad(const int32_t* expert_of, int64_t R, int32_t E, int32_t pad, int64_t M_cap,
                           int32_t* offs, int32_t* row_dst, int32_t* row_src, void* workspace, int32_t* err,
                           cudaStream_t stream);
int launch_gather_rows(const void* x, int64_t rows_in, int64_t cols, const int32_t* src, int64_t rows_out,
                       int32_t div, void* y, int32_t* err, cudaStream_t stream);

}  // namespace mx
