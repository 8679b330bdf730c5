/*
 * mxmlp.h - C ABI of the MXFP8 training-MLP library (libmxmlp.so).
 *
 * The library runs the hot path of an MXFP8 SwiGLU MLP on one Blackwell GPU
 * (sm_103a): w13 GEMM -> SwiGLU with dual MXFP8 quantization -> w2 GEMM, in
 * dense and grouped-expert form, forward and backward, as described on the
 * page "Add MXFP8 fused-MLP overrides in torchtitan" (pytorch/torchtitan PR
 * 4257), Summary section.  The per-op entry points follow the two ops the
 * page "TrainingWeightWrapperTensor base class; subclasses for FP8/MXFP8 with
 * grouped_mm and linear overrides" (pytorch/ao PR 3968) overrides: linear
 * (mx_scaled_mm) and grouped_mm (mx_grouped_mm).
 *
 * MXFP8: 32-element blocks of FP8 E4M3 codes sharing one E8M0 power-of-two
 * scale.  Scale rule (RCEIL): 2^e with e the smallest integer such that
 * amax <= 448 * 2^e, clamped to [-127,127]; byte e+127.  Codes: v*2^-e
 * rounded to nearest even, saturated to +-448.  All-zero block: scale 0x00.
 * A block holding a NaN or an infinity: scale 0xFF, every code 0x7F.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All tensor pointers are DEVICE pointers, row-major, densely packed
 *   unless a leading dimension is given.  bf16 tensors are passed as
 *   `const void*` / `void*` holding IEEE bfloat16 values.
 * - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *   only enqueues work on `stream` and returns; it never synchronizes.
 * - The caller owns every buffer.  No entry point allocates device memory
 *   (mx_mlp_workspace_size tells the caller how much to provide).
 * - Arguments are validated on the host before anything is enqueued.  On a
 *   bad argument the call returns a non-zero mx_status and enqueues nothing;
 *   mx_last_error() then holds a one-line description (thread-local).
 *   There is no fallback path: unsupported shapes return
 *   MX_ERR_UNSUPPORTED.
 * - Faults found on the device (non-monotone or unaligned group offsets, a
 *   pipeline wait that exceeded its bound, a shared-memory base without the
 *   1024-byte alignment the swizzled copies need) are OR-ed as mx_status
 *   bits into the caller's `err_word` (int32, device memory; may be NULL
 *   where noted) and the kernel skips the faulty work instead of trapping.
 *   Calls without an `err_word` (mx_quantize, mx_swiglu_quant,
 *   mx_swiglu_quant_bwd and their *_mode forms) have no device-side report:
 *   such a fault leaves part of their outputs unwritten; the composite
 *   mx_mlp_fwd / mx_mlp_bwd pass their `err_word` to every kernel they run.
 * - Scale layout MX_SCALE_MMA is the block-scaled tensor-core layout: the
 *   [R, S] scale matrix (R rows, S = cols/32 scale columns) is cut into
 *   128-row x 4-column tiles of 512 bytes; tile (rb, cb) sits at byte
 *   (rb * ceil(S/4) + cb) * 512, and inside a tile scale (r, c) sits at
 *   (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4).  Size:
 *   ceil(R/128) * ceil(S/4) * 512 bytes; padding bytes are written as 0x00.
 *   MX_SCALE_LINEAR is the plain [R, S] row-major byte matrix.
 */
#ifndef MXMLP_H
#define MXMLP_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MX_API __attribute__((visibility("default")))
#else
#define MX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes are distinct bits so that device-side faults can be OR-ed
 * into one error word. */
typedef enum {
  MX_OK = 0,
  MX_ERR_INVALID_ARG = 1,  /* null pointer, negative or zero size, bad enum */
  MX_ERR_ALIGNMENT = 2,    /* pointer or leading dimension not 16-byte aligned */
  MX_ERR_UNSUPPORTED = 4,  /* shape the kernels do not cover (no fallback) */
  MX_ERR_BAD_OFFSETS = 8,  /* group offsets decreasing, unaligned or past M */
  MX_ERR_TIMEOUT = 16,     /* a device pipeline wait exceeded its bound */
  MX_ERR_CUDA = 32         /* a CUDA runtime/driver call failed */
} mx_status;

typedef enum { MX_ROW = 1, MX_COL = 2, MX_BOTH = 3 } mx_axis;
typedef enum { MX_SCALE_LINEAR = 0, MX_SCALE_MMA = 1 } mx_scale_layout;
/* MX_RECIPE_RCEIL: every GEMM in MXFP8.  MX_RECIPE_RCEIL_WGRAD_HP: forward
 * and input-gradient GEMMs in MXFP8, weight-gradient GEMMs in bf16
 * ("wgrad_with_hp", pages "TrainingWeightWrapperTensor base class ..." and
 * "[mxfp8 training] unified MXFP8TrainingConfig ...", Autograd function
 * changes). */
typedef enum {
  MX_RECIPE_RCEIL = 0,
  MX_RECIPE_RCEIL_WGRAD_HP = 1,
  /* The same two recipes with FLOOR scales for every quantization (see
   * mx_scale_mode). */
  MX_RECIPE_FLOOR = 2,
  MX_RECIPE_FLOOR_WGRAD_HP = 3
} mx_recipe;
/* E8M0 scale rule.  MX_SCALE_RCEIL: the one above (amax/448 rounded up to a
 * power of two; "ScaleCalculationMode.RCEIL" on the ao pages).
 * MX_SCALE_FLOOR: 2^e with e = floor(log2(amax)) - 8, the shared exponent of
 * the OCP Microscaling Formats v1.0 conversion, clamped likewise; scaled
 * values in (448, 512) then saturate to +-448.  Zero and non-finite blocks
 * as for RCEIL. */
typedef enum { MX_SCALE_RCEIL = 0, MX_SCALE_FLOOR = 1 } mx_scale_mode;
typedef enum { MX_GROUP_M = 0, MX_GROUP_K = 1 } mx_grouped_mode;

/* Library version (major*10000 + minor*100 + patch). */
MX_API int mx_version(void);
/* Static string for a status code (bits OR-ed together name the first). */
MX_API const char* mx_status_string(int status);
/* Thread-local description of the last failing call on this thread. */
MX_API const char* mx_last_error(void);

/*
 * mx_quantize - MXFP8 cast of a bf16 matrix, rowwise and/or columnwise.
 * The "standalone cast" of the torchtitan page (Numerics and tests).
 *
 *   x       [rows, cols] bf16.
 *   axis    MX_ROW: blocks of 32 along cols  -> q_row [rows, cols] u8,
 *                                              s_row scales of [rows, cols/32]
 *           MX_COL: blocks of 32 along rows  -> q_col [cols, rows] u8 (the
 *                                              transposed matrix, contiguous
 *                                              along rows), s_col scales of
 *                                              [cols, rows/32]
 *           MX_BOTH: both (one read of x).
 *   layout  scale layout of s_row / s_col (MX_SCALE_LINEAR or MX_SCALE_MMA).
 * Requirements: cols % 32 == 0; for MX_COL/MX_BOTH rows % 32 == 0; x and
 * the code buffers 16-byte aligned; cols * 2 bytes a multiple of 16.
 * Unused outputs may be NULL.
 */
MX_API int mx_quantize(const void* x, int64_t rows, int64_t cols, int axis, int layout,
                void* q_row, void* s_row, void* q_col, void* s_col, void* stream);

/* mx_quantize with an explicit scale rule (mx_scale_mode). */
MX_API int mx_quantize_mode(const void* x, int64_t rows, int64_t cols, int axis, int layout, int scale_mode,
                            void* q_row, void* s_row, void* q_col, void* s_col, void* stream);

/*
 * mx_swiglu_quant - fused SwiGLU forward with dual MXFP8 quantization; the
 * bf16 activation y is never written to memory (torchtitan page, Summary:
 * "fused SwiGLU + dual MXFP8 quantization", "never materializes the BF16
 * post-activation tensor").
 *
 *   h13     [M, 2h] bf16: g = h13[:, :h] (x . w1^T), u = h13[:, h:] (x . w3^T).
 *   y       = RN_bf16(RN_f32(a * u)), a = RN_bf16(RN_f32(g * sigma)),
 *             sigma = 1/(1+exp(-g)) correctly rounded to fp32.
 *   MX_ROW  -> yq_row [M, h] u8 + ys_row scales of [M, h/32]
 *   MX_COL  -> yq_col [h, M] u8 + ys_col scales of [h, M/32]
 * Requirements: h % 64 == 0, M % 32 == 0 (M % 128 == 0 with MX_COL).
 */
MX_API int mx_swiglu_quant(const void* h13, int64_t M, int64_t h, int axis, int layout,
                    void* yq_row, void* ys_row, void* yq_col, void* ys_col, void* stream);

/*
 * mx_swiglu_quant_bwd - fused SwiGLU backward with dual MXFP8 quantization of
 * dh13 = [dg | du] (torchtitan page, Summary: "1 bwd fused op").
 *
 *   dy      [M, h] bf16 (gradient of y);  h13 [M, 2h] bf16 from the forward.
 *   du      = RN_bf16(RN_f32(dy * a));
 *   dg      = RN_bf16(dy * u * sigma * (1 + g * (1 - sigma))) rounded once
 *             from the exact value (NaN for non-finite g).
 *   MX_ROW  -> dq_row [M, 2h] u8 + ds_row scales of [M, 2h/32]
 *   MX_COL  -> dq_col [2h, M] u8 + ds_col scales of [2h, M/32]
 *   dh13_t  optional (may be NULL): dh13 in bf16, TRANSPOSED: [2h, M]
 *   y_t     optional (may be NULL): the recomputed forward y in bf16,
 *           TRANSPOSED: [h, M].  The transposed (token-contiguous) layout is
 *           the one the bf16 weight-gradient GEMM of the wgrad_with_hp recipe
 *           reads.
 * Requirements: as mx_swiglu_quant; dh13_t / y_t need M % 128 == 0.
 */
MX_API int mx_swiglu_quant_bwd(const void* dy, const void* h13, int64_t M, int64_t h, int axis,
                        int layout, void* dq_row, void* ds_row, void* dq_col, void* ds_col,
                        void* dh13_t, void* y_t, void* stream);

/* mx_swiglu_quant and mx_swiglu_quant_bwd with an explicit scale rule
 * (mx_scale_mode); the plain entry points use MX_SCALE_RCEIL. */
MX_API int mx_swiglu_quant_mode(const void* h13, int64_t M, int64_t h, int axis, int layout, int scale_mode,
                                void* yq_row, void* ys_row, void* yq_col, void* ys_col, void* stream);
MX_API int mx_swiglu_quant_bwd_mode(const void* dy, const void* h13, int64_t M, int64_t h, int axis, int layout,
                                    int scale_mode, void* dq_row, void* ds_row, void* dq_col, void* ds_col,
                                    void* dh13_t, void* y_t, void* stream);

/*
 * mx_scaled_mm - block-scaled MXFP8 GEMM on the tcgen05 tensor cores:
 *   C[M, N] (bf16, RN) = deq(A)[M, K] . deq(B)[N, K]^T, fp32 accumulation.
 *   aq [M, K] u8, as scales MX_SCALE_MMA of [M, K/32];
 *   bq [N, K] u8, bs scales MX_SCALE_MMA of [N, K/32].
 * Requirements: M % 128 == 0, N % 128 == 0, K % 128 == 0.
 * err_word may be NULL.
 */
MX_API int mx_scaled_mm(const void* aq, const void* as, const void* bq, const void* bs, int64_t M,
                 int64_t N, int64_t K, void* c, int32_t* err_word, void* stream);

/*
 * mx_grouped_mm - grouped block-scaled MXFP8 GEMM over expert-major token
 * groups (grouped_mm override, ao page; padded dispatch with pad_multiple =
 * 128, torchtitan page, Summary).
 *
 *   offs    [E] int32 device array of cumulative group ends: group e owns
 *           token rows [offs[e-1], offs[e]) (offs[-1] = 0).  Every group size
 *           must be a multiple of pad_multiple (only 128 is supported), the
 *           offsets non-decreasing and offs[E-1] <= M_total.  Read on the
 *           device: no host synchronization.
 *   MX_GROUP_M (forward / input gradient):
 *           A = aq [M_total, K] (tokens), B = bq [E, N, K] (per-expert
 *           weights, scales MX_SCALE_MMA per expert, expert stride
 *           (N/128)*(K/128)*512 bytes), C = c [M_total, N] bf16.  Rows past
 *           offs[E-1] are written as zeros.  Empty groups cost nothing.
 *   MX_GROUP_K (weight gradient):
 *           A = aq [N, M_total], B = bq [K, M_total] (columnwise copies,
 *           contiguous along tokens), C = c [E, N, K] bf16 with
 *           C[e] = A[:, group e] . B[:, group e]^T.  An empty group's C[e]
 *           is written as exact zeros.
 * Requirements: M_total, N, K multiples of 128; 1 <= E <= 1024.
 * err_word (may be NULL) receives MX_ERR_BAD_OFFSETS if offs violates the
 * rules; the offending groups are then skipped.
 */
MX_API int mx_grouped_mm(int mode, const void* aq, const void* as, const void* bq, const void* bs,
                  int64_t M_total, int64_t N, int64_t K, const int32_t* offs, int32_t E,
                  int32_t pad_multiple, void* c, int32_t* err_word, void* stream);

/*
 * mx_bf16_wgrad - bf16 weight-gradient GEMM of the wgrad_with_hp recipe on
 * the tcgen05 tensor cores (kind::f16), fp32 accumulation, bf16 RN output.
 *   a [N, M_total] bf16, b [K, M_total] bf16 (token-contiguous, e.g. the
 *   transposed outputs of mx_swiglu_quant_bwd), c [E, N, K] bf16 with
 *   C[e] = a[:, group e] . b[:, group e]^T.  offs as in mx_grouped_mm; pass
 *   offs = NULL and E = 1 for the dense case (one group of M_total tokens).
 * Requirements: M_total, N, K multiples of 128.
 */
MX_API int mx_bf16_wgrad(const void* a, const void* b, int64_t M_total, int64_t N, int64_t K,
                  const int32_t* offs, int32_t E, int32_t pad_multiple, void* c,
                  int32_t* err_word, void* stream);

/*
 * mx_mlp_workspace_size - bytes of the two caller-provided buffers of
 * mx_mlp_fwd / mx_mlp_bwd for a given problem.
 *   ctx_bytes      saved-for-backward context (written by mx_mlp_fwd, read
 *                  by mx_mlp_bwd): h13 in bf16 and the quantized operands.
 *   scratch_bytes  temporary buffer used inside one call (fwd or bwd).
 * E = 0 selects the dense MLP (weights without an expert axis).
 */
MX_API int mx_mlp_workspace_size(int64_t M_total, int64_t d, int64_t h, int32_t E, int recipe,
                          size_t* ctx_bytes, size_t* scratch_bytes);

/*
 * mx_mlp_ctx_layout - where one saved tensor lives inside the context
 * buffer of mx_mlp_fwd, for callers that inspect or checkpoint it.
 *   tensor     one of mx_ctx_tensor
 *   offset     out: byte offset from the start of ctx (256-byte aligned)
 *   bytes      out: its size in bytes
 * Returns MX_ERR_UNSUPPORTED when the recipe keeps no such tensor (the
 * columnwise x and y exist under the MXFP8 weight-gradient recipes, the
 * bf16 x^T under the wgrad_with_hp recipes).  Layouts: H13 [M_total, 2h]
 * bf16; XQ_COL [d, M_total] and YQ_COL [h, M_total] codes with MMA-layout
 * scales XS_COL / YS_COL; X_T [d, M_total] bf16; W13Q_COL [E, d, 2h] and
 * W2Q_COL [E, h, d] codes with per-expert MMA-layout scales.
 */
typedef enum {
  MX_CTX_H13 = 0, MX_CTX_XQ_COL = 1, MX_CTX_XS_COL = 2, MX_CTX_YQ_COL = 3, MX_CTX_YS_COL = 4,
  MX_CTX_X_T = 5, MX_CTX_W13Q_COL = 6, MX_CTX_W13S_COL = 7, MX_CTX_W2Q_COL = 8, MX_CTX_W2S_COL = 9
} mx_ctx_tensor;
MX_API int mx_mlp_ctx_layout(int64_t M_total, int64_t d, int64_t h, int32_t E, int recipe, int tensor,
                             size_t* offset, size_t* bytes);

/*
 * mx_mlp_fwd - forward of the MXFP8 SwiGLU MLP (torchtitan page, Summary):
 *   out = (silu(x . w1^T) * (x . w3^T)) . w2^T with every GEMM in MXFP8.
 *   x [M_total, d] bf16; dense: w1, w3 [h, d], w2 [d, h]; grouped (offs not
 *   NULL): w1, w3 [E, h, d], w2 [E, d, h] and offs/E/pad_multiple as in
 *   mx_grouped_mm.  w1 and w3 are packed into w13 = [w1; w3] while they are
 *   quantized; the caller's weights are never modified.
 *   ctx, scratch: buffers of the sizes mx_mlp_workspace_size returns (16-byte
 *   aligned).  out [M_total, d] bf16.
 * Requirements: M_total % 128 == 0, d % 128 == 0, h % 128 == 0.
 * The first call in a CUDA context that takes the fused w13 GEMM + SwiGLU
 * path (d >= 5120, or the wgrad_with_hp recipe) fills the library's table of
 * a(g) = RN_bf16(g sigma(g)) over every bf16 g (128 KB of static device
 * memory) on `stream` and waits for `stream`; later calls do not wait.
 */
MX_API int mx_mlp_fwd(const void* x, const void* w1, const void* w3, const void* w2, int64_t M_total,
               int64_t d, int64_t h, const int32_t* offs, int32_t E, int32_t pad_multiple,
               int recipe, void* ctx, void* scratch, void* out, int32_t* err_word,
               void* stream);

/*
 * mx_mlp_bwd - backward of the MXFP8 SwiGLU MLP from the context mx_mlp_fwd
 * wrote (same shapes, recipe, offs and weights as that forward call).
 *   dout [M_total, d] bf16 -> dx [M_total, d], dw1, dw3 ([h, d] or
 *   [E, h, d]) and dw2 ([d, h] or [E, d, h]), all bf16.  The weight
 *   gradients are overwritten (not accumulated).  The w13 gradient is
 *   written straight into dw1 and dw3.
 */
MX_API int mx_mlp_bwd(const void* ctx, const void* dout, const void* x, const void* w1, const void* w3,
               const void* w2, int64_t M_total, int64_t d, int64_t h, const int32_t* offs,
               int32_t E, int32_t pad_multiple, int recipe, void* scratch, void* dx, void* dw1,
               void* dw3, void* dw2, int32_t* err_word, void* stream);

/*
 * mx_linear_* - the per-linear MXFP8 path for linears outside the MLP
 * (attention projections, lm_head): the linear override of the page
 * "TrainingWeightWrapperTensor base class; subclasses for FP8/MXFP8 with
 * grouped_mm and linear overrides" (Summary), kept for non-MLP linears by the
 * page "Add MXFP8 fused-MLP overrides in torchtitan" (Summary).
 *
 *   forward   out [M, N] = x [M, K] . w [N, K]^T, x and w MX(R) along K.
 *   backward  dx [M, K] = dout [M, N] . w, dout MX(R) and w MX(C) along N;
 *             dw [N, K] = dout^T . x, both MX(C) along M (MX_RECIPE_RCEIL) or
 *             bf16 operands (MX_RECIPE_RCEIL_WGRAD_HP).
 *   ctx       caller buffer written by the forward and read by the backward
 *             (columnwise x, or bf16 x^T); scratch: caller buffer, both sized by
 *             mx_linear_workspace_size.  All bf16 in/out, fp32 accumulation,
 *             one RN to bf16.
 * Requirements: M, K, N multiples of 128; 16-byte aligned pointers.
 */
MX_API int mx_linear_workspace_size(int64_t M, int64_t K, int64_t N, int recipe, size_t* ctx_bytes,
                                    size_t* scratch_bytes);
MX_API int mx_linear_fwd(const void* x, const void* w, int64_t M, int64_t K, int64_t N, int recipe, void* ctx,
                         void* scratch, void* out, int32_t* err_word, void* stream);
MX_API int mx_linear_bwd(const void* ctx, const void* dout, const void* w, int64_t M, int64_t K, int64_t N,
                         int recipe, void* scratch, void* dx, void* dw, int32_t* err_word, void* stream);

/*
 * mx_token_group_pad - the padded expert-major row layout that the grouped
 * entry points take, built on the device from routing decisions ("[mxfp8]
 * refactor model converter; use token group padding kernels in torchao",
 * Summary: per-group padding done by kernels instead of host code; "Add
 * MXFP8 fused-MLP overrides in torchtitan", Summary: the padded dispatcher
 * with pad_multiple = 128, pad rows and the tail inert).
 *
 *   expert_of [R] int32: expert of routed row r, in [0, E) (for top-k
 *             routing of T tokens, R = T*k rows, row r belongs to token r/k).
 *   offs      [E] int32 out: cumulative padded group ends (the offs of
 *             mx_grouped_mm / mx_mlp_fwd); group e holds its rows in
 *             increasing r, padded up to a multiple of pad_multiple.
 *   row_dst   [R] int32 out: padded row of routed row r.
 *   row_src   [M_cap] int32 out: routed row held by padded row i, or -1 for
 *             a padding row and for the tail past offs[E-1].
 *   M_cap     rows of the padded buffers, a multiple of 128; the layout
 *             always fits when M_cap >= ceil(R/128)*128 + 128*E.
 *   workspace device scratch of mx_token_group_pad_workspace(R, E) bytes
 *             (may be NULL when R == 0).
 * No host synchronization: counts, offsets and ranks stay on the device.
 * Requirements: 1 <= E <= 1024, pad_multiple == 128.  err_word (may be
 * NULL) receives MX_ERR_BAD_OFFSETS if an expert id is out of range (that
 * row is left unplaced) or if the layout exceeds M_cap (then no row is
 * placed and offs is still written).
 */
MX_API size_t mx_token_group_pad_workspace(int64_t R, int32_t E);
MX_API int mx_token_group_pad(const int32_t* expert_of, int64_t R, int32_t E, int32_t pad_multiple,
                              int64_t M_cap, int32_t* offs, int32_t* row_dst, int32_t* row_src,
                              void* workspace, int32_t* err_word, void* stream);

/*
 * mx_gather_rows - y[i, :] = x[src[i] / div, :] for src[i] >= 0 and zeros
 * for src[i] < 0, i in [0, rows_out) (bf16 rows copied bit for bit).  With
 * src = row_src of mx_token_group_pad and div = k it builds the padded
 * expert-major activations from the token rows, pad and tail rows zero;
 * with src = row_dst and div = 1 it brings padded results (out, dx) back to
 * routed-row order (the same torchtitan page: dispatcher pad-row and tail
 * inertness).
 *   x [rows_in, cols], y [rows_out, cols]: bf16, 16-byte aligned, cols a
 *   multiple of 8.  err_word (may be NULL) receives MX_ERR_BAD_OFFSETS for a
 *   source row past rows_in; that output row is written as zeros.
 */
MX_API int mx_gather_rows(const void* x, int64_t rows_in, int64_t cols, const int32_t* src, int64_t rows_out,
                          int32_t div, void* y, int32_t* err_word, void* stream);

/*
 * mx_mlp_fwd_static_scratch - mx_mlp_fwd for callers that cannot allocate
 * device memory (no cudaMalloc at all: for instance code running where only
 * pre-registered buffers may be touched, or a host framework whose allocator
 * is not reachable from the call site).  The pages have no counterpart of
 * this entry point; it is a convenience of this library.
 *
 * Same arguments and results as mx_mlp_fwd, except that the temporary
 * buffer comes from a fixed device array inside the library
 * (MX_STATIC_SCRATCH_BYTES bytes, held by every GPU that loads the library
 * until the process exits) instead of from the caller.  The caller still
 * passes the inputs, ctx (as sized by mx_mlp_workspace_size) and out.
 * - Problems whose scratch_bytes (mx_mlp_workspace_size) exceed
 *   MX_STATIC_SCRATCH_BYTES are rejected with MX_ERR_UNSUPPORTED.
 * - It allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * - The array has one instance per CUDA context.  The first call in a
 *   context (the one current on the calling thread; the device's primary
 *   context if none is) looks up the array's device address there and
 *   caches it under the context's unique ID, so a device reset or a
 *   different context is looked up afresh.  Make that first call before any
 *   CUDA stream capture.
 * - All calls share the one array and the kernels overwrite every byte they
 *   read back, so no clearing is needed between calls; calls that overlap
 *   on the GPU (different streams, or different threads without ordering)
 *   race on the array and must not be issued.
 */
#define MX_STATIC_SCRATCH_BYTES (16u << 20)
MX_API int mx_mlp_fwd_static_scratch(const void* x, const void* w1, const void* w3, const void* w2,
                                     int64_t M_total, int64_t d, int64_t h, const int32_t* offs,
                                     int32_t E, int32_t pad_multiple, int recipe, void* ctx,
                                     void* out, int32_t* err_word, void* stream);

/*
 * ---- FP8 per-tensor ("tensorwise") recipe: the non-MX FP8 grouped MM
 * ("[mxfp8 training] unified MXFP8TrainingConfig and MXFP8TrainingTensor",
 * "Temporarily removed FP8GroupedMM quantize_ workflow support": FP8
 * GroupedMM is the other, non-MX recipe; its arithmetic is not given there.
 * Reading used here: one fp32 scale per tensor, or per expert for a
 * [E, N, K] weight, s = RN_f32(448 / max(amax, 2^-40)) with amax = max |x|;
 * code = E4M3 (round to nearest even, saturating) of RN_f32(x * s); the
 * dequantized value is code / s.)  A tensor's scale is carried as its amax
 * (device fp32), from which every consumer derives s.
 */

/*
 * mx_fp8_amax - amax[b] = max |x| over item b of x [batch, n] (bf16, device).
 *   x: 16-byte aligned, n % 8 == 0; batch <= 65535.
 *   amax: device fp32 [batch], overwritten (the call clears it first).  A
 *   NaN in an item makes its amax NaN.  HBM-bound: reads x once.
 * Errors: MX_ERR_INVALID_ARG (null, sizes), MX_ERR_UNSUPPORTED (n % 8),
 * MX_ERR_ALIGNMENT.
 */
MX_API int mx_fp8_amax(const void* x, int64_t batch, int64_t n, float* amax, void* stream);

/*
 * mx_fp8_quantize - FP8 per-tensor codes of x [batch, rows, cols] (bf16),
 * item b scaled by s = 448 / max(amax[b], 2^-40) (amax device fp32 [batch],
 * e.g. from mx_fp8_amax; only the device reads it).
 *   axis MX_ROW: q_row [batch, rows, cols] codes (contiguous along cols);
 *   axis MX_COL: q_col [batch, cols, rows] codes (the transpose, contiguous
 *   along rows: the K-major operand of a GEMM contracting over rows).
 *   cols % 32 == 0; rows % 32 == 0 for MX_COL; x and code buffers 16-byte
 *   aligned.  No scale bytes are written: the scale is the amax.
 */
MX_API int mx_fp8_quantize(const void* x, int64_t batch, int64_t rows, int64_t cols, const float* amax, int axis,
                           void* q_row, void* q_col, void* stream);

/*
 * mx_fp8_grouped_mm - grouped GEMM on FP8 per-tensor operands (E4M3 codes,
 * no block scales), fp32 accumulation on the tensor cores, then
 * C = RN_bf16(acc * (1/s_a) * (1/s_b)).
 *   MX_GROUP_M: A [M_total, K] codes with amax_a [1]; B [E, N, K] codes with
 *     amax_b [E] (one per expert); C [M_total, N]: rows of group e use
 *     expert e, rows past offs[E-1] are written as zeros.
 *   MX_GROUP_K: A [N, M_total] and B [K, M_total] (token-contiguous copies,
 *     e.g. mx_fp8_quantize with MX_COL), amax_a [1] and amax_b [1];
 *     C [E, N, K], C[e] = A[:, group e] . B[:, group e]^T, empty experts zero.
 *   offs, E, pad_multiple (= 128), err_word: as for mx_grouped_mm.
 *   M_total, N, K multiples of 128; buffers 16-byte aligned.
 */
MX_API int mx_fp8_grouped_mm(int mode, const void* aq, const float* amax_a, const void* bq, const float* amax_b,
                             int64_t M_total, int64_t N, int64_t K, const int32_t* offs, int32_t E,
                             int32_t pad_multiple, void* c, int32_t* err_word, void* stream);

/*
 * Kernel launch counters (observability; no counterpart on the pages).
 * The torchtitan page's GPU suite holds the fused MLP to an op-count
 * contract ("Add MXFP8 fused-MLP overrides in torchtitan", Numerics and
 * tests: one fused activation op per direction instead of the standalone
 * casts).  Every device operation the library enqueues is counted on the
 * host at launch, by family:
 */
enum mx_kernel_family {
  MX_KERNEL_QUANT = 0,        /* quant_kernel: one MX cast (rows and/or columns) */
  MX_KERNEL_SWIGLU_FWD = 1,   /* swiglu_fwd_kernel: SwiGLU + MX quantization of y */
  MX_KERNEL_SWIGLU_BWD = 2,   /* swiglu_bwd_kernel: SwiGLU backward + MX quantization of dh13 */
  MX_KERNEL_GEMM = 3,         /* gemm_kernel: MXFP8 or bf16 GEMM (dense, M- or K-grouped) */
  MX_KERNEL_GEMM_SWIGLU = 4,  /* gemm_kernel with the fused SwiGLU epilogue (w13 GEMM + y quantization) */
  MX_KERNEL_DISPATCH = 5,     /* token-group padding and row gathers */
  MX_KERNEL_MEMSET = 6,       /* cudaMemsetAsync of scale padding or dispatch maps */
  MX_KERNEL_FAMILIES = 7
};

/*
 * mx_launch_counts - copies the launch counters (totals since the library
 * was loaded, all devices and threads, counted when the launch is issued)
 * into counts[0 .. min(n, MX_KERNEL_FAMILIES)); returns MX_KERNEL_FAMILIES.
 * counts may be NULL with n = 0 to query the number of families.  Take the
 * difference of two readings around the calls of interest (calls from other
 * threads in between are counted too).
 */
MX_API int mx_launch_counts(int64_t* counts, int n);

/*
 * mx_selftest_wait_timeout - test entry of the failure detection: launches a
 * 256x256x256 MXFP8 GEMM on library-owned device buffers whose load stage
 * issues nothing, so that the MMA and epilogue pipeline waits run past their
 * 2 s bound.  The kernel then records MX_ERR_TIMEOUT in *err_word (device
 * memory, required), releases its tensor memory and returns: no trap, no
 * hang, and the CUDA context stays usable.  It exists for tests (no
 * counterpart on the pages); the call takes about 2 s of GPU time.
 */
MX_API int mx_selftest_wait_timeout(int32_t* err_word, void* stream);

/*
 * mx_selftest_silu_table - test entry of the a(g) table the fused w13 GEMM
 * epilogue reads: copies its 65536 entries (entry b = the bits of
 * RN_bf16(RN_f32(g sigma(g))) for the bf16 g with bits b; the silu rounding
 * of the page "Add MXFP8 fused-MLP overrides in torchtitan", Numerics) into
 * dst (device memory, 131072 bytes, caller-owned) on `stream`, filling the
 * table first if this context has not used it yet (which waits for
 * `stream`).  MX_ERR_INVALID_ARG if dst is NULL.
 */
MX_API int mx_selftest_silu_table(uint16_t* dst, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MXMLP_H */
