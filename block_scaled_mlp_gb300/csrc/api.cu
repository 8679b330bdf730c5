// api.cu - the C ABI of libmxmlp (include/mxmlp.h): argument validation,
// tensor-map creation, and the MLP forward/backward composites that chain
// the quantize, SwiGLU and GEMM kernels on one stream.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "kernels.h"

namespace mx {

namespace {
thread_local char g_msg[512] = "";
std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
int g_sms[64] = {0};
std::atomic<long long> g_launches[MX_KERNEL_FAMILIES];
}  // namespace

void count_launch(int family) {
  if (family >= 0 && family < MX_KERNEL_FAMILIES) g_launches[family].fetch_add(1, std::memory_order_relaxed);
}

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return MX_OK;
  return fail(MX_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (g_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

namespace {
std::once_flag g_ctx_fn_once;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

// Unique ID of the current context; false if none is current or the driver
// calls are unavailable (a per-context value is then set up on every call).
bool current_ctx_id(unsigned long long* id) {
  std::call_once(g_ctx_fn_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  if (!g_ctx_current || !g_ctx_id) return false;
  CUcontext c = nullptr;
  return g_ctx_current(&c) == CUDA_SUCCESS && c && g_ctx_id(c, id) == CUDA_SUCCESS;
}

// A device address that is set up once per CUDA context (a __device__
// array has one instance per context): cached under the context's unique
// ID, so a reset device or a caller's own non-primary context gets its own
// set-up instead of a stale address.
struct CtxCache {
  static constexpr int kSlots = 16;
  struct Slot {
    unsigned long long ctx_id;
    void* ptr;
  };
  std::mutex mu;
  Slot slots[kSlots] = {};
  int next = 0;
  template <class F>
  int lookup(void** out, F&& setup) {
    std::lock_guard<std::mutex> lock(mu);
    unsigned long long id = 0;
    if (current_ctx_id(&id))
      for (const Slot& s : slots)
        if (s.ptr && s.ctx_id == id) {
          *out = s.ptr;
          return MX_OK;
        }
    void* ptr = nullptr;
    const int rc = setup(&ptr);
    if (rc) return rc;
    if (current_ctx_id(&id)) {  // the context the set-up ran in
      slots[next] = Slot{id, ptr};
      next = (next + 1) % kSlots;
    }
    *out = ptr;
    return MX_OK;
  }
};

// a(g) = RN_bf16(RN_f32(g sigma(g))) for every bf16 g, indexed by its bits;
// filled by launch_silu_table_init the first time a context uses it.
static __device__ __align__(256) uint16_t g_silu_table[65536];
CtxCache g_silu_cache;
}  // namespace

// Device address of the a(g) table in the current context.  The first call
// in a context fills it on `stream` and waits for that stream (so the call
// must not be under stream capture); later calls only look it up.
int silu_table_address(const uint16_t** out, cudaStream_t stream) {
  void* p = nullptr;
  const int rc = g_silu_cache.lookup(&p, [stream](void** ptr) {
    cudaError_t e = cudaGetSymbolAddress(ptr, g_silu_table);
    if (e != cudaSuccess) return cuda_status(e, "cudaGetSymbolAddress(silu table)");
    const int r = launch_silu_table_init(static_cast<uint16_t*>(*ptr), stream);
    if (r) return r;
    return cuda_status(cudaStreamSynchronize(stream), "silu table fill (first use in this context)");
  });
  *out = static_cast<const uint16_t*>(p);
  return rc;
}

int make_tmap(CUtensorMap* m, CUtensorMapDataType dt, int rank, void* base, const uint64_t* dims,
              const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(MX_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t d[5];
  cuuint64_t s[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  CUresult r = g_encode(m, dt, (cuuint32_t)rank, base, d, s, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MX_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) rank %d dims %llu x %llu", (int)r, rank,
                (unsigned long long)dims[0], (unsigned long long)(rank > 1 ? dims[1] : 0));
  return MX_OK;
}

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// recipes: bit 0 = bf16 weight gradients (wgrad_with_hp), bit 1 = FLOOR scales
inline bool valid_recipe(int r) { return r >= MX_RECIPE_RCEIL && r <= MX_RECIPE_FLOOR_WGRAD_HP; }
inline bool recipe_hp(int r) { return r == MX_RECIPE_RCEIL_WGRAD_HP || r == MX_RECIPE_FLOOR_WGRAD_HP; }
inline int recipe_floor(int r) { return r == MX_RECIPE_FLOOR || r == MX_RECIPE_FLOOR_WGRAD_HP; }

inline int64_t mma_scale_bytes(int64_t rows, int64_t cols) {
  const int64_t S = cols / 32;
  return ((rows + 127) / 128) * ((S + 3) / 4) * 512;
}

// MMA-layout padding bytes must read 0x00: clear the buffer first when the
// matrix does not fill whole tiles.
int clear_padding(int layout, void* s, int64_t rows, int64_t cols, cudaStream_t st) {
  if (layout != MX_SCALE_MMA || !s) return MX_OK;
  if (rows % 128 == 0 && (cols / 32) % 4 == 0) return MX_OK;
  count_launch(MX_KERNEL_MEMSET);
  return cuda_status(cudaMemsetAsync(s, 0, (size_t)mma_scale_bytes(rows, cols), st), "cudaMemsetAsync");
}

struct Arena {
  uint8_t* base;
  size_t off = 0;
  explicit Arena(void* b) : base((uint8_t*)b) {}
  uint8_t* take(size_t bytes) {
    uint8_t* p = base ? base + off : nullptr;
    off += (bytes + 255) & ~size_t(255);
    return p;
  }
};

struct MlpBuffers {
  // context (saved for backward)
  uint8_t *h13, *xq_c, *xs_c, *yq_c, *ys_c, *x_t, *w13q_c, *w13s_c, *w2q_c, *w2s_c;
  size_t ctx_bytes;
  // forward scratch
  uint8_t *xq_r, *xs_r, *w13q_r, *w13s_r, *yq_r, *ys_r, *w2q_r, *w2s_r;
  // backward scratch
  uint8_t *dq_r, *ds_r, *dq_c, *ds_c, *dout_t, *dy, *dhq_r, *dhs_r, *dhq_c, *dhs_c, *dh13_t, *y_t;
  size_t scratch_bytes;
};

MlpBuffers carve(void* ctx, void* scratch, int64_t M, int64_t d, int64_t h, int64_t Ew, int recipe) {
  MlpBuffers b{};
  const bool hp = recipe_hp(recipe);
  Arena c(ctx);
  b.h13 = c.take(M * 2 * h * 2);
  if (hp) {
    b.x_t = c.take(d * M * 2);
  } else {
    b.xq_c = c.take(d * M);
    b.xs_c = c.take(mma_scale_bytes(d, M));
    b.yq_c = c.take(h * M);
    b.ys_c = c.take(mma_scale_bytes(h, M));
  }
  b.w13q_c = c.take(Ew * d * 2 * h);
  b.w13s_c = c.take(Ew * mma_scale_bytes(d, 2 * h));
  b.w2q_c = c.take(Ew * h * d);
  b.w2s_c = c.take(Ew * mma_scale_bytes(h, d));
  b.ctx_bytes = c.off;
  Arena f(scratch);
  b.xq_r = f.take(M * d);
  b.xs_r = f.take(mma_scale_bytes(M, d));
  b.w13q_r = f.take(Ew * 2 * h * d);
  b.w13s_r = f.take(Ew * mma_scale_bytes(2 * h, d));
  b.yq_r = f.take(M * h);
  b.ys_r = f.take(mma_scale_bytes(M, h));
  b.w2q_r = f.take(Ew * d * h);
  b.w2s_r = f.take(Ew * mma_scale_bytes(d, h));
  const size_t fwd_bytes = f.off;
  Arena g(scratch);
  b.dq_r = g.take(M * d);
  b.ds_r = g.take(mma_scale_bytes(M, d));
  if (hp) {
    b.dout_t = g.take(d * M * 2);
  } else {
    b.dq_c = g.take(d * M);
    b.ds_c = g.take(mma_scale_bytes(d, M));
  }
  b.dy = g.take(M * h * 2);
  b.dhq_r = g.take(M * 2 * h);
  b.dhs_r = g.take(mma_scale_bytes(M, 2 * h));
  if (hp) {
    b.dh13_t = g.take(2 * h * M * 2);
    b.y_t = g.take(h * M * 2);
  } else {
    b.dhq_c = g.take(2 * h * M);
    b.dhs_c = g.take(mma_scale_bytes(2 * h, M));
  }
  b.scratch_bytes = std::max(fwd_bytes, g.off);
  return b;
}

int check_mlp_args(const void* x, const void* w1, const void* w3, const void* w2, int64_t M, int64_t d,
                   int64_t h, const int32_t* offs, int32_t E, int32_t pad, int recipe, const void* ctx,
                   const void* scratch) {
  if (!x || !w1 || !w3 || !w2 || !ctx || !scratch) return fail(MX_ERR_INVALID_ARG, "null pointer argument");
  if (M <= 0 || d <= 0 || h <= 0) return fail(MX_ERR_INVALID_ARG, "sizes must be positive");
  if (M % 128 || d % 128 || h % 128)
    return fail(MX_ERR_UNSUPPORTED, "M_total, d and h must be multiples of 128 (got %lld, %lld, %lld)",
                (long long)M, (long long)d, (long long)h);
  if (!valid_recipe(recipe)) return fail(MX_ERR_INVALID_ARG, "unknown recipe %d", recipe);
  if (offs) {
    if (E < 1 || E > 1024) return fail(MX_ERR_INVALID_ARG, "E must be in [1, 1024]");
    if (pad != 128) return fail(MX_ERR_UNSUPPORTED, "pad_multiple must be 128");
  }
  if (!aligned16(x) || !aligned16(w1) || !aligned16(w3) || !aligned16(w2) || !aligned16(ctx) ||
      !aligned16(scratch))
    return fail(MX_ERR_ALIGNMENT, "tensor pointers must be 16-byte aligned");
  if ((int64_t)M * 2 * h > (int64_t)INT32_MAX * 64) return fail(MX_ERR_UNSUPPORTED, "problem too large");
  return MX_OK;
}

// ---- per-linear MXFP8 path: buffers
struct LinearBuffers {
  uint8_t *xq_c, *xs_c, *x_t;                 // ctx: columnwise x (default) or bf16 x^T (HP)
  size_t ctx_bytes;
  uint8_t *xq_r, *xs_r, *wq_r, *ws_r;         // forward scratch
  uint8_t *dq_r, *ds_r, *wq_c, *ws_c, *dq_c, *ds_c, *dout_t;  // backward scratch
  size_t scratch_bytes;
};

LinearBuffers carve_linear(void* ctx, void* scratch, int64_t M, int64_t K, int64_t N, int recipe) {
  LinearBuffers b{};
  const bool hp = recipe_hp(recipe);
  Arena c(ctx);
  if (hp) {
    b.x_t = c.take(K * M * 2);
  } else {
    b.xq_c = c.take(K * M);
    b.xs_c = c.take(mma_scale_bytes(K, M));
  }
  b.ctx_bytes = c.off;
  Arena f(scratch);
  b.xq_r = f.take(M * K);
  b.xs_r = f.take(mma_scale_bytes(M, K));
  b.wq_r = f.take(N * K);
  b.ws_r = f.take(mma_scale_bytes(N, K));
  Arena g(scratch);
  b.dq_r = g.take(M * N);
  b.ds_r = g.take(mma_scale_bytes(M, N));
  b.wq_c = g.take(K * N);
  b.ws_c = g.take(mma_scale_bytes(K, N));
  if (hp) {
    b.dout_t = g.take(N * M * 2);
  } else {
    b.dq_c = g.take(N * M);
    b.ds_c = g.take(mma_scale_bytes(N, M));
  }
  b.scratch_bytes = std::max(f.off, g.off);
  return b;
}

int check_linear_args(int64_t M, int64_t K, int64_t N, int recipe) {
  if (M <= 0 || K <= 0 || N <= 0) return fail(MX_ERR_INVALID_ARG, "sizes must be positive");
  if (M % 128 || K % 128 || N % 128)
    return fail(MX_ERR_UNSUPPORTED, "M, K and N must be multiples of 128 (got %lld, %lld, %lld)", (long long)M,
                (long long)K, (long long)N);
  if (!valid_recipe(recipe)) return fail(MX_ERR_INVALID_ARG, "unknown recipe %d", recipe);
  if (M > INT32_MAX || K > INT32_MAX || N > INT32_MAX) return fail(MX_ERR_UNSUPPORTED, "dimension too large");
  return MX_OK;
}

}  // namespace
}  // namespace mx

using namespace mx;

extern "C" {

int mx_version(void) { return 100; }

const char* mx_status_string(int s) {
  if (s == MX_OK) return "MX_OK";
  if (s & MX_ERR_INVALID_ARG) return "MX_ERR_INVALID_ARG";
  if (s & MX_ERR_ALIGNMENT) return "MX_ERR_ALIGNMENT";
  if (s & MX_ERR_UNSUPPORTED) return "MX_ERR_UNSUPPORTED";
  if (s & MX_ERR_BAD_OFFSETS) return "MX_ERR_BAD_OFFSETS";
  if (s & MX_ERR_TIMEOUT) return "MX_ERR_TIMEOUT";
  if (s & MX_ERR_CUDA) return "MX_ERR_CUDA";
  return "MX_ERR_UNKNOWN";
}

const char* mx_last_error(void) { return g_msg; }

int mx_launch_counts(int64_t* counts, int n) {
  for (int i = 0; i < n && i < MX_KERNEL_FAMILIES; ++i)
    counts[i] = counts ? (int64_t)g_launches[i].load(std::memory_order_relaxed) : 0;
  return MX_KERNEL_FAMILIES;
}

int mx_quantize(const void* x, int64_t rows, int64_t cols, int axis, int layout, void* q_row, void* s_row,
                void* q_col, void* s_col, void* stream) {
  return mx_quantize_mode(x, rows, cols, axis, layout, MX_SCALE_RCEIL, q_row, s_row, q_col, s_col, stream);
}

int mx_quantize_mode(const void* x, int64_t rows, int64_t cols, int axis, int layout, int scale_mode,
                     void* q_row, void* s_row, void* q_col, void* s_col, void* stream) {
  if (scale_mode != MX_SCALE_RCEIL && scale_mode != MX_SCALE_FLOOR)
    return fail(MX_ERR_INVALID_ARG, "unknown scale mode %d", scale_mode);
  if (!x) return fail(MX_ERR_INVALID_ARG, "x is null");
  if (rows <= 0 || cols <= 0) return fail(MX_ERR_INVALID_ARG, "rows and cols must be positive");
  if (axis < MX_ROW || axis > MX_BOTH) return fail(MX_ERR_INVALID_ARG, "axis must be MX_ROW, MX_COL or MX_BOTH");
  if (layout != MX_SCALE_LINEAR && layout != MX_SCALE_MMA) return fail(MX_ERR_INVALID_ARG, "unknown scale layout");
  if (cols % 32) return fail(MX_ERR_UNSUPPORTED, "cols must be a multiple of 32 (got %lld)", (long long)cols);
  const bool row = axis & MX_ROW, col = axis & MX_COL;
  if (col && rows % 32) return fail(MX_ERR_UNSUPPORTED, "columnwise needs rows %% 32 == 0 (got %lld)", (long long)rows);
  if (row && (!q_row || !s_row)) return fail(MX_ERR_INVALID_ARG, "rowwise outputs are null");
  if (col && (!q_col || !s_col)) return fail(MX_ERR_INVALID_ARG, "columnwise outputs are null");
  if (!aligned16(x) || (row && !aligned16(q_row)) || (col && !aligned16(q_col)))
    return fail(MX_ERR_ALIGNMENT, "x and code buffers must be 16-byte aligned");
  if (rows > INT32_MAX || cols > INT32_MAX) return fail(MX_ERR_UNSUPPORTED, "dimension too large");
  cudaStream_t st = (cudaStream_t)stream;
  int rc;
  if (row && (rc = clear_padding(layout, s_row, rows, cols, st))) return rc;
  if (col && (rc = clear_padding(layout, s_col, cols, rows, st))) return rc;
  QuantLaunch q{};
  q.x = x; q.rows = rows; q.cols = cols; q.batch = 1; q.layout = layout;
  q.q_row = row ? q_row : nullptr; q.s_row = row ? s_row : nullptr;
  q.q_col = col ? q_col : nullptr; q.s_col = col ? s_col : nullptr;
  q.qc_ld = rows; q.qc_off = 0; q.qc_bs = 0; q.sc_bs = 0;
  q.floor_scale = scale_mode == MX_SCALE_FLOOR;
  return launch_quant(q, st);
}

int mx_swiglu_quant(const void* h13, int64_t M, int64_t h, int axis, int layout, void* yq_row, void* ys_row,
                    void* yq_col, void* ys_col, void* stream) {
  return mx_swiglu_quant_mode(h13, M, h, axis, layout, MX_SCALE_RCEIL, yq_row, ys_row, yq_col, ys_col, stream);
}

int mx_swiglu_quant_mode(const void* h13, int64_t M, int64_t h, int axis, int layout, int scale_mode,
                         void* yq_row, void* ys_row, void* yq_col, void* ys_col, void* stream) {
  if (scale_mode != MX_SCALE_RCEIL && scale_mode != MX_SCALE_FLOOR)
    return fail(MX_ERR_INVALID_ARG, "unknown scale mode %d", scale_mode);
  if (!h13) return fail(MX_ERR_INVALID_ARG, "h13 is null");
  if (M <= 0 || h <= 0) return fail(MX_ERR_INVALID_ARG, "sizes must be positive");
  if (axis < MX_ROW || axis > MX_BOTH) return fail(MX_ERR_INVALID_ARG, "bad axis");
  if (layout != MX_SCALE_LINEAR && layout != MX_SCALE_MMA) return fail(MX_ERR_INVALID_ARG, "unknown scale layout");
  if (!(axis & MX_ROW)) return fail(MX_ERR_UNSUPPORTED, "the fused SwiGLU always writes the rowwise copy");
  if (h % 64 || M % 32) return fail(MX_ERR_UNSUPPORTED, "need h %% 64 == 0 and M %% 32 == 0");
  const bool col = axis & MX_COL;
  if (!yq_row || !ys_row || (col && (!yq_col || !ys_col))) return fail(MX_ERR_INVALID_ARG, "output is null");
  if (!aligned16(h13) || !aligned16(yq_row) || (col && !aligned16(yq_col)))
    return fail(MX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  int rc;
  if ((rc = clear_padding(layout, ys_row, M, h, st))) return rc;
  if (col && (rc = clear_padding(layout, ys_col, h, M, st))) return rc;
  SwigluLaunch s{};
  s.h13 = h13; s.M = M; s.h = h; s.layout = layout;
  s.q_row = yq_row; s.s_row = ys_row;
  s.q_col = col ? yq_col : nullptr; s.s_col = col ? ys_col : nullptr;
  s.floor_scale = scale_mode == MX_SCALE_FLOOR;
  if ((rc = silu_table_address(&s.silu_a, st))) return rc;
  return launch_swiglu_fwd(s, st);
}

int mx_swiglu_quant_bwd(const void* dy, const void* h13, int64_t M, int64_t h, int axis, int layout,
                        void* dq_row, void* ds_row, void* dq_col, void* ds_col, void* dh13_t, void* y_t,
                        void* stream) {
  return mx_swiglu_quant_bwd_mode(dy, h13, M, h, axis, layout, MX_SCALE_RCEIL, dq_row, ds_row, dq_col, ds_col,
                                  dh13_t, y_t, stream);
}

int mx_swiglu_quant_bwd_mode(const void* dy, const void* h13, int64_t M, int64_t h, int axis, int layout,
                             int scale_mode, void* dq_row, void* ds_row, void* dq_col, void* ds_col, void* dh13_t,
                             void* y_t, void* stream) {
  if (scale_mode != MX_SCALE_RCEIL && scale_mode != MX_SCALE_FLOOR)
    return fail(MX_ERR_INVALID_ARG, "unknown scale mode %d", scale_mode);
  if (!dy || !h13) return fail(MX_ERR_INVALID_ARG, "dy or h13 is null");
  if (M <= 0 || h <= 0) return fail(MX_ERR_INVALID_ARG, "sizes must be positive");
  if (axis < MX_ROW || axis > MX_BOTH) return fail(MX_ERR_INVALID_ARG, "bad axis");
  if (layout != MX_SCALE_LINEAR && layout != MX_SCALE_MMA) return fail(MX_ERR_INVALID_ARG, "unknown scale layout");
  if (!(axis & MX_ROW)) return fail(MX_ERR_UNSUPPORTED, "the fused SwiGLU backward always writes the rowwise copy");
  if (h % 64 || M % 32) return fail(MX_ERR_UNSUPPORTED, "need h %% 64 == 0 and M %% 32 == 0");
  const bool col = axis & MX_COL;
  if (col && (dh13_t || y_t)) return fail(MX_ERR_UNSUPPORTED, "bf16 transposed outputs come without MX_COL");
  if (!dq_row || !ds_row || (col && (!dq_col || !ds_col))) return fail(MX_ERR_INVALID_ARG, "output is null");
  if (!aligned16(dy) || !aligned16(h13) || !aligned16(dq_row) || (col && !aligned16(dq_col)) ||
      !aligned16(dh13_t) || !aligned16(y_t))
    return fail(MX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  int rc;
  if ((rc = clear_padding(layout, ds_row, M, 2 * h, st))) return rc;
  if (col && (rc = clear_padding(layout, ds_col, 2 * h, M, st))) return rc;
  SwigluLaunch s{};
  s.dy = dy; s.h13 = h13; s.M = M; s.h = h; s.layout = layout;
  s.q_row = dq_row; s.s_row = ds_row;
  s.q_col = col ? dq_col : nullptr; s.s_col = col ? ds_col : nullptr;
  s.dh13_t = dh13_t; s.y_t = y_t;
  s.floor_scale = scale_mode == MX_SCALE_FLOOR;
  return launch_swiglu_bwd(s, st);
}

int mx_scaled_mm(const void* aq, const void* as, const void* bq, const void* bs, int64_t M, int64_t N, int64_t K,
                 void* c, int32_t* err_word, void* stream) {
  if (!aq || !as || !bq || !bs || !c) return fail(MX_ERR_INVALID_ARG, "null pointer argument");
  if (M <= 0 || N <= 0 || K <= 0) return fail(MX_ERR_INVALID_ARG, "sizes must be positive");
  if (M % 128 || N % 128 || K % 128)
    return fail(MX_ERR_UNSUPPORTED, "M, N, K must be multiples of 128 (got %lld, %lld, %lld)", (long long)M,
                (long long)N, (long long)K);
  if (!aligned16(aq) || !aligned16(as) || !aligned16(bq) || !aligned16(bs) || !aligned16(c))
    return fail(MX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return fail(MX_ERR_UNSUPPORTED, "dimension too large");
  GemmLaunch g{};
  g.mx = 1; g.mode = GEMM_DENSE; g.a = aq; g.sfa = as; g.b = bq; g.sfb = bs;
  g.M = M; g.N = N; g.K = K; g.E = 1; g.c0 = c; g.err = err_word;
  return launch_gemm(g, (cudaStream_t)stream);
}

int mx_grouped_mm(int mode, const void* aq, const void* as, const void* bq, const void* bs, int64_t M_total,
                  int64_t N, int64_t K, const int32_t* offs, int32_t E, int32_t pad_multiple, void* c,
                  int32_t* err_word, void* stream) {
  if (mode != MX_GROUP_M && mode != MX_GROUP_K) return fail(MX_ERR_INVALID_ARG, "mode must be MX_GROUP_M or MX_GROUP_K");
  if (!aq || !as || !bq || !bs || !c || !offs) return fail(MX_ERR_INVALID_ARG, "null pointer argument");
  if (M_total <= 0 || N <= 0 || K <= 0) return fail(MX_ERR_INVALID_ARG, "sizes must be positive");
  if (E < 1 || E > 1024) return fail(MX_ERR_INVALID_ARG, "E must be in [1, 1024] (got %d)", E);
  if (pad_multiple != 128) return fail(MX_ERR_UNSUPPORTED, "pad_multiple must be 128 (got %d)", pad_multiple);
  if (M_total % 128 || N % 128 || K % 128)
    return fail(MX_ERR_UNSUPPORTED, "M_total, N, K must be multiples of 128");
  if (!aligned16(aq) || !aligned16(as) || !aligned16(bq) || !aligned16(bs) || !aligned16(c))
    return fail(MX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  if (M_total > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return fail(MX_ERR_UNSUPPORTED, "dimension too large");
  GemmLaunch g{};
  g.mx = 1; g.a = aq; g.sfa = as; g.b = bq; g.sfb = bs; g.offs = offs; g.E = E; g.c0 = c; g.err = err_word;
  if (mode == MX_GROUP_M) {
    g.mode = GEMM_GROUP_M; g.M = M_total; g.N = N; g.K = K;
  } else {
    g.mode = GEMM_GROUP_K; g.M = N; g.N = K; g.K = M_total;
  }
  return launch_gemm(g, (cudaStream_t)stream);
}

// ---- FP8 per-tensor recipe ("[mxfp8 training] unified MXFP8TrainingConfig
// and MXFP8TrainingTensor", FP8 GroupedMM)

int mx_fp8_amax(const void* x, int64_t batch, int64_t n, float* amax, void* stream) {
  if (!x || !amax) return fail(MX_ERR_INVALID_ARG, "null pointer argument");
  if (batch <= 0 || n <= 0) return fail(MX_ERR_INVALID_ARG, "batch and n must be positive");
  if (batch > 65535) return fail(MX_ERR_UNSUPPORTED, "at most 65535 items");
  if (n % 8) return fail(MX_ERR_UNSUPPORTED, "n must be a multiple of 8 (got %lld)", (long long)n);
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(amax) & 3)) return fail(MX_ERR_ALIGNMENT, "x must be 16-byte aligned");
  return launch_fp8_amax(x, batch, n, amax, (cudaStream_t)stream);
}

int mx_fp8_quantize(const void* x, int64_t batch, int64_t rows, int64_t cols, const float* amax, int axis,
                    void* q_row, void* q_col, void* stream) {
  if (!x || !amax) return fail(MX_ERR_INVALID_ARG, "x or amax is null");
  if (batch <= 0 || rows <= 0 || cols <= 0) return fail(MX_ERR_INVALID_ARG, "sizes must be positive");
  if (axis < MX_ROW || axis > MX_BOTH) return fail(MX_ERR_INVALID_ARG, "axis must be MX_ROW, MX_COL or MX_BOTH");
  const bool row = axis & MX_ROW, col = axis & MX_COL;
  if (cols % 32) return fail(MX_ERR_UNSUPPORTED, "cols must be a multiple of 32 (got %lld)", (long long)cols);
  if (col && rows % 32) return fail(MX_ERR_UNSUPPORTED, "columnwise needs rows %% 32 == 0 (got %lld)", (long long)rows);
  if ((row && !q_row) || (col && !q_col)) return fail(MX_ERR_INVALID_ARG, "output is null");
  if (!aligned16(x) || (row && !aligned16(q_row)) || (col && !aligned16(q_col)))
    return fail(MX_ERR_ALIGNMENT, "x and code buffers must be 16-byte aligned");
  if (rows > INT32_MAX || cols > INT32_MAX || batch > INT32_MAX) return fail(MX_ERR_UNSUPPORTED, "dimension too large");
  QuantLaunch q{};
  q.x = x; q.rows = rows; q.cols = cols; q.batch = (int32_t)batch; q.layout = MX_SCALE_LINEAR;
  q.q_row = row ? q_row : nullptr;
  q.q_col = col ? q_col : nullptr; q.qc_ld = rows; q.qc_off = 0; q.qc_bs = rows * cols;
  q.tw = 1; q.amax = amax;
  return launch_quant(q, (cudaStream_t)stream);
}

int mx_fp8_grouped_mm(int mode, const void* aq, const float* amax_a, const void* bq, const float* amax_b,
                      int64_t M_total, int64_t N, int64_t K, const int32_t* offs, int32_t E, int32_t pad_multiple,
                      void* c, int32_t* err_word, void* stream) {
  if (mode != MX_GROUP_M && mode != MX_GROUP_K) return fail(MX_ERR_INVALID_ARG, "mode must be MX_GROUP_M or MX_GROUP_K");
  if (!aq || !amax_a || !bq || !amax_b || !c || !offs) return fail(MX_ERR_INVALID_ARG, "null pointer argument");
  if (M_total <= 0 || N <= 0 || K <= 0) return fail(MX_ERR_INVALID_ARG, "sizes must be positive");
  if (E < 1 || E > 1024) return fail(MX_ERR_INVALID_ARG, "E must be in [1, 1024] (got %d)", E);
  if (pad_multiple != 128) return fail(MX_ERR_UNSUPPORTED, "pad_multiple must be 128 (got %d)", pad_multiple);
  if (M_total % 128 || N % 128 || K % 128) return fail(MX_ERR_UNSUPPORTED, "M_total, N, K must be multiples of 128");
  if (!aligned16(aq) || !aligned16(bq) || !aligned16(c)) return fail(MX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  if (M_total > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return fail(MX_ERR_UNSUPPORTED, "dimension too large");
  GemmLaunch g{};
  g.mx = 1; g.tw = 1; g.a = aq; g.b = bq; g.offs = offs; g.E = E; g.c0 = c; g.err = err_word;
  g.amax_a = amax_a; g.amax_b = amax_b;
  if (mode == MX_GROUP_M) {
    g.mode = GEMM_GROUP_M; g.M = M_total; g.N = N; g.K = K; g.amax_b_per_expert = 1;
  } else {
    g.mode = GEMM_GROUP_K; g.M = N; g.N = K; g.K = M_total; g.amax_b_per_expert = 0;
  }
  return launch_gemm(g, (cudaStream_t)stream);
}

int mx_bf16_wgrad(const void* a, const void* b, int64_t M_total, int64_t N, int64_t K, const int32_t* offs,
                  int32_t E, int32_t pad_multiple, void* c, int32_t* err_word, void* stream) {
  if (!a || !b || !c) return fail(MX_ERR_INVALID_ARG, "null pointer argument");
  if (M_total <= 0 || N <= 0 || K <= 0) return fail(MX_ERR_INVALID_ARG, "sizes must be positive");
  if (M_total % 128 || N % 128 || K % 128) return fail(MX_ERR_UNSUPPORTED, "M_total, N, K must be multiples of 128");
  if (offs) {
    if (E < 1 || E > 1024) return fail(MX_ERR_INVALID_ARG, "E must be in [1, 1024] (got %d)", E);
    if (pad_multiple != 128) return fail(MX_ERR_UNSUPPORTED, "pad_multiple must be 128 (got %d)", pad_multiple);
  } else if (E != 1) {
    return fail(MX_ERR_INVALID_ARG, "offs = NULL needs E = 1");
  }
  if (!aligned16(a) || !aligned16(b) || !aligned16(c)) return fail(MX_ERR_ALIGNMENT, "buffers must be 16-byte aligned");
  GemmLaunch g{};
  g.mx = 0; g.a = a; g.b = b; g.M = N; g.N = K; g.K = M_total; g.c0 = c; g.err = err_word;
  g.mode = offs ? GEMM_GROUP_K : GEMM_DENSE; g.offs = offs; g.E = offs ? E : 1;
  return launch_gemm(g, (cudaStream_t)stream);
}

int mx_mlp_workspace_size(int64_t M_total, int64_t d, int64_t h, int32_t E, int recipe, size_t* ctx_bytes,
                          size_t* scratch_bytes) {
  if (!ctx_bytes || !scratch_bytes) return fail(MX_ERR_INVALID_ARG, "null output pointer");
  if (M_total <= 0 || d <= 0 || h <= 0 || E < 0) return fail(MX_ERR_INVALID_ARG, "sizes must be positive");
  if (!valid_recipe(recipe)) return fail(MX_ERR_INVALID_ARG, "unknown recipe");
  const MlpBuffers b = carve(nullptr, nullptr, M_total, d, h, E > 0 ? E : 1, recipe);
  *ctx_bytes = b.ctx_bytes;
  *scratch_bytes = b.scratch_bytes;
  return MX_OK;
}

int mx_mlp_ctx_layout(int64_t M_total, int64_t d, int64_t h, int32_t E, int recipe, int tensor, size_t* offset,
                      size_t* bytes) {
  if (!offset || !bytes) return fail(MX_ERR_INVALID_ARG, "null output pointer");
  if (M_total <= 0 || d <= 0 || h <= 0 || E < 0) return fail(MX_ERR_INVALID_ARG, "sizes must be positive");
  if (!valid_recipe(recipe)) return fail(MX_ERR_INVALID_ARG, "unknown recipe");
  const int64_t Ew = E > 0 ? E : 1;
  uint8_t* const base = reinterpret_cast<uint8_t*>(uintptr_t(1) << 40);  // any non-null base: offsets only
  const MlpBuffers b = carve(base, nullptr, M_total, d, h, Ew, recipe);
  const uint8_t* p = nullptr;
  int64_t n = 0;
  switch (tensor) {
    case MX_CTX_H13: p = b.h13; n = M_total * 2 * h * 2; break;
    case MX_CTX_XQ_COL: p = b.xq_c; n = d * M_total; break;
    case MX_CTX_XS_COL: p = b.xs_c; n = mma_scale_bytes(d, M_total); break;
    case MX_CTX_YQ_COL: p = b.yq_c; n = h * M_total; break;
    case MX_CTX_YS_COL: p = b.ys_c; n = mma_scale_bytes(h, M_total); break;
    case MX_CTX_X_T: p = b.x_t; n = d * M_total * 2; break;
    case MX_CTX_W13Q_COL: p = b.w13q_c; n = Ew * d * 2 * h; break;
    case MX_CTX_W13S_COL: p = b.w13s_c; n = Ew * mma_scale_bytes(d, 2 * h); break;
    case MX_CTX_W2Q_COL: p = b.w2q_c; n = Ew * h * d; break;
    case MX_CTX_W2S_COL: p = b.w2s_c; n = Ew * mma_scale_bytes(h, d); break;
    default: return fail(MX_ERR_INVALID_ARG, "unknown context tensor %d", tensor);
  }
  if (!p) return fail(MX_ERR_UNSUPPORTED, "this recipe keeps no context tensor %d", tensor);
  *offset = (size_t)(p - base);
  *bytes = (size_t)n;
  return MX_OK;
}

int mx_mlp_fwd(const void* x, const void* w1, const void* w3, const void* w2, int64_t M, int64_t d, int64_t h,
               const int32_t* offs, int32_t E, int32_t pad_multiple, int recipe, void* ctx, void* scratch, void* out,
               int32_t* err_word, void* stream) {
  int rc = check_mlp_args(x, w1, w3, w2, M, d, h, offs, E, pad_multiple, recipe, ctx, scratch);
  if (rc) return rc;
  if (!out || !aligned16(out)) return fail(out ? MX_ERR_ALIGNMENT : MX_ERR_INVALID_ARG, "bad out pointer");
  const bool grouped = offs != nullptr;
  const int64_t Ew = grouped ? E : 1;
  const bool hp = recipe_hp(recipe);
  const int fl = recipe_floor(recipe);
  cudaStream_t st = (cudaStream_t)stream;
  MlpBuffers b = carve(ctx, scratch, M, d, h, Ew, recipe);

  // F1: x -> rowwise MX (+ columnwise MX, or bf16 transpose for the HP recipe)
  {
    QuantLaunch q{};
    q.floor_scale = fl;
    q.x = x; q.rows = M; q.cols = d; q.batch = 1; q.layout = MX_SCALE_MMA; q.err = err_word;
    q.q_row = b.xq_r; q.s_row = b.xs_r;
    if (hp) { q.t_col = b.x_t; q.tc_ld = M; }
    else { q.q_col = b.xq_c; q.s_col = b.xs_c; q.qc_ld = M; }
    if ((rc = launch_quant(q, st))) return rc;
  }
  // F2: w1, w3 -> packed w13 rowwise [2h, d] and columnwise [d, 2h], per expert
  for (int half = 0; half < 2; ++half) {
    QuantLaunch q{};
    q.floor_scale = fl;
    q.x = half ? w3 : w1; q.rows = h; q.cols = d; q.batch = (int32_t)Ew; q.layout = MX_SCALE_MMA; q.err = err_word;
    q.q_row = b.w13q_r + half * h * d;
    q.s_row = b.w13s_r + half * (h / 128) * (d / 128) * 512;
    q.qr_bs = 2 * h * d;
    q.sr_bs = mma_scale_bytes(2 * h, d);
    q.q_col = b.w13q_c; q.s_col = b.w13s_c;
    q.qc_ld = 2 * h; q.qc_off = half * h; q.qc_bs = d * 2 * h; q.sc_bs = mma_scale_bytes(d, 2 * h);
    if ((rc = launch_quant(q, st))) return rc;
  }
  // F3 + F4 in one kernel: the w13 GEMM stores h13 and, in its epilogue,
  // y = SwiGLU(h13) as rowwise MXFP8 (+ columnwise for the MXFP8-wgrad
  // recipes, whose weight gradient of w2 contracts y over tokens).  The
  // epilogue overlaps the next tile's main loop.  With a(g) from the table
  // the fused forward wins from d = 4096 on (M = 8192, h = 8192: 0.630 ms
  // against 0.714 ms for the GEMM and the SwiGLU kernel); shorter
  // contractions, where the epilogue can outlast the main loop, run the two
  // kernels instead (bit-identical).
#ifndef MX_FUSE_DUAL_MIN_K
#define MX_FUSE_DUAL_MIN_K 4096
#endif
  constexpr int64_t kFuseDualMinK = MX_FUSE_DUAL_MIN_K;
  const bool fuse = hp || d >= kFuseDualMinK;
  {
    GemmLaunch g{};
    g.mx = 1; g.mode = grouped ? GEMM_GROUP_M : GEMM_DENSE;
    g.a = b.xq_r; g.sfa = b.xs_r; g.b = b.w13q_r; g.sfb = b.w13s_r;
    g.M = M; g.N = 2 * h; g.K = d; g.offs = offs; g.E = (int32_t)Ew; g.c0 = b.h13; g.err = err_word;
    if (fuse) {
      if ((rc = silu_table_address(&g.silu_a, st))) return rc;
      g.fuse_swiglu = 1; g.yq = b.yq_r; g.ys = b.ys_r; g.floor_scale = fl;
      if (!hp) { g.yq_col = b.yq_c; g.ys_col = b.ys_c; }
    }
    if ((rc = launch_gemm(g, st))) return rc;
  }
  if (!fuse) {
    SwigluLaunch s{};
    s.floor_scale = fl;
    s.h13 = b.h13; s.M = M; s.h = h; s.layout = MX_SCALE_MMA; s.err = err_word;
    s.q_row = b.yq_r; s.s_row = b.ys_r;
    s.q_col = b.yq_c; s.s_col = b.ys_c;
    if ((rc = silu_table_address(&s.silu_a, st))) return rc;
    if ((rc = launch_swiglu_fwd(s, st))) return rc;
  }
  // F5: w2 -> rowwise [d, h] and columnwise [h, d], per expert
  {
    QuantLaunch q{};
    q.floor_scale = fl;
    q.x = w2; q.rows = d; q.cols = h; q.batch = (int32_t)Ew; q.layout = MX_SCALE_MMA; q.err = err_word;
    q.q_row = b.w2q_r; q.s_row = b.w2s_r;
    q.q_col = b.w2q_c; q.s_col = b.w2s_c;
    q.qc_ld = d; q.qc_off = 0; q.qc_bs = h * d; q.sc_bs = mma_scale_bytes(h, d);
    if ((rc = launch_quant(q, st))) return rc;
  }
  // F6: out = y . w2^T
  {
    GemmLaunch g{};
    g.mx = 1; g.mode = grouped ? GEMM_GROUP_M : GEMM_DENSE;
    g.a = b.yq_r; g.sfa = b.ys_r; g.b = b.w2q_r; g.sfb = b.w2s_r;
    g.M = M; g.N = d; g.K = h; g.offs = offs; g.E = (int32_t)Ew; g.c0 = out; g.err = err_word;
    if ((rc = launch_gemm(g, st))) return rc;
  }
  return MX_OK;
}

int mx_mlp_bwd(const void* ctx, const void* dout, const void* x, const void* w1, const void* w3, const void* w2,
               int64_t M, int64_t d, int64_t h, const int32_t* offs, int32_t E, int32_t pad_multiple, int recipe,
               void* scratch, void* dx, void* dw1, void* dw3, void* dw2, int32_t* err_word, void* stream) {
  int rc = check_mlp_args(x, w1, w3, w2, M, d, h, offs, E, pad_multiple, recipe, ctx, scratch);
  if (rc) return rc;
  if (!dout || !dx || !dw1 || !dw3 || !dw2) return fail(MX_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(dout) || !aligned16(dx) || !aligned16(dw1) || !aligned16(dw3) || !aligned16(dw2))
    return fail(MX_ERR_ALIGNMENT, "tensor pointers must be 16-byte aligned");
  const bool grouped = offs != nullptr;
  const int64_t Ew = grouped ? E : 1;
  const bool hp = recipe_hp(recipe);
  const int fl = recipe_floor(recipe);
  cudaStream_t st = (cudaStream_t)stream;
  MlpBuffers b = carve(const_cast<void*>(ctx), scratch, M, d, h, Ew, recipe);

  // B1: dout -> rowwise MX (+ columnwise MX, or bf16 transpose for HP)
  {
    QuantLaunch q{};
    q.floor_scale = fl;
    q.x = dout; q.rows = M; q.cols = d; q.batch = 1; q.layout = MX_SCALE_MMA; q.err = err_word;
    q.q_row = b.dq_r; q.s_row = b.ds_r;
    if (hp) { q.t_col = b.dout_t; q.tc_ld = M; }
    else { q.q_col = b.dq_c; q.s_col = b.ds_c; q.qc_ld = M; }
    if ((rc = launch_quant(q, st))) return rc;
  }
  // B2: dy = dout . w2  (B operand: columnwise w2, [h, d] per expert)
  {
    GemmLaunch g{};
    g.mx = 1; g.mode = grouped ? GEMM_GROUP_M : GEMM_DENSE;
    g.a = b.dq_r; g.sfa = b.ds_r; g.b = b.w2q_c; g.sfb = b.w2s_c;
    g.M = M; g.N = h; g.K = d; g.offs = offs; g.E = (int32_t)Ew; g.c0 = b.dy; g.err = err_word;
    if ((rc = launch_gemm(g, st))) return rc;
  }
  // B4: dh13 = SwiGLU'(dy, h13) -> rowwise MX (+ columnwise MX, or bf16
  // transposed dh13 and y for HP)
  {
    SwigluLaunch s{};
    s.floor_scale = fl;
    s.dy = b.dy; s.h13 = b.h13; s.M = M; s.h = h; s.layout = MX_SCALE_MMA; s.err = err_word;
    s.q_row = b.dhq_r; s.s_row = b.dhs_r;
    if (hp) { s.dh13_t = b.dh13_t; s.y_t = b.y_t; }
    else { s.q_col = b.dhq_c; s.s_col = b.dhs_c; }
    if ((rc = launch_swiglu_bwd(s, st))) return rc;
  }
  // B3: dW2 = dout^T . y (per expert over its tokens)
  {
    GemmLaunch g{};
    g.mx = hp ? 0 : 1; g.mode = grouped ? GEMM_GROUP_K : GEMM_DENSE;
    if (hp) { g.a = b.dout_t; g.b = b.y_t; }
    else { g.a = b.dq_c; g.sfa = b.ds_c; g.b = b.yq_c; g.sfb = b.ys_c; }
    g.M = d; g.N = h; g.K = M; g.offs = offs; g.E = (int32_t)Ew; g.c0 = dw2; g.err = err_word;
    if ((rc = launch_gemm(g, st))) return rc;
  }
  // B5: dx = dh13 . w13  (B operand: columnwise w13, [d, 2h] per expert)
  {
    GemmLaunch g{};
    g.mx = 1; g.mode = grouped ? GEMM_GROUP_M : GEMM_DENSE;
    g.a = b.dhq_r; g.sfa = b.dhs_r; g.b = b.w13q_c; g.sfb = b.w13s_c;
    g.M = M; g.N = d; g.K = 2 * h; g.offs = offs; g.E = (int32_t)Ew; g.c0 = dx; g.err = err_word;
    if ((rc = launch_gemm(g, st))) return rc;
  }
  // B6: dW13 = dh13^T . x, rows [0, h) -> dw1, [h, 2h) -> dw3
  {
    GemmLaunch g{};
    g.mx = hp ? 0 : 1; g.mode = grouped ? GEMM_GROUP_K : GEMM_DENSE;
    if (hp) { g.a = b.dh13_t; g.b = b.x_t; }
    else { g.a = b.dhq_c; g.sfa = b.dhs_c; g.b = b.xq_c; g.sfb = b.xs_c; }
    g.M = 2 * h; g.N = d; g.K = M; g.offs = offs; g.E = (int32_t)Ew;
    g.c0 = dw1; g.c1 = dw3; g.split = h; g.err = err_word;
    if ((rc = launch_gemm(g, st))) return rc;
  }
  return MX_OK;
}

// ---- per-linear MXFP8 path ("TrainingWeightWrapperTensor base class ...",
// linear override; "Add MXFP8 fused-MLP overrides in torchtitan": non-MLP
// linears keep the per-linear path)

int mx_linear_workspace_size(int64_t M, int64_t K, int64_t N, int recipe, size_t* ctx_bytes,
                             size_t* scratch_bytes) {
  int rc = check_linear_args(M, K, N, recipe);
  if (rc) return rc;
  if (!ctx_bytes || !scratch_bytes) return fail(MX_ERR_INVALID_ARG, "null output pointer");
  LinearBuffers b = carve_linear(nullptr, nullptr, M, K, N, recipe);
  *ctx_bytes = b.ctx_bytes;
  *scratch_bytes = b.scratch_bytes;
  return MX_OK;
}

int mx_linear_fwd(const void* x, const void* w, int64_t M, int64_t K, int64_t N, int recipe, void* ctx,
                  void* scratch, void* out, int32_t* err_word, void* stream) {
  int rc = check_linear_args(M, K, N, recipe);
  if (rc) return rc;
  if (!x || !w || !ctx || !scratch || !out) return fail(MX_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(x) || !aligned16(w) || !aligned16(ctx) || !aligned16(scratch) || !aligned16(out))
    return fail(MX_ERR_ALIGNMENT, "tensor pointers must be 16-byte aligned");
  const bool hp = recipe_hp(recipe);
  const int fl = recipe_floor(recipe);
  cudaStream_t st = (cudaStream_t)stream;
  LinearBuffers b = carve_linear(ctx, scratch, M, K, N, recipe);
  {  // x -> MX(R) along K; MX(C) along M (or bf16 x^T) saved for the weight gradient
    QuantLaunch q{};
    q.floor_scale = fl;
    q.x = x; q.rows = M; q.cols = K; q.batch = 1; q.layout = MX_SCALE_MMA; q.err = err_word;
    q.q_row = b.xq_r; q.s_row = b.xs_r;
    if (hp) { q.t_col = b.x_t; q.tc_ld = M; }
    else { q.q_col = b.xq_c; q.s_col = b.xs_c; q.qc_ld = M; }
    if ((rc = launch_quant(q, st))) return rc;
  }
  {  // w -> MX(R) along K
    QuantLaunch q{};
    q.floor_scale = fl;
    q.x = w; q.rows = N; q.cols = K; q.batch = 1; q.layout = MX_SCALE_MMA; q.err = err_word;
    q.q_row = b.wq_r; q.s_row = b.ws_r;
    if ((rc = launch_quant(q, st))) return rc;
  }
  GemmLaunch g{};
  g.mx = 1; g.mode = GEMM_DENSE;
  g.a = b.xq_r; g.sfa = b.xs_r; g.b = b.wq_r; g.sfb = b.ws_r;
  g.M = M; g.N = N; g.K = K; g.E = 1; g.c0 = out; g.err = err_word;
  return launch_gemm(g, st);
}

int mx_linear_bwd(const void* ctx, const void* dout, const void* w, int64_t M, int64_t K, int64_t N, int recipe,
                  void* scratch, void* dx, void* dw, int32_t* err_word, void* stream) {
  int rc = check_linear_args(M, K, N, recipe);
  if (rc) return rc;
  if (!ctx || !dout || !w || !scratch || !dx || !dw) return fail(MX_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned16(ctx) || !aligned16(dout) || !aligned16(w) || !aligned16(scratch) || !aligned16(dx) ||
      !aligned16(dw))
    return fail(MX_ERR_ALIGNMENT, "tensor pointers must be 16-byte aligned");
  const bool hp = recipe_hp(recipe);
  const int fl = recipe_floor(recipe);
  cudaStream_t st = (cudaStream_t)stream;
  LinearBuffers b = carve_linear(const_cast<void*>(ctx), scratch, M, K, N, recipe);
  {  // dout -> MX(R) along N; MX(C) along M (or bf16 dout^T)
    QuantLaunch q{};
    q.floor_scale = fl;
    q.x = dout; q.rows = M; q.cols = N; q.batch = 1; q.layout = MX_SCALE_MMA; q.err = err_word;
    q.q_row = b.dq_r; q.s_row = b.ds_r;
    if (hp) { q.t_col = b.dout_t; q.tc_ld = M; }
    else { q.q_col = b.dq_c; q.s_col = b.ds_c; q.qc_ld = M; }
    if ((rc = launch_quant(q, st))) return rc;
  }
  {  // w -> MX(C) along N: codes [K, N]
    QuantLaunch q{};
    q.floor_scale = fl;
    q.x = w; q.rows = N; q.cols = K; q.batch = 1; q.layout = MX_SCALE_MMA; q.err = err_word;
    q.q_col = b.wq_c; q.s_col = b.ws_c; q.qc_ld = N;
    if ((rc = launch_quant(q, st))) return rc;
  }
  {  // dx = dout . w
    GemmLaunch g{};
    g.mx = 1; g.mode = GEMM_DENSE;
    g.a = b.dq_r; g.sfa = b.ds_r; g.b = b.wq_c; g.sfb = b.ws_c;
    g.M = M; g.N = K; g.K = N; g.E = 1; g.c0 = dx; g.err = err_word;
    if ((rc = launch_gemm(g, st))) return rc;
  }
  // dw = dout^T . x
  GemmLaunch g{};
  g.mx = hp ? 0 : 1; g.mode = GEMM_DENSE;
  if (hp) { g.a = b.dout_t; g.b = b.x_t; }
  else { g.a = b.dq_c; g.sfa = b.ds_c; g.b = b.xq_c; g.sfb = b.xs_c; }
  g.M = N; g.N = K; g.K = M; g.E = 1; g.c0 = dw; g.err = err_word;
  return launch_gemm(g, st);
}

// ---- token-group padding (pages "[mxfp8] refactor model converter; use token
// group padding kernels in torchao" and "Add MXFP8 fused-MLP overrides in
// torchtitan", Summary)

size_t mx_token_group_pad_workspace(int64_t R, int32_t E) {
  if (R < 0 || E < 1) return 0;
  return token_group_pad_workspace(R, E);
}

int mx_token_group_pad(const int32_t* expert_of, int64_t R, int32_t E, int32_t pad_multiple, int64_t M_cap,
                       int32_t* offs, int32_t* row_dst, int32_t* row_src, void* workspace, int32_t* err_word,
                       void* stream) {
  if (R < 0 || M_cap < 0) return fail(MX_ERR_INVALID_ARG, "R and M_cap must be >= 0");
  if (E < 1 || E > 1024) return fail(MX_ERR_UNSUPPORTED, "need 1 <= E <= 1024 (got %d)", E);
  if (pad_multiple != 128) return fail(MX_ERR_UNSUPPORTED, "pad_multiple must be 128 (got %d)", pad_multiple);
  if (M_cap % 128) return fail(MX_ERR_UNSUPPORTED, "M_cap must be a multiple of 128");
  if (M_cap > INT32_MAX || R > INT32_MAX) return fail(MX_ERR_UNSUPPORTED, "R and M_cap must fit in int32");
  if (!offs || (M_cap > 0 && !row_src)) return fail(MX_ERR_INVALID_ARG, "offs or row_src is null");
  if (R > 0 && (!expert_of || !row_dst || !workspace))
    return fail(MX_ERR_INVALID_ARG, "expert_of, row_dst and workspace are required when R > 0");
  return launch_token_group_pad(expert_of, R, E, pad_multiple, M_cap, offs, row_dst, row_src, workspace, err_word,
                                (cudaStream_t)stream);
}

int mx_gather_rows(const void* x, int64_t rows_in, int64_t cols, const int32_t* src, int64_t rows_out,
                   int32_t div, void* y, int32_t* err_word, void* stream) {
  if (rows_in < 0 || rows_out < 0 || cols <= 0 || div < 1)
    return fail(MX_ERR_INVALID_ARG, "need rows_in, rows_out >= 0, cols > 0, div >= 1");
  if (cols % 8) return fail(MX_ERR_UNSUPPORTED, "cols must be a multiple of 8 (got %lld)", (long long)cols);
  if (rows_out > 0 && (!src || !y || (rows_in > 0 && !x))) return fail(MX_ERR_INVALID_ARG, "null pointer");
  if ((x && !aligned16(x)) || (y && !aligned16(y))) return fail(MX_ERR_ALIGNMENT, "x and y must be 16-byte aligned");
  return launch_gather_rows(x, rows_in, cols, src, rows_out, div, y, err_word, (cudaStream_t)stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Forward pass with a library-owned scratch array (no allocation anywhere).

namespace {
// The temporary buffer of mx_mlp_fwd_static_scratch.  In host code this name
// is only a host-side handle, not a device address: the device address is
// looked up with cudaGetSymbolAddress in the CUDA context that is current at
// the call (the array has one instance per context) and cached under that
// context's unique ID, so a reset device or a caller's own non-primary
// context gets its own lookup instead of a stale address.
static __device__ __align__(256) uint8_t g_static_scratch[MX_STATIC_SCRATCH_BYTES];

CtxCache g_static_cache;

// Device address of g_static_scratch in the current context (the runtime
// binds the device's primary context if none is current).
int static_scratch_address(void** out) {
  return g_static_cache.lookup(out, [](void** p) {
    const cudaError_t e = cudaGetSymbolAddress(p, g_static_scratch);
    return cuda_status(e, "cudaGetSymbolAddress(static scratch)");
  });
}
}  // namespace

extern "C" int mx_mlp_fwd_static_scratch(const void* x, const void* w1, const void* w3, const void* w2,
                                         int64_t M_total, int64_t d, int64_t h, const int32_t* offs, int32_t E,
                                         int32_t pad_multiple, int recipe, void* ctx, void* out, int32_t* err_word,
                                         void* stream) {
  size_t ctx_bytes = 0, scratch_bytes = 0;
  int rc = mx_mlp_workspace_size(M_total, d, h, offs ? E : 0, recipe, &ctx_bytes, &scratch_bytes);
  if (rc) return rc;
  if (scratch_bytes > (size_t)MX_STATIC_SCRATCH_BYTES)
    return fail(MX_ERR_UNSUPPORTED,
                "mx_mlp_fwd_static_scratch: this problem needs %zu scratch bytes, more than the static "
                "array's %u; use mx_mlp_fwd with a caller buffer",
                scratch_bytes, (unsigned)MX_STATIC_SCRATCH_BYTES);
  void* scratch = nullptr;
  if ((rc = static_scratch_address(&scratch))) return rc;
  return mx_mlp_fwd(x, w1, w3, w2, M_total, d, h, offs, E, pad_multiple, recipe, ctx, scratch, out, err_word,
                    stream);
}

// ---------------------------------------------------------------------------
// Self-test of the bounded pipeline waits (failure detection without a GPU
// fault): a 256x256x256 MXFP8 GEMM on library-owned buffers whose producer
// issues no copies, so the MMA and epilogue waits run out of their bound.

namespace {
constexpr size_t kSelftestBytes = 256 * 256 * 2 + 2 * 2048 + 256 * 256 * 2;  // A, B codes; scales; C
static __device__ __align__(256) uint8_t g_selftest[kSelftestBytes];
}  // namespace

extern "C" int mx_selftest_silu_table(uint16_t* dst, void* stream) {
  if (!dst) return fail(MX_ERR_INVALID_ARG, "dst is required");
  const uint16_t* tab = nullptr;
  int rc = silu_table_address(&tab, (cudaStream_t)stream);
  if (rc) return rc;
  return cuda_status(cudaMemcpyAsync(dst, tab, 65536 * sizeof(uint16_t), cudaMemcpyDeviceToDevice,
                                     (cudaStream_t)stream),
                     "cudaMemcpyAsync(silu table)");
}

extern "C" int mx_selftest_wait_timeout(int32_t* err_word, void* stream) {
  if (!err_word) return fail(MX_ERR_INVALID_ARG, "err_word is required");
  uint8_t* base = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&base), g_selftest);
  if (e != cudaSuccess) return cuda_status(e, "cudaGetSymbolAddress(self-test buffers)");
  GemmLaunch g{};
  g.mx = 1; g.mode = GEMM_DENSE;
  g.a = base; g.b = base + 256 * 256;
  g.sfa = base + 2 * 256 * 256; g.sfb = base + 2 * 256 * 256 + 2048;
  g.c0 = base + 2 * 256 * 256 + 2 * 2048;
  g.M = 256; g.N = 256; g.K = 256; g.E = 1;
  g.starve = 1; g.err = err_word;
  return launch_gemm(g, (cudaStream_t)stream);
}
