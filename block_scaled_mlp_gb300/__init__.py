"""MXFP8 training MLP for Blackwell sm_103a: a thin ctypes binding of the C-ABI
library ``libmxmlp.so`` (declared in ``include/mxmlp.h``).

Every function here only marshals arguments: it checks tensor devices and
dtypes, allocates output tensors with PyTorch (device memory and streams are
all PyTorch is used for), and calls the C entry point of the same name on the
current CUDA stream.  There is no other code path: if the library is missing
the calls raise ``MxError``.

Tensors:
  bf16 activations/weights     torch.bfloat16, contiguous, on a CUDA device
  MXFP8 codes                  torch.uint8 (E4M3 bit patterns)
  scales                       torch.uint8 (E8M0 bytes, MMA or linear layout)
  group offsets                torch.int32 on the device (cumulative ends)
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "MxError", "lib", "library_path", "ROW", "COL", "BOTH", "SCALE_LINEAR", "SCALE_MMA",
    "RECIPE_RCEIL", "RECIPE_RCEIL_WGRAD_HP", "RECIPE_FLOOR", "RECIPE_FLOOR_WGRAD_HP", "SCALE_RCEIL", "SCALE_FLOOR", "GROUP_M", "GROUP_K", "mma_scale_bytes",
    "quantize", "swiglu_quant", "swiglu_quant_bwd", "scaled_mm", "grouped_mm", "bf16_wgrad",
    "mlp_workspace_size", "mlp_ctx_layout", "mlp_fwd", "mlp_bwd", "mlp_fwd_static_scratch", "MlpContext", "ErrorWord",
    "token_group_pad", "token_group_capacity", "gather_rows", "linear_fwd", "linear_bwd", "LinearContext",
    "KERNEL_FAMILIES", "launch_counts", "fp8_amax", "fp8_quantize", "fp8_grouped_mm",
]

ROW, COL, BOTH = 1, 2, 3
SCALE_LINEAR, SCALE_MMA = 0, 1
RECIPE_RCEIL, RECIPE_RCEIL_WGRAD_HP, RECIPE_FLOOR, RECIPE_FLOOR_WGRAD_HP = 0, 1, 2, 3
SCALE_RCEIL, SCALE_FLOOR = 0, 1
GROUP_M, GROUP_K = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libmxmlp.so")
_lib = None

_V, _I64, _I32, _I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int
_SIGS = {
    "mx_version": ([], _I),
    "mx_status_string": ([_I], ctypes.c_char_p),
    "mx_last_error": ([], ctypes.c_char_p),
    "mx_quantize": ([_V, _I64, _I64, _I, _I, _V, _V, _V, _V, _V], _I),
    "mx_quantize_mode": ([_V, _I64, _I64, _I, _I, _I, _V, _V, _V, _V, _V], _I),
    "mx_swiglu_quant": ([_V, _I64, _I64, _I, _I, _V, _V, _V, _V, _V], _I),
    "mx_swiglu_quant_bwd": ([_V, _V, _I64, _I64, _I, _I, _V, _V, _V, _V, _V, _V, _V], _I),
    "mx_swiglu_quant_mode": ([_V, _I64, _I64, _I, _I, _I, _V, _V, _V, _V, _V], _I),
    "mx_swiglu_quant_bwd_mode": ([_V, _V, _I64, _I64, _I, _I, _I, _V, _V, _V, _V, _V, _V, _V], _I),
    "mx_scaled_mm": ([_V, _V, _V, _V, _I64, _I64, _I64, _V, _V, _V], _I),
    "mx_grouped_mm": ([_I, _V, _V, _V, _V, _I64, _I64, _I64, _V, _I32, _I32, _V, _V, _V], _I),
    "mx_bf16_wgrad": ([_V, _V, _I64, _I64, _I64, _V, _I32, _I32, _V, _V, _V], _I),
    "mx_mlp_workspace_size": ([_I64, _I64, _I64, _I32, _I, ctypes.POINTER(ctypes.c_size_t),
                               ctypes.POINTER(ctypes.c_size_t)], _I),
    "mx_mlp_ctx_layout": ([_I64, _I64, _I64, _I32, _I, _I, ctypes.POINTER(ctypes.c_size_t),
                           ctypes.POINTER(ctypes.c_size_t)], _I),
    "mx_mlp_fwd": ([_V, _V, _V, _V, _I64, _I64, _I64, _V, _I32, _I32, _I, _V, _V, _V, _V, _V], _I),
    "mx_mlp_bwd": ([_V, _V, _V, _V, _V, _V, _I64, _I64, _I64, _V, _I32, _I32, _I, _V, _V, _V, _V, _V,
                    _V, _V], _I),
    "mx_mlp_fwd_static_scratch": ([_V, _V, _V, _V, _I64, _I64, _I64, _V, _I32, _I32, _I, _V, _V, _V, _V], _I),
    "mx_token_group_pad_workspace": ([_I64, _I32], ctypes.c_size_t),
    "mx_linear_workspace_size": ([_I64, _I64, _I64, _I, ctypes.POINTER(ctypes.c_size_t),
                                  ctypes.POINTER(ctypes.c_size_t)], _I),
    "mx_linear_fwd": ([_V, _V, _I64, _I64, _I64, _I, _V, _V, _V, _V, _V], _I),
    "mx_linear_bwd": ([_V, _V, _V, _I64, _I64, _I64, _I, _V, _V, _V, _V, _V], _I),
    "mx_token_group_pad": ([_V, _I64, _I32, _I32, _I64, _V, _V, _V, _V, _V, _V], _I),
    "mx_gather_rows": ([_V, _I64, _I64, _V, _I64, _I32, _V, _V, _V], _I),
    "mx_selftest_wait_timeout": ([_V, _V], _I),
    "mx_selftest_silu_table": ([_V, _V], _I),
    "mx_launch_counts": ([ctypes.POINTER(ctypes.c_int64), _I], _I),
    "mx_fp8_amax": ([_V, _I64, _I64, _V, _V], _I),
    "mx_fp8_quantize": ([_V, _I64, _I64, _I64, _V, _I, _V, _V, _V], _I),
    "mx_fp8_grouped_mm": ([_I, _V, _V, _V, _V, _I64, _I64, _I64, _V, _I32, _I32, _V, _V, _V], _I),
}


class MxError(RuntimeError):
    """A libmxmlp call failed (status code and message from the library)."""

    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def lib():
    """Load libmxmlp.so (built in-tree by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(library_path):
            raise MxError(-1, f"{library_path} is not built; run __graft_entry__.build()")
        L = ctypes.CDLL(library_path)
        for name, (args, res) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _check(rc: int):
    if rc != 0:
        L = lib()
        raise MxError(rc, f"{L.mx_status_string(rc).decode()}: {L.mx_last_error().decode()}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t, dtype, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise MxError(1, f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise MxError(1, f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise MxError(1, f"{name} must be contiguous")


KERNEL_FAMILIES = ("quant", "swiglu_fwd", "swiglu_bwd", "gemm", "gemm_swiglu", "dispatch", "memset")


def silu_table():
    """The library's table of a(g) = RN_bf16(g sigma(g)) over every bf16 g
    (entry b for the g with bits b), as a uint16 tensor on the current
    device."""
    t = torch.empty(65536, dtype=torch.uint16, device="cuda")
    _check(lib().mx_selftest_silu_table(t.data_ptr(), _stream()))
    return t


def launch_counts() -> dict:
    """The library's launch counters by kernel family (totals since load;
    take differences around the calls of interest)."""
    n = len(KERNEL_FAMILIES)
    buf = (ctypes.c_int64 * n)()
    got = lib().mx_launch_counts(buf, n)
    if got != n:
        raise MxError(got, f"library reports {got} kernel families, binding knows {n}")
    return {k: int(buf[i]) for i, k in enumerate(KERNEL_FAMILIES)}


def mma_scale_bytes(rows: int, cols: int) -> int:
    """Bytes of the MMA-layout scales of a [rows, cols] matrix (cols/32 scales per row)."""
    s = cols // 32
    return ((rows + 127) // 128) * ((s + 3) // 4) * 512


def _scales(rows, cols, layout, device, batch=None):
    n = mma_scale_bytes(rows, cols) if layout == SCALE_MMA else rows * (cols // 32)
    shape = (n,) if batch is None else (batch, n)
    return torch.empty(shape, dtype=torch.uint8, device=device)


class ErrorWord:
    """Device int32 that kernels OR their fault bits into."""

    def __init__(self, device=None):
        self.t = torch.zeros(1, dtype=torch.int32, device=device or "cuda")

    def ptr(self):
        return ctypes.c_void_p(self.t.data_ptr())

    def value(self) -> int:
        return int(self.t.item())

    def check(self):
        v = self.value()
        if v:
            raise MxError(v, f"device fault bits 0x{v:x} ({lib().mx_status_string(v).decode()})")


# ---------------------------------------------------------------- per-op calls


def quantize(x, axis=BOTH, layout=SCALE_MMA, scale_mode=SCALE_RCEIL):
    """MXFP8 cast of a bf16 [rows, cols] matrix.  Returns a dict with
    q_row [rows, cols], s_row, q_col [cols, rows], s_col (absent axes None)."""
    _need(x, torch.bfloat16, "x")
    rows, cols = x.shape
    dev = x.device
    out = dict(q_row=None, s_row=None, q_col=None, s_col=None)
    if axis & ROW:
        out["q_row"] = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
        out["s_row"] = _scales(rows, cols, layout, dev)
    if axis & COL:
        out["q_col"] = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
        out["s_col"] = _scales(cols, rows, layout, dev)
    _check(lib().mx_quantize_mode(_ptr(x), rows, cols, axis, layout, scale_mode, _ptr(out["q_row"]),
                                  _ptr(out["s_row"]), _ptr(out["q_col"]), _ptr(out["s_col"]), _stream()))
    return out


def swiglu_quant(h13, axis=BOTH, layout=SCALE_MMA, scale_mode=SCALE_RCEIL):
    """Fused SwiGLU of h13 [M, 2h] = [g | u] with dual MXFP8 quantization of
    y [M, h].  Returns dict(q_row [M,h], s_row, q_col [h,M], s_col)."""
    _need(h13, torch.bfloat16, "h13")
    M, h2 = h13.shape
    h = h2 // 2
    dev = h13.device
    out = dict(q_row=torch.empty((M, h), dtype=torch.uint8, device=dev), s_row=_scales(M, h, layout, dev),
               q_col=None, s_col=None)
    if axis & COL:
        out["q_col"] = torch.empty((h, M), dtype=torch.uint8, device=dev)
        out["s_col"] = _scales(h, M, layout, dev)
    _check(lib().mx_swiglu_quant_mode(_ptr(h13), M, h, axis, layout, scale_mode, _ptr(out["q_row"]),
                                      _ptr(out["s_row"]), _ptr(out["q_col"]), _ptr(out["s_col"]), _stream()))
    return out


def swiglu_quant_bwd(dy, h13, axis=BOTH, layout=SCALE_MMA, bf16_transposed=False, scale_mode=SCALE_RCEIL):
    """Fused SwiGLU backward: dh13 = [dg | du] quantized rowwise (and
    columnwise with axis=BOTH).  With bf16_transposed=True (rowwise only) it
    also returns dh13_t [2h, M] and y_t [h, M] in bf16."""
    _need(dy, torch.bfloat16, "dy")
    _need(h13, torch.bfloat16, "h13")
    M, h = dy.shape
    dev = dy.device
    out = dict(q_row=torch.empty((M, 2 * h), dtype=torch.uint8, device=dev),
               s_row=_scales(M, 2 * h, layout, dev), q_col=None, s_col=None, dh13_t=None, y_t=None)
    if axis & COL:
        out["q_col"] = torch.empty((2 * h, M), dtype=torch.uint8, device=dev)
        out["s_col"] = _scales(2 * h, M, layout, dev)
    if bf16_transposed:
        out["dh13_t"] = torch.empty((2 * h, M), dtype=torch.bfloat16, device=dev)
        out["y_t"] = torch.empty((h, M), dtype=torch.bfloat16, device=dev)
    _check(lib().mx_swiglu_quant_bwd_mode(_ptr(dy), _ptr(h13), M, h, axis, layout, scale_mode, _ptr(out["q_row"]),
                                          _ptr(out["s_row"]), _ptr(out["q_col"]), _ptr(out["s_col"]),
                                          _ptr(out["dh13_t"]), _ptr(out["y_t"]), _stream()))
    return out


def scaled_mm(aq, as_, bq, bs, err: ErrorWord | None = None):
    """C[M, N] = deq(A) deq(B)^T in bf16 (MMA-layout scales)."""
    _need(aq, torch.uint8, "aq")
    _need(bq, torch.uint8, "bq")
    M, K = aq.shape
    N = bq.shape[0]
    c = torch.empty((M, N), dtype=torch.bfloat16, device=aq.device)
    _check(lib().mx_scaled_mm(_ptr(aq), _ptr(as_), _ptr(bq), _ptr(bs), M, N, K, _ptr(c),
                              err.ptr() if err else None, _stream()))
    return c


def grouped_mm(mode, aq, as_, bq, bs, offs, pad_multiple=128, err: ErrorWord | None = None):
    """Grouped MXFP8 GEMM.  GROUP_M: aq [M_total, K], bq [E, N, K] -> [M_total, N].
    GROUP_K: aq [N, M_total], bq [K, M_total] -> [E, N, K]."""
    _need(offs, torch.int32, "offs")
    E = offs.numel()
    if mode == GROUP_M:
        M_total, K = aq.shape
        N = bq.shape[1]
        c = torch.empty((M_total, N), dtype=torch.bfloat16, device=aq.device)
    else:
        N, M_total = aq.shape
        K = bq.shape[0]
        c = torch.empty((E, N, K), dtype=torch.bfloat16, device=aq.device)
    _check(lib().mx_grouped_mm(mode, _ptr(aq), _ptr(as_), _ptr(bq), _ptr(bs), M_total, N, K, _ptr(offs), E,
                               pad_multiple, _ptr(c), err.ptr() if err else None, _stream()))
    return c


def bf16_wgrad(a, b, offs=None, pad_multiple=128, err: ErrorWord | None = None):
    """bf16 weight gradient: a [N, M_total], b [K, M_total] -> [E, N, K]
    (or [N, K] with offs=None)."""
    _need(a, torch.bfloat16, "a")
    _need(b, torch.bfloat16, "b")
    N, M_total = a.shape
    K = b.shape[0]
    E = 1 if offs is None else offs.numel()
    shape = (N, K) if offs is None else (E, N, K)
    c = torch.empty(shape, dtype=torch.bfloat16, device=a.device)
    _check(lib().mx_bf16_wgrad(_ptr(a), _ptr(b), M_total, N, K, _ptr(offs), E, pad_multiple, _ptr(c),
                               err.ptr() if err else None, _stream()))
    return c


# ---------------------------------------------------------------- FP8 per-tensor


def fp8_amax(x, batch_axes=0):
    """amax = max |x| per tensor (batch_axes=0: one value) or per leading
    index (batch_axes=1: one per expert), as a device fp32 tensor."""
    _need(x, torch.bfloat16, "x")
    batch = x.shape[0] if batch_axes else 1
    amax = torch.empty(batch, dtype=torch.float32, device=x.device)
    _check(lib().mx_fp8_amax(_ptr(x), batch, x.numel() // batch, _ptr(amax), _stream()))
    return amax


def fp8_quantize(x, amax, axis=ROW):
    """FP8 per-tensor codes of x [rows, cols] or [batch, rows, cols] with
    amax [batch] (device fp32).  Returns {"q_row": [.., rows, cols],
    "q_col": [.., cols, rows]} as requested by axis."""
    _need(x, torch.bfloat16, "x")
    lead = x.shape[:-2]
    rows, cols = x.shape[-2], x.shape[-1]
    batch = x.numel() // (rows * cols)
    out = {}
    if axis & ROW:
        out["q_row"] = torch.empty(lead + (rows, cols), dtype=torch.uint8, device=x.device)
    if axis & COL:
        out["q_col"] = torch.empty(lead + (cols, rows), dtype=torch.uint8, device=x.device)
    _check(lib().mx_fp8_quantize(_ptr(x), batch, rows, cols, _ptr(amax), axis, _ptr(out.get("q_row")),
                                 _ptr(out.get("q_col")), _stream()))
    return out


def fp8_grouped_mm(mode, aq, amax_a, bq, amax_b, offs, pad_multiple=128, err: ErrorWord | None = None):
    """Grouped GEMM on FP8 per-tensor operands.  GROUP_M: aq [M_total, K]
    (amax_a [1]), bq [E, N, K] (amax_b [E]) -> [M_total, N].  GROUP_K: aq
    [N, M_total], bq [K, M_total] (amax [1] each) -> [E, N, K]."""
    _need(offs, torch.int32, "offs")
    E = offs.numel()
    if mode == GROUP_M:
        M_total, K = aq.shape
        N = bq.shape[1]
        c = torch.empty((M_total, N), dtype=torch.bfloat16, device=aq.device)
    else:
        N, M_total = aq.shape
        K = bq.shape[0]
        c = torch.empty((E, N, K), dtype=torch.bfloat16, device=aq.device)
    _check(lib().mx_fp8_grouped_mm(mode, _ptr(aq), _ptr(amax_a), _ptr(bq), _ptr(amax_b), M_total, N, K, _ptr(offs),
                                   E, pad_multiple, _ptr(c), err.ptr() if err else None, _stream()))
    return c


# ---------------------------------------------------------------- MLP


def mlp_workspace_size(M_total, d, h, E=0, recipe=RECIPE_RCEIL):
    c = ctypes.c_size_t()
    s = ctypes.c_size_t()
    _check(lib().mx_mlp_workspace_size(M_total, d, h, E, recipe, ctypes.byref(c), ctypes.byref(s)))
    return c.value, s.value


CTX_TENSORS = ("h13", "xq_col", "xs_col", "yq_col", "ys_col", "x_t", "w13q_col", "w13s_col", "w2q_col",
               "w2s_col")


def mlp_ctx_layout(M_total, d, h, E, recipe, name):
    """(byte offset, bytes) of a saved tensor inside the mlp_fwd context."""
    off, n = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().mx_mlp_ctx_layout(M_total, d, h, E, recipe, CTX_TENSORS.index(name), ctypes.byref(off),
                                   ctypes.byref(n)))
    return off.value, n.value


class MlpContext:
    """What mlp_fwd saves for mlp_bwd (a caller-owned device buffer plus the
    call's arguments)."""

    def __init__(self, buf, args):
        self.buf = buf
        self.args = args

    def h13(self):
        """The saved w13 GEMM output [M_total, 2h] (bf16), first in the context."""
        M, h = self.args["M"], self.args["h"]
        return self.buf[: M * 2 * h * 2].view(torch.bfloat16).view(M, 2 * h)

    def tensor(self, name: str):
        """A saved tensor as a flat uint8 view of the context: one of "h13",
        "xq_col", "xs_col", "yq_col", "ys_col", "x_t", "w13q_col", "w13s_col",
        "w2q_col", "w2s_col" (MxError if the recipe keeps no such tensor)."""
        a = self.args
        off, n = mlp_ctx_layout(a["M"], a["d"], a["h"], a["E"], a["recipe"], name)
        return self.buf[off:off + n]


def mlp_fwd(x, w1, w3, w2, offs=None, recipe=RECIPE_RCEIL, pad_multiple=128, scratch=None,
            err: ErrorWord | None = None, out=None):
    """MXFP8 SwiGLU MLP forward.  Dense: w1/w3 [h, d], w2 [d, h].  Grouped
    (offs given): w1/w3 [E, h, d], w2 [E, d, h].  Returns (out, ctx)."""
    for n, t in (("x", x), ("w1", w1), ("w3", w3), ("w2", w2)):
        _need(t, torch.bfloat16, n)
    M, d = x.shape
    h = w1.shape[-2]
    E = 0 if offs is None else offs.numel()
    cb, sb = mlp_workspace_size(M, d, h, E, recipe)
    ctx = torch.empty(cb, dtype=torch.uint8, device=x.device)
    if scratch is None or scratch.numel() < sb:
        scratch = torch.empty(sb, dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty((M, d), dtype=torch.bfloat16, device=x.device)
    _check(lib().mx_mlp_fwd(_ptr(x), _ptr(w1), _ptr(w3), _ptr(w2), M, d, h, _ptr(offs), max(E, 1), pad_multiple,
                            recipe, _ptr(ctx), _ptr(scratch), _ptr(out), err.ptr() if err else None, _stream()))
    return out, MlpContext(ctx, dict(x=x, w1=w1, w3=w3, w2=w2, offs=offs, recipe=recipe, M=M, d=d, h=h, E=E,
                                     pad=pad_multiple))


def mlp_fwd_static_scratch(x, w1, w3, w2, offs=None, recipe=RECIPE_RCEIL, pad_multiple=128,
                           err: ErrorWord | None = None, out=None):
    """mlp_fwd whose temporary buffer is the library's fixed device array
    (for callers that cannot allocate device memory; only problems whose
    scratch fits MX_STATIC_SCRATCH_BYTES).  Returns (out, ctx)."""
    for n, t in (("x", x), ("w1", w1), ("w3", w3), ("w2", w2)):
        _need(t, torch.bfloat16, n)
    M, d = x.shape
    h = w1.shape[-2]
    E = 0 if offs is None else offs.numel()
    cb, _ = mlp_workspace_size(M, d, h, E, recipe)
    ctx = torch.empty(cb, dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty((M, d), dtype=torch.bfloat16, device=x.device)
    _check(lib().mx_mlp_fwd_static_scratch(_ptr(x), _ptr(w1), _ptr(w3), _ptr(w2), M, d, h, _ptr(offs), max(E, 1),
                                           pad_multiple, recipe, _ptr(ctx), _ptr(out), err.ptr() if err else None,
                                           _stream()))
    return out, MlpContext(ctx, dict(x=x, w1=w1, w3=w3, w2=w2, offs=offs, recipe=recipe, M=M, d=d, h=h, E=E,
                                     pad=pad_multiple))


def mlp_bwd(ctx: MlpContext, dout, scratch=None, err: ErrorWord | None = None, grads=None):
    """MXFP8 SwiGLU MLP backward from mlp_fwd's context.  Returns (dx, dw1, dw3, dw2)."""
    a = ctx.args
    _need(dout, torch.bfloat16, "dout")
    M, d, h, E = a["M"], a["d"], a["h"], a["E"]
    _, sb = mlp_workspace_size(M, d, h, E, a["recipe"])
    if scratch is None or scratch.numel() < sb:
        scratch = torch.empty(sb, dtype=torch.uint8, device=dout.device)
    if grads is None:
        dx = torch.empty((M, d), dtype=torch.bfloat16, device=dout.device)
        dw1 = torch.empty_like(a["w1"])
        dw3 = torch.empty_like(a["w3"])
        dw2 = torch.empty_like(a["w2"])
    else:
        dx, dw1, dw3, dw2 = grads
    _check(lib().mx_mlp_bwd(_ptr(ctx.buf), _ptr(dout), _ptr(a["x"]), _ptr(a["w1"]), _ptr(a["w3"]), _ptr(a["w2"]),
                            M, d, h, _ptr(a["offs"]), max(E, 1), a["pad"], a["recipe"], _ptr(scratch), _ptr(dx),
                            _ptr(dw1), _ptr(dw3), _ptr(dw2), err.ptr() if err else None, _stream()))
    return dx, dw1, dw3, dw2


# ---------------------------------------------------------------- token-group padding


def token_group_capacity(R: int, E: int, pad_multiple: int = 128) -> int:
    """Rows of a padded buffer that holds any routing of R rows over E experts."""
    return -(-R // pad_multiple) * pad_multiple + pad_multiple * E


def token_group_pad(expert_of, E: int, m_cap: int | None = None, pad_multiple: int = 128,
                    err: ErrorWord | None = None):
    """Padded expert-major layout of routed rows (int32 expert ids on the
    device).  Returns (offs [E], row_dst [R], row_src [m_cap]), int32 on the
    device, without a host synchronization."""
    _need(expert_of, torch.int32, "expert_of")
    R = expert_of.numel()
    if m_cap is None:
        m_cap = token_group_capacity(R, E, pad_multiple)
    dev = expert_of.device
    offs = torch.empty(E, dtype=torch.int32, device=dev)
    row_dst = torch.empty(R, dtype=torch.int32, device=dev)
    row_src = torch.empty(m_cap, dtype=torch.int32, device=dev)
    ws = torch.empty(max(lib().mx_token_group_pad_workspace(R, E), 16), dtype=torch.uint8, device=dev)
    _check(lib().mx_token_group_pad(_ptr(expert_of), R, E, pad_multiple, m_cap, _ptr(offs), _ptr(row_dst),
                                    _ptr(row_src), _ptr(ws), err.ptr() if err else None, _stream()))
    return offs, row_dst, row_src


def gather_rows(x, src, div: int = 1, err: ErrorWord | None = None):
    """y[i] = x[src[i] // div] for src[i] >= 0, zero rows for src[i] < 0."""
    _need(x, torch.bfloat16, "x")
    _need(src, torch.int32, "src")
    y = torch.empty((src.numel(), x.shape[1]), dtype=torch.bfloat16, device=x.device)
    _check(lib().mx_gather_rows(_ptr(x), x.shape[0], x.shape[1], _ptr(src), src.numel(), div, _ptr(y),
                                err.ptr() if err else None, _stream()))
    return y


# ---------------------------------------------------------------- MXFP8 linear


class LinearContext:
    """What mx_linear_fwd saves for mx_linear_bwd (opaque device buffer)."""

    def __init__(self, buf, args):
        self.buf = buf
        self.args = args   # (w, M, K, N, recipe)


def linear_fwd(x, w, recipe=RECIPE_RCEIL, err: ErrorWord | None = None):
    """out = x . w^T in MXFP8 (x [M, K], w [N, K] bf16).  Returns (out, ctx)."""
    _need(x, torch.bfloat16, "x")
    _need(w, torch.bfloat16, "w")
    M, K = x.shape
    N = w.shape[0]
    c, s = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().mx_linear_workspace_size(M, K, N, recipe, ctypes.byref(c), ctypes.byref(s)))
    ctx = torch.empty(max(c.value, 16), dtype=torch.uint8, device=x.device)
    scratch = torch.empty(max(s.value, 16), dtype=torch.uint8, device=x.device)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(lib().mx_linear_fwd(_ptr(x), _ptr(w), M, K, N, recipe, _ptr(ctx), _ptr(scratch), _ptr(out),
                               err.ptr() if err else None, _stream()))
    return out, LinearContext(ctx, (w, M, K, N, recipe))


def linear_bwd(ctx: LinearContext, dout, err: ErrorWord | None = None):
    """(dx [M, K], dw [N, K]) of out = x . w^T."""
    w, M, K, N, recipe = ctx.args
    _need(dout, torch.bfloat16, "dout")
    c, s = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().mx_linear_workspace_size(M, K, N, recipe, ctypes.byref(c), ctypes.byref(s)))
    scratch = torch.empty(max(s.value, 16), dtype=torch.uint8, device=dout.device)
    dx = torch.empty((M, K), dtype=torch.bfloat16, device=dout.device)
    dw = torch.empty((N, K), dtype=torch.bfloat16, device=dout.device)
    _check(lib().mx_linear_bwd(_ptr(ctx.buf), _ptr(dout), _ptr(w), M, K, N, recipe, _ptr(scratch), _ptr(dx),
                               _ptr(dw), err.ptr() if err else None, _stream()))
    return dx, dw
