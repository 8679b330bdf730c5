"""The kernels store each 32-code block (and each 16 values of a bf16
transpose) with one 256-bit store when the destination is 32-byte aligned,
and with two 16-byte stores when it is only 16-byte aligned (the alignment
the C ABI promises to accept).  These tests write every output of the cast
and of the SwiGLU kernels at a 16-byte offset into a larger buffer and
require the same bytes as the aligned call, which the other tests compare
with the oracle."""
import ctypes

import numpy as np
import pytest
import torch

import block_scaled_mlp_gb300 as mx
from tests.util import u8

pytestmark = pytest.mark.gpu
OFF = 16


def _rand(shape, seed, std=1.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * std).to(torch.bfloat16)


def _shifted(n, dtype=torch.uint8):
    """A device buffer of n elements starting 16 bytes into an allocation."""
    esz = torch.empty((), dtype=dtype).element_size()
    base = torch.zeros(n + OFF // esz + 32, dtype=dtype, device="cuda")
    view = base[OFF // esz: OFF // esz + n]
    assert view.data_ptr() % 32 == OFF
    return view


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def test_quantize_16_byte_aligned_outputs():
    rows, cols = 384, 640
    x = _rand((rows, cols), 1)
    ref = mx.quantize(x, mx.BOTH)
    qr, qc = _shifted(rows * cols), _shifted(cols * rows)
    sr, sc = torch.zeros_like(ref["s_row"]), torch.zeros_like(ref["s_col"])
    mx._check(mx.lib().mx_quantize_mode(_p(x), rows, cols, mx.BOTH, mx.SCALE_MMA, mx.SCALE_RCEIL, _p(qr), _p(sr),
                                        _p(qc), _p(sc), mx._stream()))
    torch.cuda.synchronize()
    assert np.array_equal(u8(qr).reshape(rows, cols), u8(ref["q_row"]))
    assert np.array_equal(u8(qc).reshape(cols, rows), u8(ref["q_col"]))
    assert np.array_equal(u8(sr), u8(ref["s_row"])) and np.array_equal(u8(sc), u8(ref["s_col"]))


@pytest.mark.parametrize("axis", [mx.ROW, mx.BOTH])
def test_swiglu_fwd_16_byte_aligned_outputs(axis):
    M, h = 256, 192
    h13 = _rand((M, 2 * h), 2, std=1.3)
    ref = mx.swiglu_quant(h13, axis)
    qr = _shifted(M * h)
    qc = _shifted(h * M) if axis & mx.COL else None
    sr = torch.zeros_like(ref["s_row"])
    sc = torch.zeros_like(ref["s_col"]) if axis & mx.COL else None
    mx._check(mx.lib().mx_swiglu_quant_mode(_p(h13), M, h, axis, mx.SCALE_MMA, mx.SCALE_RCEIL, _p(qr), _p(sr),
                                            _p(qc), _p(sc), mx._stream()))
    torch.cuda.synchronize()
    assert np.array_equal(u8(qr).reshape(M, h), u8(ref["q_row"]))
    assert np.array_equal(u8(sr), u8(ref["s_row"]))
    if axis & mx.COL:
        assert np.array_equal(u8(qc).reshape(h, M), u8(ref["q_col"]))
        assert np.array_equal(u8(sc), u8(ref["s_col"]))


@pytest.mark.parametrize("hp", [False, True])
def test_swiglu_bwd_16_byte_aligned_outputs(hp):
    M, h = 256, 192
    h13 = _rand((M, 2 * h), 3, std=1.3)
    dy = _rand((M, h), 4)
    axis = mx.ROW if hp else mx.BOTH
    ref = mx.swiglu_quant_bwd(dy, h13, axis, bf16_transposed=hp)
    qr = _shifted(M * 2 * h)
    sr = torch.zeros_like(ref["s_row"])
    qc = sc = dt = yt = None
    if hp:
        dt, yt = _shifted(2 * h * M, torch.bfloat16), _shifted(h * M, torch.bfloat16)
    else:
        qc, sc = _shifted(2 * h * M), torch.zeros_like(ref["s_col"])
    mx._check(mx.lib().mx_swiglu_quant_bwd_mode(_p(dy), _p(h13), M, h, axis, mx.SCALE_MMA, mx.SCALE_RCEIL, _p(qr),
                                                _p(sr), _p(qc), _p(sc), _p(dt), _p(yt), mx._stream()))
    torch.cuda.synchronize()
    assert np.array_equal(u8(qr).reshape(M, 2 * h), u8(ref["q_row"]))
    assert np.array_equal(u8(sr), u8(ref["s_row"]))
    if hp:
        b = lambda t: t.cpu().view(torch.int16).numpy()
        assert np.array_equal(b(dt).reshape(2 * h, M), b(ref["dh13_t"]))
        assert np.array_equal(b(yt).reshape(h, M), b(ref["y_t"]))
    else:
        assert np.array_equal(u8(qc).reshape(2 * h, M), u8(ref["q_col"]))
        assert np.array_equal(u8(sc), u8(ref["s_col"]))


@pytest.mark.parametrize("d", [256, 4096])
def test_mlp_fwd_16_byte_aligned_workspaces(d):
    """The composite with its saved context, scratch and output all starting
    16 bytes into their allocations (every internal code buffer, the fused
    w13 epilogue's y included at d = 4096, then takes the 16-byte stores):
    the same output and saved context as with aligned buffers."""
    M, h = 256, 256
    x, w1, w3, w2 = _rand((M, d), 5), _rand((h, d), 6, 0.05), _rand((h, d), 7, 0.05), _rand((d, h), 8, 0.05)
    out_ref, ctx_ref = mx.mlp_fwd(x, w1, w3, w2)
    cb, sb = mx.mlp_workspace_size(M, d, h, 0, mx.RECIPE_RCEIL)
    ctx, scratch = _shifted(cb), _shifted(sb)
    out = _shifted(M * d, torch.bfloat16)
    err = mx.ErrorWord()
    mx._check(mx.lib().mx_mlp_fwd(_p(x), _p(w1), _p(w3), _p(w2), M, d, h, None, 1, 128, mx.RECIPE_RCEIL, _p(ctx),
                                  _p(scratch), _p(out), err.ptr(), mx._stream()))
    torch.cuda.synchronize()
    err.check()
    b = lambda t: t.cpu().contiguous().view(torch.int16).numpy()
    assert np.array_equal(b(out).reshape(M, d), b(out_ref))
    ctx_s = mx.MlpContext(ctx, ctx_ref.args)
    for name in ("h13", "xq_col", "xs_col", "yq_col", "ys_col", "w13q_col", "w13s_col", "w2q_col", "w2s_col"):
        assert np.array_equal(u8(ctx_s.tensor(name)), u8(ctx_ref.tensor(name))), name
