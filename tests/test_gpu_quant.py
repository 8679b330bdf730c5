"""GPU parity of the standalone MXFP8 cast (mx_quantize) against the oracle:
codes and scales must match bit for bit."""
import numpy as np
import pytest
import torch

import block_scaled_mlp_gb300 as mx
import synth
from oracle import mx_oracle as o
from tests.util import bits, to_dev, u8

pytestmark = pytest.mark.gpu


def _check_rows(res, x, layout, rows=None, scale=o.SCALE_RCEIL):
    q, s = o.quantize_rows(x if rows is None else x[rows], scale)
    got_q = u8(res["q_row"]) if rows is None else u8(res["q_row"])[rows]
    assert np.array_equal(got_q, q)
    R, C = x.shape
    flat = u8(res["s_row"])
    if layout == mx.SCALE_MMA:
        sl = o.scales_from_mma(flat, R, C // 32)
        if rows is None:
            assert np.array_equal(flat, o.scales_to_mma(s))   # padding bytes included
    else:
        sl = flat.reshape(R, C // 32)
    assert np.array_equal(sl if rows is None else sl[rows], s)


def _check_cols(res, x, layout, cols=None, scale=o.SCALE_RCEIL):
    xt = x.T if cols is None else x[:, cols].T
    q, s = o.quantize_rows(np.ascontiguousarray(xt), scale)
    got_q = u8(res["q_col"]) if cols is None else u8(res["q_col"])[cols]
    assert np.array_equal(got_q, q)
    R, C = x.shape
    flat = u8(res["s_col"])
    if layout == mx.SCALE_MMA:
        sl = o.scales_from_mma(flat, C, R // 32)
        if cols is None:
            assert np.array_equal(flat, o.scales_to_mma(s))
    else:
        sl = flat.reshape(C, R // 32)
    assert np.array_equal(sl if cols is None else sl[cols], s)


@pytest.mark.parametrize("layout", [mx.SCALE_MMA, mx.SCALE_LINEAR])
@pytest.mark.parametrize("shape", [(256, 256), (384, 640), (96, 160), (32, 32), (1024, 96)])
def test_quantize_both_matches_oracle(shape, layout):
    R, C = shape
    x = synth.quant_sweep_tensor(R, C, seed=R + C)
    res = mx.quantize(to_dev(x), mx.BOTH, layout)
    torch.cuda.synchronize()
    _check_rows(res, x, layout)
    _check_cols(res, x, layout)


@pytest.mark.parametrize("axis", [mx.ROW, mx.COL])
def test_quantize_single_axis(axis):
    x = synth.quant_sweep_tensor(512, 384, seed=3)
    res = mx.quantize(to_dev(x), axis, mx.SCALE_MMA)
    torch.cuda.synchronize()
    if axis == mx.ROW:
        assert res["q_col"] is None
        _check_rows(res, x, mx.SCALE_MMA)
    else:
        assert res["q_row"] is None
        _check_cols(res, x, mx.SCALE_MMA)


def test_quantize_ragged_rows_rowwise():
    """rows not a multiple of the 128-row tile (only rowwise allows it)."""
    x = synth.normal_bf16((200, 96), 3.0, seed=9)
    res = mx.quantize(to_dev(x), mx.ROW, mx.SCALE_LINEAR)
    torch.cuda.synchronize()
    _check_rows(res, x, mx.SCALE_LINEAR)


@pytest.mark.parametrize("layout", [mx.SCALE_MMA, mx.SCALE_LINEAR])
@pytest.mark.parametrize("shape", [(256, 256), (384, 640), (96, 160)])
def test_quantize_floor_matches_oracle(shape, layout):
    """FLOOR scales (reading R14) on the sweep recipe and on blocks whose
    amax mantissa exceeds 1.75, where saturation binds."""
    R, C = shape
    x = synth.quant_sweep_tensor(R, C, seed=R + 2 * C)
    v = o.bf16_to_f64(x)
    sat = synth.bf16_from_f32((np.sign(v) * 1.9 * 2.0 ** np.round(np.log2(np.abs(v) + 1e-30))).astype(np.float32))
    x[::3] = sat[::3]                 # every third row: magnitudes 1.9 * 2^k
    res = mx.quantize(to_dev(x), mx.BOTH, layout, mx.SCALE_FLOOR)
    torch.cuda.synchronize()
    _check_rows(res, x, layout, scale=o.SCALE_FLOOR)
    _check_cols(res, x, layout, scale=o.SCALE_FLOOR)


@pytest.mark.parametrize("scale", [o.SCALE_RCEIL, o.SCALE_FLOOR])
def test_quantize_every_bf16_amax(scale):
    """One block per non-negative bf16 amax value (plus NaN/Inf/-0 blocks):
    exhaustive E8M0 + E4M3 coverage of the kernel's scale path."""
    amax = np.arange(0, 0x7F81, dtype=np.uint32).astype(np.uint16)      # incl. +Inf
    nb = amax.size + 2
    nb += (-nb) % 128
    rng = np.random.default_rng(0)
    blocks = np.zeros((nb, 32), dtype=np.uint16)
    mags = o.bf16_to_f64(amax)
    # fill each block with values below its amax (random fractions), amax at a random slot
    fr = rng.uniform(-1, 1, size=(amax.size, 32))
    fill = o.round_to_bf16_bits(np.where(np.isfinite(mags)[:, None], fr * mags[:, None], 1.0))
    blocks[: amax.size] = fill
    blocks[np.arange(amax.size), rng.integers(0, 32, amax.size)] = amax
    blocks[amax.size] = 0x7FC0        # NaN block
    blocks[amax.size + 1, 3] = 0x8000  # -0 block
    x = blocks.reshape(-1, 128)        # 4 blocks per row
    mode = mx.SCALE_FLOOR if scale == o.SCALE_FLOOR else mx.SCALE_RCEIL
    res = mx.quantize(to_dev(x), mx.ROW, mx.SCALE_LINEAR, mode)
    torch.cuda.synchronize()
    _check_rows(res, x, mx.SCALE_LINEAR, scale=scale)


def test_quantize_golden_blocks():
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "mx_blocks.json")))
    vals = np.array([c["values"] for c in g["blocks"]], dtype=np.float32)
    n = len(vals)
    rows = ((n + 31) // 32) * 32
    x = np.zeros((rows, 32), dtype=np.uint16)
    x[:n] = synth.bf16_from_f32(vals)
    res = mx.quantize(to_dev(x), mx.ROW, mx.SCALE_LINEAR)
    torch.cuda.synchronize()
    q = u8(res["q_row"])
    s = u8(res["s_row"]).reshape(rows)
    for i, c in enumerate(g["blocks"]):
        assert int(s[i]) == c["scale"], c["name"]
        assert [int(v) for v in q[i]] == c["codes"], c["name"]


@pytest.mark.parametrize("n", [4096, 32768])
def test_quantize_sweep_full_size_sampled(n):
    """The quantize-sweep workload at its full size, in the launch the bench
    times (MX_BOTH, MMA layout); the oracle checks sampled rows and columns."""
    x = synth.quant_sweep_tensor(n, n, seed=n)
    xd = to_dev(x)
    res = mx.quantize(xd, mx.BOTH, mx.SCALE_MMA)
    torch.cuda.synchronize()
    rng = np.random.default_rng(n)
    rows = np.sort(rng.choice(n, 48, replace=False))
    cols = np.sort(rng.choice(n, 48, replace=False))
    _check_rows(res, x, mx.SCALE_MMA, rows=rows)
    _check_cols(res, x, mx.SCALE_MMA, cols=cols)
