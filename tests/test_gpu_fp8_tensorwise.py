"""GPU parity of the FP8 per-tensor recipe (reading R15; page "[mxfp8
training] unified MXFP8TrainingConfig and MXFP8TrainingTensor", FP8
GroupedMM) against the oracle:

* mx_fp8_amax equals max |x| exactly, per tensor and per expert;
* mx_fp8_quantize codes are bit-exact, by rows and by columns, per expert,
  including an all-zero expert (the 2^-40 floor);
* mx_fp8_grouped_mm (M- and K-grouped) within the normwise 2e-3 bar of the
  float64 GEMM of the dequantized operands, with an empty expert (exact
  zeros), tail rows (zeros), ragged group sizes and several tiles.
"""
import numpy as np
import pytest
import torch

import block_scaled_mlp_gb300 as mx
import synth
from oracle import mx_oracle as o
from tests.util import bits, to_dev, u8

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _rand_bf16(shape, seed, scale=1.0, wide=False):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(shape)
    if wide:
        v = v * np.exp(rng.uniform(-6, 6, shape))
    return synth.bf16_from_f32((v * scale).astype(np.float32))


def test_amax_exact_per_tensor_and_per_expert():
    x = _rand_bf16((640, 384), 1, wide=True)
    amax = mx.fp8_amax(to_dev(x))
    torch.cuda.synchronize()
    assert amax.cpu().numpy()[0] == o.fp8_tensor_amax(x)
    w = _rand_bf16((5, 256, 128), 2) * 1
    w[3] = 0                                                # an all-zero expert
    w = w.astype(np.uint16)
    wa = mx.fp8_amax(to_dev(w), batch_axes=1)
    torch.cuda.synchronize()
    assert np.array_equal(wa.cpu().numpy(), o.fp8_tensor_amax(w, batch_axes=1))


@pytest.mark.parametrize("axis", [mx.ROW, mx.COL, mx.BOTH])
def test_quantize_bit_exact(axis):
    x = _rand_bf16((384, 640), 3, wide=True)
    amax = mx.fp8_amax(to_dev(x))
    res = mx.fp8_quantize(to_dev(x), amax, axis)
    torch.cuda.synchronize()
    ref, s, _ = o.fp8_quantize_tensor(x)
    if axis & mx.ROW:
        assert np.array_equal(u8(res["q_row"]), ref)
    if axis & mx.COL:
        refc, _, _ = o.fp8_quantize_tensor(x.T.copy())
        assert np.array_equal(u8(res["q_col"]), refc)


def test_quantize_per_expert_with_zero_expert():
    w = _rand_bf16((4, 256, 384), 4)
    w[1] = 0
    w[2] = _rand_bf16((256, 384), 5, scale=1e-4)
    dw = to_dev(w)
    amax = mx.fp8_amax(dw, batch_axes=1)
    res = mx.fp8_quantize(dw, amax, mx.BOTH)
    torch.cuda.synchronize()
    ref, s, _ = o.fp8_quantize_tensor(w, batch_axes=1)
    assert np.array_equal(u8(res["q_row"]), ref)
    refc, _, _ = o.fp8_quantize_tensor(np.swapaxes(w, 1, 2).copy(), batch_axes=1)
    assert np.array_equal(u8(res["q_col"]), refc)
    assert not u8(res["q_row"])[1].any()


def _grouped_inputs(counts, K, N, seed, tail=0):
    inp = synth.grouped_mlp_inputs(np.array(counts), K, N, seed, tail_rows=tail)
    if tail:
        end = int(inp["offs"][-1])
        inp["x"][end:] = synth.normal_bf16((tail, K), 1.0, seed * 1000 + 9)
    return inp


@pytest.mark.parametrize("counts,K,N,tail", [([100, 0, 300, 28], 256, 384, 128),
                                             ([700, 5, 0, 1200, 64], 512, 768, 0)])
def test_grouped_m_vs_oracle(counts, K, N, tail):
    inp = _grouped_inputs(counts, K, N, seed=11, tail=tail)
    x, w = inp["x"], inp["w1"]                       # x [M_total, K], w1 [E, N, K]
    offs = to_dev(inp["offs"], torch.int32)
    dx, dw = to_dev(x), to_dev(w)
    ax, aw = mx.fp8_amax(dx), mx.fp8_amax(dw, batch_axes=1)
    xq = mx.fp8_quantize(dx, ax, mx.ROW)["q_row"]
    wq = mx.fp8_quantize(dw, aw, mx.ROW)["q_row"]
    err = mx.ErrorWord()
    c = mx.fp8_grouped_mm(mx.GROUP_M, xq, ax, wq, aw, offs, err=err)
    torch.cuda.synchronize()
    err.check()
    aq, sa, _ = o.fp8_quantize_tensor(x)
    bq, sb, _ = o.fp8_quantize_tensor(w, batch_axes=1)
    assert np.array_equal(u8(xq), aq) and np.array_equal(u8(wq), bq)
    ref = o.fp8_grouped_mm_m(aq, sa, bq, sb, inp["offs"])
    got = o.bf16_to_f64(bits(c))
    e = o.normwise_rel_err(got, ref)
    print("fp8 grouped M normwise", e)
    assert e <= TOL
    end = int(inp["offs"][-1])
    assert not got[end:].any(), "tail rows must be zero"
    for gi, (s, t) in enumerate(o.group_bounds(inp["offs"])):   # each group within the bar on its own
        if t > s:
            assert o.normwise_rel_err(got[s:t], ref[s:t]) <= TOL, gi


@pytest.mark.parametrize("counts,N,K", [([100, 0, 300, 28], 256, 384), ([700, 5, 0, 1200, 64], 384, 256)])
def test_grouped_k_vs_oracle(counts, N, K):
    inp = _grouped_inputs(counts, N, K, seed=12)
    dout, x = inp["x"], synth.normal_bf16((inp["x"].shape[0], K), 1.0, 77)   # [M_total, N], [M_total, K]
    x[~inp["real_rows"]] = 0
    offs = to_dev(inp["offs"], torch.int32)
    dd, dx = to_dev(dout), to_dev(x)
    ad, ax = mx.fp8_amax(dd), mx.fp8_amax(dx)
    dq = mx.fp8_quantize(dd, ad, mx.COL)["q_col"]      # [N, M_total]
    xq = mx.fp8_quantize(dx, ax, mx.COL)["q_col"]      # [K, M_total]
    err = mx.ErrorWord()
    c = mx.fp8_grouped_mm(mx.GROUP_K, dq, ad, xq, ax, offs, err=err)
    torch.cuda.synchronize()
    err.check()
    aq, sa, _ = o.fp8_quantize_tensor(dout.T.copy())
    bq, sb, _ = o.fp8_quantize_tensor(x.T.copy())
    assert np.array_equal(u8(dq), aq) and np.array_equal(u8(xq), bq)
    ref = o.fp8_grouped_mm_k(aq, sa, bq, sb, inp["offs"])
    got = o.bf16_to_f64(bits(c))
    for e_, (s, t) in enumerate(o.group_bounds(inp["offs"])):
        if t == s:
            assert not got[e_].any(), "an empty expert's weight gradient is exact zeros"
        else:
            assert o.normwise_rel_err(got[e_], ref[e_]) <= TOL, e_
    print("fp8 grouped K normwise", o.normwise_rel_err(got, ref))
