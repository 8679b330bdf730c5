"""Pins of the MXFP8 linear oracle (reading R13): exact on inputs the MX
format represents exactly, within MX quantization error of the textbook fp64
linear otherwise (a transposed operand or a swapped gradient would be O(1)
off), and the wgrad_hp weight gradient within bf16 rounding of fp64."""
import numpy as np
import pytest

import synth
from oracle import mx_oracle as o


def _small_ints(shape, seed):
    """Integers in [-7, 7] (exact in E4M3 under any power-of-two scale that
    keeps them in range) as bf16 bits."""
    v = np.random.default_rng(seed).integers(-7, 8, shape).astype(np.float32)
    return synth.bf16_from_f32(v)


@pytest.mark.parametrize("recipe", [o.RECIPE_RCEIL, o.RECIPE_RCEIL_WGRAD_HP])
def test_exact_on_exactly_representable_inputs(recipe):
    x, w, dout = _small_ints((64, 96), 1), _small_ints((32, 96), 2), _small_ints((64, 32), 3)
    X, W, D = (o.bf16_to_f64(a) for a in (x, w, dout))
    out = o.linear_fwd(x, w)
    dx, dw = o.linear_bwd(x, w, dout, recipe)
    # quantization is exact on these inputs: each result is the exact integer
    # sum rounded once to bf16
    assert np.array_equal(o.bf16_to_f64(out), o.bf16_to_f64(o.round_to_bf16_bits(X @ W.T)))
    assert np.array_equal(o.bf16_to_f64(dx), o.bf16_to_f64(o.round_to_bf16_bits(D @ W)))
    assert np.array_equal(o.bf16_to_f64(dw), o.bf16_to_f64(o.round_to_bf16_bits(D.T @ X)))


@pytest.mark.parametrize("recipe", [o.RECIPE_RCEIL, o.RECIPE_RCEIL_WGRAD_HP])
def test_close_to_plain_fp64_linear(recipe):
    x = synth.normal_bf16((128, 256), 1.0, 5)
    w = synth.normal_bf16((64, 256), 0.02, 6)
    dout = synth.normal_bf16((128, 64), 1.0, 7)
    X, W, D = (o.bf16_to_f64(a) for a in (x, w, dout))
    out = o.linear_fwd(x, w)
    dx, dw = o.linear_bwd(x, w, dout, recipe)
    for got, ref in ((out, X @ W.T), (dx, D @ W), (dw, D.T @ X)):
        assert o.normwise_rel_err(o.bf16_to_f64(got), ref) < 0.1
    if recipe == o.RECIPE_RCEIL_WGRAD_HP:
        assert o.normwise_rel_err(o.bf16_to_f64(dw), D.T @ X) < 4e-3


def test_transposed_operand_is_far_off():
    """The pins above would catch a swapped operand: w^T in place of w is O(1) away."""
    x = synth.normal_bf16((128, 128), 1.0, 8)
    w = synth.normal_bf16((128, 128), 0.02, 9)
    X, W = o.bf16_to_f64(x), o.bf16_to_f64(w)
    assert o.normwise_rel_err(o.bf16_to_f64(o.linear_fwd(x, w)), X @ W) > 0.5
