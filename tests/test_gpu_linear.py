"""Parity of the per-linear MXFP8 path (mx_linear_fwd / mx_linear_bwd,
reading R13) with the oracle: bit-exact where the MX format represents the
inputs exactly, normwise within 2e-3 of the exact float64 products
otherwise, bit-identical to the op chain (mx_quantize + mx_scaled_mm /
mx_bf16_wgrad), and sampled at the lm_head size (8192 tokens, 4096 ->
128256)."""
import numpy as np
import pytest
import torch

import block_scaled_mlp_gb300 as mx
import synth
from oracle import mx_oracle as o
from tests.util import bits, to_dev

pytestmark = pytest.mark.gpu
TOL = 2e-3
RECIPES = [(mx.RECIPE_RCEIL, o.RECIPE_RCEIL), (mx.RECIPE_RCEIL_WGRAD_HP, o.RECIPE_RCEIL_WGRAD_HP),
           (mx.RECIPE_FLOOR, o.RECIPE_FLOOR), (mx.RECIPE_FLOOR_WGRAD_HP, o.RECIPE_FLOOR_WGRAD_HP)]


def _run(x, w, dout, recipe):
    err = mx.ErrorWord()
    out, ctx = mx.linear_fwd(to_dev(x), to_dev(w), recipe, err=err)
    dx, dw = mx.linear_bwd(ctx, to_dev(dout), err=err)
    torch.cuda.synchronize()
    err.check()
    return bits(out), bits(dx), bits(dw)


@pytest.mark.parametrize("recipe,orec", RECIPES)
def test_exact_inputs_bit_exact(recipe, orec):
    rng = np.random.default_rng(1)
    ints = lambda *s: synth.bf16_from_f32(rng.integers(-7, 8, s).astype(np.float32))
    x, w, dout = ints(256, 384), ints(512, 384), ints(256, 512)
    out, dx, dw = _run(x, w, dout, recipe)
    r_out = o.linear_fwd(x, w, recipe=orec)
    r_dx, r_dw = o.linear_bwd(x, w, dout, orec)
    assert np.array_equal(out, r_out) and np.array_equal(dx, r_dx) and np.array_equal(dw, r_dw)


@pytest.mark.parametrize("recipe,orec", RECIPES)
@pytest.mark.parametrize("M,K,N", [(256, 384, 512), (384, 256, 128), (128, 1024, 640)])
def test_matches_oracle(M, K, N, recipe, orec):
    x = synth.normal_bf16((M, K), 1.0, M + K)
    w = synth.normal_bf16((N, K), 0.02, N + 1)
    dout = synth.normal_bf16((M, N), 1.0, N + 2)
    out, dx, dw = _run(x, w, dout, recipe)
    r_out = o.linear_fwd(x, w, rounded=False, recipe=orec)
    r_dx, r_dw = o.linear_bwd(x, w, dout, orec, rounded=False)
    for got, ref in ((out, r_out), (dx, r_dx), (dw, r_dw)):
        assert o.normwise_rel_err(o.bf16_to_f64(got), ref) <= TOL


@pytest.mark.parametrize("recipe", [mx.RECIPE_RCEIL, mx.RECIPE_RCEIL_WGRAD_HP])
def test_composite_equals_op_chain(recipe):
    M, K, N = 256, 384, 512
    x = to_dev(synth.normal_bf16((M, K), 1.0, 3))
    w = to_dev(synth.normal_bf16((N, K), 0.02, 4))
    dout = to_dev(synth.normal_bf16((M, N), 1.0, 5))
    out, ctx = mx.linear_fwd(x, w, recipe)
    dx, dw = mx.linear_bwd(ctx, dout)
    qx, qw, qd = mx.quantize(x), mx.quantize(w), mx.quantize(dout)
    c_out = mx.scaled_mm(qx["q_row"], qx["s_row"], qw["q_row"], qw["s_row"])
    c_dx = mx.scaled_mm(qd["q_row"], qd["s_row"], qw["q_col"], qw["s_col"])
    if recipe == mx.RECIPE_RCEIL:
        c_dw = mx.scaled_mm(qd["q_col"], qd["s_col"], qx["q_col"], qx["s_col"])
    else:
        c_dw = mx.bf16_wgrad(dout.t().contiguous(), x.t().contiguous())
    torch.cuda.synchronize()
    for a, b in ((out, c_out), (dx, c_dx), (dw, c_dw)):
        assert np.array_equal(bits(a), bits(b))


def test_lm_head_size_sampled():
    """8192 tokens, 4096 -> 128256 (a Llama-3 lm_head), default recipe."""
    M, K, N = 8192, 4096, 128256
    x = synth.normal_bf16((M, K), 1.0, 31)
    w = synth.normal_bf16((N, K), 0.02, 32)
    dout = synth.normal_bf16((M, N), 1.0, 33)
    out, ctx = mx.linear_fwd(to_dev(x), to_dev(w), mx.RECIPE_RCEIL)
    dx, dw = mx.linear_bwd(ctx, to_dev(dout))
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    R = np.sort(rng.choice(M, 16, replace=False))
    J = np.sort(rng.choice(N, 64, replace=False))
    Jk = np.sort(rng.choice(K, 64, replace=False))
    ref = o.linear_fwd(x[R], w[J], rounded=False)
    assert o.normwise_rel_err(o.bf16_to_f64(bits(out[torch.as_tensor(R, device="cuda")][:, torch.as_tensor(J, device="cuda")])), ref) <= TOL
    # dx rows R: every output needs all of N, columns Jk of w's columnwise copy
    dq, ds = o.quantize_rows(dout[R])
    wq_c, ws_c = o.quantize_cols(w[:, Jk])
    ref = o.mx_mm(dq, ds, wq_c, ws_c)
    assert o.normwise_rel_err(o.bf16_to_f64(bits(dx)[R][:, Jk]), ref) <= TOL
    # dw rows J, columns Jk: contraction over all tokens
    aq, as_ = o.quantize_cols(dout[:, J])
    bq, bs = o.quantize_cols(x[:, Jk])
    ref = o.mx_mm(aq, as_, bq, bs)
    assert o.normwise_rel_err(o.bf16_to_f64(bits(dw)[J][:, Jk]), ref) <= TOL
