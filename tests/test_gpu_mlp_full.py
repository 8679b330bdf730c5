"""Full-size parity of the MLP composite on the bench workloads (the launch
configuration bench.py times): the Llama-3-8B FFN (dense, wgrad_with_hp)
and the two routed-expert MoE layers (grouped, default recipe).

The oracle cannot redo these steps whole on the host, so it recomputes
sampled outputs one by one from the same inputs: per sampled group (the
smallest, the median and the largest non-empty expert; the whole matrix
for the dense layer) 32 rows x 128 columns of h13, out and dx, and 32 x 64
entries of each weight gradient over the group's tokens, each to the
normwise 2e-3 bar against fp64 accumulation; the quantized activations it
needs along the way are recomputed from the GPU's own h13 (stage-wise, as
in the small tests).  Padding rows must be exact zeros, and so must an
empty expert's weight gradients."""
import numpy as np
import pytest
import torch

import block_scaled_mlp_gb300 as mx
import synth
from oracle import mx_oracle as o
from tests.util import bits, to_dev

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _make(name):
    w = dict(synth.WORKLOADS[name])
    if w["kind"] == "dense":
        inp = synth.dense_mlp_inputs(w["M"], w["d"], w["h"], w["seed"])
        inp["offs"] = None
    else:
        if w["counts"] == "zipf":
            counts = synth.zipf_group_counts(w["E"], w["tokens"], w["s"], w["seed"], w["n_empty"])
        else:
            counts = synth.dirichlet_group_counts(w["E"], w["tokens"], w["alpha"], w["seed"], w["n_empty"])
        inp = synth.grouped_mlp_inputs(counts, w["d"], w["h"], w["seed"])
    return w, inp


def _row_q(a):
    return o.quantize_rows(np.ascontiguousarray(a))


@pytest.mark.parametrize("name", ["llama3_8b_ffn", "moe_16e", "moe_64e"])
def test_full_size_sampled(name):
    w, inp = _make(name)
    hp = w.get("recipe") == "wgrad_hp"
    recipe = mx.RECIPE_RCEIL_WGRAD_HP if hp else mx.RECIPE_RCEIL
    grouped = inp["offs"] is not None
    t = {k: to_dev(inp[k]) for k in ("x", "w1", "w3", "w2", "dout")}
    offs_d = to_dev(inp["offs"], torch.int32) if grouped else None
    err = mx.ErrorWord()
    out, ctx = mx.mlp_fwd(t["x"], t["w1"], t["w3"], t["w2"], offs=offs_d, recipe=recipe, err=err)
    dx, dw1, dw3, dw2 = mx.mlp_bwd(ctx, t["dout"], err=err)
    torch.cuda.synchronize()
    err.check()
    h13_gpu = ctx.h13()
    if grouped:
        bounds = o.group_bounds(inp["offs"])
        real = inp["real_rows"]
        assert not bits(out)[~real].any() and not bits(dx)[~real].any(), "padding rows must be zero"
        assert not bits(out)[int(inp["offs"][-1]):].any()
        for ee, (a, b) in enumerate(bounds):
            if a == b:
                assert not bits(dw1[ee]).any() and not bits(dw2[ee]).any(), "empty expert"
        # the groups (experts) whose rows and weight gradients are sampled:
        # the smallest, the median and the largest non-empty group
        live = sorted((b - a, i) for i, (a, b) in enumerate(bounds) if b > a)
        groups = sorted({live[0][1], live[len(live) // 2][1], live[-1][1]})
    else:
        groups = [0]
    for e in groups:
        _check_group(e, inp, grouped, hp, h13_gpu, out, dx, dw1, dw3, dw2, np.random.default_rng(7 + e))


def _check_group(e, inp, grouped, hp, h13_gpu, out, dx, dw1, dw3, dw2, rng):
    """Sampled entries of h13, out, dx (rows of group e) and of expert e's
    weight gradients against the oracle, each to the normwise bar."""
    x, dout = inp["x"], inp["dout"]
    M, d = x.shape
    h = inp["w1"].shape[-2]
    if grouped:
        s0, s1 = o.group_bounds(inp["offs"])[e]
        W1, W3, W2 = inp["w1"][e], inp["w3"][e], inp["w2"][e]
    else:
        s0, s1 = 0, M
        W1, W3, W2 = inp["w1"], inp["w3"], inp["w2"]
    real_rows = np.arange(s0, s1)
    if grouped:
        real_rows = real_rows[inp["real_rows"][s0:s1]]
    R = np.sort(rng.choice(real_rows, min(32, len(real_rows)), replace=False))
    J = np.sort(rng.choice(2 * h, 128, replace=False))
    Jd = np.sort(rng.choice(d, 128, replace=False))
    W13 = np.concatenate([W1, W3], axis=0)

    # F3: h13[R, J]
    xq, xs = _row_q(x[R])
    wq, ws = _row_q(W13[J])
    ref = o.mx_mm(xq, xs, wq, ws)
    h13_s = bits(h13_gpu[torch.as_tensor(R, device="cuda")][:, torch.as_tensor(J, device="cuda")])
    assert o.normwise_rel_err(o.bf16_to_f64(h13_s), ref) <= TOL, ("h13", e)

    # F4 + F6: out[R, Jd] from the GPU's h13 rows
    h13_R = bits(h13_gpu[torch.as_tensor(R, device="cuda")])
    y_R = o.swiglu_fwd(*o.split_h13(h13_R))
    yq, ys = _row_q(y_R)
    w2q, w2s = _row_q(W2[Jd])
    ref = o.mx_mm(yq, ys, w2q, w2s)
    out_s = bits(out)[R][:, Jd]
    assert o.normwise_rel_err(o.bf16_to_f64(out_s), ref) <= TOL, ("out", e)

    # B2 + B4 + B5: dx[R, Jd]
    dq, ds = _row_q(dout[R])
    w2qc, w2sc = _row_q(W2.T)                        # [h, d] columnwise copy of w2
    dy_R = o.round_to_bf16_bits(o.mx_mm(dq, ds, w2qc, w2sc))
    dg, du = o.swiglu_bwd(dy_R, *o.split_h13(h13_R))
    dhq, dhs = _row_q(np.concatenate([dg, du], axis=1))
    w13qc, w13sc = _row_q(W13.T[Jd])                 # rows Jd of the columnwise w13
    ref = o.mx_mm(dhq, dhs, w13qc, w13sc)
    dx_s = bits(dx)[R][:, Jd]
    assert o.normwise_rel_err(o.bf16_to_f64(dx_s), ref) <= TOL, ("dx", e)

    # B3 / B6: sampled weight-gradient entries over the group's tokens
    # (a thousand or more entries each, so that the normwise bar is not
    # dominated by the bf16 rounding of a handful of values)
    I2 = np.sort(rng.choice(d, 32, replace=False))   # rows of dw2
    J2 = np.sort(rng.choice(h, 64, replace=False))   # cols of dw2
    I1 = np.sort(rng.choice(h, 32, replace=False))   # rows of dw1 / dw3
    J1 = np.sort(rng.choice(d, 64, replace=False))
    tok = slice(s0, s1)
    h13_cols = bits(h13_gpu[s0:s1])                   # [T, 2h] of the group
    g_all, u_all = o.split_h13(h13_cols)
    y_cols = o.swiglu_fwd(g_all[:, J2], u_all[:, J2])  # [T, |J2|]
    dout_g = dout[tok]
    if hp:
        ref2 = o.bf16_to_f64(dout_g[:, I2]).T @ o.bf16_to_f64(y_cols)
    else:
        aq, as_ = o.quantize_cols(dout_g[:, I2])      # [|I2|, T]
        bq, bs = o.quantize_cols(y_cols)
        ref2 = o.mx_mm(aq, as_, bq, bs)
    dw2_s = bits(dw2[e] if grouped else dw2)[I2][:, J2]
    assert o.normwise_rel_err(o.bf16_to_f64(dw2_s), ref2) <= TOL, ("dw2", e)

    # dh13 columns I1 (dg) and h + I1 (du) for all tokens of the group
    dqg, dsg = _row_q(dout_g)
    w2c_I, w2cs_I = _row_q(W2.T[I1])
    dy_g = o.round_to_bf16_bits(o.mx_mm(dqg, dsg, w2c_I, w2cs_I))   # [T, |I1|]
    dg_g, du_g = o.swiglu_bwd(dy_g, g_all[:, I1], u_all[:, I1])
    x_g = x[tok]
    for name_w, dcol, dw in (("dw1", dg_g, dw1), ("dw3", du_g, dw3)):
        if hp:
            ref1 = o.bf16_to_f64(dcol).T @ o.bf16_to_f64(x_g[:, J1])
        else:
            aq, as_ = o.quantize_cols(dcol)
            bq, bs = o.quantize_cols(x_g[:, J1])
            ref1 = o.mx_mm(aq, as_, bq, bs)
        got = bits(dw[e] if grouped else dw)[I1][:, J1]
        assert o.normwise_rel_err(o.bf16_to_f64(got), ref1) <= TOL, (name_w, e)
