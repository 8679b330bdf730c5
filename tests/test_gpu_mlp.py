"""GPU parity of the MXFP8 SwiGLU MLP composites (mx_mlp_fwd / mx_mlp_bwd).

1. The composite equals, bit for bit, the same computation spelled out as a
   chain of per-op entry points (the kernels are deterministic).
2. That chain is checked stage by stage against the oracle, each stage fed
   the GPU's own upstream tensors: quantized codes/scales bit-exact, GEMM
   outputs within the normwise 2e-3 bar against fp64 accumulation.
3. End to end against the oracle's own fp64 chain (normwise) at the tiny
   dense config, both recipes, and a small grouped config.
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


def _cat_tiles(sa, sb, rows, cols_each):
    """Concatenate two MMA-layout scale blocks side by side (along columns)."""
    rt, ct = rows // 128, cols_each // 128
    a = sa.view(rt, ct, 512)
    b = sb.view(rt, ct, 512)
    return torch.cat([a, b], dim=1).reshape(-1)


def _quant_weights(w1, w3, w2, sm=0):
    """Per-expert MX quantization of the weights exactly as the composite
    lays them out: w13 rowwise [E,2h,d], w13 columnwise [E,d,2h], w2
    rowwise [E,d,h], w2 columnwise [E,h,d]."""
    grouped = w1.dim() == 3
    E = w1.shape[0] if grouped else 1
    W1 = w1 if grouped else w1[None]
    W3 = w3 if grouped else w3[None]
    W2 = w2 if grouped else w2[None]
    h, d = W1.shape[1], W1.shape[2]
    r = dict(w13q=[], w13s=[], w13qc=[], w13sc=[], w2q=[], w2s=[], w2qc=[], w2sc=[])
    for e in range(E):
        a = mx.quantize(W1[e].contiguous(), scale_mode=sm)
        b = mx.quantize(W3[e].contiguous(), scale_mode=sm)
        c = mx.quantize(W2[e].contiguous(), scale_mode=sm)
        r["w13q"].append(torch.cat([a["q_row"], b["q_row"]], 0))
        r["w13s"].append(torch.cat([a["s_row"], b["s_row"]], 0))
        r["w13qc"].append(torch.cat([a["q_col"], b["q_col"]], 1))
        r["w13sc"].append(_cat_tiles(a["s_col"], b["s_col"], d, h))
        r["w2q"].append(c["q_row"]); r["w2s"].append(c["s_row"])
        r["w2qc"].append(c["q_col"]); r["w2sc"].append(c["s_col"])
    out = {k: torch.stack(v) for k, v in r.items()}
    if not grouped:
        out = {k: v[0] for k, v in out.items()}
    return out


def _chain(x, w1, w3, w2, dout, offs, recipe):
    """The MLP forward+backward as a chain of per-op entry points."""
    hp = recipe in (mx.RECIPE_RCEIL_WGRAD_HP, mx.RECIPE_FLOOR_WGRAD_HP)
    sm = mx.SCALE_FLOOR if recipe in (mx.RECIPE_FLOOR, mx.RECIPE_FLOOR_WGRAD_HP) else mx.SCALE_RCEIL
    grouped = offs is not None
    W = _quant_weights(w1, w3, w2, sm)
    h = w1.shape[-2]
    xq = mx.quantize(x, mx.BOTH, scale_mode=sm)

    def mm(aq, as_, bq, bs):
        if grouped:
            return mx.grouped_mm(mx.GROUP_M, aq, as_, bq, bs, offs)
        return mx.scaled_mm(aq, as_, bq, bs)

    def wg(aq, as_, bq, bs):
        if grouped:
            return mx.grouped_mm(mx.GROUP_K, aq, as_, bq, bs, offs)
        return mx.scaled_mm(aq, as_, bq, bs)

    h13 = mm(xq["q_row"], xq["s_row"], W["w13q"], W["w13s"])
    y = mx.swiglu_quant(h13, mx.ROW if hp else mx.BOTH, scale_mode=sm)
    out = mm(y["q_row"], y["s_row"], W["w2q"], W["w2s"])
    dq = mx.quantize(dout, mx.BOTH, scale_mode=sm)
    dy = mm(dq["q_row"], dq["s_row"], W["w2qc"], W["w2sc"])
    if hp:
        dh = mx.swiglu_quant_bwd(dy, h13, mx.ROW, bf16_transposed=True, scale_mode=sm)
        dout_t = dout.t().contiguous()
        x_t = x.t().contiguous()
        dw2 = mx.bf16_wgrad(dout_t, dh["y_t"], offs)
        dw13 = mx.bf16_wgrad(dh["dh13_t"], x_t, offs)
    else:
        dh = mx.swiglu_quant_bwd(dy, h13, mx.BOTH, scale_mode=sm)
        dw2 = wg(dq["q_col"], dq["s_col"], y["q_col"], y["s_col"])
        dw13 = wg(dh["q_col"], dh["s_col"], xq["q_col"], xq["s_col"])
    dx = mm(dh["q_row"], dh["s_row"], W["w13qc"], W["w13sc"])
    dw1, dw3 = dw13[..., :h, :], dw13[..., h:, :]
    return dict(W=W, xq=xq, h13=h13, y=y, out=out, dq=dq, dy=dy, dh=dh, dx=dx, dw1=dw1, dw3=dw3, dw2=dw2)


def _inputs_dense(M, d, h, seed):
    inp = synth.dense_mlp_inputs(M, d, h, seed)
    return inp, {k: to_dev(v) for k, v in inp.items()}, None


def _inputs_grouped(counts, d, h, seed):
    inp = synth.grouped_mlp_inputs(np.array(counts), d, h, seed)
    dev = {k: to_dev(inp[k]) for k in ("x", "w1", "w3", "w2", "dout")}
    return inp, dev, to_dev(inp["offs"], torch.int32)


CASES = [
    ("dense", mx.RECIPE_RCEIL),
    ("dense", mx.RECIPE_RCEIL_WGRAD_HP),
    ("grouped", mx.RECIPE_RCEIL),
    ("grouped", mx.RECIPE_RCEIL_WGRAD_HP),
    ("dense", mx.RECIPE_FLOOR),
    ("grouped", mx.RECIPE_FLOOR_WGRAD_HP),
]
ORACLE_RECIPE = {mx.RECIPE_RCEIL: o.RECIPE_RCEIL, mx.RECIPE_RCEIL_WGRAD_HP: o.RECIPE_RCEIL_WGRAD_HP,
                 mx.RECIPE_FLOOR: o.RECIPE_FLOOR, mx.RECIPE_FLOOR_WGRAD_HP: o.RECIPE_FLOOR_WGRAD_HP}


def _inputs_grouped_tail(counts, d, h, seed, tail):
    """Grouped inputs with `tail` rows past the last group whose x values are
    not zero (the tail must stay inert whatever it holds)."""
    inp = synth.grouped_mlp_inputs(np.array(counts), d, h, seed, tail_rows=tail)
    end = int(inp["offs"][-1])
    inp["x"][end:] = synth.normal_bf16((tail, d), 1.0, seed * 1000 + 9)
    dev = {k: to_dev(inp[k]) for k in ("x", "w1", "w3", "w2", "dout")}
    return inp, dev, to_dev(inp["offs"], torch.int32)


def _setup(kind):
    if kind == "dense":
        return _inputs_dense(256, 256, 512, seed=0)           # the tiny dense config
    if kind == "grouped_tail":
        return _inputs_grouped_tail([100, 0, 300, 28], 256, 384, seed=4, tail=128)
    # d = 5120 (>= 4096): long enough a contraction that the w13 GEMM also carries the
    # columnwise quantization of y under the MXFP8-wgrad recipes
    if kind == "dense_wide":
        return _inputs_dense(256, 5120, 256, seed=6)
    if kind == "grouped_tail_wide":
        return _inputs_grouped_tail([100, 0, 300, 28], 5120, 256, seed=7, tail=128)
    return _inputs_grouped([100, 0, 300, 28], 256, 384, seed=4)


@pytest.mark.parametrize("kind,recipe", CASES)
def test_composite_equals_op_chain(kind, recipe):
    inp, t, offs = _setup(kind)
    err = mx.ErrorWord()
    out, ctx = mx.mlp_fwd(t["x"], t["w1"], t["w3"], t["w2"], offs=offs, recipe=recipe, err=err)
    dx, dw1, dw3, dw2 = mx.mlp_bwd(ctx, t["dout"], err=err)
    ch = _chain(t["x"], t["w1"], t["w3"], t["w2"], t["dout"], offs, recipe)
    torch.cuda.synchronize()
    err.check()
    assert torch.equal(ctx.h13(), ch["h13"])
    for name, a, b in [("out", out, ch["out"]), ("dx", dx, ch["dx"]), ("dw1", dw1, ch["dw1"]),
                       ("dw3", dw3, ch["dw3"]), ("dw2", dw2, ch["dw2"])]:
        assert torch.equal(a, b), name


@pytest.mark.parametrize("kind,recipe", CASES)
def test_op_chain_stagewise_vs_oracle(kind, recipe):
    inp, t, offs = _setup(kind)
    orc = ORACLE_RECIPE[recipe]
    hp = o.recipe_hp(orc)
    sc = o.recipe_scale(orc)
    ch = _chain(t["x"], t["w1"], t["w3"], t["w2"], t["dout"], offs, recipe)
    torch.cuda.synchronize()
    offs_h = inp.get("offs")
    grouped = offs_h is not None
    x, w1, w3, w2, dout = (inp[k] for k in ("x", "w1", "w3", "w2", "dout"))
    h = w1.shape[-2]
    M, d = x.shape
    # F1/F2/F5: quantization bit-exact
    xq, xs = o.quantize_rows(x, sc)
    assert np.array_equal(u8(ch["xq"]["q_row"]), xq)
    w13 = np.concatenate([w1, w3], axis=-2)
    w13q, w13s = o.quantize_rows(w13, sc)
    assert np.array_equal(u8(ch["W"]["w13q"]), w13q)
    assert np.array_equal(u8(ch["W"]["w13s"]), o.scales_to_mma(w13s))
    w13qc, w13sc = o.quantize_cols(w13, sc)
    assert np.array_equal(u8(ch["W"]["w13qc"]), w13qc)
    assert np.array_equal(u8(ch["W"]["w13sc"]), o.scales_to_mma(w13sc))
    # F3: h13 from the (bit-exact) quantized operands
    ref = o.mx_grouped_mm_m(xq, xs, w13q, w13s, offs_h) if grouped else o.mx_mm(xq, xs, w13q, w13s)
    h13 = bits(ch["h13"])
    assert o.normwise_rel_err(o.bf16_to_f64(h13), ref) <= TOL
    # F4: SwiGLU of the GPU's h13, bit-exact codes
    y = o.swiglu_fwd(*o.split_h13(h13))
    yq, ys = o.quantize_rows(y, sc)
    assert np.array_equal(u8(ch["y"]["q_row"]), yq)
    assert np.array_equal(u8(ch["y"]["s_row"]), o.scales_to_mma(ys))
    if not hp:
        yqc, ysc = o.quantize_cols(y, sc)
        assert np.array_equal(u8(ch["y"]["q_col"]), yqc)
    # F6
    w2q, w2s = o.quantize_rows(w2, sc)
    ref = o.mx_grouped_mm_m(yq, ys, w2q, w2s, offs_h) if grouped else o.mx_mm(yq, ys, w2q, w2s)
    assert o.normwise_rel_err(o.bf16_to_f64(bits(ch["out"])), ref) <= TOL
    # B2: dy
    dq, ds = o.quantize_rows(dout, sc)
    assert np.array_equal(u8(ch["dq"]["q_row"]), dq)
    w2qc, w2sc = o.quantize_cols(w2, sc)
    ref = o.mx_grouped_mm_m(dq, ds, w2qc, w2sc, offs_h) if grouped else o.mx_mm(dq, ds, w2qc, w2sc)
    dy = bits(ch["dy"])
    assert o.normwise_rel_err(o.bf16_to_f64(dy), ref) <= TOL
    # B4: SwiGLU backward of the GPU's dy and h13, bit-exact
    dg, du = o.swiglu_bwd(dy, *o.split_h13(h13))
    dh13 = np.concatenate([dg, du], axis=-1)
    dhq, dhs = o.quantize_rows(dh13, sc)
    assert np.array_equal(u8(ch["dh"]["q_row"]), dhq)
    # B5: dx
    ref = (o.mx_grouped_mm_m(dhq, dhs, w13qc, w13sc, offs_h) if grouped
           else o.mx_mm(dhq, dhs, w13qc, w13sc))
    assert o.normwise_rel_err(o.bf16_to_f64(bits(ch["dx"])), ref) <= TOL
    # B3 / B6: weight gradients
    go = offs_h if grouped else np.array([M], np.int32)
    if hp:
        assert np.array_equal(bits(ch["dh"]["dh13_t"]).T, dh13)
        assert np.array_equal(bits(ch["dh"]["y_t"]).T, y)
        ref2 = o.bf16_grouped_mm_k(dout.T, y.T, go)
        ref13 = o.bf16_grouped_mm_k(dh13.T, x.T, go)
    else:
        dqc, dsc = o.quantize_cols(dout, sc)
        dhqc, dhsc = o.quantize_cols(dh13, sc)
        assert np.array_equal(u8(ch["dh"]["q_col"]), dhqc)
        xqc, xsc = o.quantize_cols(x, sc)
        ref2 = o.mx_grouped_mm_k(dqc, dsc, yqc, ysc, go)
        ref13 = o.mx_grouped_mm_k(dhqc, dhsc, xqc, xsc, go)
    if not grouped:
        ref2, ref13 = ref2[0], ref13[0]
    assert o.normwise_rel_err(o.bf16_to_f64(bits(ch["dw2"])), ref2) <= TOL
    assert o.normwise_rel_err(o.bf16_to_f64(bits(ch["dw1"])), ref13[..., :h, :]) <= TOL
    assert o.normwise_rel_err(o.bf16_to_f64(bits(ch["dw3"])), ref13[..., h:, :]) <= TOL
    if grouped:
        for e, (s, t_) in enumerate(o.group_bounds(offs_h)):
            if s == t_:
                assert not bits(ch["dw1"])[e].any() and not bits(ch["dw2"])[e].any()


@pytest.mark.parametrize("kind,recipe", CASES)
def test_end_to_end_vs_oracle(kind, recipe):
    inp, t, offs = _setup(kind)
    out, ctx = mx.mlp_fwd(t["x"], t["w1"], t["w3"], t["w2"], offs=offs, recipe=recipe)
    dx, dw1, dw3, dw2 = mx.mlp_bwd(ctx, t["dout"])
    torch.cuda.synchronize()
    offs_h = inp.get("offs")
    orc = ORACLE_RECIPE[recipe]
    f = o.mlp_fwd(inp["x"], inp["w1"], inp["w3"], inp["w2"], offs=offs_h, recipe=orc)
    b = o.mlp_bwd(inp["x"], inp["w1"], inp["w3"], inp["w2"], inp["dout"], offs=offs_h, recipe=orc, fwd=f)
    h = inp["w1"].shape[-2]
    errs = {}
    for name, got, ref in [("out", out, f["out_f"]), ("dx", dx, b["dx_f"]), ("dw2", dw2, b["dw2_f"]),
                           ("dw1", dw1, b["dw13_f"][..., :h, :]), ("dw3", dw3, b["dw13_f"][..., h:, :])]:
        errs[name] = o.normwise_rel_err(o.bf16_to_f64(bits(got)), ref)
    print(kind, recipe, {k: f"{v:.2e}" for k, v in errs.items()})
    assert max(errs.values()) <= 2e-3, errs
    if offs_h is not None:
        assert not bits(out)[~inp["real_rows"]].any(), "padding rows must stay zero"


@pytest.mark.parametrize("kind,recipe", [("dense", mx.RECIPE_RCEIL), ("grouped_tail", mx.RECIPE_RCEIL),
                                         ("grouped_tail", mx.RECIPE_FLOOR), ("dense_wide", mx.RECIPE_RCEIL),
                                         ("grouped_tail_wide", mx.RECIPE_RCEIL),
                                         ("grouped_tail_wide", mx.RECIPE_FLOOR)])
def test_saved_columnwise_operands_vs_oracle(kind, recipe):
    """Under the MXFP8 weight-gradient recipes the forward saves y and x
    quantized by columns; at d >= 4096 the w13 GEMM's epilogue writes the
    columnwise y (each 32-row block of its tile), below it the SwiGLU kernel
    does.  Both equal the oracle bit for bit, including the rows past the
    last group (zero codes, scale 0x00)."""
    inp, t, offs = _setup(kind)
    sc = o.recipe_scale(ORACLE_RECIPE[recipe])
    err = mx.ErrorWord()
    out, ctx = mx.mlp_fwd(t["x"], t["w1"], t["w3"], t["w2"], offs=offs, recipe=recipe, err=err)
    torch.cuda.synchronize()
    err.check()
    M, d = inp["x"].shape
    h = inp["w1"].shape[-2]
    h13 = bits(ctx.h13())
    if offs is not None:
        end = int(inp["offs"][-1])
        assert not h13[end:].any() and not bits(out)[end:].any(), "tail rows must be zero"
    y = o.swiglu_fwd(*o.split_h13(h13))
    yqc, ysc = o.quantize_cols(y, sc)
    assert np.array_equal(u8(ctx.tensor("yq_col")).reshape(h, M), yqc)
    assert np.array_equal(u8(ctx.tensor("ys_col")), o.scales_to_mma(ysc))
    xqc, xsc = o.quantize_cols(inp["x"], sc)
    assert np.array_equal(u8(ctx.tensor("xq_col")).reshape(d, M), xqc)
    assert np.array_equal(u8(ctx.tensor("xs_col")), o.scales_to_mma(xsc))


@pytest.mark.parametrize("kind,recipe", [("dense_wide", mx.RECIPE_RCEIL), ("grouped_tail_wide", mx.RECIPE_FLOOR),
                                         ("dense_wide", mx.RECIPE_RCEIL_WGRAD_HP)])
def test_fused_forward_equals_op_chain(kind, recipe):
    """At d >= 4096 the composite's w13 GEMM carries SwiGLU and both
    quantizations of y; its outputs equal the per-op chain bit for bit."""
    inp, t, offs = _setup(kind)
    err = mx.ErrorWord()
    out, ctx = mx.mlp_fwd(t["x"], t["w1"], t["w3"], t["w2"], offs=offs, recipe=recipe, err=err)
    dx, dw1, dw3, dw2 = mx.mlp_bwd(ctx, t["dout"], err=err)
    ch = _chain(t["x"], t["w1"], t["w3"], t["w2"], t["dout"], offs, recipe)
    torch.cuda.synchronize()
    err.check()
    assert torch.equal(ctx.h13(), ch["h13"])
    for name, a, b in [("out", out, ch["out"]), ("dx", dx, ch["dx"]), ("dw1", dw1, ch["dw1"]),
                       ("dw3", dw3, ch["dw3"]), ("dw2", dw2, ch["dw2"])]:
        assert torch.equal(a, b), name


@pytest.mark.parametrize("recipe", [mx.RECIPE_RCEIL, mx.RECIPE_RCEIL_WGRAD_HP])
def test_all_experts_empty(recipe):
    """Every group empty (offs all zero), 128 tail rows holding non-zero x:
    the output, the input gradient and every expert's weight gradients are
    exact zeros."""
    inp, t, offs = _inputs_grouped_tail([0, 0, 0, 0], 256, 256, seed=21, tail=128)
    inp["dout"][:] = synth.normal_bf16(inp["dout"].shape, 1.0, 22)
    t["dout"] = to_dev(inp["dout"])
    err = mx.ErrorWord()
    out, ctx = mx.mlp_fwd(t["x"], t["w1"], t["w3"], t["w2"], offs=offs, recipe=recipe, err=err)
    dx, dw1, dw3, dw2 = mx.mlp_bwd(ctx, t["dout"], err=err)
    torch.cuda.synchronize()
    err.check()
    for name, a in (("out", out), ("dx", dx), ("dw1", dw1), ("dw3", dw3), ("dw2", dw2)):
        assert not bits(a).any(), name


@pytest.mark.parametrize("recipe", [mx.RECIPE_RCEIL, mx.RECIPE_RCEIL_WGRAD_HP])
def test_single_expert_equals_dense(recipe):
    """One expert holding every row (E = 1, no padding) is the dense layer:
    the grouped forms give the dense forms' outputs and gradients bit for
    bit (the same products summed in the same order)."""
    M, d, h = 256, 256, 384
    inp, t, _ = _inputs_dense(M, d, h, seed=23)
    offs = to_dev(np.array([M], dtype=np.int32), torch.int32)
    err = mx.ErrorWord()
    out_d, ctx_d = mx.mlp_fwd(t["x"], t["w1"], t["w3"], t["w2"], recipe=recipe, err=err)
    grads_d = mx.mlp_bwd(ctx_d, t["dout"], err=err)
    w1g, w3g, w2g = (t[k].unsqueeze(0).contiguous() for k in ("w1", "w3", "w2"))
    out_g, ctx_g = mx.mlp_fwd(t["x"], w1g, w3g, w2g, offs=offs, recipe=recipe, err=err)
    grads_g = mx.mlp_bwd(ctx_g, t["dout"], err=err)
    torch.cuda.synchronize()
    err.check()
    assert np.array_equal(bits(out_g), bits(out_d))
    for name, a, b in zip(("dx", "dw1", "dw3", "dw2"), grads_g, grads_d):
        assert np.array_equal(bits(a).reshape(bits(b).shape), bits(b)), name
