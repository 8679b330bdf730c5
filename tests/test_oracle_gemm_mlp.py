"""Pins for the oracle's block-scaled GEMMs (dense, M-grouped, K-grouped) and
for the composed MLP forward/backward.

References: a pure-Python triple loop with its own E4M3 decoding, exact
permutation/identity cases, the textbook fp64 SwiGLU MLP and its analytic
gradients, and structural identities (grouped == per-group dense, padding
rows inert, empty experts give zero gradients)."""
import numpy as np
import pytest

from oracle import mx_oracle as o
import synth


def _decode_e4m3_py(c: int) -> float:
    s = -1.0 if c & 0x80 else 1.0
    e, m = (c >> 3) & 0xF, c & 7
    if e == 0:
        return s * m / 512.0
    return s * (1 + m / 8.0) * 2.0 ** (e - 7)


def test_mx_mm_vs_triple_loop():
    rng = np.random.default_rng(0)
    M, N, K = 3, 4, 96
    a = synth.bf16_from_f32(rng.standard_normal((M, K)).astype(np.float32) * 5)
    b = synth.bf16_from_f32(rng.standard_normal((N, K)).astype(np.float32) * 0.1)
    aq, as_ = o.quantize_rows(a)
    bq, bs = o.quantize_rows(b)
    got = o.mx_mm(aq, as_, bq, bs)
    for i in range(M):
        for j in range(N):
            acc = 0.0
            for k in range(K):
                va = _decode_e4m3_py(int(aq[i, k])) * 2.0 ** (int(as_[i, k // 32]) - 127)
                vb = _decode_e4m3_py(int(bq[j, k])) * 2.0 ** (int(bs[j, k // 32]) - 127)
                acc += va * vb
            assert got[i, j] == pytest.approx(acc, rel=1e-14, abs=1e-300)


def test_mx_mm_permutation_is_exact():
    """B = a permutation matrix (entries 1.0 quantize exactly: amax 1 ->
    scale 2^-8, code 2^8): C = deq(A)[:, perm]."""
    rng = np.random.default_rng(1)
    K = 64
    a = synth.bf16_from_f32(rng.standard_normal((5, K)).astype(np.float32))
    perm = rng.permutation(K)
    P = np.zeros((K, K), dtype=np.float32)
    P[np.arange(K), perm] = 1.0
    aq, as_ = o.quantize_rows(a)
    bq, bs = o.quantize_rows(synth.bf16_from_f32(P))
    C = o.mx_mm(aq, as_, bq, bs)
    assert np.array_equal(C, o.dequantize(aq, as_)[:, perm])


def _grouped_setup(counts, d=64, h=64, seed=7, tail=0):
    inp = synth.grouped_mlp_inputs(np.array(counts), d, h, seed, tail_rows=tail)
    return inp


def test_grouped_m_equals_per_group_dense_and_tail_zero():
    inp = _grouped_setup([100, 0, 300, 28], tail=64)
    x, w1, offs = inp["x"], inp["w1"], inp["offs"]
    xq, xs = o.quantize_rows(x)
    wq, ws = o.quantize_rows(w1)
    C = o.mx_grouped_mm_m(xq, xs, wq, ws, offs)
    for e, (s, t) in enumerate(o.group_bounds(offs)):
        if t > s:
            assert np.array_equal(C[s:t], o.mx_mm(xq[s:t], xs[s:t], wq[e], ws[e]))
    assert not C[int(offs[-1]):].any()
    # padding rows of x are zero, so their output rows are zero
    assert not C[~inp["real_rows"]].any()


def test_grouped_k_sums_to_dense_and_empty_is_zero():
    inp = _grouped_setup([128, 0, 256, 100])
    x, dout, offs = inp["x"], inp["dout"], inp["offs"]
    aq, as_ = o.quantize_cols(dout)   # [d, M]
    bq, bs = o.quantize_cols(x)       # [d, M]
    C = o.mx_grouped_mm_k(aq, as_, bq, bs, offs)
    assert C.shape == (4, 64, 64)
    assert not C[1].any()
    dense = o.mx_mm(aq, as_, bq, bs)
    assert np.allclose(C.sum(axis=0), dense, rtol=1e-12, atol=1e-12)


def _plain_mlp(x, w1, w3, w2, dout):
    """Textbook fp64 SwiGLU MLP with analytic gradients (no quantization)."""
    X, W1, W3, W2, D = (o.bf16_to_f64(t) for t in (x, w1, w3, w2, dout))
    g = X @ W1.T
    u = X @ W3.T
    s = 1 / (1 + np.exp(-g))
    a = g * s
    y = a * u
    out = y @ W2.T
    dy = D @ W2
    dW2 = D.T @ y
    dg = dy * u * s * (1 + g * (1 - s))
    du = dy * a
    dx = dg @ W1 + du @ W3
    return dict(out=out, dx=dx, dw1=dg.T @ X, dw3=du.T @ X, dw2=dW2)


@pytest.mark.parametrize("recipe", [o.RECIPE_RCEIL, o.RECIPE_RCEIL_WGRAD_HP])
def test_mlp_close_to_plain_fp64_mlp(recipe):
    """MXFP8 quantization error only: a transposed operand, swapped w1/w3 or
    a wrong gradient would be O(1) off."""
    inp = synth.dense_mlp_inputs(128, 128, 256, seed=11)
    x, w1, w3, w2, dout = (inp[k] for k in ("x", "w1", "w3", "w2", "dout"))
    f = o.mlp_fwd(x, w1, w3, w2, recipe=recipe)
    b = o.mlp_bwd(x, w1, w3, w2, dout, recipe=recipe, fwd=f)
    ref = _plain_mlp(x, w1, w3, w2, dout)
    for name, got in [("out", f["out"]), ("dx", b["dx"]), ("dw1", b["dw1"]),
                      ("dw3", b["dw3"]), ("dw2", b["dw2"])]:
        err = o.normwise_rel_err(o.bf16_to_f64(got), ref[name])
        assert err < 0.1, (name, err)
    # the HP recipe's weight gradients are bf16 GEMMs of the bf16 operands:
    # only the final bf16 rounding separates them from fp64 dout^T . y
    if recipe == o.RECIPE_RCEIL_WGRAD_HP:
        hp = o.bf16_to_f64(dout).T @ o.bf16_to_f64(f["y"])
        assert o.normwise_rel_err(o.bf16_to_f64(b["dw2"]), hp) < 4e-3
        hp1 = o.bf16_to_f64(b["dg"]).T @ o.bf16_to_f64(x)
        assert o.normwise_rel_err(o.bf16_to_f64(b["dw1"]), hp1) < 4e-3


def test_grouped_mlp_equals_per_expert_dense():
    inp = _grouped_setup([128, 0, 200, 60], d=64, h=96, seed=3)
    x, w1, w3, w2, dout, offs = (inp[k] for k in ("x", "w1", "w3", "w2", "dout", "offs"))
    f = o.mlp_fwd(x, w1, w3, w2, offs=offs)
    b = o.mlp_bwd(x, w1, w3, w2, dout, offs=offs, fwd=f)
    for e, (s, t) in enumerate(o.group_bounds(offs)):
        if t == s:
            assert not b["dw1"][e].any() and not b["dw3"][e].any() and not b["dw2"][e].any()
            continue
        fe = o.mlp_fwd(x[s:t], w1[e], w3[e], w2[e])
        be = o.mlp_bwd(x[s:t], w1[e], w3[e], w2[e], dout[s:t], fwd=fe)
        assert np.array_equal(f["out"][s:t], fe["out"])
        assert np.array_equal(b["dx"][s:t], be["dx"])
        assert np.array_equal(b["dw1"][e], be["dw1"])
        assert np.array_equal(b["dw3"][e], be["dw3"])
        assert np.array_equal(b["dw2"][e], be["dw2"])


def test_padding_rows_are_inert():
    """Zero padding rows give zero output rows, and padding a group with more
    zero rows leaves its weight gradients bit-identical."""
    d, h = 64, 64
    inp = _grouped_setup([100], d=d, h=h, seed=5)
    x, w1, w3, w2, dout, offs = (inp[k] for k in ("x", "w1", "w3", "w2", "dout", "offs"))
    assert int(offs[-1]) == 128
    f = o.mlp_fwd(x, w1, w3, w2, offs=offs)
    b = o.mlp_bwd(x, w1, w3, w2, dout, offs=offs, fwd=f)
    assert not f["out"][100:].any() and not b["dx"][100:].any()
    x2 = np.zeros((384, d), dtype=np.uint16)
    d2 = np.zeros((384, d), dtype=np.uint16)
    x2[:128], d2[:128] = x, dout
    offs2 = np.array([384], dtype=np.int32)
    f2 = o.mlp_fwd(x2, w1, w3, w2, offs=offs2)
    b2 = o.mlp_bwd(x2, w1, w3, w2, d2, offs=offs2, fwd=f2)
    assert not f2["out"][100:].any()
    for k in ("dw1", "dw3", "dw2"):
        assert np.array_equal(b[k], b2[k])
    assert np.array_equal(f["out"][:100], f2["out"][:100])
