"""Pins for the oracle's SwiGLU forward (correctly rounded sigmoid, bf16 SiLU,
y = a*u) and backward (du, dg).  References: mpmath at high precision with
its own rounding, torch's bf16 CPU arithmetic, and central differences."""
import mpmath
import numpy as np
import pytest
import torch

from oracle import mx_oracle as o


def _all_bf16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return bits, o.bf16_to_f64(bits)


def _mp_sigmoid_f32(g: float) -> float:
    """Independent reference: sigmoid at 200 bits, rounded by mpmath to a
    24-bit significand (round-half-even).  Valid where the result is a
    normal float32 (g > -87)."""
    with mpmath.workprec(200):
        s = 1 / (1 + mpmath.exp(-mpmath.mpf(g)))
    with mpmath.workprec(24):
        r = +s          # rounds to 24 bits, nearest-even
    return float(r)


@pytest.mark.slow
def test_sigmoid_correctly_rounded_every_bf16():
    bits, g = _all_bf16()
    m = np.isfinite(g) & (g > -87.0) & (g < 40.0)
    gs = g[m]
    got = o.sigmoid_rn_f32(gs)
    ref = np.array([_mp_sigmoid_f32(float(x)) for x in gs])
    assert np.array_equal(got, ref)


def test_sigmoid_tails_and_specials():
    # float32 below 2^-149 rounds to zero; above the 1 - 2^-25 midpoint to 1
    got = o.sigmoid_rn_f32(np.array([0.0, -0.0, 200.0, -200.0, np.inf, -np.inf, 17.5]))
    assert list(got[:6]) == [0.5, 0.5, 1.0, 0.0, 1.0, 0.0]
    assert got[6] == 1.0  # e^-17.5 = 2.5e-8 < 2^-25 = 2.98e-8
    # deep negative side: float32 subnormal results, checked with mpmath at
    # an explicit 2^-149 quantum
    for g in [-88.0, -95.5, -100.0, -103.0]:
        with mpmath.workprec(200):
            s = 1 / (1 + mpmath.exp(-mpmath.mpf(g)))
            q = mpmath.mpf(2) ** -149
            n = s / q
            fl = mpmath.floor(n)
            frac = n - fl
            k = fl + 1 if frac > 0.5 or (frac == 0.5 and int(fl) % 2 == 1) else fl
            ref = float(k * q)
        assert o.sigmoid_rn_f32(np.array([g]))[0] == ref


def test_sigmoid_monotone_over_bf16():
    bits, g = _all_bf16()
    m = np.isfinite(g)
    gs = np.unique(g[m])
    s = o.sigmoid_rn_f32(gs)
    assert np.all(np.diff(s) >= 0)


@pytest.mark.slow
def test_silu_every_bf16_vs_torch_roundings():
    """a = RN_bf16(RN_f32(g * sigma_f32)), with sigma from mpmath and both
    roundings done by torch casts."""
    bits, g = _all_bf16()
    m = np.isfinite(g) & (g > -87.0) & (g < 40.0)
    gs = g[m]
    sig = np.array([_mp_sigmoid_f32(float(x)) for x in gs])
    p = torch.from_numpy(gs * sig).to(torch.float32).to(torch.bfloat16)
    ref = p.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(o.silu_bf16(bits[m]), ref)


def test_silu_specials():
    b = o.round_to_bf16_bits(np.array([0.0, -0.0, 100.0, -200.0, -1e30]))
    a = o.silu_bf16(b)
    assert list(a) == [0x0000, 0x8000, int(o.round_to_bf16_bits(100.0)), 0x8000, 0x8000]
    # g = -90: sigma = e^-90 = 8.2e-40 is a float32 subnormal, yet
    # g*sigma = -7.4e-38 is a normal bf16, so a is not -0
    a90 = o.bf16_to_f64(o.silu_bf16(o.round_to_bf16_bits(np.array([-90.0]))))[0]
    assert -7.5e-38 < a90 < -7.3e-38
    # g = -100: g*sigma = -3.7e-42 is below half the smallest bf16 subnormal
    # (2^-133 = 9.2e-41), so a = -0
    assert o.silu_bf16(o.round_to_bf16_bits(np.array([-100.0])))[0] == 0x8000


def test_swiglu_fwd_matches_torch_bf16_mul():
    rng = np.random.default_rng(3)
    g = o.round_to_bf16_bits(rng.standard_normal(50000) * 3)
    u = o.round_to_bf16_bits(rng.standard_normal(50000) * 3)
    a = o.silu_bf16(g)
    ta = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    tu = torch.from_numpy(u.view(np.int16)).view(torch.bfloat16)
    ref = (ta * tu).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(o.swiglu_fwd(g, u), ref)


def test_du_matches_torch_bf16_mul():
    rng = np.random.default_rng(4)
    g = o.round_to_bf16_bits(rng.standard_normal(50000) * 3)
    u = o.round_to_bf16_bits(rng.standard_normal(50000))
    dy = o.round_to_bf16_bits(rng.standard_normal(50000))
    _, du = o.swiglu_bwd(dy, g, u)
    ta = torch.from_numpy(o.silu_bf16(g).view(np.int16)).view(torch.bfloat16)
    tdy = torch.from_numpy(dy.view(np.int16)).view(torch.bfloat16)
    ref = (tdy * ta).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(du, ref)


def test_dsilu_factor_vs_central_differences():
    """f(g) = d/dg [g*sigma(g)], checked against mpmath's numerical
    derivative of g*sigma(g) (not the closed form)."""
    gs = np.concatenate([np.linspace(-30, 30, 241), [-1.2784645, -1.25, 0.0, 1e-3]])
    f, _ = o._dsilu_factor_f64(gs)
    for gi, fi in zip(gs, f):
        with mpmath.workprec(120):
            ref = mpmath.diff(lambda t: t / (1 + mpmath.exp(-t)), mpmath.mpf(float(gi)))
        ref = float(ref)
        assert abs(fi - ref) <= 1e-12 * max(abs(ref), 1e-3), (gi, fi, ref)


def test_dg_g_zero_is_half_dy_u():
    """g = 0: sigma = 1/2, 1 + g(1-sigma) = 1, so dg = RN_bf16(dy*u/2),
    including exact ties (rounded here by torch)."""
    rng = np.random.default_rng(5)
    dy = o.round_to_bf16_bits(rng.standard_normal(20000))
    u = o.round_to_bf16_bits(rng.standard_normal(20000))
    g = np.zeros(20000, dtype=np.uint16)
    dg, _ = o.swiglu_bwd(dy, g, u)
    half = o.bf16_to_f64(dy) * o.bf16_to_f64(u) / 2  # exact, fits float32
    ref = torch.from_numpy(half).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(dg, ref)


def test_dg_vs_mpmath_sample():
    rng = np.random.default_rng(6)
    n = 3000
    g = o.round_to_bf16_bits(rng.standard_normal(n) * 4)
    u = o.round_to_bf16_bits(rng.standard_normal(n))
    dy = o.round_to_bf16_bits(rng.standard_normal(n))
    dg, _ = o.swiglu_bwd(dy, g, u)
    gv, uv, dyv = o.bf16_to_f64(g), o.bf16_to_f64(u), o.bf16_to_f64(dy)
    checked = 0
    for i in range(n):
        with mpmath.workprec(200):
            x = mpmath.mpf(float(gv[i]))
            s = 1 / (1 + mpmath.exp(-x))
            exact = mpmath.mpf(float(dyv[i])) * mpmath.mpf(float(uv[i])) * s * (1 + x * (1 - s))
        with mpmath.workprec(8):          # bf16 significand, nearest-even
            r = float(+exact)
        if r == 0.0 or not np.isfinite(r) or abs(r) < 2.0**-126:
            continue
        ref = o.round_to_bf16_bits(np.array([r]))[0]
        assert dg[i] == ref, (gv[i], uv[i], dyv[i])
        checked += 1
    assert checked > n * 0.9


def test_dg_nonfinite_g_is_nan_and_deep_negative_is_signed_zero():
    g = o.round_to_bf16_bits(np.array([np.inf, -np.inf, np.nan, -1000.0, -1000.0]))
    u = o.round_to_bf16_bits(np.array([1.0, 1.0, 1.0, 2.0, -2.0]))
    dy = o.round_to_bf16_bits(np.array([1.0, 1.0, 1.0, 1.0, 1.0]))
    dg, _ = o.swiglu_bwd(dy, g, u)
    v = o.bf16_to_f64(dg)
    assert np.isnan(v[:3]).all()
    # f(g) < 0 for g << 0: dy*u*f has the sign opposite to dy*u
    assert dg[3] == 0x8000 and dg[4] == 0x0000
