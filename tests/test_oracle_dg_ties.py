"""Pins of the oracle's exact-tie handling in the SwiGLU backward (reading R5:
dg = RN_bf16 of the exact dy*u*f(g), f(g) = sigma(g)*(1 + g*(1 - sigma(g))),
rounded once; page "Add MXFP8 fused-MLP overrides in torchtitan", Numerics
and tests).

dy*u is a product of two bf16 values, so it can sit exactly on a bf16
rounding midpoint.  Whether dg then rounds up or down is decided by how f
deviates from a simple value, which float64 cannot see:

* large g: f - 1 = (1 - sigma)(g*sigma - 1) > 0 for g > 1.28, so the exact
  product lies just beyond the midpoint, away from zero;
* tiny g: f - 1/2 ~ g/2, so the sign of g decides; at g = 0 the tie is exact
  and goes to the even neighbour.

Worked case: dy = 1.5, u = 131/128 gives dy*u = 393/256 = 1.53515625, the
midpoint of the bf16 values 1.53125 (0x3FC4, even) and 1.5390625 (0x3FC5).
Ties-to-even would give 0x3FC4; the exact rule gives 0x3FC5 for large g.
The expected codes below are derived by hand from these facts, and each is
also confirmed by an independent 4000-bit mpmath evaluation of the
closed form f - 1 = (1 - sigma)(g sigma - 1).
"""
import mpmath
import numpy as np
import pytest

from oracle import mx_oracle as o

BF = {1.5: 0x3FC0, -1.5: 0xBFC0, 3.0: 0x4040, 131 / 128: 0x3F83, 130 / 128: 0x3F82,
      132 / 128: 0x3F84, 200.0: 0x4348, 2000.0: 0x44FA, 2.0 ** -100: 0x0D80, -(2.0 ** -100): 0x8D80, 0.0: 0x0000}


def _bits(v):
    b = BF[v]
    assert float(o.bf16_to_f64(np.uint16(b))) == v, v   # the table's encodings are the values
    return b


def _dg(dy, g, u):
    dg, _ = o.swiglu_bwd(np.array([_bits(dy)], np.uint16), np.array([_bits(g)], np.uint16),
                         np.array([_bits(u)], np.uint16))
    return int(dg[0])


def _mp_sign_vs(dyu, g, target):
    """sign(dy*u*f(g) - target) at 4000 bits, from f = 1 + (1 - s)(g s - 1)."""
    with mpmath.workprec(4000):
        x = mpmath.mpf(g)
        e = mpmath.exp(-x)
        s = 1 / (1 + e)
        f = 1 + (e / (1 + e)) * (x * s - 1)
        d = mpmath.mpf(dyu) * f - mpmath.mpf(target)
        return 0 if d == 0 else (1 if d > 0 else -1)


@pytest.mark.parametrize("g", [200.0, 2000.0])
def test_large_g_tie_rounds_away_from_zero(g):
    mid = 393 / 256
    assert 1.5 * (131 / 128) == mid
    assert _mp_sign_vs(mid, g, mid) == 1            # the exact value lies beyond the midpoint
    assert _dg(1.5, g, 131 / 128) == 0x3FC5         # away from zero, not ties-to-even (0x3FC4)
    assert _dg(-1.5, g, 131 / 128) == 0xBFC5


@pytest.mark.parametrize("g", [200.0, 2000.0])
def test_large_g_non_ties_round_to_the_product(g):
    # dy*u exactly representable: f - 1 is far too small to move it
    assert _dg(1.5, g, 130 / 128) == 0x3FC3         # 1.5234375
    assert _dg(1.5, g, 132 / 128) == 0x3FC6         # 1.546875
    assert _dg(-1.5, g, 130 / 128) == 0xBFC3
    with mpmath.workprec(4000):
        for u, code in ((130 / 128, 0x3FC3), (132 / 128, 0x3FC6)):
            v = float(o.bf16_to_f64(np.uint16(code)))
            ulp = 2.0 ** -7
            assert _mp_sign_vs(1.5 * u, g, v + ulp / 2) == -1 and _mp_sign_vs(1.5 * u, g, v - ulp / 2) == 1


def test_tiny_g_tie_follows_the_sign_of_g():
    # dy*u = 3.0703125, dy*u/2 = 1.53515625 (the same midpoint); f - 1/2 ~ g/2
    mid = 393 / 256
    assert _mp_sign_vs(3.0 * (131 / 128), 2.0 ** -100, mid) == 1
    assert _mp_sign_vs(3.0 * (131 / 128), -(2.0 ** -100), mid) == -1
    assert _dg(3.0, 2.0 ** -100, 131 / 128) == 0x3FC5     # away from zero
    assert _dg(3.0, -(2.0 ** -100), 131 / 128) == 0x3FC4  # towards zero
    assert _dg(3.0, 0.0, 131 / 128) == 0x3FC4             # exact tie: the even neighbour
