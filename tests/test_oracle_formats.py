"""Pins for the oracle's number formats: bf16 rounding, E8M0 (RCEIL) scales,
E4M3 codes, MX quantization and the MMA scale layout.

Each check compares the oracle with something other than itself: a library
cast, an exhaustive brute-force search, exact rational rounding, or values
worked out by hand from the OCP MX v1.0 definitions (tests/golden/).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import mx_oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits_of(vals):
    t = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- bf16


def test_round_to_bf16_matches_torch_cast():
    rng = np.random.default_rng(0)
    # random float32 bit patterns covering normals, subnormals, huge values
    bits = rng.integers(0, 2**32, size=200000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    # add ties and edge cases
    extra = np.array([1.0 + 2**-8, 1.0 + 3 * 2**-8, -(1.0 + 2**-8), 3.3895314e38,
                      3.4e38, 2**-133, 2**-134, 3 * 2**-134, 1e-45, -0.0, 0.0],
                     dtype=np.float32)
    f = np.concatenate([f, extra])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = o.round_to_bf16_bits(f.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_decode_roundtrip_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = o.bf16_to_f64(bits)
    fin = np.isfinite(v)
    back = o.round_to_bf16_bits(v[fin])
    assert np.array_equal(back, bits[fin])
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(v[fin], ref[fin])


# ---------------------------------------------------------------- E8M0


def _all_nonneg_finite_bf16():
    bits = np.arange(0, 0x7F80, dtype=np.uint16)
    return bits, o.bf16_to_f64(bits)


def test_e8m0_exhaustive_brute_force():
    """Every non-negative finite bf16 amax: the oracle's scale byte is the
    smallest e in [-127,127] with amax <= 448*2^e (brute-force search)."""
    bits, a = _all_nonneg_finite_bf16()
    es = np.arange(-127, 128)
    ok = a[:, None] <= 448.0 * np.power(2.0, es)[None, :]
    # smallest e satisfying the bound (always exists: 448*2^127 > bf16 max)
    e_min = es[np.argmax(ok, axis=1)]
    assert ok.any(axis=1).all()
    got = o.e8m0_rceil(a)
    assert np.array_equal(got.astype(np.int64), e_min + 127)


def test_e8m0_exhaustive_bit_rule():
    """Closed form on the bf16 bits: byte = E - 8 + (mantissa > 0x60),
    clamped at 0 (E = biased exponent field).  448 = 1.75 * 2^8 and
    1.75 is mantissa 0x60."""
    bits, a = _all_nonneg_finite_bf16()
    E = (bits.astype(np.int64) >> 7) & 0xFF
    m = bits.astype(np.int64) & 0x7F
    rule = np.where(E == 0, 0, np.maximum(E - 8 + (m > 0x60), 0))
    assert np.array_equal(o.e8m0_rceil(a).astype(np.int64), rule)


@pytest.mark.parametrize("k", [-20, -8, -1, 0, 1, 5, 20])
def test_e8m0_powers_of_two_at_448(k):
    amax = 448.0 * 2.0**k
    assert int(o.e8m0_rceil(np.array([amax]))[0]) == 127 + k
    # the next bf16 above 448*2^k needs the next scale
    nxt = o.bf16_to_f64(np.array([o.round_to_bf16_bits(amax) + 1], dtype=np.uint16))
    assert int(o.e8m0_rceil(nxt)[0]) == 128 + k


def test_e8m0_specials():
    got = o.e8m0_rceil(np.array([0.0, 2.0**-133, 450.0, 1.0, np.nan, np.inf]))
    # 1.0: ceil(log2(1/448)) = ceil(-8.807) = -8 -> 119
    assert list(got) == [0, 0, 128, 119, 255, 255]


# ---------------------------------------------------------------- E4M3


def _e4m3_grid():
    """All non-negative finite E4M3fn values with their codes, built from
    the format definition independently of the oracle."""
    vals, codes = [], []
    for c in range(0x7F):  # 0x7F is NaN
        ef, m = c >> 3, c & 7
        if ef == 0:
            v = Fraction(m, 512)
        else:
            v = (1 + Fraction(m, 8)) * Fraction(2) ** (ef - 7)
        vals.append(v)
        codes.append(c)
    return vals, codes


def _rne_exact(x: Fraction, grid, codes):
    """Nearest grid value, ties to the even code; saturate above the max."""
    if x >= grid[-1]:
        return codes[-1]
    import bisect
    i = bisect.bisect_left(grid, x)
    if grid[i] == x:
        return codes[i]
    lo, hi = i - 1, i
    dl, dh = x - grid[lo], grid[hi] - x
    if dl < dh:
        return codes[lo]
    if dh < dl:
        return codes[hi]
    return codes[lo] if codes[lo] % 2 == 0 else codes[hi]


def test_e4m3_exhaustive_vs_exact_rational():
    """Every finite bf16 value (these include every v*2^-e the quantizer can
    form, up to the exponent shift) rounded by exact rational arithmetic."""
    grid, codes = _e4m3_grid()
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = o.bf16_to_f64(bits)
    fin = np.isfinite(v)
    v = v[fin]
    got = o.e4m3_encode(v)
    # exact reference on magnitudes, vectorised by unique magnitudes
    mags = np.unique(np.abs(v))
    ref_mag = {}
    for m in mags:
        ref_mag[m] = _rne_exact(Fraction(float(m)), grid, codes)
    ref = np.array([ref_mag[abs(x)] | (0x80 if np.signbit(x) else 0) for x in v], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_matches_torch_in_range():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = o.bf16_to_f64(bits)
    m = np.isfinite(v) & (np.abs(v) <= 448.0)
    v = v[m]
    ref = torch.from_numpy(v).to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(o.e4m3_encode(v), ref)


def test_e4m3_worked_values():
    v = np.array([0.53125, 464.0, 1000.0, -0.0, 2.0**-9, 2.0**-10, 1.5 * 2.0**-10,
                  3 * 2.0**-10, 448.0, -448.0, 1.0, 0.0, np.inf, np.nan])
    want = [0x30, 0x7E, 0x7E, 0x80, 0x01, 0x00, 0x01, 0x02, 0x7E, 0xFE, 0x38, 0x00, 0x7E, 0x7F]
    assert list(o.e4m3_encode(v)) == want
    # powers of two inside the range map exactly
    for k in range(-9, 9):
        c = int(o.e4m3_encode(np.array([2.0**k]))[0])
        assert o.e4m3_decode(np.array([c]))[0] == 2.0**k


# ---------------------------------------------------------------- MX blocks


def _load_golden():
    with open(os.path.join(GOLDEN, "mx_blocks.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _load_golden()["blocks"], ids=lambda c: c["name"])
def test_golden_blocks(case):
    vals = case["values"]
    bits = _bf16_bits_of(vals).reshape(1, 32)
    q, s = o.quantize_rows(bits)
    assert int(s[0, 0]) == case["scale"], case["why"]
    assert [int(c) for c in q[0]] == case["codes"], case["why"]


def test_quantize_error_bound_and_scale_range():
    """|deq - v| <= half an E4M3 step (relative 2^-4 on normals), and every
    block's max code is in the top binade unless the block is zero."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, 256)).astype(np.float32) * np.exp(rng.uniform(-30, 30, (64, 1))).astype(np.float32)
    bits = _bf16_bits_of(x)
    q, s = o.quantize_rows(bits)
    deq = o.dequantize(q, s)
    v = o.bf16_to_f64(bits)
    e = (s.astype(np.int64) - 127).repeat(32, axis=1)
    step = np.ldexp(np.ones_like(v), e)  # scale
    rel = np.abs(deq - v)
    # bound: half the quantum of the e4m3 binade of v/scale (>= 2^-10 * scale)
    vs = np.abs(v) / step
    _, ex = np.frexp(np.maximum(vs, 2.0**-6))
    quantum = np.ldexp(1.0, np.maximum(ex - 1, -6) - 3) * step
    assert np.all(rel <= quantum / 2 + 0)
    # RCEIL puts the scaled block amax in (224, 448]; RNE may take it to 224
    amax_code = np.max(np.abs(o.e4m3_decode(q)).reshape(64, 8, 32), axis=2)
    assert np.all((amax_code >= 224) & (amax_code <= 448))


def test_columnwise_blocks_run_along_rows():
    """A matrix whose column j holds j+1 in row 5 and zeros elsewhere: every
    column block of rows 0..31 has amax j+1; other row blocks are zero."""
    R, C = 64, 32
    x = np.zeros((R, C), dtype=np.float32)
    x[5, :] = np.arange(1, C + 1)
    q, s = o.quantize_cols(_bf16_bits_of(x))
    assert q.shape == (C, R) and s.shape == (C, R // 32)
    for j in range(C):
        assert int(s[j, 0]) == int(o.e8m0_rceil(np.array([j + 1.0]))[0])
        assert int(s[j, 1]) == 0
        assert np.count_nonzero(q[j]) == 1 and q[j, 5] != 0


def test_mma_layout_positions_and_roundtrip():
    R, Cs = 256, 12
    rng = np.random.default_rng(2)
    s = rng.integers(0, 255, size=(R, Cs), dtype=np.uint8)
    flat = o.scales_to_mma(s)
    assert flat.size == 2 * 3 * 512
    # hand-computed positions: tile (rb, cb) at (rb*3 + cb)*512, inside
    # (r%32)*16 + ((r%128)//32)*4 + c%4
    assert flat[0] == s[0, 0]
    assert flat[(0 * 3 + 1) * 512 + 1 * 16 + 1 * 4 + 1] == s[33, 5]
    assert flat[(1 * 3 + 2) * 512 + 31 * 16 + 3 * 4 + 3] == s[255, 11]
    assert np.array_equal(o.scales_from_mma(flat, R, Cs), s)


def test_mma_layout_padding_is_zero():
    s = np.full((100, 5), 7, dtype=np.uint8)
    flat = o.scales_to_mma(s)
    assert flat.size == 1 * 2 * 512
    assert np.count_nonzero(flat) == 100 * 5
