"""Pins of the FLOOR scale mode (reading R14): the E8M0 byte against a
brute-force search on every non-negative bf16 amax, worked values where
saturation binds, and its relation to RCEIL."""
import numpy as np

import synth
from oracle import mx_oracle as o


def _all_amax():
    bits = np.arange(0, 0x7F81, dtype=np.uint16)            # +0 .. +Inf
    return bits, o.bf16_to_f64(bits)


def test_floor_against_brute_force_every_bf16_amax():
    bits, a = _all_amax()
    got = o.e8m0_floor(a)
    for i in range(0, a.size, 97):                          # brute force on a spread sample
        v = a[i]
        if not np.isfinite(v):
            assert got[i] == 255
            continue
        if v == 0:
            assert got[i] == 0
            continue
        k = -200
        while 2.0 ** (k + 1) <= v:                          # largest k with 2^k <= amax
            k += 1
        assert got[i] == min(max(k - 8, -127), 127) + 127, (i, v)
    # closed form on every value: the bf16 exponent field minus 8
    E = (bits.astype(np.int64) >> 7) & 0xFF
    fin = np.isfinite(a) & (a > 0)
    normal = fin & (E > 0)
    assert np.array_equal(got[normal], np.maximum(E[normal] - 8, 0).astype(np.uint8))
    assert np.all(got[fin & (E == 0)] == 0)                  # subnormal amax clamps


def test_floor_worked_values_and_saturation():
    assert o.e8m0_floor([448.0, 480.0, 511.0, 512.0, 1.0, 0.0, 2.0 ** -140]).tolist() == \
        [127, 127, 127, 128, 119, 0, 0]
    assert o.e8m0_floor([np.nan, np.inf]).tolist() == [255, 255]
    block = np.zeros(32, np.float32)
    block[0], block[1], block[2] = 480.0, 1.0, -500.0
    bits = synth.bf16_from_f32(block)[None]
    q, s = o.quantize_rows(bits, o.SCALE_FLOOR)
    assert s[0, 0] == 127 and q[0, 0] == 0x7E and q[0, 2] == 0xFE     # +-448: saturation binds
    q, s = o.quantize_rows(bits, o.SCALE_RCEIL)
    assert s[0, 0] == 128 and q[0, 0] == 0x77                         # 240 = 1.875 * 2^7, exact


def test_floor_relation_to_rceil():
    bits, a = _all_amax()
    fin = np.isfinite(a) & (a >= 2.0 ** -100)
    f, r = o.e8m0_floor(a[fin]).astype(int), o.e8m0_rceil(a[fin]).astype(int)
    mant = bits[fin].astype(np.int64) & 0x7F
    assert np.all((r - f) == (mant > 0x60))                  # RCEIL rounds up iff amax/2^E > 1.75
