"""Pins of the oracle's FP8 per-tensor ("tensorwise") scaling and its grouped
GEMMs (reading R15; page "[mxfp8 training] unified MXFP8TrainingConfig and
MXFP8TrainingTensor", FP8 GroupedMM, the non-MX FP8 recipe).

* Hand-worked cases (tests/golden/fp8_tensorwise.json): scale bits and
  codes, including an fp32 tie inside x*s, an E4M3 tie, a subnormal code,
  signed zeros and the all-zero floor.
* Invariant: the element that attains amax maps to +-448 (0x7E / 0xFE) for
  every magnitude of amax.
* In-range codes against torch's float8_e4m3fn cast of the same fp32
  products (an independent rounding routine).
* GEMMs against a pure-Python triple loop with its own E4M3 decoder;
  grouped == per-group dense; K-grouped sums to the dense product; empty
  experts and tail rows give zeros; close to the unquantized product.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import mx_oracle as o
import synth

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = json.load(open(os.path.join(HERE, "golden", "fp8_tensorwise.json")))


@pytest.mark.parametrize("case", GOLD["cases"], ids=[c["name"] for c in GOLD["cases"]])
def test_worked_cases(case):
    x = synth.bf16_from_f32(np.array(case["values"], np.float32))
    codes, s, amax = o.fp8_quantize_tensor(x)
    assert int(np.float32(s).view(np.uint32)) == int(case["scale_bits"], 16)
    assert [int(c) for c in codes] == [int(c, 16) for c in case["codes"]]


def _decode_py(c: int) -> Fraction:
    sign = -1 if c & 0x80 else 1
    e, m = (c >> 3) & 0xF, c & 7
    if e == 0:
        return sign * Fraction(m, 512)
    return sign * (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)


def test_amax_element_maps_to_448_at_every_magnitude():
    rng = np.random.default_rng(5)
    for k in range(-30, 31, 3):
        v = rng.standard_normal(256).astype(np.float32) * np.float32(2.0 ** k)
        x = synth.bf16_from_f32(v)
        codes, s, amax = o.fp8_quantize_tensor(x)
        i = int(np.argmax(np.abs(o.bf16_to_f64(x))))
        assert codes[i] & 0x7F == 0x7E, (k, hex(codes[i]))
        assert np.all((codes & 0x7F) <= 0x7E)            # never NaN for finite input


def test_codes_equal_torch_e4m3_cast_of_the_fp32_products():
    rng = np.random.default_rng(6)
    x = synth.bf16_from_f32((rng.standard_normal((64, 96)) * np.exp(rng.uniform(-4, 4, (64, 96)))).astype(np.float32))
    codes, s, _ = o.fp8_quantize_tensor(x)
    prod = torch.from_numpy(o.bf16_to_f64(x).astype(np.float32)) * torch.tensor(float(s), dtype=torch.float32)
    ref = prod.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.abs(prod.numpy()).max() <= 448.0 * (1 + 2.0 ** -23)
    assert np.array_equal(codes, ref)


def test_per_expert_scales_equal_separate_tensors():
    rng = np.random.default_rng(7)
    w = synth.bf16_from_f32((rng.standard_normal((3, 16, 32)) * np.array([1e-3, 1.0, 50.0])[:, None, None])
                            .astype(np.float32))
    codes, s, amax = o.fp8_quantize_tensor(w, batch_axes=1)
    assert s.shape == (3,)
    for e in range(3):
        ce, se, _ = o.fp8_quantize_tensor(w[e])
        assert np.array_equal(codes[e], ce) and np.float32(se) == s[e]


def test_grouped_m_against_triple_loop():
    rng = np.random.default_rng(8)
    x = synth.bf16_from_f32(rng.standard_normal((5, 7)).astype(np.float32))
    w = synth.bf16_from_f32((rng.standard_normal((2, 3, 7)) * 0.1).astype(np.float32))
    aq, sa, _ = o.fp8_quantize_tensor(x)
    bq, sb, _ = o.fp8_quantize_tensor(w, batch_axes=1)
    offs = np.array([2, 4], np.int32)                  # rows 0-1 expert 0, 2-3 expert 1, row 4 tail
    got = o.fp8_grouped_mm_m(aq, sa, bq, sb, offs)
    for i in range(5):
        e = 0 if i < 2 else (1 if i < 4 else None)
        for j in range(3):
            if e is None:
                assert got[i, j] == 0.0
                continue
            acc = sum(_decode_py(int(aq[i, k])) * _decode_py(int(bq[e, j, k])) for k in range(7))
            ref = acc / (Fraction(float(sa)) * Fraction(float(sb[e])))
            assert abs(got[i, j] - float(ref)) <= 1e-12 * max(1.0, abs(float(ref)))


def test_grouped_k_sums_to_dense_and_empty_expert_is_zero():
    rng = np.random.default_rng(9)
    M, N, K = 384, 16, 24
    a = synth.bf16_from_f32(rng.standard_normal((N, M)).astype(np.float32))
    b = synth.bf16_from_f32(rng.standard_normal((K, M)).astype(np.float32))
    aq, sa, _ = o.fp8_quantize_tensor(a)
    bq, sb, _ = o.fp8_quantize_tensor(b)
    offs = np.array([128, 128, 384], np.int32)
    C = o.fp8_grouped_mm_k(aq, sa, bq, sb, offs)
    assert not C[1].any()
    dense = o.fp8_dequantize(aq, sa) @ o.fp8_dequantize(bq, sb).T
    assert np.allclose(C.sum(axis=0), dense, rtol=1e-12, atol=1e-12)
    # grouped M of the transposes per group equals the K-grouped slices
    for e, (s, t) in enumerate(o.group_bounds(offs)):
        if t > s:
            ref = o.fp8_dequantize(aq[:, s:t], sa) @ o.fp8_dequantize(bq[:, s:t], sb).T
            assert np.allclose(C[e], ref, rtol=1e-12, atol=1e-12)


def test_close_to_unquantized_product_and_transposition_is_caught():
    rng = np.random.default_rng(10)
    x = synth.bf16_from_f32(rng.standard_normal((256, 128)).astype(np.float32))
    w = synth.bf16_from_f32((rng.standard_normal((1, 128, 128)) * 0.02).astype(np.float32))
    aq, sa, _ = o.fp8_quantize_tensor(x)
    bq, sb, _ = o.fp8_quantize_tensor(w, batch_axes=1)
    got = o.fp8_grouped_mm_m(aq, sa, bq, sb, np.array([256], np.int32))
    ref = o.bf16_to_f64(x) @ o.bf16_to_f64(w[0]).T
    err = o.normwise_rel_err(got, ref)
    assert err < 0.06, err                                   # E4M3 rounding of both operands
    assert o.normwise_rel_err(got, o.bf16_to_f64(x) @ o.bf16_to_f64(w[0])) > 0.5
