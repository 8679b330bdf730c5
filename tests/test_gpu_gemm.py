"""GPU parity of the tcgen05 GEMMs (block-scaled MXFP8 dense / M-grouped /
K-grouped, and the bf16 weight-gradient GEMM) against the oracle's exact
fp64 accumulation.

Bar: normwise ||C - C_ref|| / ||C_ref|| <= 2e-3 against the fp64 value
before rounding, and every element within one bf16 step of RN_bf16(C_ref)."""
import numpy as np
import pytest
import torch

import block_scaled_mlp_gb300 as mx
import synth
from oracle import mx_oracle as o
from tests.util import bits, to_dev, u8

pytestmark = pytest.mark.gpu
TOL = 2e-3


def _rand_codes(rng, shape):
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x3F          # no NaN codes
    return c


def _rand_scales(rng, rows, cols, lo=122, hi=133):
    return rng.integers(lo, hi, size=(rows, cols // 32), dtype=np.uint8)


def _bf16_ulp(v):
    """Spacing of bf16 values at |v| (subnormal spacing below 2^-126)."""
    a = np.abs(v)
    _, ex = np.frexp(np.maximum(a, 2.0**-126))
    return np.ldexp(1.0, ex - 1 - 7)


def _assert_close(got_bits, ref_f, what="", absdot=None, K=None):
    """Normwise bar, plus an elementwise bound: one bf16 step of the exact
    value plus K * 2^-23 * sum_k |a_k b_k| for the fp32 accumulation."""
    got = o.bf16_to_f64(got_bits)
    err = o.normwise_rel_err(got, ref_f)
    ref_b = o.round_to_bf16_bits(ref_f)
    frac = float((got_bits != ref_b).mean())
    print(f"{what}: normwise {err:.3e}, not-RN fraction {frac:.3e}")
    assert err <= TOL, (what, err)
    if absdot is not None:
        bound = _bf16_ulp(ref_f) + K * 2.0**-23 * absdot
        bad = np.abs(got - ref_f) > bound
        assert not bad.any(), (what, int(bad.sum()), got[bad][:4], ref_f[bad][:4])


def _dev_scales(s):
    return to_dev(o.scales_to_mma(s), dtype=torch.uint8)


@pytest.mark.parametrize("scales", ["uniform", "varying"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 512, 384), (384, 384, 256)])
def test_scaled_mm_random_codes(M, N, K, scales):
    rng = np.random.default_rng(M * 7 + N + K)
    aq, bq = _rand_codes(rng, (M, K)), _rand_codes(rng, (N, K))
    if scales == "uniform":
        as_ = np.full((M, K // 32), 127, np.uint8)
        bs = np.full((N, K // 32), 127, np.uint8)
    else:
        as_, bs = _rand_scales(rng, M, K), _rand_scales(rng, N, K)
    c = mx.scaled_mm(to_dev(aq, torch.uint8), _dev_scales(as_), to_dev(bq, torch.uint8), _dev_scales(bs))
    torch.cuda.synchronize()
    _assert_close(bits(c), o.mx_mm(aq, as_, bq, bs), f"scaled_mm {M}x{N}x{K} {scales}",
                  o.mx_mm(aq & 0x7F, as_, bq & 0x7F, bs), K)


def test_scaled_mm_quantized_operands():
    M, N, K = 256, 1024, 512
    a = synth.normal_bf16((M, K), 1.0, 31)
    b = synth.normal_bf16((N, K), 0.02, 32)
    (aq, as_), (bq, bs) = o.quantize_rows(a), o.quantize_rows(b)
    c = mx.scaled_mm(to_dev(aq, torch.uint8), _dev_scales(as_), to_dev(bq, torch.uint8), _dev_scales(bs))
    torch.cuda.synchronize()
    _assert_close(bits(c), o.mx_mm(aq, as_, bq, bs), "scaled_mm quantized",
                  o.mx_mm(aq & 0x7F, as_, bq & 0x7F, bs), K)


def _grouped_offs(counts):
    pc = synth.pad_counts(np.array(counts))
    return synth.offsets_from_counts(pc)


def test_grouped_m_with_empty_groups_and_tail():
    rng = np.random.default_rng(5)
    counts = [100, 0, 250, 128, 0]
    offs = _grouped_offs(counts)
    M_total = int(offs[-1]) + 128            # one tail tile
    N, K, E = 256, 256, len(counts)
    aq = _rand_codes(rng, (M_total, K))
    as_ = _rand_scales(rng, M_total, K)
    bq = _rand_codes(rng, (E, N, K))
    bs = np.stack([_rand_scales(rng, N, K) for _ in range(E)])
    err = mx.ErrorWord()
    c = mx.grouped_mm(mx.GROUP_M, to_dev(aq, torch.uint8), _dev_scales(as_), to_dev(bq, torch.uint8),
                      to_dev(o.scales_to_mma(bs), torch.uint8), to_dev(offs, torch.int32), err=err)
    torch.cuda.synchronize()
    err.check()
    ref = o.mx_grouped_mm_m(aq, as_, bq, bs, offs)
    got = bits(c)
    assert not got[int(offs[-1]):].any(), "tail rows must be zero"
    _assert_close(got, ref, "grouped_m", o.mx_grouped_mm_m(aq & 0x7F, as_, bq & 0x7F, bs, offs), K)


def test_grouped_k_with_empty_group():
    rng = np.random.default_rng(6)
    counts = [128, 0, 300, 60]
    offs = _grouped_offs(counts)
    T = int(offs[-1])
    N, K, E = 256, 384, len(counts)
    aq, bq = _rand_codes(rng, (N, T)), _rand_codes(rng, (K, T))
    as_, bs = _rand_scales(rng, N, T), _rand_scales(rng, K, T)
    err = mx.ErrorWord()
    c = mx.grouped_mm(mx.GROUP_K, to_dev(aq, torch.uint8), _dev_scales(as_), to_dev(bq, torch.uint8),
                      _dev_scales(bs), to_dev(offs, torch.int32), err=err)
    torch.cuda.synchronize()
    err.check()
    got = bits(c)
    assert not got[1].any(), "empty expert must get exact zeros"
    _assert_close(got, o.mx_grouped_mm_k(aq, as_, bq, bs, offs), "grouped_k",
                  o.mx_grouped_mm_k(aq & 0x7F, as_, bq & 0x7F, bs, offs), T)


def test_grouped_bad_offsets_flagged():
    rng = np.random.default_rng(7)
    offs = np.array([256, 128, 384], dtype=np.int32)      # decreasing
    M_total, N, K = 384, 256, 128
    aq = _rand_codes(rng, (M_total, K))
    bq = _rand_codes(rng, (3, N, K))
    err = mx.ErrorWord()
    mx.grouped_mm(mx.GROUP_M, to_dev(aq, torch.uint8), _dev_scales(_rand_scales(rng, M_total, K)),
                  to_dev(bq, torch.uint8),
                  to_dev(o.scales_to_mma(np.stack([_rand_scales(rng, N, K)] * 3)), torch.uint8),
                  to_dev(offs, torch.int32), err=err)
    torch.cuda.synchronize()
    assert err.value() & 8


@pytest.mark.parametrize("grouped", [False, True])
def test_bf16_wgrad(grouped):
    rng = np.random.default_rng(8)
    counts = [128, 0, 256]
    offs = _grouped_offs(counts) if grouped else np.array([384], np.int32)
    T = int(offs[-1])
    N, K = 256, 512
    a = o.round_to_bf16_bits(rng.standard_normal((N, T)))
    b = o.round_to_bf16_bits(rng.standard_normal((K, T)) * 0.1)
    c = mx.bf16_wgrad(to_dev(a), to_dev(b), to_dev(offs, torch.int32) if grouped else None)
    torch.cuda.synchronize()
    ref = o.bf16_grouped_mm_k(a, b, offs)
    absdot = o.bf16_grouped_mm_k(a & 0x7FFF, b & 0x7FFF, offs)
    got = bits(c)
    if not grouped:
        ref, absdot = ref[0], absdot[0]
    else:
        assert not got[1].any()
    _assert_close(got, ref, f"bf16_wgrad grouped={grouped}", absdot, T)
