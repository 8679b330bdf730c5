"""Failure detection on the GPU without a fault: a pipeline wait that runs
past its bound ends the kernel with MX_ERR_TIMEOUT in the error word, and the
context stays usable (the next GEMM is exact)."""
import numpy as np
import pytest
import torch

import block_scaled_mlp_gb300 as mx
import synth
from oracle import mx_oracle as o
from tests.util import bits, to_dev

pytestmark = pytest.mark.gpu


def test_expired_wait_reports_timeout_and_context_survives():
    err = mx.ErrorWord()
    mx._check(mx.lib().mx_selftest_wait_timeout(err.ptr(), mx._stream()))
    torch.cuda.synchronize()
    assert err.value() & 16, f"expected MX_ERR_TIMEOUT, got {err.value()}"
    # the same context runs a GEMM correctly afterwards
    rng = np.random.default_rng(2)
    ints = lambda *s: synth.bf16_from_f32(rng.integers(-7, 8, s).astype(np.float32))
    a, b = ints(256, 256), ints(128, 256)
    qa, qb = mx.quantize(to_dev(a), mx.ROW), mx.quantize(to_dev(b), mx.ROW)
    c = mx.scaled_mm(qa["q_row"], qa["s_row"], qb["q_row"], qb["s_row"])
    torch.cuda.synchronize()
    ref = o.round_to_bf16_bits(o.bf16_to_f64(a) @ o.bf16_to_f64(b).T)
    assert np.array_equal(bits(c), ref)
