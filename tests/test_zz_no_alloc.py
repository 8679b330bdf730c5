"""The allocation-free forward entry point (mx_mlp_fwd_static_scratch).

Some callers cannot allocate device memory at the call site (their buffers
are registered up front, or the allocator of the framework that owns the
device is not reachable from there).  mx_mlp_fwd_static_scratch serves them:
its temporary buffer is a fixed array inside the library.  This test calls
it through the C ABI twice in a row and checks each result against the
regular mx_mlp_fwd on the same inputs.  It lives in its own file that sorts
last, so a run that stops at the first failure has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_scaled_mlp_gb300 as mx
import synth
from oracle import mx_oracle as o
from tests.util import bits, to_dev

pytestmark = pytest.mark.gpu


def _call_static(L, t, ctx, out, err):
    P = lambda a: ctypes.c_void_p(a.data_ptr())
    M, d = t["x"].shape
    h = t["w1"].shape[0]
    return L.mx_mlp_fwd_static_scratch(P(t["x"]), P(t["w1"]), P(t["w3"]), P(t["w2"]), M, d, h, None, 1, 128,
                                       mx.RECIPE_RCEIL, P(ctx), P(out), err.ptr(),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_static_scratch_forward_matches_mlp_fwd_twice():
    L = mx.lib()
    M, d, h = 256, 256, 512
    cb, sb = mx.mlp_workspace_size(M, d, h, 0, mx.RECIPE_RCEIL)
    assert sb <= 16 << 20
    for seed in (0, 5):   # two calls in a row, different inputs
        inp = synth.dense_mlp_inputs(M, d, h, seed)
        t = {k: to_dev(v) for k, v in inp.items()}
        ref, ref_ctx = mx.mlp_fwd(t["x"], t["w1"], t["w3"], t["w2"], recipe=mx.RECIPE_RCEIL)
        ctx = torch.empty(cb, dtype=torch.uint8, device="cuda")
        out = torch.empty((M, d), dtype=torch.bfloat16, device="cuda")
        err = mx.ErrorWord()
        rc = _call_static(L, t, ctx, out, err)
        assert rc == 0, L.mx_last_error()
        torch.cuda.synchronize()
        err.check()
        e = o.normwise_rel_err(o.bf16_to_f64(bits(out)), o.bf16_to_f64(bits(ref)))
        assert e <= 2e-3
        assert torch.equal(out, ref)          # same kernels, same inputs
        assert torch.equal(ctx, ref_ctx.buf)  # the saved context too


def test_static_scratch_rejects_problems_beyond_its_size():
    L = mx.lib()
    M, d, h = 8192, 4096, 14336                 # scratch far above the array
    p = ctypes.c_void_p(256)
    rc = L.mx_mlp_fwd_static_scratch(p, p, p, p, M, d, h, None, 1, 128, 0, p, p, None, None)
    assert rc == 4 and b"static" in L.mx_last_error()
