"""The allocation-free forward entry point (mx_mlp_fwd_static_scratch).

Some callers cannot allocate device memory at the call site (their buffers
are registered up front, or the allocator of the framework that owns the
device is not reachable from there).  mx_mlp_fwd_static_scratch serves them:
its temporary buffer is a fixed array inside the library.  These tests call
it through the C ABI and check its output and saved context against the
regular mx_mlp_fwd on the same inputs, on two calls in a row; that the call
leaves the device's free memory unchanged; that a problem whose scratch
nearly fills the array is accepted and correct; and that one beyond it is
rejected.  The file sorts last, so a run that stops at the first failure has
run everything else.
"""
import ctypes

import pytest
import torch

import block_scaled_mlp_gb300 as mx
import synth
from oracle import mx_oracle as o
from tests.util import bits, to_dev

pytestmark = pytest.mark.gpu

LIMIT = 16 << 20   # MX_STATIC_SCRATCH_BYTES


def _call_static(L, t, ctx, out, err):
    P = lambda a: ctypes.c_void_p(a.data_ptr())
    M, d = t["x"].shape
    h = t["w1"].shape[0]
    return L.mx_mlp_fwd_static_scratch(P(t["x"]), P(t["w1"]), P(t["w3"]), P(t["w2"]), M, d, h, None, 1, 128,
                                       mx.RECIPE_RCEIL, P(ctx), P(out), err.ptr(),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _check_against_mlp_fwd(L, M, d, h, seed):
    cb, sb = mx.mlp_workspace_size(M, d, h, 0, mx.RECIPE_RCEIL)
    assert sb <= LIMIT
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
    return t, ctx, out, err


def test_static_scratch_forward_matches_mlp_fwd_twice():
    L = mx.lib()
    for seed in (0, 5):   # two calls in a row, different inputs
        _check_against_mlp_fwd(L, 256, 256, 512, seed)


def test_static_scratch_call_leaves_free_device_memory_unchanged():
    L = mx.lib()
    t, ctx, out, err = _check_against_mlp_fwd(L, 256, 256, 512, 3)   # module loaded, address cached
    same = False
    for _ in range(3):   # the device is shared with other processes: one clean reading suffices
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        alloc0 = torch.cuda.memory_allocated()
        assert _call_static(L, t, ctx, out, err) == 0, L.mx_last_error()
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        assert torch.cuda.memory_allocated() == alloc0
        if free1 == free0:
            same = True
            break
    assert same, "the device's free memory changed across the call"
    err.check()


def test_static_scratch_accepts_a_problem_that_nearly_fills_the_array():
    L = mx.lib()
    M, d, h = 1024, 256, 2560            # scratch 16,596,992 bytes: 98.9% of the array
    sb = mx.mlp_workspace_size(M, d, h, 0, mx.RECIPE_RCEIL)[1]
    assert 0.95 * LIMIT <= sb <= LIMIT
    _check_against_mlp_fwd(L, M, d, h, 11)


def test_static_scratch_rejects_problems_beyond_its_size():
    L = mx.lib()
    p = ctypes.c_void_p(256)
    for M, d, h in ((1024, 256, 2688), (8192, 4096, 14336)):   # just beyond, and far beyond
        assert mx.mlp_workspace_size(M, d, h, 0, mx.RECIPE_RCEIL)[1] > LIMIT
        rc = L.mx_mlp_fwd_static_scratch(p, p, p, p, M, d, h, None, 1, 128, 0, p, p, None, None)
        assert rc == 4 and b"static" in L.mx_last_error()
