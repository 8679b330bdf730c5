"""C-ABI checks that need no GPU: the library loads, exports every entry
point the header declares, and rejects bad arguments on the host (before
any CUDA call) with the documented status codes."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxmlp.h")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    import block_scaled_mlp_gb300 as mx
    return mx.lib()


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"MX_API\s+(?:const\s+char\*|int|size_t)\s+(mx_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for want in ["mx_quantize", "mx_swiglu_quant", "mx_swiglu_quant_bwd", "mx_scaled_mm", "mx_grouped_mm",
                 "mx_bf16_wgrad", "mx_mlp_workspace_size", "mx_mlp_fwd", "mx_mlp_bwd",
                 "mx_token_group_pad_workspace", "mx_token_group_pad", "mx_gather_rows",
                 "mx_linear_workspace_size", "mx_linear_fwd", "mx_linear_bwd", "mx_quantize_mode",
                 "mx_swiglu_quant_mode", "mx_swiglu_quant_bwd_mode", "mx_mlp_fwd_static_scratch",
                 "mx_selftest_wait_timeout", "mx_selftest_silu_table", "mx_mlp_ctx_layout"]:
        assert want in names


def test_library_exports_every_declared_symbol(L):
    for name in _declared():
        assert hasattr(L, name), name


def test_launch_counters_readable_without_a_gpu(L):
    import block_scaled_mlp_gb300 as mx
    assert L.mx_launch_counts(None, 0) == len(mx.KERNEL_FAMILIES)
    before = mx.launch_counts()
    p = ctypes.c_void_p(0x10000)
    assert L.mx_quantize(None, 64, 64, 3, 1, p, p, p, p, None) == 1   # rejected on the host: nothing launched
    assert mx.launch_counts() == before


def test_status_strings(L):
    assert L.mx_status_string(0) == b"MX_OK"
    assert L.mx_status_string(8) == b"MX_ERR_BAD_OFFSETS"
    assert L.mx_status_string(16) == b"MX_ERR_TIMEOUT"
    assert L.mx_version() >= 100


def _fake(addr=0x10000):
    return ctypes.c_void_p(addr)


def test_quantize_rejects_bad_arguments(L):
    p = _fake()
    assert L.mx_quantize(None, 64, 64, 3, 1, p, p, p, p, None) == 1           # null x
    assert L.mx_quantize(p, 64, 48, 1, 1, p, p, None, None, None) == 4        # cols % 32
    assert L.mx_quantize(p, 48, 64, 2, 1, None, None, p, p, None) == 4        # rows % 32 for COL
    assert L.mx_quantize(p, 64, 64, 5, 1, p, p, p, p, None) == 1              # bad axis
    assert L.mx_quantize(_fake(0x10001), 64, 64, 1, 1, p, p, None, None, None) == 2  # alignment
    assert b"aligned" in L.mx_last_error()


def test_gemm_rejects_bad_arguments(L):
    p = _fake()
    assert L.mx_scaled_mm(p, p, p, p, 100, 128, 128, p, None, None) == 4
    assert L.mx_grouped_mm(0, p, p, p, p, 256, 128, 128, p, 4, 64, p, None, None) == 4   # pad 64
    assert L.mx_grouped_mm(0, p, p, p, p, 256, 128, 128, p, 0, 128, p, None, None) == 1  # E = 0
    assert L.mx_grouped_mm(7, p, p, p, p, 256, 128, 128, p, 4, 128, p, None, None) == 1  # mode
    assert L.mx_bf16_wgrad(p, p, 256, 128, 128, None, 3, 128, p, None, None) == 1         # dense needs E=1


def test_mlp_workspace_and_validation(L):
    c, s = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.mx_mlp_workspace_size(256, 256, 512, 0, 0, ctypes.byref(c), ctypes.byref(s)) == 0
    # ctx holds at least h13 (bf16) and the columnwise copies
    assert c.value >= 256 * 1024 * 2 + 256 * 256 + 512 * 256
    assert s.value > 0
    c2, s2 = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.mx_mlp_workspace_size(256, 256, 512, 0, 1, ctypes.byref(c2), ctypes.byref(s2)) == 0
    p = _fake()
    assert L.mx_mlp_fwd(p, p, p, p, 200, 256, 512, None, 0, 128, 0, p, p, p, None, None) == 4
    assert L.mx_mlp_fwd(p, p, p, p, 0, 256, 512, None, 0, 128, 0, p, p, p, None, None) == 1   # no rows
    assert L.mx_mlp_fwd(p, p, p, p, 256, 256, 512, p, 4, 128, 9, p, p, p, None, None) == 1
    assert L.mx_mlp_bwd(p, None, p, p, p, p, 256, 256, 512, None, 0, 128, 0, p, p, p, p, p, None, None) == 1


def test_token_group_pad_rejects_bad_arguments(L):
    p = _fake()
    assert L.mx_token_group_pad_workspace(4096, 16) == 16 + 4 * 16 * 4     # 4 chunks of 1024 rows
    assert L.mx_token_group_pad(p, 100, 0, 128, 256, p, p, p, p, None, None) == 4       # E = 0
    assert L.mx_token_group_pad(p, 100, 2000, 128, 256, p, p, p, p, None, None) == 4    # E > 1024
    assert L.mx_token_group_pad(p, 100, 4, 64, 256, p, p, p, p, None, None) == 4        # pad 64
    assert L.mx_token_group_pad(p, 100, 4, 128, 200, p, p, p, p, None, None) == 4       # M_cap % 128
    assert L.mx_token_group_pad(p, -1, 4, 128, 256, p, p, p, p, None, None) == 1        # R < 0
    assert L.mx_token_group_pad(None, 100, 4, 128, 256, p, p, p, p, None, None) == 1    # no expert ids
    assert L.mx_token_group_pad(p, 100, 4, 128, 256, p, p, p, None, None, None) == 1    # no workspace
    assert L.mx_gather_rows(p, 10, 12, p, 10, 1, p, None, None) == 4                      # cols % 8
    assert L.mx_gather_rows(p, 10, 16, p, 10, 0, p, None, None) == 1                      # div 0
    assert L.mx_gather_rows(ctypes.c_void_p(0x1008), 10, 16, p, 10, 1, p, None, None) == 2  # alignment


def test_scale_modes_and_recipes(L):
    p = _fake()
    assert L.mx_quantize_mode(p, 64, 64, 3, 1, 2, p, p, p, p, None) == 1                 # scale mode 2
    assert L.mx_swiglu_quant_mode(p, 64, 64, 1, 1, 5, p, p, None, None, None) == 1
    assert L.mx_swiglu_quant_bwd_mode(p, p, 64, 64, 1, 1, -1, p, p, None, None, None, None, None) == 1
    c, s = ctypes.c_size_t(), ctypes.c_size_t()
    for recipe in (2, 3):                                                                  # FLOOR recipes
        assert L.mx_mlp_workspace_size(256, 256, 512, 0, recipe, ctypes.byref(c), ctypes.byref(s)) == 0
        assert L.mx_linear_workspace_size(256, 256, 512, recipe, ctypes.byref(c), ctypes.byref(s)) == 0
    assert L.mx_mlp_workspace_size(256, 256, 512, 0, 4, ctypes.byref(c), ctypes.byref(s)) == 1


def test_linear_rejects_bad_arguments(L):
    p = _fake()
    c, s = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.mx_linear_workspace_size(256, 384, 512, 0, ctypes.byref(c), ctypes.byref(s)) == 0
    assert c.value >= 384 * 256 and s.value >= 256 * 384 + 512 * 384
    assert L.mx_linear_workspace_size(256, 384, 500, 0, ctypes.byref(c), ctypes.byref(s)) == 4   # N % 128
    assert L.mx_linear_fwd(p, p, 256, 384, 512, 7, p, p, p, None, None) == 1                     # recipe
    assert L.mx_linear_fwd(p, None, 256, 384, 512, 0, p, p, p, None, None) == 1                  # no w
    assert L.mx_linear_bwd(p, p, p, 0, 384, 512, 0, p, p, p, None, None) == 1                    # M = 0
    assert L.mx_linear_bwd(p, p, ctypes.c_void_p(0x10008), 256, 384, 512, 0, p, p, p, None, None) == 2


def test_python_binding_fails_loudly_without_cuda_tensors():
    import torch
    import block_scaled_mlp_gb300 as mx
    with pytest.raises(mx.MxError):
        mx.quantize(torch.zeros(64, 64, dtype=torch.bfloat16))


def test_mlp_context_layout(L):
    """Saved tensors tile the context without overlap, 256-byte aligned, and
    exist exactly under the recipes that keep them."""
    import block_scaled_mlp_gb300 as mx
    M, d, h = 1024, 256, 384
    for E in (0, 4):
        for recipe in (mx.RECIPE_RCEIL, mx.RECIPE_RCEIL_WGRAD_HP, mx.RECIPE_FLOOR, mx.RECIPE_FLOOR_WGRAD_HP):
            ctx_bytes, _ = mx.mlp_workspace_size(M, d, h, E, recipe)
            hp = recipe in (mx.RECIPE_RCEIL_WGRAD_HP, mx.RECIPE_FLOOR_WGRAD_HP)
            spans = []
            for name in mx.CTX_TENSORS:
                cols = name in ("xq_col", "xs_col", "yq_col", "ys_col")
                if (name == "x_t" and not hp) or (cols and hp):
                    with pytest.raises(mx.MxError):
                        mx.mlp_ctx_layout(M, d, h, E, recipe, name)
                    continue
                off, n = mx.mlp_ctx_layout(M, d, h, E, recipe, name)
                assert off % 256 == 0 and off + n <= ctx_bytes
                spans.append((off, n, name))
            spans.sort()
            assert spans[0][0] == 0 and spans[0][2] == "h13" and spans[0][1] == M * 2 * h * 2
            for (o0, n0, _), (o1, _, _) in zip(spans, spans[1:]):
                assert o0 + n0 <= o1
            Ew = max(E, 1)
            sizes = {nm: n for _, n, nm in spans}
            assert sizes["w13q_col"] == Ew * d * 2 * h and sizes["w2q_col"] == Ew * h * d
            if not hp:
                assert sizes["yq_col"] == h * M and sizes["ys_col"] == mx.mma_scale_bytes(h, M)
    off, n = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.mx_mlp_ctx_layout(M, d, h, 0, 0, 10, ctypes.byref(off), ctypes.byref(n)) == 1


def test_silu_table_needs_a_destination(L):
    assert L.mx_selftest_silu_table(None, None) == 1  # MX_ERR_INVALID_ARG, before any device call


def test_selftest_needs_an_error_word(L):
    """The wait-timeout self-test rejects a missing error word on the host,
    before touching the device."""
    assert L.mx_selftest_wait_timeout(None, None) == 1  # MX_ERR_INVALID_ARG
