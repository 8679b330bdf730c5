"""Parity of the token-group padding kernels with the oracle (reading R12):
offsets and row maps bit-exact, gathered activations bit-exact, pad and
tail rows zero, on small and full-size (MoE 64E: 16384 tokens x top-8)
routings, plus the degenerate and faulty cases."""
import numpy as np
import pytest
import torch

import block_scaled_mlp_gb300 as mx
import synth
from oracle import mx_oracle as o
from tests.util import bits, to_dev

pytestmark = pytest.mark.gpu


def _run(ids, E, m_cap=None):
    err = mx.ErrorWord()
    offs, dst, src = mx.token_group_pad(torch.as_tensor(ids, dtype=torch.int32, device="cuda"), E, m_cap, err=err)
    torch.cuda.synchronize()
    return offs.cpu().numpy(), dst.cpu().numpy(), src.cpu().numpy(), err.value()


@pytest.mark.parametrize("R,E,seed", [(1, 1, 0), (31, 3, 1), (1000, 16, 2), (1025, 7, 3), (5000, 64, 4),
                                      (20000, 1000, 5), (4096, 1, 6)])
def test_layout_matches_oracle(R, E, seed):
    ids = np.random.default_rng(seed).integers(0, E, R).astype(np.int32)
    m_cap = mx.token_group_capacity(R, E)
    offs, dst, src, err = _run(ids, E, m_cap)
    o_offs, o_dst, o_src = o.token_group_pad(ids, E, 128, m_cap)
    assert err == 0
    assert np.array_equal(offs, o_offs) and np.array_equal(dst, o_dst) and np.array_equal(src, o_src)


def test_empty_experts_and_single_expert():
    counts = np.array([0, 300, 0, 0, 128, 1, 0])
    ids = synth.routed_expert_ids(counts, 9)
    offs, dst, src, err = _run(ids, len(counts))
    o_offs, o_dst, o_src = o.token_group_pad(ids, len(counts), 128, src.size)
    assert err == 0 and np.array_equal(offs, o_offs) and np.array_equal(dst, o_dst) and np.array_equal(src, o_src)
    offs, dst, src, err = _run(np.full(777, 3, np.int32), 5)
    assert offs.tolist() == [0, 0, 0, 896, 896] and dst.tolist() == list(range(777))


def test_no_rows():
    offs, dst, src, err = _run(np.zeros(0, np.int32), 4, 256)
    assert err == 0 and offs.tolist() == [0, 0, 0, 0] and dst.size == 0 and np.all(src == -1)


def test_capacity_overflow_is_reported_and_places_nothing():
    ids = np.arange(4, dtype=np.int32)                 # 4 groups of one row need 512 padded rows
    offs, dst, src, err = _run(ids, 4, 256)
    assert err & 8
    assert offs.tolist() == [128, 256, 384, 512] and np.all(dst == -1) and np.all(src == -1)


def test_bad_expert_id_is_reported_and_skipped():
    ids = np.array([0, 5, 1, -2, 0, 1], np.int32)
    offs, dst, src, err = _run(ids, 3, 512)
    assert err & 8
    valid = np.where((ids >= 0) & (ids < 3))[0]
    s_offs, s_dst, s_src = o.token_group_pad(ids[valid], 3, 128, 512)
    assert np.array_equal(offs, s_offs)
    assert np.all(dst[[1, 3]] == -1) and np.array_equal(dst[valid], s_dst)
    live = s_src >= 0
    assert np.array_equal(src[live], valid[s_src[live]]) and np.all(src[~live] == -1)


def test_full_size_topk_dispatch_and_gather():
    """MoE 64E shape: 16384 tokens x top-8 = 131072 routed rows, d=7168."""
    T, E, k, d = 16384, 64, 8, 7168
    ids = synth.topk_expert_ids(T, E, k, 17)
    m_cap = mx.token_group_capacity(ids.size, E)
    offs, dst, src, err = _run(ids, E, m_cap)
    o_offs, o_dst, o_src = o.token_group_pad(ids, E, 128, m_cap)
    assert err == 0
    assert np.array_equal(offs, o_offs) and np.array_equal(dst, o_dst) and np.array_equal(src, o_src)
    x = synth.normal_bf16((T, d), 1.0, 23)
    xd = to_dev(x)
    err = mx.ErrorWord()
    xp = mx.gather_rows(xd, torch.as_tensor(src, device="cuda"), div=k, err=err)
    back = mx.gather_rows(xp, torch.as_tensor(dst, device="cuda"), div=1, err=err)
    torch.cuda.synchronize()
    err.check()
    rows = np.random.default_rng(5).choice(m_cap, 4096, replace=False)  # sampled padded rows
    ref = o.gather_rows(x, src[rows], div=k)
    assert np.array_equal(bits(xp)[rows], ref)
    assert not bits(xp)[src < 0].any()                               # pad and tail rows are zero
    assert np.array_equal(bits(back), x[np.arange(ids.size) // k])  # routed order restored


def test_gather_out_of_range_source_gives_zero_and_flag():
    x = to_dev(synth.normal_bf16((4, 16), 1.0, 1))
    err = mx.ErrorWord()
    y = mx.gather_rows(x, torch.tensor([0, 9, -1, 3], dtype=torch.int32, device="cuda"), err=err)
    torch.cuda.synchronize()
    assert err.value() & 8
    yb, xb = bits(y), bits(x)
    assert np.array_equal(yb[0], xb[0]) and np.array_equal(yb[3], xb[3])
    assert not yb[1].any() and not yb[2].any()
