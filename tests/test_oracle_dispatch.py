"""Pins of the token-group padding oracle (reading R12): a hand-derived
worked example, a brute-force restatement on small inputs, the layout
invariants, and the degenerate cases."""
import json
import os

import numpy as np
import pytest

from oracle import mx_oracle as o

HERE = os.path.dirname(os.path.abspath(__file__))


def _brute(expert_of, E, pad, m_cap):
    """Place rows by walking experts in order and rows in order (plain loops)."""
    offs, row_dst, row_src = [], [0] * len(expert_of), [-1] * m_cap
    pos = 0
    for e in range(E):
        n = 0
        for r, x in enumerate(expert_of):
            if x == e:
                row_dst[r] = pos + n
                row_src[pos + n] = r
                n += 1
        pos += -(-n // pad) * pad
        offs.append(pos)
    return offs, row_dst, row_src


def test_golden_small_example():
    g = json.load(open(os.path.join(HERE, "golden", "token_pad_small.json")))
    offs, dst, src = o.token_group_pad(g["expert_of"], g["E"], g["pad_multiple"], g["m_cap"])
    assert offs.tolist() == g["offs"]
    assert dst.tolist() == g["row_dst"]
    assert src.tolist() == g["row_src"]


@pytest.mark.parametrize("seed", range(6))
def test_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 9))
    R = int(rng.integers(0, 60))
    pad = int(rng.choice([1, 4, 8, 128]))
    ex = rng.integers(0, E, R).tolist()
    m_cap = -(-R // pad) * pad + E * pad + pad
    offs, dst, src = o.token_group_pad(ex, E, pad, m_cap)
    b_offs, b_dst, b_src = _brute(ex, E, pad, m_cap)
    assert offs.tolist() == b_offs and dst.tolist() == b_dst and src.tolist() == b_src


def test_layout_invariants_on_a_routed_batch():
    rng = np.random.default_rng(11)
    E, T, k = 16, 3000, 2
    ex = np.stack([rng.permutation(E)[:k] for _ in range(T)]).reshape(-1)   # top-2 routing
    m_cap = -(-ex.size // 128) * 128 + 128 * E
    offs, dst, src = o.token_group_pad(ex, E, 128, m_cap)
    assert np.all(offs % 128 == 0) and np.all(np.diff(offs) >= 0)
    counts = np.bincount(ex, minlength=E)
    assert np.array_equal(np.diff(np.concatenate([[0], offs])), -(-counts // 128) * 128)
    assert np.array_equal(src[dst], np.arange(ex.size))                   # inverse maps
    assert (src >= 0).sum() == ex.size
    starts = np.concatenate([[0], offs[:-1]])
    for e in range(E):                                                    # stable, contiguous, padded
        rows = src[starts[e]:offs[e]]
        live = rows[rows >= 0]
        assert np.all(ex[live] == e) and np.all(np.diff(live) > 0)
        assert np.all(rows[:counts[e]] >= 0) and np.all(rows[counts[e]:] == -1)
    assert np.all(src[offs[-1]:] == -1)                                   # tail


def test_degenerate_cases():
    offs, dst, src = o.token_group_pad([], 3, 128, 256)                   # no rows
    assert offs.tolist() == [0, 0, 0] and dst.size == 0 and np.all(src == -1)
    offs, dst, src = o.token_group_pad([1] * 128, 3, 128, 128)            # one full group, exact fit
    assert offs.tolist() == [0, 128, 128] and dst.tolist() == list(range(128))
    offs, _, _ = o.token_group_pad([0, 2], 3, 128, 256)                   # empty middle expert
    assert offs.tolist() == [128, 128, 256]
    with pytest.raises(ValueError):
        o.token_group_pad([0, 1, 2], 3, 128, 256)                         # capacity too small
    with pytest.raises(ValueError):
        o.token_group_pad([0, 3], 3, 128, 512)                            # expert id out of range


def test_gather_rows_tokens_and_zeros():
    x = np.arange(5 * 4, dtype=np.uint16).reshape(5, 4)                   # 5 tokens
    src = np.array([3, -1, 0, 9, -1])                                     # routed rows, topk 2
    y = o.gather_rows(x, src, div=2)
    assert y[0].tolist() == x[1].tolist() and y[2].tolist() == x[0].tolist()
    assert y[3].tolist() == x[4].tolist()
    assert not y[1].any() and not y[4].any()
