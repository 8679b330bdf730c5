"""Seeded synthetic inputs for the MXFP8 training MLP.

This module only draws random data and lays it out; it holds none of the
quantization, activation or GEMM arithmetic.  Both the CUDA path (through the
tests and the bench) and the CPU oracle receive the arrays it returns, so the
two sides always see identical bits.

Every tensor is returned as a numpy ``uint16`` array of bfloat16 bit patterns
(or ``int32`` for group offsets).  Sampling happens in float32 on the host and
is rounded to bfloat16 by ``torch.Tensor.to(torch.bfloat16)``.

Workload recipes (shapes and distributions of the MXFP8 fused-MLP workloads
the torchtitan "Add MXFP8 fused-MLP overrides" page describes, Summary and
Usage sections; the sizes are those of a Llama-3-8B FFN and two routed-expert
MoE layers):

* dense MLP: x ~ N(0,1) [M,d]; w1, w3 ~ N(0,0.02) [h,d]; w2 ~ N(0,0.02) [d,h];
  upstream gradient ~ N(0,1) [M,d].
* quantize sweep: N(0,1) with 1% of elements scaled x100, 2% of 32x32 tiles
  all zero, 1% of 1x32 row blocks "pinned" at U(-1,1)*448*2^k with one
  element exactly +-448*2^k, k ~ U{-20..20}.
* routed experts: expert-major token rows, each group padded with zero rows
  to a multiple of ``pad_multiple`` (128); group sizes from a Zipf(1.1)
  multinomial (one expert forced empty) or a Dirichlet(0.3) multinomial (four
  experts forced empty), then the expert order is shuffled.
"""
from __future__ import annotations

import numpy as np
import torch

__all__ = [
    "bf16_from_f32",
    "normal_bf16",
    "quant_sweep_tensor",
    "dense_mlp_inputs",
    "zipf_group_counts",
    "dirichlet_group_counts",
    "pad_counts",
    "offsets_from_counts",
    "grouped_mlp_inputs",
    "WORKLOADS",
]


def bf16_from_f32(a: np.ndarray) -> np.ndarray:
    """float32 array -> bfloat16 bit patterns (uint16), RNE via torch."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, std: float, seed: int) -> np.ndarray:
    """N(0, std^2) samples as bfloat16 bits."""
    t = torch.randn(tuple(shape), generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def quant_sweep_tensor(rows: int, cols: int, seed: int) -> np.ndarray:
    """The quantize-sweep recipe (see module docstring) for a [rows, cols] tensor.

    rows and cols must be multiples of 32.
    """
    assert rows % 32 == 0 and cols % 32 == 0
    g = _gen(seed)
    x = torch.randn((rows, cols), generator=g, dtype=torch.float32)
    # 1% outliers x100
    out_mask = torch.rand((rows, cols), generator=g) < 0.01
    x[out_mask] *= 100.0
    # 2% of 32x32 tiles all zero
    tr, tc = rows // 32, cols // 32
    zt = torch.rand((tr, tc), generator=g) < 0.02
    zmask = zt.repeat_interleave(32, 0).repeat_interleave(32, 1)
    x[zmask] = 0.0
    # 1% of 1x32 row blocks pinned at +-448*2^k
    nb = cols // 32
    pin = (torch.rand((rows, nb), generator=g) < 0.01) & ~zmask[:, ::32]
    idx = pin.nonzero()
    if idx.numel():
        n = idx.shape[0]
        k = torch.randint(-20, 21, (n,), generator=g).to(torch.float32)
        mag = 448.0 * torch.pow(2.0, k)
        vals = (torch.rand((n, 32), generator=g) * 2.0 - 1.0) * mag[:, None]
        which = torch.randint(0, 32, (n,), generator=g)
        sgn = torch.where(torch.rand((n,), generator=g) < 0.5, -1.0, 1.0)
        vals[torch.arange(n), which] = sgn * mag
        xv = x.view(rows, nb, 32)
        xv[idx[:, 0], idx[:, 1], :] = vals
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def dense_mlp_inputs(M: int, d: int, h: int, seed: int) -> dict:
    """x [M,d], w1/w3 [h,d], w2 [d,h], dout [M,d] as bfloat16 bits."""
    return {
        "x": normal_bf16((M, d), 1.0, seed * 1000 + 1),
        "w1": normal_bf16((h, d), 0.02, seed * 1000 + 2),
        "w3": normal_bf16((h, d), 0.02, seed * 1000 + 3),
        "w2": normal_bf16((d, h), 0.02, seed * 1000 + 4),
        "dout": normal_bf16((M, d), 1.0, seed * 1000 + 5),
    }


def zipf_group_counts(E: int, tokens: int, s: float, seed: int, n_empty: int = 1) -> np.ndarray:
    """Per-expert token counts: multinomial(tokens, p ~ rank^-s) over E-n_empty
    experts, the last n_empty experts forced to zero, then the order shuffled."""
    rng = np.random.default_rng(seed)
    live = E - n_empty
    p = np.arange(1, live + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    c = np.zeros(E, dtype=np.int64)
    c[:live] = rng.multinomial(tokens, p)
    return c[rng.permutation(E)]


def dirichlet_group_counts(E: int, rows: int, alpha: float, seed: int, n_empty: int = 4) -> np.ndarray:
    """Per-expert row counts: multinomial(rows, Dirichlet(alpha)) over E-n_empty
    experts, n_empty experts forced to zero, then the order shuffled."""
    rng = np.random.default_rng(seed)
    live = E - n_empty
    p = rng.dirichlet(np.full(live, alpha))
    c = np.zeros(E, dtype=np.int64)
    c[:live] = rng.multinomial(rows, p)
    return c[rng.permutation(E)]


def routed_expert_ids(counts: np.ndarray, seed: int) -> np.ndarray:
    """Expert id of every routed row (int32): counts[e] rows of expert e, in a
    seeded random order (the routing decisions of a batch, before dispatch)."""
    rng = np.random.default_rng(seed)
    ids = np.repeat(np.arange(len(counts), dtype=np.int32), np.asarray(counts, dtype=np.int64))
    return ids[rng.permutation(ids.size)]


def topk_expert_ids(tokens: int, E: int, k: int, seed: int) -> np.ndarray:
    """Top-k routing: k distinct experts per token, flattened token-major
    (routed row r belongs to token r // k)."""
    rng = np.random.default_rng(seed)
    keys = rng.random((tokens, E))
    return np.argsort(keys, axis=1)[:, :k].astype(np.int32).reshape(-1)


def pad_counts(counts: np.ndarray, pad_multiple: int = 128) -> np.ndarray:
    return ((np.asarray(counts) + pad_multiple - 1) // pad_multiple) * pad_multiple


def offsets_from_counts(padded_counts: np.ndarray) -> np.ndarray:
    """Cumulative group ends (int32), the torch grouped_mm convention."""
    return np.cumsum(np.asarray(padded_counts, dtype=np.int64)).astype(np.int32)


def grouped_mlp_inputs(counts: np.ndarray, d: int, h: int, seed: int,
                       pad_multiple: int = 128, tail_rows: int = 0) -> dict:
    """Expert-major routed rows with zero padding rows.

    Returns x [M_total,d], w1/w3 [E,h,d], w2 [E,d,h], dout [M_total,d], offs
    [E] int32, the real counts and a boolean row mask of real rows.  Padding
    rows (and ``tail_rows`` extra rows after the last group) are zero in x and
    dout.
    """
    counts = np.asarray(counts, dtype=np.int64)
    E = counts.shape[0]
    pc = pad_counts(counts, pad_multiple)
    offs = offsets_from_counts(pc)
    M_total = int(offs[-1]) + int(tail_rows)
    real = np.zeros(M_total, dtype=bool)
    start = 0
    for e in range(E):
        real[start:start + counts[e]] = True
        start += int(pc[e])
    x = normal_bf16((M_total, d), 1.0, seed * 1000 + 1)
    dout = normal_bf16((M_total, d), 1.0, seed * 1000 + 5)
    x[~real] = 0
    dout[~real] = 0
    return {
        "x": x,
        "w1": normal_bf16((E, h, d), 0.02, seed * 1000 + 2),
        "w3": normal_bf16((E, h, d), 0.02, seed * 1000 + 3),
        "w2": normal_bf16((E, d, h), 0.02, seed * 1000 + 4),
        "dout": dout,
        "offs": offs,
        "counts": counts,
        "real_rows": real,
    }


# Named workloads with their sizes (used by the tests and the bench).
WORKLOADS = {
    "tiny_dense": dict(kind="dense", M=256, d=256, h=512, seed=0),
    "llama3_8b_ffn": dict(kind="dense", M=8192, d=4096, h=14336, seed=1, recipe="wgrad_hp"),
    "moe_16e": dict(kind="grouped", E=16, d=5120, h=8192, tokens=32768, seed=2,
                    counts="zipf", s=1.1, n_empty=1, topk=1),
    "moe_64e": dict(kind="grouped", E=64, d=7168, h=2048, tokens=131072, seed=3,
                    counts="dirichlet", alpha=0.3, n_empty=4, topk=8),
}
