"""Plain CPU oracle for the MXFP8 training MLP (w13 GEMM -> SwiGLU with dual
MXFP8 quantization -> w2 GEMM, dense and grouped, forward and backward).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  It shares no code,
table or constant with the CUDA library in ``block_scaled_mlp_gb300`` and
never imports it.

Sources, by the pages' titles:

* "Add MXFP8 fused-MLP overrides in torchtitan" (pytorch/torchtitan PR 4257),
  Summary: the composite is "w13 GEMM -> fused SwiGLU + dual MXFP8
  quantization -> w2 GEMM", dense and grouped; w1 and w3 are packed into one
  fused w13 at forward time; grouped token rows are expert-major and padded
  to pad_multiple=128.  Numerics and tests: the fused forward is bitwise equal
  to "standalone-cast quantization" and the backward is within one e4m3 code;
  the kernel computes a correctly-rounded sigmoid.
* "TrainingWeightWrapperTensor base class ..." (pytorch/ao PR 3968) and
  "[mxfp8 training] unified MXFP8TrainingConfig ..." (pytorch/ao PR 3948),
  Autograd function changes: the ``wgrad_with_hp`` recipe keeps the weight
  gradient GEMM in high precision (bf16 operands); ``ScaleCalculationMode.RCEIL``
  names the scale mode.
* The MX block format itself (32-element blocks, E8M0 power-of-two shared
  scale, FP8 E4M3 elements) is the one of the OCP Microscaling Formats v1.0
  specification, which the pages name by "MXFP8" only.

Readings where the pages are silent:

R1  RCEIL: the block scale is 2^e with e the smallest integer such that
    amax <= 448 * 2^e, clamped to [-127, 127]; the E8M0 byte is e + 127.
    An all-zero block gets byte 0x00.  A block holding a NaN or an infinity
    gets scale 0xFF and every code 0x7F.
R2  Element code: v * 2^-e rounded to the E4M3 (fn) grid with
    round-to-nearest-even, saturated to +-448; the sign of zero is kept.
R3  Columnwise ("dual") quantization of X[R,C] is the rowwise quantization
    of X^T: codes [C,R], scales [C,R/32].
R4  SwiGLU forward ("standalone-cast" reading): sigma = RN_f32(1/(1+e^-g))
    correctly rounded; a = RN_bf16(RN_f32(g*sigma)); y = RN_bf16(RN_f32(a*u));
    y is then quantized.  h13 = [g | u] along the hidden axis.
R5  SwiGLU backward: du = RN_bf16(RN_f32(dy*a)); dg = RN_bf16 of the exact
    real dy*u*sigma(g)*(1+g*(1-sigma(g))), one rounding; non-finite g gives
    NaN; the sign of a zero result follows IEEE multiplication of the signs.
R6  GEMMs: C = deq(A) deq(B)^T, every product exact in float64 and summed
    in float64 (BLAS order: not exact, but its error is far below the 2e-3
    normwise bar), then RN_bf16 for the stored result.  Grouped forward/dgrad: rows of group
    e are [offs[e-1], offs[e]); rows past offs[E-1] (the tail) are zero.
    Grouped wgrad: dW[e] sums over group e's rows only; an empty group gives
    exact zeros.
R7  Scale layout "MMA": the 128-row x 4-scale-column tiled layout of the
    block-scaled tensor-core MMA (public PTX / cuBLAS documentation), padded
    with 0x00.
R12 Token-group padding ("[mxfp8] refactor model converter; use token group
    padding kernels in torchao": per-group padding done by kernels instead of
    host code; "Add MXFP8 fused-MLP overrides in torchtitan": the padded
    dispatcher, pad_multiple=128, inert pad and tail rows).  Routed row r has
    expert expert_of[r] in [0, E).  The padded layout places groups in expert
    order, the rows of a group in increasing r (a stable sort by expert),
    each group padded with zero rows to a multiple of pad_multiple; offs[e]
    is the cumulative padded end of group e; padded rows past offs[E-1] up
    to the buffer's capacity (the tail) are zero as well.  A routed row's
    activations are those of token r // topk.
R14 FLOOR scale mode (the pages name ScaleCalculationMode.RCEIL as one mode
    of several, defining none): the shared exponent of the OCP MX v1.0
    conversion, e = floor(log2(amax)) - 8 (8 = the exponent of E4M3's largest
    power of two), clamped to [-127, 127], byte e + 127; zero and non-finite
    blocks as in R1; elements as in R2, where saturation now binds (scaled
    values in (448, 512) become +-448).  Recipes "floor" and
    "floor_wgrad_hp" use it for every quantization of the MLP and linear.
R15 FP8 per-tensor ("tensorwise") grouped MM ("[mxfp8 training] unified
    MXFP8TrainingConfig and MXFP8TrainingTensor": FP8 GroupedMM is the
    non-MX FP8 recipe, its workflow temporarily removed there, arithmetic
    not given).  One fp32 scale per tensor (per expert for [E, ...] weight
    tensors): amax = max |x| (NaN propagates), s = RN_f32(448 /
    max(amax, 2^-40)) by IEEE fp32 division (the floor keeps an all-zero
    tensor finite); code = E4M3 of RN_f32(x * s), RNE and saturating as in
    R2.  Dequantized value code / s.  GEMMs as in R6 on the dequantized
    operands: M-grouped with one activation scale and one scale per expert
    weight, K-grouped (weight gradient) with one scale per operand.
R13 Per-linear MXFP8 path ("TrainingWeightWrapperTensor base class ...",
    linear override; "Add MXFP8 fused-MLP overrides in torchtitan": non-MLP
    linears keep the per-linear MXFP8 path): out = x w^T with both operands
    MX(R) along the contraction; dx = dout w with dout MX(R) and w MX(C);
    dw = dout^T x with both MX(C) along the tokens, or in bf16 under the
    wgrad_hp recipe; each GEMM rounded once to bf16.

Every function here that has a pin in ``tests/test_oracle_*.py`` says so.
"""
from __future__ import annotations

import math
from functools import lru_cache

import mpmath
import numpy as np

E4M3_MAX = 448.0
BLOCK = 32

# --------------------------------------------------------------------------
# bfloat16 / float32 helpers (exact decode, RNE encode)
# --------------------------------------------------------------------------


def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bfloat16 bit patterns (bf16 is the top half of an fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def round_to_f32(x) -> np.ndarray:
    """RN_f32 (numpy's float64->float32 cast is round-to-nearest-even with
    subnormals and overflow to infinity), returned as float64."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_to_bf16_bits(x) -> np.ndarray:
    """RN_bf16: round float64 values to the nearest bfloat16, ties to even.

    bfloat16: 8 significant bits, normal exponents -126..127, subnormal
    quantum 2^-133, overflow to infinity.  NaN -> 0x7FC0.
    Pinned against torch's float32->bfloat16 cast (tests/test_oracle_formats.py).
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint16)
    sign = np.signbit(x).astype(np.uint16) << 15
    a = np.abs(x)
    nan = np.isnan(x)
    inf = np.isinf(a)
    fin = ~nan & ~inf & (a > 0)
    if fin.any():
        af = a[fin]
        _, ex = np.frexp(af)            # af = m * 2^ex, m in [0.5, 1)
        unb = ex - 1                     # floor(log2(af))
        qe = np.maximum(unb, -126) - 7   # quantum exponent
        n = np.rint(np.ldexp(af, -qe))   # exact scaling, RNE
        val = np.ldexp(n, qe)
        over = val >= 2.0 ** 128
        # encode
        _, ex2 = np.frexp(val)
        unb2 = ex2 - 1
        sub = unb2 < -126
        with np.errstate(invalid="ignore", over="ignore"):
            mant_sub = np.where(sub, np.ldexp(val, 133), 0.0).astype(np.int64)
            mant_nrm = (np.ldexp(val, -unb2) - 1.0) * 128.0
        code = np.where(sub, mant_sub,
                        ((unb2 + 127).astype(np.int64) << 7) | mant_nrm.astype(np.int64))
        code = np.where(val == 0, 0, code)
        code = np.where(over, 0x7F80, code)
        out[fin] = code.astype(np.uint16)
    out[inf] = 0x7F80
    out = np.asarray(out | sign, dtype=np.uint16)
    out[nan] = 0x7FC0
    return out


# --------------------------------------------------------------------------
# E8M0 scale (RCEIL) and E4M3 codes
# --------------------------------------------------------------------------


def e8m0_rceil(amax) -> np.ndarray:
    """Reading R1.  Pinned exhaustively over every non-negative bf16 amax."""
    amax = np.asarray(amax, dtype=np.float64)
    out = np.full(amax.shape, 255, dtype=np.uint8)
    fin = np.isfinite(amax)
    a = amax[fin]
    with np.errstate(divide="ignore"):
        cand = np.where(a > 0, np.ceil(np.log2(a / E4M3_MAX)), -127.0)
    cand = np.clip(cand, -127, 127).astype(np.int64)
    # fix up so that the defining inequalities hold exactly
    for _ in range(4):
        up = (a > np.ldexp(E4M3_MAX, cand)) & (cand < 127)
        cand = cand + up
        down = (cand > -127) & (a <= np.ldexp(E4M3_MAX, cand - 1))
        cand = cand - down
    out[fin] = (cand + 127).astype(np.uint8)
    return out


def e8m0_floor(amax) -> np.ndarray:
    """Reading R14: e = floor(log2 amax) - 8, clamped; byte e + 127; zero
    amax -> 0x00, non-finite -> 0xFF.  Pinned exhaustively over every
    non-negative bf16 amax in tests/test_oracle_floor.py."""
    amax = np.asarray(amax, dtype=np.float64)
    out = np.full(amax.shape, 255, dtype=np.uint8)
    fin = np.isfinite(amax)
    a = amax[fin]
    _, ex = np.frexp(a)                       # a = m 2^ex, m in [0.5, 1): floor(log2 a) = ex - 1
    e = np.where(a > 0, ex - 1 - 8, -127)
    out[fin] = (np.clip(e, -127, 127) + 127).astype(np.uint8)
    return out


def e4m3_encode(v) -> np.ndarray:
    """Reading R2: RNE onto the E4M3fn grid (bias 7, subnormal quantum 2^-9,
    max 448), saturating to +-448, sign of zero kept, NaN -> 0x7F.
    Pinned exhaustively against exact rational rounding and against torch's
    float8_e4m3fn cast for in-range values."""
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros(v.shape, dtype=np.uint8)
    sign = (np.signbit(v).astype(np.uint8) << 7)
    a = np.abs(v)
    nan = np.isnan(v)
    pos = ~nan & (a > 0)
    if pos.any():
        ap = np.minimum(a[pos], 1e300)  # infinities saturate below
        _, ex = np.frexp(ap)
        unb = np.maximum(ex - 1, -6)
        qe = unb - 3
        n = np.rint(np.ldexp(ap, -qe))
        q = np.minimum(np.ldexp(n, qe), E4M3_MAX)
        _, ex2 = np.frexp(q)
        unb2 = ex2 - 1
        sub = unb2 < -6
        m_sub = np.ldexp(q, 9).astype(np.int64)
        m_nrm = ((np.ldexp(q, -unb2) - 1.0) * 8.0).astype(np.int64)
        code = np.where(sub, m_sub, ((unb2 + 7).astype(np.int64) << 3) | m_nrm)
        code = np.where(q == 0, 0, code)
        out[pos] = code.astype(np.uint8)
    out = np.asarray(out | sign, dtype=np.uint8)
    out[nan] = 0x7F
    return out


@lru_cache(maxsize=1)
def _e4m3_table() -> np.ndarray:
    t = np.empty(256, dtype=np.float64)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        ef = (c >> 3) & 0xF
        m = c & 0x7
        if ef == 0xF and m == 0x7:
            t[c] = np.nan
        elif ef == 0:
            t[c] = s * m * 2.0 ** -9
        else:
            t[c] = s * (1.0 + m / 8.0) * 2.0 ** (ef - 7)
    return t


def e4m3_decode(codes) -> np.ndarray:
    return _e4m3_table()[np.asarray(codes, dtype=np.uint8)]


# --------------------------------------------------------------------------
# MX quantization (rowwise / columnwise) and scale layouts
# --------------------------------------------------------------------------


SCALE_RCEIL = "rceil"
SCALE_FLOOR = "floor"


def quantize_rows(bits, scale: str = SCALE_RCEIL):
    """MX(R): 32-element blocks along the last axis (scale mode R1 or R14).

    bits: bf16 bit patterns [..., C] with C % 32 == 0.
    Returns (codes uint8 [..., C], scales uint8 [..., C/32]) in the linear
    scale layout.
    """
    bits = np.asarray(bits, dtype=np.uint16)
    C = bits.shape[-1]
    assert C % BLOCK == 0
    v = bf16_to_f64(bits).reshape(bits.shape[:-1] + (C // BLOCK, BLOCK))
    amax = np.max(np.abs(v), axis=-1)        # NaN propagates
    s = e8m0_floor(amax) if scale == SCALE_FLOOR else e8m0_rceil(amax)
    e = s.astype(np.int64) - 127
    scaled = np.ldexp(v, -e[..., None])      # exact power-of-two scaling
    codes = e4m3_encode(scaled)
    bad = s == 255
    codes[bad] = 0x7F
    return codes.reshape(bits.shape), s


def quantize_cols(bits, scale: str = SCALE_RCEIL):
    """MX(C) of X[R,C] = MX(R) of X^T (reading R3): codes [C,R], scales [C,R/32].
    Leading batch axes (experts) are kept."""
    bits = np.asarray(bits, dtype=np.uint16)
    return quantize_rows(np.swapaxes(bits, -1, -2), scale)


def dequantize(codes, scales) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    C = codes.shape[-1]
    v = e4m3_decode(codes).reshape(codes.shape[:-1] + (C // BLOCK, BLOCK))
    s = np.asarray(scales, dtype=np.int64)
    e = np.where(s == 255, 0, s - 127)
    out = np.ldexp(v, e[..., None])
    out[s == 255] = np.nan
    return out.reshape(codes.shape)


def mma_scale_bytes(rows: int, scale_cols: int) -> int:
    return ((rows + 127) // 128) * ((scale_cols + 3) // 4) * 512


def _mma_index(rows: int, scale_cols: int):
    r = np.arange(rows)[:, None]
    c = np.arange(scale_cols)[None, :]
    ct = (scale_cols + 3) // 4
    tile = (r // 128) * ct + c // 4
    return tile * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)


def scales_to_mma(s) -> np.ndarray:
    """Reading R7.  s: linear scales [R, Cs] (or [E, R, Cs]); returns the
    flat tiled layout (per expert, if batched), padding bytes 0x00."""
    s = np.asarray(s, dtype=np.uint8)
    if s.ndim == 3:
        return np.stack([scales_to_mma(si) for si in s])
    R, Cs = s.shape
    out = np.zeros(mma_scale_bytes(R, Cs), dtype=np.uint8)
    out[_mma_index(R, Cs)] = s
    return out


def scales_from_mma(flat, rows: int, scale_cols: int) -> np.ndarray:
    flat = np.asarray(flat, dtype=np.uint8)
    if flat.ndim == 2:
        return np.stack([scales_from_mma(f, rows, scale_cols) for f in flat])
    return flat[_mma_index(rows, scale_cols)]


# --------------------------------------------------------------------------
# Correctly rounded sigmoid and the SwiGLU forward/backward
# --------------------------------------------------------------------------

_MP_PREC = 240


def _mp_sigmoid(g: float):
    with mpmath.workprec(_MP_PREC):
        x = mpmath.mpf(g)
        return 1 / (1 + mpmath.exp(-x))


def _mp_round(x, f32: bool, prec: int = _MP_PREC) -> float:
    """Round an mpf to the nearest float32 (f32=True) or bfloat16 value, ties
    to even, deciding the direction in `prec`-bit precision."""
    with mpmath.workprec(prec):
        approx = float(x)
        if f32:
            c = np.float32(approx)
            lo = float(np.nextafter(c, np.float32(-np.inf)))
            hi = float(np.nextafter(c, np.float32(np.inf)))
            cands = [lo, float(c), hi]
        else:
            cb = int(round_to_bf16_bits(approx))
            def nb(b, d):
                # neighbour bf16 values through the bit pattern
                if b & 0x8000:
                    d = -d
                return (b + d) & 0xFFFF
            cands = [float(bf16_to_f64(np.uint16(nb(cb, -1)))),
                     float(bf16_to_f64(np.uint16(cb))),
                     float(bf16_to_f64(np.uint16(nb(cb, 1))))]
        cands = [c for c in cands if math.isfinite(c)]
        best = None
        for c in cands:
            dist = abs(x - mpmath.mpf(c))
            if best is None or dist < best[0]:
                best = (dist, c, [c])
            elif dist == best[0]:
                best[2].append(c)
        ties = best[2]
        if len(ties) == 1:
            return ties[0]
        # tie: pick the even significand
        for c in ties:
            if f32:
                b = int(np.float32(c).view(np.uint32))
            else:
                b = int(round_to_bf16_bits(c))
            if b & 1 == 0:
                return c
        return ties[0]


def sigmoid_rn_f32(g) -> np.ndarray:
    """Reading R4: RN_f32(1/(1+exp(-g))), correctly rounded.

    float64 evaluation (relative error far below 2^-45); values within
    2^-40 (relative) of an fp32 rounding midpoint are recomputed in 240-bit
    precision with mpmath.  Pinned against mpmath for every bf16 input.
    """
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        t = np.exp(-g)
        s = 1.0 / (1.0 + t)
    c = s.astype(np.float32)
    c64 = c.astype(np.float64)
    lo = np.nextafter(c, np.float32(-np.inf)).astype(np.float64)
    hi = np.nextafter(c, np.float32(np.inf)).astype(np.float64)
    with np.errstate(invalid="ignore"):
        dist = np.minimum(np.abs(s - (c64 + lo) / 2), np.abs(s - (c64 + hi) / 2))
        amb = np.isfinite(g) & (s > 0) & (dist <= np.abs(s) * 2.0 ** -40)
    out = c64.copy()
    for i in zip(*np.nonzero(amb)):
        out[i] = _mp_round(_mp_sigmoid(float(g[i])), f32=True)
    return out


@lru_cache(maxsize=1)
def _silu_table() -> np.ndarray:
    """a(g) = RN_bf16(RN_f32(g * sigmoid_rn_f32(g))) for all 65536 bf16 g."""
    gb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    g = bf16_to_f64(gb)
    sig = sigmoid_rn_f32(g)
    with np.errstate(invalid="ignore"):
        p = round_to_f32(g * sig)     # g*sig is exact in float64 (8 x 24 bits)
    return round_to_bf16_bits(p)


def silu_bf16(g_bits) -> np.ndarray:
    """Reading R4: the bf16 SiLU a(g) of bf16 inputs (bit patterns)."""
    return _silu_table()[np.asarray(g_bits, dtype=np.uint16)]


def swiglu_fwd(g_bits, u_bits) -> np.ndarray:
    """Reading R4: y = RN_bf16(RN_f32(a(g) * u)) as bf16 bits."""
    a = bf16_to_f64(silu_bf16(g_bits))
    u = bf16_to_f64(u_bits)
    with np.errstate(invalid="ignore"):
        return round_to_bf16_bits(round_to_f32(a * u))  # a*u exact in float64


def _mp_dsilu_factor(g: float, prec: int = _MP_PREC):
    """sigma(g) * (1 + g*(1 - sigma(g))) in `prec`-bit precision, with 1 - sigma
    formed as e^-g/(1+e^-g) so that no cancellation occurs for large g."""
    with mpmath.workprec(prec):
        x = mpmath.mpf(g)
        t = mpmath.exp(-x)
        s = 1 / (1 + t)
        oms = t / (1 + t)
        return s * (1 + x * oms)


def _dg_exact_bf16(dyu: float, g: float) -> int:
    """RN_bf16 of the exact dyu * f(g) (dyu = dy*u, an exact float64) for the
    few products the float64 evaluation cannot round with certainty.

    f(g) - 1 ~ g*e^-g for large g and f(g) - 1/2 ~ g/2 for tiny g, so the
    working precision grows with |g| until the exact value is resolved; for
    g > 1000 the deviation of f from 1 is below 2^-1400 and only decides
    exact ties of dyu, always away from zero (f > 1 for g > 1.28)."""
    if g > 1000.0:
        b = int(round_to_bf16_bits(dyu))
        lo = float(bf16_to_f64(_bf16_step(np.uint16(b), -1)))
        hi = float(bf16_to_f64(_bf16_step(np.uint16(b), +1)))
        v = float(bf16_to_f64(np.uint16(b)))
        for w in (lo, hi):
            if dyu == (v + w) / 2:           # exact tie of dyu: f > 1 breaks it
                return int(round_to_bf16_bits(max(v, w, key=abs)))
        return b
    prec = _MP_PREC + 160 + int(2 * max(0.0, 1.45 * g))
    with mpmath.workprec(prec):
        exact = mpmath.mpf(dyu) * _mp_dsilu_factor(g, prec)
        return int(round_to_bf16_bits(_mp_round(exact, f32=False, prec=prec)))


def _dsilu_factor_f64(g):
    """float64 evaluation of f(g) = sigma*(1+g*(1-sigma)) and a bound on its
    relative error (see swiglu_bwd)."""
    g = np.asarray(g, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        t = np.exp(-g)
        s = 1.0 / (1.0 + t)
        oms = t * s                       # 1 - sigma without cancellation
        go = g * oms
        inner = 1.0 + go
        f = s * inner
        rel = 2.0 ** -44 * (1.0 + np.abs(go) / np.abs(inner))
    deep = g < -700.0                     # sigma underflows: f is a tiny negative
    f = np.where(deep, -0.0, f)
    rel = np.where(deep, 0.0, rel)
    return f, rel


def swiglu_bwd(dy_bits, g_bits, u_bits):
    """Reading R5.  Returns (dg_bits, du_bits).

    dg is RN_bf16 of the exact dy*u*f(g): dy*u is exact in float64; f(g) is
    evaluated in float64 with a relative error bound; products whose
    float64 value lies within that bound of a bf16 rounding midpoint are
    recomputed in 240-bit precision.  Pinned against mpmath and against
    central differences of silu(g)*u (tests/test_oracle_swiglu.py).
    """
    dy_bits = np.asarray(dy_bits, dtype=np.uint16)
    g_bits = np.asarray(g_bits, dtype=np.uint16)
    u_bits = np.asarray(u_bits, dtype=np.uint16)
    dy = bf16_to_f64(dy_bits)
    g = bf16_to_f64(g_bits)
    u = bf16_to_f64(u_bits)
    a = bf16_to_f64(silu_bf16(g_bits))
    with np.errstate(invalid="ignore", over="ignore"):
        du_bits = round_to_bf16_bits(round_to_f32(dy * a))
        dyu = dy * u                      # exact (8 x 8 bits)
        f, rel = _dsilu_factor_f64(g)
        p = dyu * f
    dg_bits = round_to_bf16_bits(p)
    # ambiguity: distance from p to the nearest bf16 rounding midpoint
    lo_b = _bf16_step(dg_bits, -1)
    hi_b = _bf16_step(dg_bits, +1)
    c = bf16_to_f64(dg_bits)
    with np.errstate(invalid="ignore"):
        dist = np.minimum(np.abs(p - (c + bf16_to_f64(lo_b)) / 2),
                          np.abs(p - (c + bf16_to_f64(hi_b)) / 2))
        amb = np.isfinite(p) & (p != 0) & (dist <= np.abs(p) * (rel + 2.0 ** -50))
    for i in zip(*np.nonzero(amb)):
        dg_bits[i] = _dg_exact_bf16(float(dyu[i]), float(g[i]))
    dg_bits[~np.isfinite(g)] = 0x7FC0
    return dg_bits, du_bits


def _bf16_step(bits, d):
    """Neighbouring bf16 magnitude (towards +inf in magnitude for d=+1)."""
    b = np.asarray(bits, dtype=np.int64)
    mag = (b & 0x7FFF) + d
    mag = np.clip(mag, 0, 0x7F7F)
    return ((b & 0x8000) | mag).astype(np.uint16)


def split_h13(h13_bits):
    """h13 = [g | u] along the last axis (w13 = [w1; w3])."""
    h13_bits = np.asarray(h13_bits, dtype=np.uint16)
    h = h13_bits.shape[-1] // 2
    return h13_bits[..., :h], h13_bits[..., h:]


# --------------------------------------------------------------------------
# GEMMs (exact accumulation)
# --------------------------------------------------------------------------


def mx_mm(aq, as_, bq, bs) -> np.ndarray:
    """Reading R6: C[M,N] = deq(A)[M,K] . deq(B)[N,K]^T in float64 (products of
    E4M3 codes and powers of two are exact; float64 accumulation).  Linear
    scale layout.  Pinned against a pure-Python triple loop."""
    A = dequantize(aq, as_)
    B = dequantize(bq, bs)
    return A @ B.T


def bf16_mm(a_bits, b_bits) -> np.ndarray:
    """C = A . B^T from bf16 operands, float64 accumulation."""
    return bf16_to_f64(a_bits) @ bf16_to_f64(b_bits).T


def group_bounds(offs):
    offs = [int(o) for o in np.asarray(offs).reshape(-1)]
    out, start = [], 0
    for end in offs:
        out.append((start, end))
        start = end
    return out


def mx_grouped_mm_m(aq, as_, bq, bs, offs) -> np.ndarray:
    """M-grouped: A [M_total,K]; B [E,N,K]; rows of group e use B[e]; tail rows 0."""
    A = dequantize(aq, as_)
    M = A.shape[0]
    N = bq.shape[1]
    C = np.zeros((M, N), dtype=np.float64)
    for e, (s, t) in enumerate(group_bounds(offs)):
        if t > s:
            C[s:t] = A[s:t] @ dequantize(bq[e], bs[e]).T
    return C


def mx_grouped_mm_k(aq, as_, bq, bs, offs) -> np.ndarray:
    """K-grouped (weight gradient): A [N, M_total], B [K, M_total] (columnwise
    copies, contraction along tokens); C[e] = A[:, group e] . B[:, group e]^T;
    an empty group gives exact zeros."""
    A = dequantize(aq, as_)
    B = dequantize(bq, bs)
    offs = np.asarray(offs)
    C = np.zeros((len(offs), A.shape[0], B.shape[0]), dtype=np.float64)
    for e, (s, t) in enumerate(group_bounds(offs)):
        if t > s:
            C[e] = A[:, s:t] @ B[:, s:t].T
    return C


# --------------------------------------------------------------------------
# FP8 per-tensor scaling and its grouped GEMMs (reading R15)
# --------------------------------------------------------------------------

FP8_AMAX_FLOOR = 2.0 ** -40


def fp8_tensor_amax(bits, batch_axes: int = 0) -> np.ndarray:
    """max |x| over each tensor: over everything (batch_axes=0) or over all
    but the leading batch axis (batch_axes=1, one amax per expert).  Exact
    (bf16 values); NaN propagates.  Returned as float32."""
    v = np.abs(bf16_to_f64(bits))
    if batch_axes:
        return v.reshape(v.shape[0], -1).max(axis=1).astype(np.float32)
    return np.float32(v.max())


def fp8_tensor_scale(amax) -> np.ndarray:
    """Reading R15: s = RN_f32(448 / max(amax, 2^-40)), IEEE fp32 division
    (numpy float32 arithmetic is correctly rounded).  Pinned on hand-worked
    values (tests/golden/fp8_tensorwise.json)."""
    a = np.maximum(np.asarray(amax, dtype=np.float32), np.float32(FP8_AMAX_FLOOR))
    with np.errstate(invalid="ignore", divide="ignore"):
        return (np.float32(E4M3_MAX) / a).astype(np.float32)


def fp8_quantize_tensor(bits, batch_axes: int = 0):
    """Reading R15: codes of RN_f32(x * s), s from the tensor's (or each
    expert's) amax.  Returns (codes uint8, s float32 scalar or [E], amax)."""
    bits = np.asarray(bits, dtype=np.uint16)
    amax = fp8_tensor_amax(bits, batch_axes)
    s = fp8_tensor_scale(amax)
    x = bf16_to_f64(bits).astype(np.float32)             # exact
    sb = s.reshape((-1,) + (1,) * (bits.ndim - 1)) if batch_axes else s
    with np.errstate(invalid="ignore", over="ignore"):
        prod = (x * sb).astype(np.float32)               # one fp32 rounding
    return e4m3_encode(prod.astype(np.float64)), s, amax


def fp8_dequantize(codes, s) -> np.ndarray:
    """code / s in float64 (s per tensor, or per leading index when s has one
    entry per row of the leading axis)."""
    v = e4m3_decode(codes)
    s = np.asarray(s, dtype=np.float64)
    if s.ndim == 1:
        s = s.reshape((-1,) + (1,) * (v.ndim - 1))
    return v / s


def fp8_grouped_mm_m(aq, sa, bq, sb, offs) -> np.ndarray:
    """M-grouped: A [M_total, K] with one scale; B [E, N, K] with one scale per
    expert; rows of group e use B[e]; tail rows are zero (as R6)."""
    A = fp8_dequantize(aq, sa)
    B = fp8_dequantize(bq, sb)
    C = np.zeros((A.shape[0], B.shape[1]), dtype=np.float64)
    for e, (s, t) in enumerate(group_bounds(offs)):
        if t > s:
            C[s:t] = A[s:t] @ B[e].T
    return C


def fp8_grouped_mm_k(aq, sa, bq, sb, offs) -> np.ndarray:
    """K-grouped (weight gradient): A [N, M_total], B [K, M_total], one scale
    each; C[e] = A[:, group e] . B[:, group e]^T; an empty group is zero."""
    A = fp8_dequantize(aq, sa)
    B = fp8_dequantize(bq, sb)
    offs = np.asarray(offs)
    C = np.zeros((len(offs), A.shape[0], B.shape[0]), dtype=np.float64)
    for e, (s, t) in enumerate(group_bounds(offs)):
        if t > s:
            C[e] = A[:, s:t] @ B[:, s:t].T
    return C


def bf16_grouped_mm_k(a_bits, b_bits, offs) -> np.ndarray:
    """bf16 weight gradient, K-grouped: a [N, M_total], b [K, M_total]."""
    A = bf16_to_f64(a_bits)
    B = bf16_to_f64(b_bits)
    offs = np.asarray(offs)
    C = np.zeros((len(offs), A.shape[0], B.shape[0]), dtype=np.float64)
    for e, (s, t) in enumerate(group_bounds(offs)):
        if t > s:
            C[e] = A[:, s:t] @ B[:, s:t].T
    return C


# --------------------------------------------------------------------------
# Full MLP, forward and backward
# --------------------------------------------------------------------------

RECIPE_RCEIL = "rceil"
RECIPE_RCEIL_WGRAD_HP = "wgrad_hp"
RECIPE_FLOOR = "floor"
RECIPE_FLOOR_WGRAD_HP = "floor_wgrad_hp"


def recipe_hp(recipe) -> bool:
    """Weight-gradient GEMMs in bf16 (wgrad_with_hp)."""
    return recipe in (RECIPE_RCEIL_WGRAD_HP, RECIPE_FLOOR_WGRAD_HP)


def recipe_scale(recipe) -> str:
    return SCALE_FLOOR if recipe in (RECIPE_FLOOR, RECIPE_FLOOR_WGRAD_HP) else SCALE_RCEIL


def mlp_fwd(x, w1, w3, w2, offs=None, recipe=RECIPE_RCEIL):
    """Forward of the MXFP8 SwiGLU MLP, every intermediate returned.

    Dense: x [M,d], w1/w3 [h,d], w2 [d,h].  Grouped: w* carry a leading
    expert axis and ``offs`` holds cumulative group ends.
    Steps: quantize x (MX(R) along d); pack w13 = [w1; w3] and quantize along
    d; h13 = RN_bf16(x . w13^T); y = SwiGLU(h13) quantized MX(R) along h and
    (default recipe) MX(C) along tokens; w2 quantized along h;
    out = RN_bf16(y . w2^T).
    """
    x = np.asarray(x, dtype=np.uint16)
    grouped = offs is not None
    sc = recipe_scale(recipe)
    w13 = np.concatenate([w1, w3], axis=-2)          # [.., 2h, d]
    xq, xs = quantize_rows(x, sc)
    w13q, w13s = quantize_rows(w13, sc)
    w2q, w2s = quantize_rows(w2, sc)
    if grouped:
        h13_f = mx_grouped_mm_m(xq, xs, w13q, w13s, offs)
    else:
        h13_f = mx_mm(xq, xs, w13q, w13s)
    h13 = round_to_bf16_bits(h13_f)
    g, u = split_h13(h13)
    y = swiglu_fwd(g, u)
    yq, ys = quantize_rows(y, sc)
    if grouped:
        out_f = mx_grouped_mm_m(yq, ys, w2q, w2s, offs)
    else:
        out_f = mx_mm(yq, ys, w2q, w2s)
    out = round_to_bf16_bits(out_f)
    res = dict(xq=xq, xs=xs, w13q=w13q, w13s=w13s, h13_f=h13_f, h13=h13, y=y,
               yq=yq, ys=ys, w2q=w2q, w2s=w2s, out_f=out_f, out=out)
    if not recipe_hp(recipe):
        res["yq_c"], res["ys_c"] = quantize_cols(y, sc)
        res["xq_c"], res["xs_c"] = quantize_cols(x, sc)
    return res


def mlp_bwd(x, w1, w3, w2, dout, offs=None, recipe=RECIPE_RCEIL, fwd=None):
    """Backward of the MXFP8 SwiGLU MLP.

    dy = RN_bf16(dout . w2)            (MX(R) dout, MX(C) w2 along d)
    dW2 = RN_bf16(dout^T . y)          (MX(C) dout and y along tokens; HP: bf16)
    dh13 = [dg | du] = SwiGLU'(dy, h13) quantized MX(R) along 2h, MX(C) along tokens
    dx = RN_bf16(dh13 . w13)           (MX(C) w13 along 2h)
    dW13 = RN_bf16(dh13^T . x)         (MX(C) dh13 and x along tokens; HP: bf16)
    """
    if fwd is None:
        fwd = mlp_fwd(x, w1, w3, w2, offs, recipe)
    grouped = offs is not None
    x = np.asarray(x, dtype=np.uint16)
    dout = np.asarray(dout, dtype=np.uint16)
    w13 = np.concatenate([w1, w3], axis=-2)
    h = np.asarray(w1).shape[-2]
    sc = recipe_scale(recipe)
    dq, ds = quantize_rows(dout, sc)
    w2q_c, w2s_c = quantize_cols(w2, sc)             # [.., h, d]
    w13q_c, w13s_c = quantize_cols(w13, sc)          # [.., d, 2h]
    if grouped:
        dy_f = mx_grouped_mm_m(dq, ds, w2q_c, w2s_c, offs)
    else:
        dy_f = mx_mm(dq, ds, w2q_c, w2s_c)
    dy = round_to_bf16_bits(dy_f)
    g, u = split_h13(fwd["h13"])
    dg, du = swiglu_bwd(dy, g, u)
    dh13 = np.concatenate([dg, du], axis=-1)
    dhq, dhs = quantize_rows(dh13, sc)
    if grouped:
        dx_f = mx_grouped_mm_m(dhq, dhs, w13q_c, w13s_c, offs)
    else:
        dx_f = mx_mm(dhq, dhs, w13q_c, w13s_c)
    dx = round_to_bf16_bits(dx_f)
    res = dict(dq=dq, ds=ds, w2q_c=w2q_c, w2s_c=w2s_c, w13q_c=w13q_c, w13s_c=w13s_c,
               dy_f=dy_f, dy=dy, dg=dg, du=du, dh13=dh13, dhq=dhq, dhs=dhs,
               dx_f=dx_f, dx=dx)
    go = offs if grouped else np.array([x.shape[0]], dtype=np.int32)
    if not recipe_hp(recipe):
        dq_c, ds_c = quantize_cols(dout, sc)         # [d, M]
        dhq_c, dhs_c = quantize_cols(dh13, sc)       # [2h, M]
        dw2_f = mx_grouped_mm_k(dq_c, ds_c, fwd["yq_c"], fwd["ys_c"], go)
        dw13_f = mx_grouped_mm_k(dhq_c, dhs_c, fwd["xq_c"], fwd["xs_c"], go)
        res.update(dq_c=dq_c, ds_c=ds_c, dhq_c=dhq_c, dhs_c=dhs_c)
    else:
        dw2_f = bf16_grouped_mm_k(dout.T, fwd["y"].T, go)
        dw13_f = bf16_grouped_mm_k(dh13.T, x.T, go)
    if not grouped:
        dw2_f = dw2_f[0]
        dw13_f = dw13_f[0]
    dw2 = round_to_bf16_bits(dw2_f)
    dw13 = round_to_bf16_bits(dw13_f)
    res.update(dw2_f=dw2_f, dw2=dw2, dw13_f=dw13_f, dw13=dw13,
               dw1=dw13[..., :h, :], dw3=dw13[..., h:, :])
    return res


# --------------------------------------------------------------------------
# Comparison helpers used by the tests
# --------------------------------------------------------------------------


def normwise_rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(got - ref)
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return float(num / den)


def e4m3_code_distance(c1, c2) -> np.ndarray:
    """Distance between two E4M3 codes counted in representable steps
    (crossing zero counts +0/-0 as one point)."""
    def ordinal(c):
        c = np.asarray(c, dtype=np.int64)
        mag = c & 0x7F
        return np.where(c & 0x80, -mag, mag)
    return np.abs(ordinal(c1) - ordinal(c2))


# --------------------------------------------------------------------------
# MXFP8 linear (reading R13)
# --------------------------------------------------------------------------


def linear_fwd(x, w, rounded: bool = True, recipe=RECIPE_RCEIL):
    """out = RN_bf16(x . w^T) with x [M,K] and w [N,K] both quantized MX(R)
    along K (the per-linear MXFP8 path, reading R13); rounded=False returns
    the exact float64 product before the bf16 rounding.  Pinned in
    tests/test_oracle_linear.py."""
    xq, xs = quantize_rows(np.asarray(x, dtype=np.uint16), recipe_scale(recipe))
    wq, ws = quantize_rows(np.asarray(w, dtype=np.uint16), recipe_scale(recipe))
    out = mx_mm(xq, xs, wq, ws)
    return round_to_bf16_bits(out) if rounded else out


def linear_bwd(x, w, dout, recipe=RECIPE_RCEIL, rounded: bool = True):
    """Gradients of out = x . w^T (reading R13).

    dx = RN_bf16(dout . w): dout MX(R) along N, w MX(C) along N.
    dw = RN_bf16(dout^T . x): default recipe dout and x MX(C) along M;
    wgrad_hp recipe bf16 operands, float64 accumulation.
    Returns (dx, dw) as bf16 bits.  Pinned in tests/test_oracle_linear.py."""
    x = np.asarray(x, dtype=np.uint16)
    w = np.asarray(w, dtype=np.uint16)
    dout = np.asarray(dout, dtype=np.uint16)
    sc = recipe_scale(recipe)
    dq, ds = quantize_rows(dout, sc)
    wq_c, ws_c = quantize_cols(w, sc)                    # [K, N], blocks along N
    dx = mx_mm(dq, ds, wq_c, ws_c)
    if recipe_hp(recipe):
        dw = bf16_mm(dout.T, x.T)
    else:
        dq_c, ds_c = quantize_cols(dout, sc)             # [N, M], blocks along M
        xq_c, xs_c = quantize_cols(x, sc)                # [K, M]
        dw = mx_mm(dq_c, ds_c, xq_c, xs_c)
    if rounded:
        return round_to_bf16_bits(dx), round_to_bf16_bits(dw)
    return dx, dw


# --------------------------------------------------------------------------
# Token-group padding (reading R12)
# --------------------------------------------------------------------------


def token_group_pad(expert_of, E: int, pad_multiple: int = 128, m_cap: int | None = None):
    """Padded expert-major layout of routed rows (R12).

    Returns (offs, row_dst, row_src): offs[e] the cumulative padded end of
    group e (int32 [E]); row_dst[r] the padded row of routed row r (int32
    [R]); row_src[i] the routed row held by padded row i, or -1 for padding
    and tail rows (int32 [m_cap], m_cap defaulting to offs[-1]).  Pinned in
    tests/test_oracle_dispatch.py."""
    expert_of = np.asarray(expert_of, dtype=np.int64).reshape(-1)
    R = expert_of.size
    if R and (expert_of.min() < 0 or expert_of.max() >= E):
        raise ValueError("expert id out of range")
    counts = np.bincount(expert_of, minlength=E)[:E]
    padded = (counts + pad_multiple - 1) // pad_multiple * pad_multiple
    ends = np.cumsum(padded)
    starts = ends - padded
    if m_cap is None:
        m_cap = int(ends[-1]) if E else 0
    if E and ends[-1] > m_cap:
        raise ValueError("padded layout exceeds the capacity")
    order = np.argsort(expert_of, kind="stable")        # expert-major, r increasing within a group
    row_dst = np.empty(R, dtype=np.int64)
    rank = np.arange(R) - np.repeat(np.cumsum(counts) - counts, counts)  # position within the group
    row_dst[order] = starts[expert_of[order]] + rank
    row_src = np.full(m_cap, -1, dtype=np.int64)
    row_src[row_dst] = np.arange(R)
    return ends.astype(np.int32), row_dst.astype(np.int32), row_src.astype(np.int32)


def gather_rows(x_bits, src, div: int = 1):
    """y[i] = x[src[i] // div] for src[i] >= 0, zero rows otherwise (bf16 bit
    patterns, copied exactly).  Pinned in tests/test_oracle_dispatch.py."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    src = np.asarray(src, dtype=np.int64)
    y = np.zeros((src.size, x_bits.shape[1]), dtype=np.uint16)
    live = src >= 0
    y[live] = x_bits[src[live] // div]
    return y
