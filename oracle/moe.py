"""The MoE steps either side of the grouped GEMM (oracle; test infrastructure).

"Low Precision RL", section "3. Unified MXFP8 (Blackwell)": MoE layers run
their own GEMM backend on routed tokens (the routed MoE runners), so each
expert's rows of the grouped GEMM are the tokens routed to it, in expert
order, quantised along K like any activation; between the gate+up and the
down projection of the expert MLP (SwiGLU in the Qwen3 MoE models the pages
train) the activation is formed and quantised again.  The pages describe
neither step; the readings here:

  gather + quantise:   A = quantize(X[token_index]) row by row -- exactly
                       the gathered BF16 rows, quantised.
  SwiGLU + requantise: H = [gate | up] (gate = H[:, :I], up = H[:, I:2I]),
                       y = BF16(silu(gate) * up), silu(g) = g / (1 + e^-g),
                       then quantize(y) row by row.

y is the plain definition: silu(g) * up evaluated in float64 (numpy's exp,
well below a float64 ulp of error at these sizes) and rounded once to
nearest-even BF16.  A GPU that evaluates y in float32 lands on the same BF16
value except where the exact value lies within its float32 error of a BF16
rounding boundary; bf16_tie_neighbour names those elements and the other
admissible BF16 value, so a test can accept either outcome there and demand
bit-exact codes everywhere else.
"""
from __future__ import annotations

import numpy as np

from . import quantize as Q
from .formats import round_to_bf16

F32 = np.float32

ROWWISE = {
    "1x128": Q.quantize_1x128,
    "mxfp8": Q.quantize_mxfp8,
    "1x128_pow2": Q.quantize_1x128_pow2,
}


def quantize_gathered(x: np.ndarray, token_index: np.ndarray, gran: str):
    """Codes and scales of the rows x[token_index] (in that order)."""
    rows = np.asarray(x, dtype=F32)[np.asarray(token_index, dtype=np.int64)]
    return ROWWISE[gran](rows)


def swiglu_exact(h: np.ndarray, inter: int) -> np.ndarray:
    """silu(gate) * up in float64 for H = [gate | up] of width 2 * inter,
    silu(g) = g / (1 + e^-g).  e^-g overflows float64 only for g < -709,
    where the quotient is -0 and the exact value rounds to -0 in BF16 too."""
    h = np.asarray(h, dtype=np.float64)
    assert h.shape[1] >= 2 * inter
    gate, up = h[:, :inter], h[:, inter:2 * inter]
    with np.errstate(over="ignore"):
        return gate / (1.0 + np.exp(-gate)) * up


def swiglu_bf16(h: np.ndarray, inter: int) -> np.ndarray:
    """y = BF16(silu(gate) * up): the float64 value rounded once to nearest-even
    BF16.  Returns float32 values that are exactly BF16."""
    return round_to_bf16(swiglu_exact(h, inter)).astype(F32)


def swiglu_quantize(h: np.ndarray, inter: int, gran: str):
    """Codes and scales of the SwiGLU activation, quantised row by row."""
    return ROWWISE[gran](swiglu_bf16(h, inter))


def bf16_tie_neighbour(y: np.ndarray, f32_ulps: float, abs_floor: float = 2.0 ** -146):
    """For exact values y (float64): (near, alt, tie).  near = BF16_RNE(y);
    tie marks the values that lie within f32_ulps float32 ulps of |y| (or
    within abs_floor, for results in the subnormal range) of the BF16 rounding
    boundary between near and its other neighbour alt; alt is that neighbour
    (equal to near where tie is False).  A float32 evaluation of y with at most
    that error rounds to near or, only where tie is True, to alt."""
    y = np.asarray(y, dtype=np.float64)
    near = round_to_bf16(y)
    _, e = np.frexp(np.abs(near))
    # BF16 spacing at near (2^-133 for subnormals and for 0), and the boundary on y's side of near
    q = np.where(near == 0, 2.0 ** -133, np.ldexp(1.0, np.maximum(e - 8, -133)))
    below = y < near
    # the step below a power of two is half as wide
    mag = np.abs(near)
    pow2 = (mag > 0) & (np.frexp(mag)[0] == 0.5) & (e - 9 >= -133)
    step_down_mag = np.where(pow2, q / 2, q)
    toward_zero = np.where(near >= 0, below, ~below)
    step = np.where(toward_zero, step_down_mag, q)
    alt = near + np.where(below, -step, step)
    boundary = (near + alt) / 2
    _, ey = np.frexp(np.abs(y))
    f32_ulp = np.ldexp(1.0, np.maximum(ey - 24, -149))
    tie = np.abs(y - boundary) <= np.maximum(f32_ulps * f32_ulp, abs_floor)
    tie &= np.isfinite(y) & (y != near)
    return near, np.where(tie, alt, near), tie


GROUP = {"1x128": 128, "mxfp8": 32, "1x128_pow2": 128}


def _scale_of_amax(amax, gran: str):
    """Step 1 for the granularity: float32 S, or the UE8M0 byte."""
    if gran == "1x128":
        return Q.fp32_scale(amax)
    return (Q.mxfp8_exponent(amax) + 127).astype(np.uint8)


def _scale_value(s, gran: str) -> np.float32:
    if gran == "1x128":
        return F32(s)
    return F32(np.ldexp(1.0, int(s) - 127))


def swiglu_check(codes, scales, h: np.ndarray, inter: int, gran: str, f32_ulps: float = 8.0):
    """Compare quantised SwiGLU output (codes, scales, e.g. from a GPU) with
    the definition.  Groups with no element near a BF16 rounding boundary
    (bf16_tie_neighbour) must match quantize(BF16(exact y)) bit for bit.  In
    the other groups the scale must be the scale of an amax that some
    admissible choice of the near-boundary elements gives, and every code must
    be the cast, under that scale, of the element's admissible BF16 value(s).
    Returns (mismatching code and scale entries, near-boundary elements,
    groups holding one)."""
    y = swiglu_exact(h, inter)
    near, alt, tie = bf16_tie_neighbour(y, f32_ulps)
    rq, rs = ROWWISE[gran](near.astype(F32))
    g = GROUP[gran]
    rows, cols = near.shape
    ng = -(-cols // g)
    pad = np.zeros((rows, ng * g), bool)
    pad[:, :cols] = tie
    tie_g = pad.reshape(rows, ng, g).any(axis=2)
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales)
    elem_in_tie_group = tie_g[:, np.arange(cols) // g]
    mism = int(((codes != rq) & ~elem_in_tie_group).sum()) + int(((scales != rs) & ~tie_g).sum())
    for r, gi in zip(*np.nonzero(tie_g)):
        c0, c1 = gi * g, min(cols, gi * g + g)
        yn, ya = near[r, c0:c1], alt[r, c0:c1]
        floor = np.max(np.minimum(np.abs(yn), np.abs(ya)))
        cands = np.unique(np.concatenate([np.abs(yn), np.abs(ya)]))
        cands = cands[cands >= floor]
        allowed = {np.asarray(_scale_of_amax(a, gran)).tobytes() for a in cands}
        sg = scales[r, gi]
        if np.asarray(sg).tobytes() not in allowed:
            mism += 1
            continue
        sv = _scale_value(sg, gran)
        cn = Q.cast_e4m3(yn.astype(F32), sv)
        ca = Q.cast_e4m3(ya.astype(F32), sv)
        got = codes[r, c0:c1]
        mism += int(((got != cn) & (got != ca)).sum())
    return mism, int(tie.sum()), int(tie_g.sum())
