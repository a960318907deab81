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

A quantised code is an integer decided by floating point, so the oracle
takes that decision in the precision the GPU computes y in: float32, by the
fixed sequence of exp_f32 / silu_f32 below (each operation one IEEE float32
rounding, no fused multiply-add), then one round-to-nearest-even to BF16.
The tests pin that sequence to float64 mathematics (a few float32 ulps).
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


# ---------------------------------------------------------------- e^x in float32
# Cody and Waite's reduction ("Software Manual for the Elementary Functions",
# 1980): x = n ln2 + r with n = rint(x / ln2) and ln2 split in two parts
# (LN2_HI has 16 significant bits, so n * LN2_HI is exact for |n| < 2^8),
# then e^r by its Taylor series to r^7 (|r| <= ln2 / 2: truncation below
# 2^-27 relative) in Horner form, then the scaling by 2^n.
LOG2E = F32(1.4426950408889634)
LN2_HI = F32(0.693145751953125)          # 0x3F317200
LN2_LO = F32(0.6931471805599453 - 0.693145751953125)
TAYLOR = [F32(1.0 / f) for f in (5040.0, 720.0, 120.0, 24.0, 6.0, 2.0, 1.0, 1.0)]   # 1/7! .. 1/0!
X_MAX = F32(89.0)     # above: +inf (e^x overflows float32 from 88.72)
X_MIN = F32(-87.0)    # below: 0 (and 1 + e^x == 1 in float32 long before)


def exp_f32(x) -> np.ndarray:
    x = np.asarray(x, dtype=F32)
    with np.errstate(over="ignore", invalid="ignore"):
        n = np.rint((x * LOG2E).astype(F32)).astype(F32)
        r = ((x - (n * LN2_HI).astype(F32)).astype(F32) - (n * LN2_LO).astype(F32)).astype(F32)
        p = np.full_like(r, TAYLOR[0])
        for c in TAYLOR[1:]:
            p = ((p * r).astype(F32) + c).astype(F32)
        ni = np.clip(n, -126, 128).astype(np.int32) - 1          # 2^(n-1) stays a float32 (>= 2^-127)
        half = np.ldexp(np.ones_like(p), ni).astype(F32)
        e = ((p * half).astype(F32) * F32(2.0)).astype(F32)
    e = np.where(x > X_MAX, F32(np.inf), e)
    e = np.where(x < X_MIN, F32(0.0), e)
    return e.astype(F32)


def silu_f32(g) -> np.ndarray:
    """silu(g) = g / (1 + e^-g), float32."""
    g = np.asarray(g, dtype=F32)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        return (g / (F32(1.0) + exp_f32(-g)).astype(F32)).astype(F32)


def swiglu_bf16(h: np.ndarray, inter: int) -> np.ndarray:
    """y = BF16(silu(gate) * up) for H = [gate | up] of width 2 * inter.
    Returns float32 values that are exactly BF16."""
    h = np.asarray(h, dtype=F32)
    assert h.shape[1] >= 2 * inter
    gate, up = h[:, :inter], h[:, inter:2 * inter]
    y = (silu_f32(gate) * up).astype(F32)
    return round_to_bf16(y.astype(np.float64)).astype(F32)


def swiglu_quantize(h: np.ndarray, inter: int, gran: str):
    """Codes and scales of the SwiGLU activation, quantised row by row."""
    return ROWWISE[gran](swiglu_bf16(h, inter))
