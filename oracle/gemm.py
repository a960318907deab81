"""Block-scaled GEMM reference (oracle; test infrastructure).

The layer's forward and backward GEMMs run on the quantised operands with
the scales applied per block ("Low Precision RL", "Unified training recipe":
a matching low-precision GEMM in the trainer forward; section "3. Unified
MXFP8 (Blackwell)": MXFP8 also for the weight-gradient and data-gradient
GEMMs).  The exact value such a GEMM approximates is

    D[m, n] = sum_k  deq_A[m, k] * deq_B[n, k]

where deq = decode(code) * scale of the block holding (row, k).  Each
dequantised value (a code with at most 4 significant bits times an FP32 or
power-of-two scale) is exact in float64; the products and the sum are taken
with a float64 matrix product (library routine), and the result is rounded
once to BF16, the output type.

Operand convention: A is [M, K], B is [N, K] (both K-major), D = A . B^T.
"""
from __future__ import annotations

import numpy as np

from .formats import e2m1_decode, e4m3_decode, round_to_bf16, ue8m0_decode, unpack_e2m1


def _expand(scale: np.ndarray, rows: int, cols: int, rg: int, cg: int) -> np.ndarray:
    s = np.asarray(scale, dtype=np.float64)
    if s.ndim == 0:
        return np.full((rows, cols), float(s))
    return np.repeat(np.repeat(s, rg, axis=0), cg, axis=1)[:rows, :cols]


def dequant_per_tensor(codes, s):
    return e4m3_decode(codes) * np.float64(s)


def dequant_1x128(codes, s, group: int = 128):
    r, c = codes.shape
    return e4m3_decode(codes) * _expand(s, r, c, 1, group)


def dequant_128x128(codes, s, block: int = 128):
    r, c = codes.shape
    return e4m3_decode(codes) * _expand(s, r, c, block, block)


def dequant_mxfp8(codes, e8, group: int = 32):
    r, c = codes.shape
    return e4m3_decode(codes) * _expand(ue8m0_decode(e8), r, c, 1, group)


def dequant_1x128_pow2(codes, e8, group: int = 128):
    r, c = codes.shape
    return e4m3_decode(codes) * _expand(ue8m0_decode(e8), r, c, 1, group)


def dequant_128x128_pow2(codes, e8, block: int = 128):
    r, c = codes.shape
    return e4m3_decode(codes) * _expand(ue8m0_decode(e8), r, c, block, block)


def dequant_nvfp4(packed, sb, s_g, group: int = 16):
    """value = E2M1(code) * E4M3(block scale) * S_g, all exact in float64.
    S_g is one outer scale, or one per row ([R]) for per-token scaling."""
    q = unpack_e2m1(packed)
    r, c = q.shape
    g = np.asarray(s_g, dtype=np.float64)
    if g.ndim == 1:
        g = g.reshape(r, 1)
    return e2m1_decode(q) * _expand(e4m3_decode(sb), r, c, 1, group) * g


DEQUANT = {
    "per_tensor": dequant_per_tensor,
    "1x128": dequant_1x128,
    "128x128": dequant_128x128,
    "mxfp8": dequant_mxfp8,
    "1x128_pow2": dequant_1x128_pow2,
    "128x128_pow2": dequant_128x128_pow2,
}


def dequantize_bf16(codes, scales, gran, s_g=None):
    """BF16 dequantisation of quantised operands (the "dequantized backward"
    of "Low Precision RL", "Advanced: dequantized backward": the BF16 backward
    GEMMs consume BF16 dequantisations of the low-precision forward operands).
    Reading: the exact dequantised value, rounded once to BF16 (nearest even).
    Returns float64 values that are exactly BF16."""
    if gran == "nvfp4":
        return round_to_bf16(dequant_nvfp4(codes, scales, s_g))
    return round_to_bf16(DEQUANT[gran](codes, scales))


def gemm_f64(a64: np.ndarray, b64: np.ndarray) -> np.ndarray:
    """D64 = A . B^T in float64."""
    return np.asarray(a64, dtype=np.float64) @ np.asarray(b64, dtype=np.float64).T


def gemm_bf16(a64: np.ndarray, b64: np.ndarray) -> np.ndarray:
    """The reference output: the float64 product rounded once to BF16."""
    return round_to_bf16(gemm_f64(a64, b64))


def block_gemm(a_codes, a_s, a_gran, b_codes, b_s, b_gran):
    """D = deq(A) . deq(B)^T rounded to BF16, for the FP32/UE8M0-scaled FP8 modes."""
    return gemm_bf16(DEQUANT[a_gran](a_codes, a_s), DEQUANT[b_gran](b_codes, b_s))


def grouped_gemm(a64: np.ndarray, b64_per_expert, offsets) -> np.ndarray:
    """MoE grouped GEMM: rows offsets[e] .. offsets[e+1] of A use expert e's B."""
    offsets = np.asarray(offsets, dtype=np.int64)
    n = b64_per_expert[0].shape[0]
    out = np.zeros((a64.shape[0], n), dtype=np.float64)
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            out[lo:hi] = gemm_bf16(a64[lo:hi], b64_per_expert[e])
    return out
