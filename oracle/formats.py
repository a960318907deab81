"""Number formats used by the low-precision linear layer (oracle; test infrastructure).

E4M3 ("FP8 Format" section of the Unified FP8 review: 4-bit exponent,
3-bit mantissa) in its OCP "FN" variant: exponent bias 7, no infinities,
the single NaN pattern S.1111.111, largest finite magnitude 448.
E2M1 (NVFP4 elements, "Low Precision RL", section "4. NVFP4 (Blackwell)"):
exponent bias 1, no inf/NaN, magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}.
UE8M0 (MXFP8 block scale, "Low Precision RL", table "Choose a precision"):
an unsigned biased exponent, value 2^(code-127), code 0xFF is NaN.

Decoding is written straight from the bit fields.  Encoding is done by
brute force: the nearest representable magnitude, ties to the code with an
even mantissa (round-to-nearest-even), magnitudes beyond the largest finite
value clamp to it (saturating cast), the sign bit is copied (so -0 -> 0x80).
All comparisons happen in float64, where every code value and every
midpoint between neighbouring codes is exact.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E2M1_MAX = 6.0
E4M3_NAN = 0x7F


def e4m3_value(code: int) -> float:
    """Value of one E4M3 code, from its sign / exponent / mantissa fields."""
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        mag = (m / 8.0) * 2.0 ** (1 - 7)          # subnormal: 0.m * 2^(1-bias)
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)    # normal: 1.m * 2^(e-bias)
    return -mag if s else mag


def e2m1_value(code: int) -> float:
    """Value of one E2M1 code (4 bits), from its fields."""
    s = (code >> 3) & 1
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        mag = (m / 2.0) * 2.0 ** (1 - 1)
    else:
        mag = (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if s else mag


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
# magnitudes of the non-negative finite codes, in code order (increasing)
_E4M3_MAGS = E4M3_TABLE[:0x7F]
_E2M1_MAGS = E2M1_TABLE[:8]


def _encode_nearest(t: np.ndarray, mags: np.ndarray, sign_bit: int) -> np.ndarray:
    a = np.abs(t.astype(np.float64))
    top = len(mags) - 1
    idx = np.searchsorted(mags, a, side="right") - 1       # mags[idx] <= a
    idx = np.clip(idx, 0, top)
    nxt = np.minimum(idx + 1, top)
    mid = (mags[idx] + mags[nxt]) * 0.5
    go_up = (a > mid) | ((a == mid) & (idx % 2 == 1))       # tie -> even code
    code = np.where(go_up & (idx < top), idx + 1, idx)      # >= max: saturate
    code = code | np.where(np.signbit(t), sign_bit, 0)
    return code.astype(np.uint8)


def e4m3_encode(t) -> np.ndarray:
    """Saturating round-to-nearest-even cast of float values to E4M3 codes.

    NaN maps to 0x7F; +-inf and |t| > 448 map to +-448 (0x7E / 0xFE).
    """
    t = np.asarray(t, dtype=np.float32)
    code = _encode_nearest(t, _E4M3_MAGS, 0x80)
    return np.where(np.isnan(t), np.uint8(E4M3_NAN), code).astype(np.uint8)


def e4m3_decode(codes) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e2m1_encode(t) -> np.ndarray:
    """Saturating round-to-nearest-even cast to 4-bit E2M1 codes (uint8 0..15)."""
    t = np.asarray(t, dtype=np.float32)
    return _encode_nearest(t, _E2M1_MAGS, 0x8)


def e2m1_decode(codes) -> np.ndarray:
    return E2M1_TABLE[np.asarray(codes, dtype=np.uint8) & 0xF]


def ue8m0_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.int64)
    v = np.ldexp(1.0, c - 127)
    return np.where(c == 0xFF, np.nan, v)


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """Pack pairs of 4-bit codes along the last axis: element 2j -> low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def bf16_bits_to_f32(bits) -> np.ndarray:
    """BF16 is the top half of an IEEE binary32: widen by a 16-bit shift."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32)
    return (b << np.uint32(16)).view(np.float32)


def round_to_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest BF16 value (ties to even), as float64.

    BF16 keeps 8 significant bits; its smallest exponent quantum is 2^-133
    (subnormals).  The value is scaled by a power of two (exact), rounded to
    an integer with numpy's half-to-even rint, and scaled back.  Overflow to
    +-inf follows IEEE (anything at or beyond the rounding boundary of the
    largest finite BF16 value).
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)                      # x = m * 2^e, 0.5 <= |m| < 1
    q = np.maximum(e - 8, -133)             # quantum 2^q of x's binade
    r = np.rint(np.ldexp(x, -q))
    y = np.ldexp(r, q)
    big = 2.0 ** 128 * (1 - 2.0 ** -9)      # rounding boundary above max finite
    y = np.where(np.abs(x) >= big, np.copysign(np.inf, x), y)
    return np.where(x == 0, x, y)


def f64_to_bf16_bits(x) -> np.ndarray:
    y = round_to_bf16(x).astype(np.float32)   # exact: y is a bf16 value
    return (y.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
