"""Quantisers of the low-precision linear layer (oracle; test infrastructure).

Every function takes the BF16 input already widened to float32, shape
[R, C], and returns codes plus scales.  Arithmetic follows the two steps of
the Unified FP8 review, section "FP8 Quantization":

  Step 1  S = max|X| / V_max       (over the tensor, or over one block)
  Step 2  Q(x) = round(x / S)

read as: the amax is exact (a max of absolute values), S is an IEEE float32
division, x / S is an IEEE float32 division, and "round" is the saturating
round-to-nearest-even cast to the target format (E4M3, V_max = 448; E2M1,
V_max = 6).  numpy float32 arithmetic is IEEE binary32 with
round-to-nearest-even and gradual underflow, which is exactly that.

Granularities (review, "FP8 Quantization": per-tensor, per-token for
activations and gradients, per-block for weights; "Low Precision RL",
table "Choose a precision"):
  per-tensor        one FP32 scale
  1x128 (per token) one FP32 scale per row and 128 consecutive columns
  128x128 (block)   one FP32 scale per 128x128 tile
  MXFP8 1x32        one UE8M0 (power-of-two) scale per row and 32 columns
  NVFP4 1x16        one E4M3 scale per row and 16 columns, times one FP32
                    tensor scale; elements are E2M1

A last group that runs past the edge of the tensor is not padded: its amax
is taken over the elements that exist.

Scale layouts returned: row-major [R, ceil(C/g)] for 1-D groups, [ceil(R/128),
ceil(C/128)] for 128x128, a 0-d float32 for per-tensor.
"""
from __future__ import annotations

import numpy as np

from .formats import E2M1_MAX, E4M3_MAX, e2m1_decode, e2m1_encode, e4m3_decode, e4m3_encode, pack_e2m1

F32 = np.float32


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def fp32_scale(amax):
    """Step 1 with an FP32 scale: S = amax / 448 (IEEE float32 division).

    An all-zero block has no defined S on the pages; S = 1 is used, which
    leaves every code +-0 (parity unpinned reading).
    """
    amax = np.asarray(amax, dtype=F32)
    s = amax / F32(E4M3_MAX)
    return np.where(amax == 0, F32(1.0), s).astype(F32)


def cast_e4m3(x, s):
    """Step 2: Q(x) = E4M3(x / S) with IEEE float32 division."""
    return e4m3_encode(np.asarray(x, dtype=F32) / np.asarray(s, dtype=F32))


def _group_amax_1d(x: np.ndarray, g: int) -> np.ndarray:
    """max|x| over groups of g consecutive columns; ragged last group allowed."""
    r, c = x.shape
    n = _ceil_div(c, g)
    pad = np.zeros((r, n * g), dtype=F32)
    pad[:, :c] = np.abs(x)
    return pad.reshape(r, n, g).max(axis=2)


def _expand_cols(s: np.ndarray, g: int, c: int) -> np.ndarray:
    return np.repeat(s, g, axis=1)[:, :c]


def quantize_per_tensor(x: np.ndarray):
    x = np.asarray(x, dtype=F32)
    amax = np.abs(x).max() if x.size else F32(0)
    s = fp32_scale(amax)
    return cast_e4m3(x, s), s


def quantize_1x128(x: np.ndarray, group: int = 128):
    """Per-token scaling with groups of `group` columns (group = C gives one
    scale per row, the "rowwise" scaling of the full-pipeline FP8 RL paper)."""
    x = np.asarray(x, dtype=F32)
    s = fp32_scale(_group_amax_1d(x, group))
    return cast_e4m3(x, _expand_cols(s, group, x.shape[1])), s


def quantize_128x128(x: np.ndarray, block: int = 128):
    x = np.asarray(x, dtype=F32)
    r, c = x.shape
    nr, nc = _ceil_div(r, block), _ceil_div(c, block)
    pad = np.zeros((nr * block, nc * block), dtype=F32)
    pad[:r, :c] = np.abs(x)
    amax = pad.reshape(nr, block, nc, block).max(axis=(1, 3))
    s = fp32_scale(amax)
    s_full = np.repeat(np.repeat(s, block, axis=0), block, axis=1)[:r, :c]
    return cast_e4m3(x, s_full), s


def mxfp8_exponent(amax) -> np.ndarray:
    """Smallest integer e with 448 * 2^e >= amax, clamped to [-127, 127].

    This is S = 2^ceil(log2(amax / 448)) evaluated exactly: write
    amax = m * 2^E with 0.5 <= m < 1 and 448 = 0.875 * 2^9; then
    448 * 2^(E-9) >= amax iff m <= 0.875, and 448 * 2^(E-10) < amax always.
    amax = 0 gives the smallest scale, e = -127 (parity unpinned reading).
    """
    a = np.asarray(amax, dtype=np.float64)
    m, big_e = np.frexp(a)
    e = np.where(m <= 0.875, big_e - 9, big_e - 8)
    e = np.where(a == 0, -127, e)
    return np.clip(e, -127, 127).astype(np.int64)


def quantize_mxfp8(x: np.ndarray, group: int = 32):
    """MXFP8: 1x32 groups of E4M3 sharing one UE8M0 scale ("Low Precision RL",
    "3. Unified MXFP8 (Blackwell)").  Returns (codes, ue8m0 codes [R, C/32])."""
    x = np.asarray(x, dtype=F32)
    e = mxfp8_exponent(_group_amax_1d(x, group))
    s = np.ldexp(np.float64(1.0), e).astype(F32)            # 2^e, exact in f32
    codes = cast_e4m3(x, _expand_cols(s, group, x.shape[1]))
    return codes, (e + 127).astype(np.uint8)


def quantize_1x128_pow2(x: np.ndarray, group: int = 128):
    """Block-wise recipe with power-of-two scales: 1x128 groups, the MXFP8
    scale rule (smallest 2^e with 448 * 2^e >= amax) applied per group.  The
    "Low Precision RL" page (section "2. Unified block-wise FP8") notes that on
    Blackwell TransformerEngine runs the block-wise recipe through MXFP8 with
    power-of-two scales.  Returns (codes, UE8M0 codes [R, ceil(C/128)])."""
    x = np.asarray(x, dtype=F32)
    e = mxfp8_exponent(_group_amax_1d(x, group))
    s = np.ldexp(np.float64(1.0), e).astype(F32)
    codes = cast_e4m3(x, _expand_cols(s, group, x.shape[1]))
    return codes, (e + 127).astype(np.uint8)


def quantize_128x128_pow2(x: np.ndarray, block: int = 128):
    """128x128 blocks with power-of-two scales (see quantize_1x128_pow2).
    Returns (codes, UE8M0 codes [ceil(R/128), ceil(C/128)])."""
    x = np.asarray(x, dtype=F32)
    r, c = x.shape
    nr, nc = _ceil_div(r, block), _ceil_div(c, block)
    pad = np.zeros((nr * block, nc * block), dtype=F32)
    pad[:r, :c] = np.abs(x)
    e = mxfp8_exponent(pad.reshape(nr, block, nc, block).max(axis=(1, 3)))
    s = np.ldexp(np.float64(1.0), e).astype(F32)
    s_full = np.repeat(np.repeat(s, block, axis=0), block, axis=1)[:r, :c]
    return cast_e4m3(x, s_full), (e + 127).astype(np.uint8)


NVFP4_GLOBAL_DIV = F32(E4M3_MAX * E2M1_MAX)   # 448 * 6 = 2688
# Four-over-six keeps the largest block scale at 256 (not 448) for the map-to-6
# choice, so the map-to-4 choice of the same block (1.5x larger, 384) still fits
# E4M3: S_g = amax / (256 * 6).
NVFP4_GLOBAL_DIV_4OVER6 = F32(256.0 * E2M1_MAX)   # 1536


def _outer_scale(amax, four_over_six: bool):
    """S_g = amax / (V_max(E4M3) * 6) in float32; 1 where amax == 0."""
    div = NVFP4_GLOBAL_DIV_4OVER6 if four_over_six else NVFP4_GLOBAL_DIV
    amax = np.asarray(amax, dtype=F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        s = (amax / div).astype(F32)
    return np.where(amax == 0, F32(1.0), s).astype(F32)


def nvfp4_tensor_scale(x: np.ndarray, four_over_six: bool = False):
    """Outer FP32 scale of the whole tensor: S_g = amax_T / (448 * 6)
    (amax_T / (256 * 6) with four-over-six); S_g = 1 for an all-zero tensor."""
    x = np.asarray(x, dtype=F32)
    amax = np.abs(x).max() if x.size else F32(0)
    return F32(_outer_scale(F32(amax), four_over_six))


def nvfp4_row_scales(x: np.ndarray, four_over_six: bool = False) -> np.ndarray:
    """Per-token outer scales ("4. NVFP4 (Blackwell)": activation scaling is
    computed per token): S_g[r] = amax(row r) / (448 * 6), or / (256 * 6) with
    four-over-six; 1 for an all-zero row.  Shape [R], float32."""
    x = np.asarray(x, dtype=F32)
    amax = np.abs(x).max(axis=1) if x.shape[1] else np.zeros(x.shape[0], dtype=F32)
    return _outer_scale(amax, four_over_six)


def _nvfp4_candidate(x, amax_b, s_col, v_map, group):
    """Block scales and codes when the block amax is mapped to the E2M1
    magnitude v_map (6 = the format's maximum, or 4)."""
    c = x.shape[1]
    sb = e4m3_encode((amax_b / F32(v_map)) / s_col)
    big_s = (e4m3_decode(sb).astype(F32) * s_col).astype(F32)
    big_s_full = _expand_cols(big_s, group, c)
    zero = big_s_full == 0
    with np.errstate(divide="ignore", invalid="ignore"):
        t = x / np.where(zero, F32(1.0), big_s_full)
    q = np.where(zero, np.uint8(0), e2m1_encode(t)).astype(np.uint8)
    return sb, q, big_s_full


def nvfp4_block_sq_error(x, q, big_s_full, group: int = 16):
    """Squared quantisation error of each 16-element block, in float32:
    y = E2M1(q) * S_b, d = x - y, and d*d summed over elements 0..7 and 8..15
    of the block in order, the two half sums then added (each operation one
    IEEE float32 rounding; the summation order is fixed so that the choice it
    decides is reproducible).  Returns [R, C/16] float32."""
    assert group == 16
    r, c = x.shape
    with np.errstate(over="ignore"):      # squares of values near the float32 limit are +inf, as in IEEE
        y = (e2m1_decode(q).astype(F32) * big_s_full).astype(F32)
        d = (x - y).astype(F32)
        sq = (d * d).astype(F32).reshape(r, c // 16, 2, 8)
        acc = sq[..., 0].copy()
        for i in range(1, 8):
            acc = (acc + sq[..., i]).astype(F32)
        return (acc[..., 0] + acc[..., 1]).astype(F32)


def quantize_nvfp4(x: np.ndarray, group: int = 16, s_g=None, row_scaled: bool = False,
                   four_over_six: bool = False):
    """NVFP4: E2M1 values in 1x16 blocks, an E4M3 scale per block and an outer
    FP32 scale ("Low Precision RL", "4. NVFP4 (Blackwell)"; RHT, 2-D blocks and
    stochastic rounding are switched off there, so plain RNE 1-D blocks).

    Reading of the two-level scale, applying Step 1 twice:
      S_g = amax_T / (448 * 6)                    (float32)
      s_b = E4M3( (amax_b / 6) / S_g )            (float32 divisions, then cast)
      S_b = decode(s_b) * S_g                     (float32 multiply)
      q   = E2M1( x / S_b )                       (float32 division, then cast)
    A block whose s_b decodes to 0 gets all-zero codes (0x0).

    row_scaled: the outer scale is per row (per token), S_g[r] from the row's
    amax, instead of one per tensor.

    four_over_six ("Advanced: four-over-six"): every block is quantised twice,
    with its amax mapped to 6 (s_b from amax_b / 6) and to 4 (s_b from
    amax_b / 4), under S_g = amax / (256 * 6); the block keeps the choice with
    the smaller squared error (nvfp4_block_sq_error), the map-to-6 choice on a
    tie.

    s_g, when given, is used as the outer scale (a scalar, or [R] when
    row_scaled).  Returns (packed codes [R, C/2], block scale codes [R, C/16],
    S_g as a float32 scalar or [R] array).
    """
    x = np.asarray(x, dtype=F32)
    r, c = x.shape
    assert c % group == 0 and group % 2 == 0
    if s_g is None:
        s_g = nvfp4_row_scales(x, four_over_six) if row_scaled else nvfp4_tensor_scale(x, four_over_six)
    if row_scaled:
        s_g = np.asarray(s_g, dtype=F32).reshape(r)
        s_col = s_g[:, None]
    else:
        s_g = F32(s_g)
        s_col = s_g
    amax_b = _group_amax_1d(x, group)
    sb, q, big_s_full = _nvfp4_candidate(x, amax_b, s_col, E2M1_MAX, group)
    if four_over_six:
        sb4, q4, big_s4 = _nvfp4_candidate(x, amax_b, s_col, 4.0, group)
        err6 = nvfp4_block_sq_error(x, q, big_s_full, group)
        err4 = nvfp4_block_sq_error(x, q4, big_s4, group)
        use4 = err4 < err6
        sb = np.where(use4, sb4, sb).astype(np.uint8)
        q = np.where(_expand_cols(use4, group, c), q4, q).astype(np.uint8)
    return pack_e2m1(q), sb, s_g


def transposed(fn, x: np.ndarray, **kw):
    """Column-wise variant used by dgrad/wgrad: quantise X^T from the same BF16
    source (not a re-quantisation of already-rounded codes)."""
    return fn(np.ascontiguousarray(np.asarray(x, dtype=F32).T), **kw)
