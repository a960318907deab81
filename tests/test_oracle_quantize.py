"""Pins for the oracle's quantisers (CPU only).

Checked against: the hand-worked examples in tests/golden (each cites the
page section whose formula it works through), a pure-Python loop
restatement of Step 1 / Step 2 on tiny inputs, and invariants the
mathematics fixes (the amax element lands on +-V_max, the rounding error
bound, power-of-two scale invariance, minimality of the MXFP8 exponent,
transpose invariance of 128x128 blocks, reductions between granularities).
"""
import json
import math
import os

import numpy as np
import pytest

import synth
from oracle import formats as F
from oracle import quantize as Q

F32 = np.float32


def load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- worked examples

def test_per_tensor_worked_example(golden_dir):
    g = load(golden_dir, "per_tensor_worked.json")
    x = F.bf16_bits_to_f32(np.array(g["x_bf16_bits"], dtype=np.uint16))[None, :]
    codes, s = Q.quantize_per_tensor(x)
    assert float(s) == g["scale"]
    assert codes.ravel().tolist() == g["codes"]
    assert (F.e4m3_decode(codes) * float(s)).ravel().tolist() == g["dequant"]


def test_mxfp8_worked_example(golden_dir):
    g = load(golden_dir, "mxfp8_worked.json")
    for key in ("block_a", "block_b"):
        b = g[key]
        x = np.zeros((1, 32), dtype=F32)
        x[0, : len(b["x"])] = b["x"]
        codes, e8 = Q.quantize_mxfp8(x)
        assert int(Q.mxfp8_exponent(np.abs(x).max())) == b["e"]
        assert int(e8[0, 0]) == b["ue8m0"]
        assert codes[0, : len(b["x"])].tolist() == b["codes"]


def test_nvfp4_worked_example(golden_dir):
    g = load(golden_dir, "nvfp4_worked.json")
    x = np.array(g["x"], dtype=F32)[None, :]
    packed, sb, s_g = Q.quantize_nvfp4(x)
    assert s_g == F32(3.0) / F32(2688.0)
    assert int(sb[0, 0]) == g["block_scale_code"]
    assert F.unpack_e2m1(packed)[0].tolist() == g["e2m1_codes"]


# ---------------------------------------------------------------- loop restatement

def loop_quantize_groups(x, rg, cg):
    """Step 1 and Step 2 written as plain loops over blocks of rg x cg."""
    r, c = x.shape
    codes = np.zeros((r, c), dtype=np.uint8)
    nr, nc = math.ceil(r / rg), math.ceil(c / cg)
    scales = np.zeros((nr, nc), dtype=F32)
    for bi in range(nr):
        for bj in range(nc):
            amax = 0.0
            for i in range(bi * rg, min(r, bi * rg + rg)):
                for j in range(bj * cg, min(c, bj * cg + cg)):
                    amax = max(amax, abs(float(x[i, j])))
            s = F32(1.0) if amax == 0 else F32(F32(amax) / F32(448.0))
            scales[bi, bj] = s
            for i in range(bi * rg, min(r, bi * rg + rg)):
                for j in range(bj * cg, min(c, bj * cg + cg)):
                    t = F32(x[i, j]) / s
                    codes[i, j] = int(F.e4m3_encode(t))
    return codes, scales


@pytest.fixture(scope="module")
def tiny():
    bits = synth.activations((5, 200), seed=7, outlier_frac=0.05, outlier_mult=50.0)
    return F.bf16_bits_to_f32(bits)


def test_1x128_matches_loops(tiny):
    c, s = Q.quantize_1x128(tiny)
    lc, ls = loop_quantize_groups(tiny, 1, 128)
    assert np.array_equal(c, lc) and np.array_equal(s, ls)
    assert s.shape == (5, 2)                       # ragged last group: 72 columns


def test_128x128_matches_loops():
    x = F.bf16_bits_to_f32(synth.activations((130, 260), seed=8))
    c, s = Q.quantize_128x128(x)
    lc, ls = loop_quantize_groups(x, 128, 128)
    assert np.array_equal(c, lc) and np.array_equal(s, ls)
    assert s.shape == (2, 3)


def test_per_tensor_matches_loops(tiny):
    c, s = Q.quantize_per_tensor(tiny)
    lc, ls = loop_quantize_groups(tiny, tiny.shape[0], tiny.shape[1])
    assert np.array_equal(c, lc) and float(s) == float(ls[0, 0])


def test_mxfp8_matches_loops(tiny):
    c, e8 = Q.quantize_mxfp8(tiny)
    r, cc = tiny.shape
    for i in range(r):
        for bj in range(math.ceil(cc / 32)):
            blk = tiny[i, bj * 32: bj * 32 + 32]
            amax = max(abs(float(v)) for v in blk)
            e = -127
            while 448.0 * 2.0 ** e < amax:      # smallest e with 448*2^e >= amax
                e += 1
            assert int(e8[i, bj]) == e + 127
            for j, v in enumerate(blk):
                assert int(c[i, bj * 32 + j]) == int(F.e4m3_encode(F32(v) / F32(2.0 ** e)))


def test_nvfp4_matches_loops():
    x = F.bf16_bits_to_f32(synth.activations((3, 64), seed=9, outlier_frac=0.05, outlier_mult=100.0))
    packed, sb, s_g = Q.quantize_nvfp4(x)
    amax_t = max(abs(float(v)) for v in x.ravel())
    assert s_g == F32(F32(amax_t) / F32(2688.0))
    codes = F.unpack_e2m1(packed)
    for i in range(3):
        for b in range(4):
            blk = x[i, b * 16:(b + 1) * 16]
            amax_b = max(abs(float(v)) for v in blk)
            want_sb = int(F.e4m3_encode(F32(F32(amax_b) / F32(6.0)) / s_g))
            assert int(sb[i, b]) == want_sb
            big_s = F32(F32(F.E4M3_TABLE[want_sb]) * s_g)
            for j, v in enumerate(blk):
                want = 0 if big_s == 0 else int(F.e2m1_encode(F32(v) / big_s))
                assert int(codes[i, b * 16 + j]) == want


# ---------------------------------------------------------------- invariants

@pytest.fixture(scope="module")
def act():
    return F.bf16_bits_to_f32(synth.activations((256, 512), seed=11, outlier_frac=0.01, outlier_mult=50.0))


@pytest.mark.parametrize("fn", ["1x128", "128x128", "per_tensor"])
def test_amax_element_maps_to_vmax(act, fn):
    if fn == "1x128":
        c, s = Q.quantize_1x128(act)
        groups = [(slice(i, i + 1), slice(j, j + 128)) for i in range(256) for j in range(0, 512, 128)]
    elif fn == "128x128":
        c, s = Q.quantize_128x128(act)
        groups = [(slice(i, i + 128), slice(j, j + 128)) for i in range(0, 256, 128) for j in range(0, 512, 128)]
    else:
        c, s = Q.quantize_per_tensor(act)
        groups = [(slice(None), slice(None))]
    dec = F.e4m3_decode(c)
    for sl in groups:
        blk = np.abs(act[sl])
        pos = np.unravel_index(np.argmax(blk), blk.shape)
        assert abs(dec[sl][pos]) == 448.0
        assert np.abs(dec[sl]).max() == 448.0


def test_rounding_error_bound(act):
    c, s = Q.quantize_1x128(act)
    s_full = np.repeat(s, 128, axis=1).astype(np.float64)
    t = act.astype(np.float64) / s_full
    dec = F.e4m3_decode(c)
    # E4M3 spacing at |t|: 2^(floor(log2|t|) - 3) for normals, 2^-9 below 2^-6
    with np.errstate(divide="ignore"):
        ex = np.floor(np.log2(np.maximum(np.abs(t), 2.0 ** -6)))
    spacing = 2.0 ** (ex - 3)
    f32_ulp = np.abs(t) * 2.0 ** -23
    assert np.all(np.abs(t - dec) <= spacing / 2 + f32_ulp)


def test_power_of_two_scale_invariance(act):
    for k in (-20, -3, 5, 40):
        x2 = (act.astype(np.float64) * 2.0 ** k).astype(F32)
        for fn in (Q.quantize_1x128, Q.quantize_128x128):
            c1, s1 = fn(act)
            c2, s2 = fn(x2)
            assert np.array_equal(c1, c2)
            assert np.array_equal(s2, (s1.astype(np.float64) * 2.0 ** k).astype(F32))
        c1, e1 = Q.quantize_mxfp8(act)
        c2, e2 = Q.quantize_mxfp8(x2)
        assert np.array_equal(c1, c2) and np.array_equal(e2.astype(int), e1.astype(int) + k)


def test_mxfp8_exponent_minimal_and_no_saturation(act):
    amax = Q._group_amax_1d(act, 32).astype(np.float64)
    e = Q.mxfp8_exponent(amax)
    assert np.all(448.0 * np.ldexp(1.0, e) >= amax)
    assert np.all(448.0 * np.ldexp(1.0, e - 1) < amax)
    c, e8 = Q.quantize_mxfp8(act)
    dec = np.abs(F.e4m3_decode(c)).reshape(256, 16, 32)
    top = dec.max(axis=2)
    assert np.all((top >= 224) & (top <= 448))
    t = np.abs(act.astype(np.float64)).reshape(256, 16, 32) / np.ldexp(1.0, e)[..., None]
    assert np.all(t <= 448.0)


def test_mxfp8_exponent_edges():
    assert int(Q.mxfp8_exponent(0.0)) == -127
    assert int(Q.mxfp8_exponent(448.0)) == 0
    assert int(Q.mxfp8_exponent(448.0 * (1 + 2.0 ** -7))) == 1
    assert int(Q.mxfp8_exponent(2.0 ** -133)) == -127       # clamped below
    assert int(Q.mxfp8_exponent(3.0e38)) == 120


def test_128x128_transpose_invariance(act):
    c, s = Q.quantize_128x128(act)
    ct, st = Q.transposed(Q.quantize_128x128, act)
    assert np.array_equal(ct, c.T) and np.array_equal(st, s.T)


def test_granularity_reductions():
    x = F.bf16_bits_to_f32(synth.activations((128, 128), seed=12))
    c1, s1 = Q.quantize_per_tensor(x)
    c2, s2 = Q.quantize_128x128(x)
    assert np.array_equal(c1, c2) and float(s1) == float(s2[0, 0])
    y = F.bf16_bits_to_f32(synth.activations((4, 384), seed=13))
    cr, sr = Q.quantize_1x128(y, group=384)                 # one scale per row
    for i in range(4):
        ci, si = Q.quantize_per_tensor(y[i:i + 1])
        assert np.array_equal(cr[i:i + 1], ci) and float(sr[i, 0]) == float(si)


def test_zero_block_conventions():
    x = np.zeros((2, 128), dtype=F32)
    x[1, 5] = -0.0
    c, s = Q.quantize_1x128(x)
    assert np.all(s == 1.0) and c[0].max() == 0 and c[1, 5] == 0x80
    c8, e8 = Q.quantize_mxfp8(x)
    assert np.all(e8 == 0) and c8[1, 5] == 0x80
    p, sb, sg = Q.quantize_nvfp4(np.zeros((1, 32), dtype=F32))
    assert sg == 1.0 and np.all(sb == 0) and np.all(p == 0)


def test_nvfp4_invariants():
    x = F.bf16_bits_to_f32(synth.activations((64, 256), seed=14, outlier_frac=0.001, outlier_mult=100.0))
    packed, sb, s_g = Q.quantize_nvfp4(x)
    codes = F.unpack_e2m1(packed)
    deq = F.e2m1_decode(codes) * np.repeat(F.e4m3_decode(sb), 16, axis=1) * float(s_g)
    # the tensor's amax element: its block scale saturates at 448, so it lands on +-6
    i, j = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert abs(F.e2m1_decode(codes[i, j])) == 6.0
    assert int(sb[i, j // 16]) & 0x7F == 0x7E
    # every block scale is finite and positive
    assert not np.any((sb & 0x7F) == 0x7F)
    # relative reconstruction error is bounded by E2M1 and E4M3 rounding
    err = np.abs(deq - x) / np.abs(x).reshape(64, 16, 16).max(axis=2).repeat(16, axis=1)
    assert err.max() < 0.35


def test_transposed_is_quantize_of_transpose(act):
    c, s = Q.transposed(Q.quantize_1x128, act)
    c2, s2 = Q.quantize_1x128(np.ascontiguousarray(act.T))
    assert np.array_equal(c, c2) and np.array_equal(s, s2) and c.shape == (512, 256)


# ---------------------------------------------------------------- power-of-two block-wise
def test_pow2_1x128_matches_loops_and_mxfp8(tiny):
    c, e8 = Q.quantize_1x128_pow2(tiny)
    r, cc = tiny.shape
    for i in range(r):
        for bj in range((cc + 127) // 128):
            blk = tiny[i, bj * 128: bj * 128 + 128]
            amax = max(abs(float(v)) for v in blk)
            e = -127
            while 448.0 * 2.0 ** e < amax:
                e += 1
            assert int(e8[i, bj]) == e + 127
            for j, v in enumerate(blk):
                assert int(c[i, bj * 128 + j]) == int(F.e4m3_encode(F32(v) / F32(2.0 ** e)))
    # the 1x128 exponent is the largest of its four 1x32 MXFP8 exponents
    _, e32 = Q.quantize_mxfp8(tiny)
    for i in range(r):
        for bj in range((cc + 127) // 128):
            assert int(e8[i, bj]) == int(e32[i, 4 * bj: 4 * bj + 4].max())


def test_pow2_128x128_matches_loops():
    x = F.bf16_bits_to_f32(synth.activations((130, 260), seed=15))
    c, e8 = Q.quantize_128x128_pow2(x)
    assert e8.shape == (2, 3)
    for bi in range(2):
        for bj in range(3):
            blk = x[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            e = int(Q.mxfp8_exponent(np.abs(blk).max()))
            assert int(e8[bi, bj]) == e + 127
            want = F.e4m3_encode(blk / np.float32(2.0 ** e))
            assert np.array_equal(c[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128], want)
    ct, et = Q.transposed(Q.quantize_128x128_pow2, x)
    assert np.array_equal(ct, c.T) and np.array_equal(et, e8.T)


def test_pow2_amax_element_range_and_no_saturation(act):
    c, e8 = Q.quantize_1x128_pow2(act)
    dec = np.abs(F.e4m3_decode(c)).reshape(256, 4, 128)
    top = dec.max(axis=2)
    assert np.all((top >= 224) & (top <= 448))


# ---------------------------------------------------------------- NVFP4 per-token scale, four-over-six
def test_nvfp4_row_scaled_is_per_row_tensor_scaling():
    """Per-token outer scale: each row is quantised exactly as a one-row tensor
    would be, with S_g[r] = row amax / 2688 (2688 -> 1 exactly; zero row -> 1)."""
    x = F.bf16_bits_to_f32(synth.activations((6, 64), seed=51, outlier_frac=0.05, outlier_mult=100.0))
    x[2] *= F32(1e-3)
    x[3] = 0.0
    x[4, 7] = F32(2688.0)
    x[4, 8:] = 0.0
    p, sb, sg = Q.quantize_nvfp4(x, row_scaled=True)
    assert sg.shape == (6,) and sg[3] == 1.0 and sg[4] == 1.0
    for r in range(6):
        pr, sbr, sgr = Q.quantize_nvfp4(x[r:r + 1])
        assert sg[r] == sgr
        assert np.array_equal(p[r:r + 1], pr) and np.array_equal(sb[r:r + 1], sbr)
    # a row 1000x smaller than the tensor keeps its resolution only with row scales
    pt, sbt, _ = Q.quantize_nvfp4(x)
    assert np.count_nonzero(F.unpack_e2m1(p)[2]) > np.count_nonzero(F.unpack_e2m1(pt)[2])


def test_nvfp4_four_over_six_worked_example(golden_dir):
    g = load(golden_dir, "nvfp4_4over6_worked.json")
    x = np.array(g["x"], dtype=F32)[None, :]
    p, sb, sg = Q.quantize_nvfp4(x, four_over_six=True)
    assert sg == F32(g["tensor_scale"])
    assert sb[0].tolist() == g["block_scale_codes"]
    deq = F.e2m1_decode(F.unpack_e2m1(p)) * np.repeat(F.e4m3_decode(sb), 16, axis=1) * float(sg)
    assert np.array_equal(deq, x.astype(np.float64))
    # the same row without four-over-six cannot represent block 1 exactly
    p6, sb6, sg6 = Q.quantize_nvfp4(x)
    deq6 = F.e2m1_decode(F.unpack_e2m1(p6)) * np.repeat(F.e4m3_decode(sb6), 16, axis=1) * float(sg6)
    assert not np.array_equal(deq6[0, 16:32], x[0, 16:32].astype(np.float64))


def _exact_block_sq_error(blk, s_g, v_map):
    """Squared error of one block mapped to v_map, in exact rational arithmetic,
    with the scale and codes built by per-element loops."""
    from fractions import Fraction
    amax = max(abs(float(v)) for v in blk)
    sb = int(F.e4m3_encode(F32(F32(amax) / F32(v_map)) / s_g))
    big_s = F32(F32(F.E4M3_TABLE[sb]) * s_g)
    err = Fraction(0)
    for v in blk:
        q = 0 if big_s == 0 else int(F.e2m1_encode(F32(v) / big_s))
        d = Fraction(float(v)) - Fraction(float(F.E2M1_TABLE[q])) * Fraction(float(big_s))
        err += d * d
    return err, sb


def test_nvfp4_four_over_six_picks_smaller_error():
    """Against exact squared errors: wherever the two choices differ by more
    than float32 summation can blur, the oracle keeps the one with the smaller
    error; its scale code is that choice's code."""
    x = F.bf16_bits_to_f32(synth.activations((8, 256), seed=52, outlier_frac=0.02, outlier_mult=30.0))
    for row_scaled in (False, True):
        p, sb, sg = Q.quantize_nvfp4(x, row_scaled=row_scaled, four_over_six=True)
        chose4 = decided = 0
        for i in range(8):
            s_g = F32(sg[i] if row_scaled else sg)
            if row_scaled:
                assert s_g == F32(F32(np.abs(x[i]).max()) / F32(1536.0))
            for b in range(16):
                blk = x[i, 16 * b:16 * b + 16]
                e6, sb6 = _exact_block_sq_error(blk, s_g, 6.0)
                e4, sb4 = _exact_block_sq_error(blk, s_g, 4.0)
                if abs(e6 - e4) <= 1e-4 * max(e6, e4):
                    continue
                decided += 1
                want = sb4 if e4 < e6 else sb6
                chose4 += int(e4 < e6)
                assert int(sb[i, b]) == want
        assert decided > 100 and 0 < chose4 < decided


def test_nvfp4_four_over_six_error_never_worse():
    """The kept choice's squared error is at most that of the map-to-6 choice
    under the same outer scale, block by block."""
    x = F.bf16_bits_to_f32(synth.activations((32, 512), seed=53, outlier_frac=0.01, outlier_mult=50.0))
    s_g = Q.nvfp4_tensor_scale(x, four_over_six=True)
    p, sb, _ = Q.quantize_nvfp4(x, four_over_six=True)
    p6, sb6, _ = Q.quantize_nvfp4(x, s_g=s_g)
    def block_err(pk, s):
        deq = F.e2m1_decode(F.unpack_e2m1(pk)) * np.repeat(F.e4m3_decode(s), 16, axis=1) * float(s_g)
        return ((deq - x) ** 2).reshape(32, 32, 16).sum(axis=2)
    e, e6 = block_err(p, sb), block_err(p6, sb6)
    assert np.all(e <= e6 * (1 + 1e-5) + 1e-30)
    assert np.mean(e) < np.mean(e6)
    # the largest block scale is 384 (map-to-4 of the amax block) or 256, never above
    assert F.e4m3_decode(sb).max() <= 384.0
