"""Pins for the oracle's MoE steps (CPU only).

SwiGLU is the float64 definition silu(g) * up rounded once to BF16.  It is
pinned by values that do not come from the oracle's own evaluation: scipy's
logistic function (a separate implementation of 1 / (1 + e^-g)), the
identity silu(g) - silu(-g) = g, exact special values, cases where a
float32 evaluation rounded twice would give another BF16 value, and the
[gate | up] layout.  The near-boundary classifier is checked against a
bit-level construction of the two BF16 values that bracket each input.  The
gathered quantisation is checked against per-row quantisation of the
indexed tokens and against indexing the quantised matrix.
"""
import numpy as np
import pytest

import synth
from oracle import formats as F
from oracle import moe as M
from oracle import quantize as Q

F32 = np.float32


def test_silu_against_scipy_logistic():
    special = pytest.importorskip("scipy.special")
    g = np.concatenate([np.linspace(-700, 700, 200001), -np.logspace(-30, 2.8, 3000), np.logspace(-30, 2.8, 3000)])
    up = np.linspace(-3.0, 3.0, g.size)
    h = np.stack([g, up], axis=1)
    got = M.swiglu_exact(h, 1)[:, 0]
    ref = g * special.expit(g) * up
    nz = ref != 0
    assert np.max(np.abs(got[nz] - ref[nz]) / np.abs(ref[nz])) < 1e-13
    assert np.all(got[~nz] == 0)


def test_silu_odd_part_identity():
    g = np.linspace(-60, 60, 12001)
    h_pos = np.stack([g, np.ones_like(g)], axis=1)
    h_neg = np.stack([-g, np.ones_like(g)], axis=1)
    diff = M.swiglu_exact(h_pos, 1)[:, 0] - M.swiglu_exact(h_neg, 1)[:, 0]
    assert np.max(np.abs(diff - g)) <= 1e-13 * np.max(np.abs(g))


def test_silu_special_values():
    h = np.array([[0.0, 5.0], [-0.0, 1.0], [100.0, 0.5], [-800.0, 1.0], [-800.0, -1.0], [1.0, 1.0], [-1.0, 1.0],
                  [2.0, 1.0]])
    y = M.swiglu_exact(h, 1)[:, 0]
    assert y[0] == 0.0 and y[1] == 0.0
    assert y[2] == 50.0                               # 1 + e^-100 == 1 in float64
    assert y[3] == 0.0 and np.signbit(y[3])           # g e^g underflows: -0 * 1
    assert y[4] == 0.0 and not np.signbit(y[4])
    assert abs(y[5] - 0.7310585786300049) < 1e-16     # sigma(1), a textbook constant
    assert abs(y[6] + 0.2689414213699951) < 1e-16
    assert abs(y[7] - 1.7615941559557649) < 1e-15


def test_far_negative_gate_keeps_tiny_bf16_values():
    """For g below -88.7, e^-g overflows float32, yet silu(g) * up is still
    a normal or subnormal BF16 number; the definition keeps it."""
    g = np.array([-88.0, -89.0, -92.0, -96.0, -100.0, -104.0])
    up = np.array([1.0, 1.0, 1.0, 1.0, 100.0, 1e4])
    y = M.swiglu_bf16(np.stack([g, up], axis=1), 1)[:, 0]
    exact = g * np.exp(g) * up
    assert np.all(y < 0)
    assert np.all(np.abs(y - exact) <= np.abs(exact) * 2.0 ** -7 + 2.0 ** -134)


def test_swiglu_rounds_once_from_the_exact_value():
    """On two million random BF16 (gate, up) pairs, find those where a float32
    evaluation (rounded to float32, then to BF16) lands on another BF16 value
    than the exact value rounded once; the oracle must give the once-rounded
    value there."""
    rng = synth.rng(66)
    gb = rng.integers(0, 65536, 2_000_000).astype(np.uint16)
    ub = rng.integers(0, 65536, 2_000_000).astype(np.uint16)
    g = F.bf16_bits_to_f32(gb).astype(np.float64)
    u = F.bf16_bits_to_f32(ub).astype(np.float64)
    keep = np.isfinite(g) & np.isfinite(u) & (np.abs(g) < 80) & (np.abs(u) < 1e30) & (np.abs(u) > 1e-30)
    g, u = g[keep], u[keep]
    exact = g / (1.0 + np.exp(-g)) * u
    twice = F.round_to_bf16(exact.astype(F32).astype(np.float64))
    once = F.round_to_bf16(exact)
    y = M.swiglu_bf16(np.stack([g, u], axis=1), 1)[:, 0].astype(np.float64)
    assert np.array_equal(y, once)
    differ = twice != once
    # such cases exist, so this pin distinguishes the two readings
    assert differ.sum() > 0


def test_swiglu_layout_gate_then_up():
    inter = 32
    h = np.zeros((2, 2 * inter), F32)
    h[0, :inter] = 0.0            # gate 0 -> silu 0 -> y 0 whatever up is
    h[0, inter:] = 5.0
    h[1, :inter] = 20.0           # silu(20) = 20 (to BF16) -> y = 20 * up
    h[1, inter:] = 0.5
    y = M.swiglu_bf16(h, inter)
    assert np.all(y[0] == 0.0)
    assert np.all(y[1] == 10.0)
    # the swapped reading, silu(up) * gate, gives silu(0.5) * 20 = 6.22...
    assert M.swiglu_bf16(np.array([[0.5, 20.0]]), 1)[0, 0] != 10.0


def _bracket_bf16(y):
    """The BF16 values just below and above |y| by bit manipulation of the
    float32 pattern (independent of the oracle's frexp construction)."""
    a = np.abs(y).astype(F32)
    lo_bits = (a.view(np.uint32) >> 16).astype(np.uint32)
    lo = F.bf16_bits_to_f32(lo_bits.astype(np.uint16)).astype(np.float64)
    hi = F.bf16_bits_to_f32((lo_bits + 1).astype(np.uint16)).astype(np.float64)
    return lo, hi, lo_bits


def test_tie_neighbour_against_bit_brackets():
    rng = synth.rng(64)
    y = rng.standard_normal(200000) * np.exp2(rng.integers(-140, 100, 200000).astype(np.float64))
    # exact float32 values (so the float32 truncation in _bracket_bf16 is exact) plus midpoints
    y = y.astype(F32).astype(np.float64)
    lo, hi, lo_bits = _bracket_bf16(y)
    mids = (lo + hi) / 2 * np.sign(y)
    y = np.concatenate([y, mids, mids + np.spacing(mids.astype(F32)).astype(np.float64)])
    lo, hi, lo_bits = _bracket_bf16(y)
    near, alt, tie = M.bf16_tie_neighbour(y, 8.0)
    a = np.abs(y)
    mid = (lo + hi) / 2
    nearest = np.where(a < mid, lo, np.where(a > mid, hi, np.where(lo_bits % 2 == 0, lo, hi)))
    assert np.array_equal(np.abs(near), nearest)
    other = np.where(nearest == lo, hi, lo)
    exact_bf16 = a == lo
    other = np.where(exact_bf16, nearest, other)
    f32ulp = np.spacing(a.astype(F32)).astype(np.float64)
    want_tie = (np.abs(a - mid) <= np.maximum(8 * f32ulp, 2.0 ** -146)) & ~exact_bf16
    # a value just above the largest finite BF16 rounds to it or to inf; keep those out
    ok = np.isfinite(hi)
    assert np.array_equal(tie[ok], want_tie[ok])
    assert np.array_equal(np.abs(alt[ok & tie]), other[ok & tie])


def test_swiglu_check_accepts_either_neighbour_and_rejects_others():
    h = F.bf16_bits_to_f32(synth.activations((8, 256), seed=65)).astype(np.float64)
    inter = 128
    y = M.swiglu_exact(h, inter)
    near, alt, tie = M.bf16_tie_neighbour(y, 8.0)
    # plant a near-boundary element and take its other neighbour
    h2 = h.copy()
    h2[3, 5] = 1.0
    h2[3, inter + 5] = (1.0 + 2.0 ** -8) / (1.0 / (1.0 + np.exp(-1.0)))   # y = 1 + 2^-8, a BF16 tie
    y2 = M.swiglu_exact(h2, inter)
    n2, a2, t2 = M.bf16_tie_neighbour(y2, 8.0)
    assert t2[3, 5]
    c_near, s_near = Q.quantize_mxfp8(n2.astype(F32))
    c_alt, s_alt = Q.quantize_mxfp8(np.where(t2, a2, n2).astype(F32))
    assert M.swiglu_check(c_near, s_near, h2, inter, "mxfp8")[0] == 0
    assert M.swiglu_check(c_alt, s_alt, h2, inter, "mxfp8")[0] == 0
    bad = c_near.copy()
    bad[0, 0] ^= 1
    assert M.swiglu_check(bad, s_near, h2, inter, "mxfp8")[0] == 1
    bad_s = s_near.copy()
    bad_s[1, 1] += 1
    assert M.swiglu_check(c_near, bad_s, h2, inter, "mxfp8")[0] == 1


@pytest.mark.parametrize("gran", ["1x128", "mxfp8", "1x128_pow2"])
def test_quantize_gathered_is_indexing_the_tokens(gran):
    x = F.bf16_bits_to_f32(synth.activations((40, 384), seed=62, outlier_frac=0.02, outlier_mult=50.0))
    idx = np.array([3, 3, 0, 39, 17, 17, 17, 5, 38, 1], np.int64)
    c, s = M.quantize_gathered(x, idx, gran)
    call, sall = M.ROWWISE[gran](x)
    assert np.array_equal(c, call[idx]) and np.array_equal(s, sall[idx])
    for r, t in enumerate(idx):
        cr, sr = M.ROWWISE[gran](x[t:t + 1])
        assert np.array_equal(c[r:r + 1], cr) and np.array_equal(s[r:r + 1], sr)


def test_swiglu_quantize_is_quantize_of_activation():
    h = F.bf16_bits_to_f32(synth.activations((16, 768), seed=63))
    c, s = M.swiglu_quantize(h, 384, "mxfp8")
    c2, s2 = Q.quantize_mxfp8(M.swiglu_bf16(h, 384))
    assert np.array_equal(c, c2) and np.array_equal(s, s2)
