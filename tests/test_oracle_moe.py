"""Pins for the oracle's MoE steps (CPU only).

The float32 e^x / silu sequence is checked against float64 mathematics
(ulp bounds, exact special values); the SwiGLU activation against the
float64 definition rounded once to BF16 (equal except at BF16 rounding
ties); the layout of [gate | up] by inputs whose swapped reading gives a
different result; the gathered quantisation against per-row quantisation of
the indexed tokens and against indexing the quantised matrix.
"""
import numpy as np
import pytest

import synth
from oracle import formats as F
from oracle import moe as M
from oracle import quantize as Q
from tests._util import bf16_ulp

F32 = np.float32


def ulps(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return np.abs(got - ref) / np.spacing(np.abs(ref).astype(F32)).astype(np.float64)


def test_exp_f32_within_two_ulps():
    x = np.linspace(-87.0, 88.7, 400001).astype(F32)
    assert ulps(M.exp_f32(x), np.exp(x.astype(np.float64))).max() <= 2.0
    e = M.exp_f32(np.array([0.0, 1.0, -1.0, 89.5, -90.0], F32))
    assert e[0] == 1.0 and e[3] == np.inf and e[4] == 0.0
    assert ulps(e[1:3], np.exp([1.0, -1.0])).max() <= 1.0


def test_silu_f32_within_four_ulps():
    g = np.concatenate([np.linspace(-80, 80, 200001), -np.logspace(-30, 1.9, 2000), np.logspace(-30, 1.9, 2000)]).astype(F32)
    ref = g.astype(np.float64) / (1.0 + np.exp(-g.astype(np.float64)))
    got = M.silu_f32(g)
    nz = ref != 0
    assert ulps(got[nz], ref[nz]).max() <= 4.0
    s = M.silu_f32(np.array([0.0, 100.0, -0.0], F32))
    assert s[0] == 0.0 and s[1] == 100.0 and s[2] == 0.0


def test_swiglu_bf16_is_the_definition_rounded_once():
    h = F.bf16_bits_to_f32(synth.activations((64, 512), seed=61, outlier_frac=0.02, outlier_mult=8.0))
    inter = 256
    y = M.swiglu_bf16(h, inter).astype(np.float64)
    gate, up = h[:, :inter].astype(np.float64), h[:, inter:].astype(np.float64)
    exact = gate / (1.0 + np.exp(-gate)) * up
    ref = F.round_to_bf16(exact)
    diff = y != ref
    # differences only where the exact value sits within float32 error of a BF16 tie: one BF16 ulp
    assert diff.mean() < 1e-3
    assert np.all(np.abs(y[diff] - ref[diff]) <= bf16_ulp(ref[diff]))
    # every value is a BF16 number
    assert np.array_equal(F.round_to_bf16(y), y)


def test_swiglu_layout_gate_then_up():
    inter = 32
    h = np.zeros((2, 2 * inter), F32)
    h[0, :inter] = 0.0            # gate 0 -> silu 0 -> y 0 whatever up is
    h[0, inter:] = 5.0
    h[1, :inter] = 20.0           # silu(20) = 20 (to float32) -> y = 20 * up
    h[1, inter:] = 0.5
    y = M.swiglu_bf16(h, inter)
    assert np.all(y[0] == 0.0)
    assert np.all(y[1] == 10.0)
    # the swapped reading (silu(up) * gate) would give silu(5)*0 = 0 and silu(0.5)*20 != 10
    assert M.silu_f32(np.float32(0.5)) * 20 != 10.0


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
