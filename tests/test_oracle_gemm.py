"""Pins for the oracle's block-scaled GEMM (CPU only).

Checked against: a pure-Python triple loop that sums per K-block and applies
the two scales the way the blockwise GEMM is defined, an exact integer GEMM
(unit scales, small integer codes), PyTorch's float32->bfloat16 cast for the
output rounding, a per-expert loop for the grouped GEMM with ragged and
empty experts, and the quantisation error budget for the transposed
operands of dgrad and wgrad.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import formats as F
from oracle import gemm as G
from oracle import quantize as Q


def loop_block_gemm(qa, sa_of, qb, sb_of, k, kb=128):
    """D[m,n] = sum_kb sa(m,kb) * sb(n,kb) * sum_{k in kb} dec(qa) * dec(qb)."""
    m, n = qa.shape[0], qb.shape[0]
    out = np.zeros((m, n))
    ta, tb = F.E4M3_TABLE, F.E4M3_TABLE
    for i in range(m):
        for j in range(n):
            acc = 0.0
            for b in range(0, k, kb):
                part = 0.0
                for t in range(b, min(k, b + kb)):
                    part += float(ta[qa[i, t]]) * float(tb[qb[j, t]])
                acc += float(sa_of(i, b // kb)) * float(sb_of(j, b // kb)) * part
            out[i, j] = acc
    return out


def test_blockwise_gemm_matches_loops():
    x = F.bf16_bits_to_f32(synth.activations((3, 384), seed=21))
    w = F.bf16_bits_to_f32(synth.weights((5, 384), seed=22))
    qa, sa = Q.quantize_1x128(x)
    qb, sb = Q.quantize_128x128(w)
    ref = loop_block_gemm(qa, lambda i, b: sa[i, b], qb, lambda j, b: sb[j // 128, b], 384)
    d64 = G.gemm_f64(G.dequant_1x128(qa, sa), G.dequant_128x128(qb, sb))
    assert np.allclose(d64, ref, rtol=1e-12, atol=1e-15)
    assert np.array_equal(G.block_gemm(qa, sa, "1x128", qb, sb, "128x128"), F.round_to_bf16(d64))


def test_mxfp8_gemm_matches_loops():
    x = F.bf16_bits_to_f32(synth.activations((2, 96), seed=23))
    w = F.bf16_bits_to_f32(synth.weights((3, 96), seed=24))
    qa, ea = Q.quantize_mxfp8(x)
    qb, eb = Q.quantize_mxfp8(w)
    ref = loop_block_gemm(qa, lambda i, b: 2.0 ** (int(ea[i, b]) - 127),
                          qb, lambda j, b: 2.0 ** (int(eb[j, b]) - 127), 96, kb=32)
    d64 = G.gemm_f64(G.dequant_mxfp8(qa, ea), G.dequant_mxfp8(qb, eb))
    assert np.allclose(d64, ref, rtol=1e-12, atol=1e-15)


def test_nvfp4_gemm_matches_loops():
    x = F.bf16_bits_to_f32(synth.activations((2, 64), seed=25))
    w = F.bf16_bits_to_f32(synth.weights((3, 64), seed=26))
    pa, sba, ga = Q.quantize_nvfp4(x)
    pb, sbb, gb = Q.quantize_nvfp4(w)
    qa, qb = F.unpack_e2m1(pa), F.unpack_e2m1(pb)
    ref = np.zeros((2, 3))
    for i in range(2):
        for j in range(3):
            for t in range(64):
                ref[i, j] += (F.E2M1_TABLE[qa[i, t]] * F.E4M3_TABLE[sba[i, t // 16]] * float(ga)
                              * F.E2M1_TABLE[qb[j, t]] * F.E4M3_TABLE[sbb[j, t // 16]] * float(gb))
    d64 = G.gemm_f64(G.dequant_nvfp4(pa, sba, ga), G.dequant_nvfp4(pb, sbb, gb))
    assert np.allclose(d64, ref, rtol=1e-12, atol=1e-20)


def test_integer_gemm_is_exact():
    g = np.random.Generator(np.random.PCG64(27))
    ia = g.integers(-3, 4, size=(16, 256))
    ib = g.integers(-3, 4, size=(8, 256))
    qa = F.e4m3_encode(ia.astype(np.float32))
    qb = F.e4m3_encode(ib.astype(np.float32))
    ones_a = np.ones((16, 2), dtype=np.float32)
    ones_b = np.ones((1, 2), dtype=np.float32)
    d = G.block_gemm(qa, ones_a, "1x128", qb, ones_b, "128x128")
    want = ia @ ib.T                    # |want| <= 9*256 < 2^12; bf16 holds integers < 256 exactly
    small = np.abs(want) < 256
    assert np.array_equal(d[small], want[small].astype(np.float64))
    assert np.array_equal(d, F.round_to_bf16(want.astype(np.float64)))


def test_output_rounding_matches_torch_bf16():
    x = F.bf16_bits_to_f32(synth.activations((64, 256), seed=28))
    w = F.bf16_bits_to_f32(synth.weights((32, 256), seed=29))
    qa, sa = Q.quantize_1x128(x)
    qb, sb = Q.quantize_1x128(w)
    d64 = G.gemm_f64(G.dequant_1x128(qa, sa), G.dequant_1x128(qb, sb))
    d32 = d64.astype(np.float32)
    exact32 = d32.astype(np.float64) == d64       # values float32 holds exactly
    ref = torch.from_numpy(d32).to(torch.bfloat16).double().numpy()
    got = G.block_gemm(qa, sa, "1x128", qb, sb, "1x128")
    assert np.array_equal(got[exact32], ref[exact32])


def test_grouped_gemm_ragged_experts():
    counts = [0, 1, 127, 129, 0, 3]
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    rows = int(offsets[-1])
    x = F.bf16_bits_to_f32(synth.activations((rows, 64), seed=30))
    qa, ea = Q.quantize_mxfp8(x)
    a64 = G.dequant_mxfp8(qa, ea)
    bs = []
    for e in range(len(counts)):
        w = F.bf16_bits_to_f32(synth.weights((48, 64), seed=100 + e))
        qb, eb = Q.quantize_mxfp8(w)
        bs.append(G.dequant_mxfp8(qb, eb))
    d = G.grouped_gemm(a64, bs, offsets)
    for e in range(len(counts)):
        for r in range(int(offsets[e]), int(offsets[e + 1])):
            want = F.round_to_bf16(np.array([sum(a64[r, t] * bs[e][j, t] for t in range(64)) for j in range(48)]))
            assert np.allclose(d[r], want, rtol=2 ** -7, atol=0)


def test_transposed_operands_track_bf16_products():
    """dgrad = dY.W and wgrad = dY^T.X built from transposed quantisations stay
    within the quantisation error of the BF16 products (a transposed or
    mis-scaled operand would be off by O(1))."""
    x = F.bf16_bits_to_f32(synth.activations((256, 256), seed=31))
    w = F.bf16_bits_to_f32(synth.weights((384, 256), seed=32))
    dy = F.bf16_bits_to_f32(synth.activations((256, 384), seed=33))
    qdy, sdy = Q.quantize_1x128(dy)
    qwt, swt = Q.transposed(Q.quantize_128x128, w)
    dgrad = G.block_gemm(qdy, sdy, "1x128", qwt, swt, "128x128")
    qdyt, sdyt = Q.transposed(Q.quantize_1x128, dy)
    qxt, sxt = Q.transposed(Q.quantize_1x128, x)
    wgrad = G.block_gemm(qdyt, sdyt, "1x128", qxt, sxt, "1x128")
    for got, want in ((dgrad, dy.astype(np.float64) @ w), (wgrad, dy.astype(np.float64).T @ x)):
        rel = np.linalg.norm(got - want) / np.linalg.norm(want)
        assert rel < 0.05, rel


def rational_bf16(q):
    """Round a Fraction to the nearest BF16 value (ties to even), exactly."""
    from fractions import Fraction
    if q == 0:
        return 0.0
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 7)          # 8 significant bits
    n, r = divmod(a, quantum)
    n = int(n)
    if r * 2 > quantum or (r * 2 == quantum and n % 2 == 1):
        n += 1
    return sign * float(n * quantum)


def test_dequantize_bf16_single_rounding():
    """Each dequantised value is the exact code x scale rounded once to BF16,
    checked with rational arithmetic; the sample includes values where a
    float32 intermediate would round twice and land elsewhere."""
    from fractions import Fraction
    g = np.random.Generator(np.random.PCG64(41))
    codes = np.arange(0, 0x7F, dtype=np.uint8)[None, :]
    double_rounding_cases = 0
    # random scales, plus scales built so that code * S lands just above a
    # BF16 rounding tie by less than half a float32 ulp
    scales = [np.float32(g.uniform(0.5, 2.0)) * np.float32(2.0 ** g.integers(-20, 20)) for _ in range(200)]
    for c in (1.125, 1.375, 1.625, 1.875, 3.5, 7.0):
        for d_ in (2.0 ** -26, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -27):
            scales.append(np.float32((1 + 2.0 ** -8 + d_) / c))
    for s in scales:
        d = G.dequantize_bf16(codes, np.array(s, dtype=np.float32), "per_tensor")
        for c, v in zip(codes[0], d[0]):
            exact = Fraction(float(F.E4M3_TABLE[c])) * Fraction(float(s))
            assert v == rational_bf16(exact)
            via_f32 = F.round_to_bf16(np.float64(np.float32(F.E4M3_TABLE[c]) * s))
            double_rounding_cases += int(via_f32 != v)
    assert double_rounding_cases > 0
    # NVFP4 values: E2M1 x E4M3 x S_g, each rounded once
    x = F.bf16_bits_to_f32(synth.activations((2, 64), seed=40))
    p, sb, sg = Q.quantize_nvfp4(x)
    d = G.dequantize_bf16(p, sb, "nvfp4", s_g=sg)
    q = F.unpack_e2m1(p)
    for i in range(2):
        for j in range(64):
            exact = (Fraction(float(F.E2M1_TABLE[q[i, j]])) * Fraction(float(F.E4M3_TABLE[sb[i, j // 16]]))
                     * Fraction(float(sg)))
            assert d[i, j] == rational_bf16(exact)


def test_nvfp4_row_scaled_gemm_matches_loops():
    """Per-token outer scales on A (one S_g per row), one per tensor on B:
    D[i, j] = sum_t E2M1(qa) s_b(a) S_g[i] * E2M1(qb) s_b(b) S_g(B)."""
    x = F.bf16_bits_to_f32(synth.activations((3, 64), seed=42))
    x[1] *= np.float32(1e-2)
    w = F.bf16_bits_to_f32(synth.weights((2, 64), seed=43))
    for fos in (False, True):
        pa, sba, ga = Q.quantize_nvfp4(x, row_scaled=True, four_over_six=fos)
        pb, sbb, gb = Q.quantize_nvfp4(w, four_over_six=fos)
        assert ga.shape == (3,)
        qa, qb = F.unpack_e2m1(pa), F.unpack_e2m1(pb)
        ref = np.zeros((3, 2))
        for i in range(3):
            for j in range(2):
                for t in range(64):
                    ref[i, j] += (F.E2M1_TABLE[qa[i, t]] * F.E4M3_TABLE[sba[i, t // 16]] * float(ga[i])
                                  * F.E2M1_TABLE[qb[j, t]] * F.E4M3_TABLE[sbb[j, t // 16]] * float(gb))
        d64 = G.gemm_f64(G.dequant_nvfp4(pa, sba, ga), G.dequant_nvfp4(pb, sbb, gb))
        assert np.allclose(d64, ref, rtol=1e-12, atol=1e-20)
