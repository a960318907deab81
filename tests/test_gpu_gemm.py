"""GPU block-scaled GEMMs vs the CPU oracle.

The oracle quantises the BF16 inputs itself (never the GPU's codes),
dequantises exactly in float64, multiplies in float64 and rounds once to
BF16.  The GPU output must satisfy, per compared block of outputs,
relative Frobenius error <= 1e-3 and every |error| <= max(2e-2 * rms(reference),
one BF16 ulp of the reference element): the reference is the exact sum rounded
once to BF16 and the GPU rounds its FP32 sum to BF16, so near a rounding tie
two correct results differ by one output ulp, which for elements above about
2.5 rms exceeds 2e-2 * rms (tests/_util.py, assert_gemm_close).
Small and ragged shapes are compared in full; the full-size linear-layer
workloads on sampled rows and columns (the oracle quantises just the
operand rows those outputs depend on; 128x128 weight blocks in full).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import formats as OF
from oracle import gemm as OG
from oracle import quantize as OQ
from tests._util import assert_gemm_close, bf16_to_f64, to_dev_bf16, to_f32

pytestmark = pytest.mark.gpu
fp = pytest.importorskip("fp8_block_scaled_03_gb300")

Q_FN = {"per_tensor": OQ.quantize_per_tensor, "1x128": OQ.quantize_1x128, "128x128": OQ.quantize_128x128}
DQ_FN = {"per_tensor": OG.dequant_per_tensor, "1x128": OG.dequant_1x128, "128x128": OG.dequant_128x128}


@pytest.fixture(scope="module", autouse=True)
def built():
    from fp8_block_scaled_03_gb300 import build
    build.build()
    fp.load_library()
    fp.clear_status()


def oracle_deq(x_f32, gran):
    c, s = Q_FN[gran](x_f32)
    return DQ_FN[gran](c, s)


def gpu_block_gemm(a_bits, a_gran, b_bits, b_gran):
    qa, sa, _ = fp.fp8_quantize(to_dev_bf16(a_bits), a_gran)
    qb, sb, _ = fp.fp8_quantize(to_dev_bf16(b_bits), b_gran)
    return fp.fp8_block_gemm(qa, sa, a_gran, qb, sb, b_gran)


# ------------------------------------------------------------------ FP32-scaled (blockwise) GEMM
def test_tiny_blockwise_linear():
    """X [128,256] 1x128 times W [256,256] 128x128, compared in full."""
    xb = synth.activations((128, 256), seed=0, outlier_frac=0.01, outlier_mult=50.0)
    wb = synth.weights((256, 256), seed=1, std=0.02)
    d = gpu_block_gemm(xb, "1x128", wb, "128x128")
    ref = OG.gemm_bf16(oracle_deq(to_f32(xb), "1x128"), oracle_deq(to_f32(wb), "128x128"))
    assert_gemm_close(bf16_to_f64(d), ref)
    assert fp.read_status() == 0


@pytest.mark.parametrize("a_gran,b_gran", [("1x128", "128x128"), ("1x128", "1x128"), ("128x128", "128x128"),
                                           ("per_tensor", "per_tensor"), ("per_tensor", "128x128"),
                                           ("128x128", "1x128"), ("1x128", "per_tensor")])
@pytest.mark.parametrize("m,n,k", [(300, 520, 384), (128, 256, 128), (1, 8, 256), (513, 264, 1024)])
def test_blockwise_modes_and_ragged_shapes(a_gran, b_gran, m, n, k):
    ab = synth.activations((m, k), seed=m + k, outlier_frac=0.01, outlier_mult=50.0)
    bb = synth.weights((n, k), seed=n + k + 1, std=0.02)
    d = gpu_block_gemm(ab, a_gran, bb, b_gran)
    ref = OG.gemm_bf16(oracle_deq(to_f32(ab), a_gran), oracle_deq(to_f32(bb), b_gran))
    assert_gemm_close(bf16_to_f64(d), ref)


@pytest.mark.parametrize("a_gran,b_gran", [("1x128", "128x128"), ("1x128", "1x128"), ("per_tensor", "128x128")])
@pytest.mark.parametrize("m,n,k", [(2048, 2304, 640), (129, 8, 128)])
def test_blockwise_partial_tiles(a_gran, b_gran, m, n, k):
    """Several tiles per CTA with a ragged last row and column tile, and a
    single row tile narrower than one N tile."""
    ab = synth.activations((m, k), seed=m + 2 * k, outlier_frac=0.01, outlier_mult=50.0)
    bb = synth.weights((n, k), seed=n + 3 * k, std=0.02)
    d = gpu_block_gemm(ab, a_gran, bb, b_gran)
    ref = OG.gemm_bf16(oracle_deq(to_f32(ab), a_gran), oracle_deq(to_f32(bb), b_gran))
    assert_gemm_close(bf16_to_f64(d), ref)
    assert fp.read_status() == 0


def test_blockwise_grouped_ragged_experts():
    """FP32-scale grouped GEMM with empty, one-row, ragged and multi-tile experts."""
    counts = [0, 1, 127, 129, 0, 3, 256, 300]
    n, k = 264, 384
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    rows, e = int(offsets[-1]), len(counts)
    ab = synth.activations((rows, k), seed=77, outlier_frac=0.01, outlier_mult=50.0)
    bb = synth.weights((e * n, k), seed=78)
    qa, sa, _ = fp.fp8_quantize(to_dev_bf16(ab), "1x128")
    qbs, sbs = [], []
    for i in range(e):
        q_, s_, _ = fp.fp8_quantize(to_dev_bf16(bb[i * n:(i + 1) * n]), "128x128")
        qbs.append(q_); sbs.append(s_)
    d = fp.fp8_grouped_gemm(qa, sa, torch.stack(qbs), torch.stack(sbs), torch.from_numpy(offsets).cuda(), "1x128")
    got = bf16_to_f64(d)
    a64 = oracle_deq(to_f32(ab), "1x128")
    for i in range(e):
        lo, hi = offsets[i], offsets[i + 1]
        if hi > lo:
            ref = OG.gemm_bf16(a64[lo:hi], oracle_deq(to_f32(bb[i * n:(i + 1) * n]), "128x128"))
            assert_gemm_close(got[lo:hi], ref)
    assert fp.read_status() == 0


def test_blockwise_many_tiles_persistent():
    """More tiles than SMs: every CTA walks several tiles and K blocks."""
    m, n, k = 2048, 2304, 640
    ab = synth.activations((m, k), seed=41)
    bb = synth.weights((n, k), seed=42)
    d = gpu_block_gemm(ab, "1x128", bb, "128x128")
    ref = OG.gemm_bf16(oracle_deq(to_f32(ab), "1x128"), oracle_deq(to_f32(bb), "128x128"))
    assert_gemm_close(bf16_to_f64(d), ref)
    assert fp.read_status() == 0


# ------------------------------------------------------------------ full-size dense linear, fwd + bwd
M3, H3, I3 = 8192, 2560, 9728


@pytest.fixture(scope="module")
def dense_inputs():
    x = synth.activations((M3, H3), seed=0, outlier_frac=0.01, outlier_mult=50.0)
    w = synth.weights((I3, H3), seed=1, std=0.02)
    dy = synth.activations((M3, I3), seed=2, outlier_frac=0.01, outlier_mult=50.0)
    return x, w, dy


def sampled(rows_total, cols_total, seed, nr=48, nc=256):
    g = np.random.Generator(np.random.PCG64(seed))
    rows = np.sort(g.choice(rows_total, nr, replace=False))
    rows[-1] = rows_total - 1
    blocks = np.sort(g.choice(cols_total // 128, max(1, nc // 128), replace=False))
    return rows, blocks


def test_dense_fprop_dgrad_wgrad_sampled(dense_inputs):
    x, w, dy = dense_inputs
    xd, wd, dyd = to_dev_bf16(x), to_dev_bf16(w), to_dev_bf16(dy)
    # the step as the bench runs it: dual quantisers, then three GEMMs
    qxt, sxt, qx, sx = fp.fp8_quantize_transposed(xd, "1x128", also_rowwise=True)
    qwt, swt, qw, sw = fp.fp8_quantize_transposed(wd, "128x128", also_rowwise=True)
    qdyt, sdyt, qdy, sdy = fp.fp8_quantize_transposed(dyd, "1x128", also_rowwise=True)
    y = fp.fp8_block_gemm(qx, sx, "1x128", qw, sw, "128x128")
    dx = fp.fp8_block_gemm(qdy, sdy, "1x128", qwt, swt, "128x128")
    dw = fp.fp8_block_gemm(qdyt, sdyt, "1x128", qxt, sxt, "1x128")
    torch.cuda.synchronize()
    assert fp.read_status() == 0
    xf, wf, dyf = to_f32(x), to_f32(w), to_f32(dy)

    # fprop: rows of X, 128-row blocks of W
    rows, blocks = sampled(M3, I3, 10)
    a64 = oracle_deq(xf[rows], "1x128")
    for nb in blocks:
        b64 = oracle_deq(wf[nb * 128:(nb + 1) * 128], "128x128")
        assert_gemm_close(bf16_to_f64(y[torch.from_numpy(rows).cuda(), nb * 128:(nb + 1) * 128]),
                          OG.gemm_bf16(a64, b64))
    # dgrad: rows of dY, 128-row blocks of W^T (= 128-column blocks of W)
    rows, blocks = sampled(M3, H3, 11)
    a64 = oracle_deq(dyf[rows], "1x128")
    for nb in blocks:
        wt_blk = np.ascontiguousarray(wf[:, nb * 128:(nb + 1) * 128].T)
        b64 = oracle_deq(wt_blk, "128x128")
        assert_gemm_close(bf16_to_f64(dx[torch.from_numpy(rows).cuda(), nb * 128:(nb + 1) * 128]),
                          OG.gemm_bf16(a64, b64))
    # wgrad: rows of dY^T (= columns of dY), rows of X^T (= columns of X), both 1x128 along M
    rows, blocks = sampled(I3, H3, 12)
    a64 = oracle_deq(np.ascontiguousarray(dyf[:, rows].T), "1x128")
    for nb in blocks:
        b64 = oracle_deq(np.ascontiguousarray(xf[:, nb * 128:(nb + 1) * 128].T), "1x128")
        assert_gemm_close(bf16_to_f64(dw[torch.from_numpy(rows).cuda(), nb * 128:(nb + 1) * 128]),
                          OG.gemm_bf16(a64, b64))


# ------------------------------------------------------------------ MXFP8 (hardware block scale)
def mx_deq(x_f32):
    c, e = OQ.quantize_mxfp8(x_f32)
    return OG.dequant_mxfp8(c, e)


@pytest.mark.parametrize("m,n,k", [(128, 256, 128), (300, 520, 384), (1, 8, 128), (1000, 1536, 2048)])
def test_mxfp8_dense(m, n, k):
    ab = synth.activations((m, k), seed=m + 3, outlier_frac=0.001, outlier_mult=100.0)
    bb = synth.weights((n, k), seed=n + 4)
    qa, sa, _ = fp.fp8_quantize(to_dev_bf16(ab), "mxfp8")
    qb, sb, _ = fp.fp8_quantize(to_dev_bf16(bb), "mxfp8")
    d = fp.fp8_block_gemm(qa, sa, "mxfp8", qb, sb, "mxfp8")
    ref = OG.gemm_bf16(mx_deq(to_f32(ab)), mx_deq(to_f32(bb)))
    assert_gemm_close(bf16_to_f64(d), ref)
    assert fp.read_status() == 0


def grouped_case(counts, n, k, seed, gran="mxfp8"):
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    rows = int(offsets[-1])
    e = len(counts)
    ab = synth.activations((max(rows, 1), k), seed=seed, outlier_frac=0.001, outlier_mult=100.0)[:rows]
    bb = synth.weights((e * n, k), seed=seed + 1)
    qa, sa, _ = fp.fp8_quantize(to_dev_bf16(ab), gran)
    qb, sb, _ = fp.fp8_quantize(to_dev_bf16(bb), gran)
    off_d = torch.from_numpy(offsets).cuda()
    if gran == "mxfp8":
        d = fp.fp8_grouped_gemm(qa, sa, qb.view(e, n, k), sb.view(e, n, k // 32), off_d, "mxfp8")
    return ab, bb, offsets, d


@pytest.mark.parametrize("counts", [[0, 1, 127, 129, 0, 3, 256, 64], [300], [0, 0, 5], [128] * 16])
def test_mxfp8_grouped_ragged(counts):
    n, k = 264, 256
    ab, bb, offsets, d = grouped_case(counts, n, k, seed=len(counts) + sum(counts))
    a64 = mx_deq(to_f32(ab)) if ab.shape[0] else np.zeros((0, k))
    bs = [mx_deq(to_f32(bb[i * n:(i + 1) * n])) for i in range(len(counts))]
    ref = OG.grouped_gemm(a64, bs, offsets)
    got = bf16_to_f64(d)
    for e in range(len(counts)):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            assert_gemm_close(got[lo:hi], ref[lo:hi])
    assert fp.read_status() == 0


GROUPED_B_GRAN = {"mxfp8": "mxfp8", "1x128": "128x128", "1x128_pow2": "128x128_pow2"}


@pytest.mark.parametrize("gran", ["mxfp8", "1x128", "1x128_pow2"])
@pytest.mark.parametrize("case", ["past_end", "decreasing", "negative_first"])
def test_grouped_malformed_offsets_clamped(gran, case):
    """Offsets that break the contract must not reach outside D (a guard
    region after D stays untouched) and must set FP8BS_EOFFSETS; rows that
    the well-formed experts cover are computed as with correct offsets."""
    total, n, k, experts = 300, 256, 256, 4
    ab = synth.activations((total, k), seed=141)
    bb = synth.weights((experts * n, k), seed=142)
    qa, sa, _ = fp.fp8_quantize(to_dev_bf16(ab), gran)
    gb = GROUPED_B_GRAN[gran]
    qb, sb, _ = fp.fp8_quantize(to_dev_bf16(bb), gb)
    qb = qb.view(experts, n, k)
    sb = sb.view(experts, n, k // 32) if gb == "mxfp8" else sb.view(experts, n // 128, k // 128)
    good = torch.tensor([0, 100, 100, 250, total], dtype=torch.int64, device="cuda")
    fp.clear_status()
    ref = fp.fp8_grouped_gemm(qa, sa, qb, sb, good, gran)
    assert fp.read_status() == 0
    bad = {"past_end": [0, 100, 100, 250, total + 5000], "decreasing": [0, 200, 100, 250, total],
           "negative_first": [-64, 100, 100, 250, total]}[case]
    buf = torch.full((total + 64, n), 7.0, dtype=torch.bfloat16, device="cuda")
    fp.fp8_grouped_gemm(qa, sa, qb, sb, torch.tensor(bad, dtype=torch.int64, device="cuda"), gran, out=buf[:total])
    assert fp.read_status() == -8                                    # FP8BS_EOFFSETS
    fp.clear_status()
    assert torch.all(buf[total:] == 7.0), "rows after D were written"
    same = {"past_end": [(0, total)], "decreasing": [(0, 100), (250, total)], "negative_first": [(0, total)]}[case]
    for lo, hi in same:
        assert torch.equal(buf[lo:hi].view(torch.int16), ref[lo:hi].view(torch.int16))


def test_moe_grouped_full_size_sampled():
    """Qwen3-30B-A3B-shaped MoE: 16384 tokens, top-8 of 128 experts, gate+up
    [1536, 2048] and down [2048, 768] per expert; sampled experts and rows."""
    tokens, experts, hidden, inter = 16384, 128, 2048, 768
    token_index, offsets = synth.moe_routing(tokens, experts, 8, seed=0)
    x = synth.activations((tokens, hidden), seed=3, outlier_frac=0.001, outlier_mult=100.0)
    a_bits = x[token_index]
    w_gu = synth.weights((experts * 2 * inter, hidden), seed=4)
    h = synth.activations((a_bits.shape[0], inter), seed=5, outlier_frac=0.001, outlier_mult=100.0)
    w_dn = synth.weights((experts * hidden, inter), seed=6)
    off_d = torch.from_numpy(offsets).cuda()
    qa, sa, _ = fp.fp8_quantize(to_dev_bf16(a_bits), "mxfp8")
    qb, sb, _ = fp.fp8_quantize(to_dev_bf16(w_gu), "mxfp8")
    d_gu = fp.fp8_grouped_gemm(qa, sa, qb.view(experts, 2 * inter, hidden), sb.view(experts, 2 * inter, hidden // 32),
                               off_d, "mxfp8")
    qh, sh_, _ = fp.fp8_quantize(to_dev_bf16(h), "mxfp8")
    qd, sd, _ = fp.fp8_quantize(to_dev_bf16(w_dn), "mxfp8")
    d_dn = fp.fp8_grouped_gemm(qh, sh_, qd.view(experts, hidden, inter), sd.view(experts, hidden, inter // 32),
                               off_d, "mxfp8")
    torch.cuda.synchronize()
    assert fp.read_status() == 0
    counts = np.diff(offsets)
    g = np.random.Generator(np.random.PCG64(7))
    picks = list(g.choice(np.nonzero(counts)[0], 6, replace=False)) + [int(np.argmax(counts)), int(np.argmin(counts))]
    for e in picks:
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        rows = np.unique(np.concatenate([g.integers(lo, hi, 8), [lo, hi - 1]]))
        for d, a_src, w_src, n in ((d_gu, a_bits, w_gu, 2 * inter), (d_dn, h, w_dn, hidden)):
            a64 = mx_deq(to_f32(a_src[rows]))
            b64 = mx_deq(to_f32(w_src[e * n:(e + 1) * n]))
            assert_gemm_close(bf16_to_f64(d[torch.from_numpy(rows).cuda()]), OG.gemm_bf16(a64, b64))


# ------------------------------------------------------------------ NVFP4
def nv_deq(x_f32, s_g=None, **kw):
    p, sb, sg = OQ.quantize_nvfp4(x_f32, s_g=s_g, **kw)
    return OG.dequant_nvfp4(p, sb, sg)


@pytest.mark.parametrize("m,n,k", [(128, 256, 256), (300, 520, 512), (1, 8, 256), (1000, 1024, 2048)])
def test_nvfp4_dense(m, n, k):
    ab = synth.activations((m, k), seed=m + 5, outlier_frac=0.0)
    bb = synth.weights((n, k), seed=n + 6)
    qa, sa, ta = fp.fp8_quantize(to_dev_bf16(ab), "nvfp4")
    qb, sb, tb = fp.fp8_quantize(to_dev_bf16(bb), "nvfp4")
    d = fp.fp8_block_gemm(qa, sa, "nvfp4", qb, sb, "nvfp4", ta, tb, k=k)
    ref = OG.gemm_bf16(nv_deq(to_f32(ab)), nv_deq(to_f32(bb)))
    assert_gemm_close(bf16_to_f64(d), ref)
    assert fp.read_status() == 0


@pytest.mark.parametrize("fos", [False, True])
@pytest.mark.parametrize("m,n,k", [(128, 256, 256), (300, 520, 512), (1, 8, 256), (1000, 1024, 2048)])
def test_nvfp4_row_scaled_activation(m, n, k, fos):
    """Per-token outer scales on A (rows spanning six orders of magnitude),
    one outer scale on B; optionally four-over-six block scales on both."""
    ab = synth.activations((m, k), seed=m + 7, outlier_frac=0.01, outlier_mult=20.0)
    mag = np.float32(10.0) ** np.random.Generator(np.random.PCG64(m)).integers(-3, 3, m).astype(np.float32)
    af = to_f32(ab) * mag[:, None]
    ab = synth.f32_to_bf16_bits(af)
    bb = synth.weights((n, k), seed=n + 8)
    flags = fp.FLAG_NVFP4_4OVER6 if fos else 0
    qa, sa, ta = fp.fp8_quantize(to_dev_bf16(ab), "nvfp4_row", flags=flags)
    qb, sb, tb = fp.fp8_quantize(to_dev_bf16(bb), "nvfp4", flags=flags)
    assert ta.shape == (m,)
    d = fp.fp8_block_gemm(qa, sa, "nvfp4_row", qb, sb, "nvfp4", ta, tb, k=k)
    ref = OG.gemm_bf16(nv_deq(to_f32(ab), row_scaled=True, four_over_six=fos),
                       nv_deq(to_f32(bb), four_over_six=fos))
    # rows differ in scale by up to 1e5: compare each magnitude class on its own
    got = bf16_to_f64(d)
    for e in np.unique(mag):
        sel = mag == e
        assert_gemm_close(got[sel], ref[sel])
    assert fp.read_status() == 0


@pytest.mark.parametrize("form", ["nvfp4", "nvfp4_row+4o6"])
def test_nvfp4_full_size_sampled(form):
    """Qwen2.5-32B MLP-shaped NVFP4 linear: X [16384,5120], W [27648,5120];
    one outer activation scale, or per-token outer scales with four-over-six."""
    m, n, k = 16384, 27648, 5120
    a_gran, _, opt = form.partition("+")
    fos = opt == "4o6"
    flags = fp.FLAG_NVFP4_4OVER6 if fos else 0
    xb = synth.activations((m, k), seed=0, outlier_frac=0.0)
    wb = synth.weights((n, k), seed=1)
    qa, sa, ta = fp.fp8_quantize(to_dev_bf16(xb), a_gran, flags=flags)
    qb, sb, tb = fp.fp8_quantize(to_dev_bf16(wb), "nvfp4", flags=flags)
    d = fp.fp8_block_gemm(qa, sa, a_gran, qb, sb, "nvfp4", ta, tb, k=k)
    torch.cuda.synchronize()
    assert fp.read_status() == 0
    xf, wf = to_f32(xb), to_f32(wb)
    row = a_gran == "nvfp4_row"
    sg_x = OQ.nvfp4_row_scales(xf, fos) if row else OQ.nvfp4_tensor_scale(xf, fos)
    sg_w = OQ.nvfp4_tensor_scale(wf, fos)
    assert np.array_equal(ta.cpu().numpy(), np.atleast_1d(sg_x)) and float(tb.item()) == float(sg_w)
    g = np.random.Generator(np.random.PCG64(8))
    rows = np.sort(g.choice(m, 32, replace=False))
    cols = np.sort(g.choice(n, 512, replace=False))
    a64 = nv_deq(xf[rows], s_g=sg_x[rows] if row else sg_x, row_scaled=row, four_over_six=fos)
    b64 = nv_deq(wf[cols], s_g=sg_w, four_over_six=fos)
    got = bf16_to_f64(d[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()])
    assert_gemm_close(got, OG.gemm_bf16(a64, b64))


def nv_grouped_case(counts, n, k, seed, a_gran="nvfp4", fos=False):
    """Per-expert NVFP4 weights, each with its own outer scale (quantised one
    expert at a time), and the routed rows of A; returns what the oracle needs
    and the GPU output."""
    e = len(counts)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    rows = int(offsets[-1])
    flags = fp.FLAG_NVFP4_4OVER6 if fos else 0
    ab = synth.activations((rows, k), seed=seed, outlier_frac=0.01, outlier_mult=20.0)
    bb = synth.weights((e * n, k), seed=seed + 1)
    qa, sa, ta = fp.fp8_quantize(to_dev_bf16(ab), a_gran, flags=flags)
    qbs, sbs, tbs = [], [], []
    for i in range(e):
        qb, sb, tb = fp.fp8_quantize(to_dev_bf16(bb[i * n:(i + 1) * n]), "nvfp4", flags=flags)
        qbs.append(qb)
        sbs.append(sb)
        tbs.append(tb)
    d = fp.fp8_grouped_gemm(qa, sa, torch.stack(qbs), torch.stack(sbs), torch.from_numpy(offsets).cuda(), a_gran,
                            a_tensor_scale=ta, b_tensor_scale=torch.cat(tbs), k=k)
    torch.cuda.synchronize()
    return ab, bb, offsets, d


@pytest.mark.parametrize("counts", [[0, 1, 127, 129, 0, 3, 256, 64], [300], [0, 0, 5], [128] * 6])
@pytest.mark.parametrize("form", ["nvfp4", "nvfp4_row+4o6"])
def test_nvfp4_grouped_ragged(counts, form):
    """The NVFP4 recipe on a MoE ("Low Precision RL", table "Choose a
    precision"): each expert's weight has its own outer scale; A has one outer
    scale, or one per row with four-over-six blocks."""
    n, k = 264, 512
    a_gran, _, opt = form.partition("+")
    fos = opt == "4o6"
    ab, bb, offsets, d = nv_grouped_case(counts, n, k, seed=len(counts) * 7 + sum(counts), a_gran=a_gran, fos=fos)
    row = a_gran == "nvfp4_row"
    a64 = nv_deq(to_f32(ab), row_scaled=row, four_over_six=fos) if ab.shape[0] else np.zeros((0, k))
    bs = [nv_deq(to_f32(bb[i * n:(i + 1) * n]), four_over_six=fos) for i in range(len(counts))]
    ref = OG.grouped_gemm(a64, bs, offsets)
    got = bf16_to_f64(d)
    for e in range(len(counts)):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            if row:   # per-row outer scales: rows differ in magnitude, so compare row by row blocks
                for r0 in range(lo, hi, 64):
                    assert_gemm_close(got[r0:min(hi, r0 + 64)], ref[r0:min(hi, r0 + 64)])
            else:
                assert_gemm_close(got[lo:hi], ref[lo:hi])
    assert fp.read_status() == 0


def test_nvfp4_grouped_moe_full_size_sampled():
    """Qwen3-30B-A3B-shaped MoE in NVFP4: 16384 tokens, top-8 of 128 experts,
    gate+up [1536, 2048] per expert; per-token outer activation scales with
    four-over-six; sampled experts and rows against the oracle."""
    tokens, experts, hidden, inter = 16384, 128, 2048, 768
    token_index, offsets = synth.moe_routing(tokens, experts, 8, seed=0)
    x = synth.activations((tokens, hidden), seed=13, outlier_frac=0.001, outlier_mult=100.0)
    a_bits = x[token_index]
    w_gu = synth.weights((experts * 2 * inter, hidden), seed=14)
    flags = fp.FLAG_NVFP4_4OVER6
    qa, sa, ta = fp.fp8_quantize(to_dev_bf16(a_bits), "nvfp4_row", flags=flags)
    wd = to_dev_bf16(w_gu).view(experts, 2 * inter, hidden)
    qb = torch.empty((experts, 2 * inter, hidden // 2), dtype=torch.uint8, device="cuda")
    sb = torch.empty((experts, 2 * inter, hidden // 16), dtype=torch.uint8, device="cuda")
    tb = torch.empty((experts,), dtype=torch.float32, device="cuda")
    for e in range(experts):    # gate and up of one expert share one outer scale (their concatenation's)
        fp.fp8_quantize(wd[e], "nvfp4", q=qb[e], scales=sb[e], tensor_scale=tb[e:e + 1], flags=flags)
    off_d = torch.from_numpy(offsets).cuda()
    d = fp.fp8_grouped_gemm(qa, sa, qb, sb, off_d, "nvfp4_row", a_tensor_scale=ta, b_tensor_scale=tb, k=hidden)
    torch.cuda.synchronize()
    assert fp.read_status() == 0
    counts = np.diff(offsets)
    g = np.random.Generator(np.random.PCG64(17))
    picks = list(g.choice(np.nonzero(counts)[0], 5, replace=False)) + [int(np.argmax(counts))]
    for e in picks:
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        rows = np.unique(np.concatenate([g.integers(lo, hi, 8), [lo, hi - 1]]))
        a64 = nv_deq(to_f32(a_bits[rows]), row_scaled=True, four_over_six=True)
        b64 = nv_deq(to_f32(w_gu[e * 2 * inter:(e + 1) * 2 * inter]), four_over_six=True)
        got = bf16_to_f64(d[torch.from_numpy(rows).cuda()])
        ref = OG.gemm_bf16(a64, b64)
        for i in range(len(rows)):    # each row has its own outer scale
            assert_gemm_close(got[i:i + 1], ref[i:i + 1])


# ------------------------------------------------------------------ block-wise with power-of-two scales
P2_Q = {"1x128_pow2": OQ.quantize_1x128_pow2, "128x128_pow2": OQ.quantize_128x128_pow2}


def p2_deq(x_f32, gran):
    c, e = P2_Q[gran](x_f32)
    return OG.DEQUANT[gran](c, e)


@pytest.mark.parametrize("a_gran,b_gran", [("1x128_pow2", "128x128_pow2"), ("1x128_pow2", "1x128_pow2"),
                                           ("128x128_pow2", "128x128_pow2"), ("128x128_pow2", "1x128_pow2")])
# k = 1152 and 896: 9 and 7 K blocks, so the scale rows' pitch is not a multiple
# of 4 bytes and the rows start at every byte offset of a word
@pytest.mark.parametrize("m,n,k", [(300, 520, 384), (128, 256, 128), (1, 8, 256), (1000, 1536, 2048),
                                   (300, 520, 1152), (130, 264, 896)])
def test_pow2_blockwise(a_gran, b_gran, m, n, k):
    ab = synth.activations((m, k), seed=m + k + 9, outlier_frac=0.01, outlier_mult=50.0)
    bb = synth.weights((n, k), seed=n + k + 10, std=0.02)
    d = gpu_block_gemm(ab, a_gran, bb, b_gran)
    ref = OG.gemm_bf16(p2_deq(to_f32(ab), a_gran), p2_deq(to_f32(bb), b_gran))
    assert_gemm_close(bf16_to_f64(d), ref)
    assert fp.read_status() == 0


@pytest.mark.parametrize("k", [384, 1152])   # 1152: 9 K blocks, scale rows at every byte offset of a word
@pytest.mark.parametrize("counts", [[0, 1, 127, 129, 0, 3, 256, 64], [300], [128] * 12])
def test_pow2_grouped_ragged(counts, k):
    n = 264
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    rows, e = int(offsets[-1]), len(counts)
    ab = synth.activations((rows, k), seed=rows + 1, outlier_frac=0.01, outlier_mult=50.0)
    bb = synth.weights((e * n, k), seed=rows + 2)
    qa, sa, _ = fp.fp8_quantize(to_dev_bf16(ab), "1x128_pow2")
    qbs, sbs = [], []
    for i in range(e):   # per-expert 128x128 grids, stacked along the expert axis
        q_, s_, _ = fp.fp8_quantize(to_dev_bf16(bb[i * n:(i + 1) * n]), "128x128_pow2")
        qbs.append(q_); sbs.append(s_)
    qb, sb = torch.stack(qbs), torch.stack(sbs)
    d = fp.fp8_grouped_gemm(qa, sa, qb, sb, torch.from_numpy(offsets).cuda(), "1x128_pow2")
    got = bf16_to_f64(d)
    a64 = p2_deq(to_f32(ab), "1x128_pow2")
    for i in range(e):
        lo, hi = offsets[i], offsets[i + 1]
        if hi > lo:
            ref = OG.gemm_bf16(a64[lo:hi], p2_deq(to_f32(bb[i * n:(i + 1) * n]), "128x128_pow2"))
            assert_gemm_close(got[lo:hi], ref)
    assert fp.read_status() == 0


def test_pow2_dense_linear_sampled(dense_inputs):
    """The full-size fwd+bwd step on the power-of-two path, sampled outputs."""
    x, w, dy = dense_inputs
    xd, wd, dyd = to_dev_bf16(x), to_dev_bf16(w), to_dev_bf16(dy)
    qxt, sxt, qx, sx = fp.fp8_quantize_transposed(xd, "1x128_pow2", also_rowwise=True)
    qwt, swt, qw, sw = fp.fp8_quantize_transposed(wd, "128x128_pow2", also_rowwise=True)
    qdyt, sdyt, qdy, sdy = fp.fp8_quantize_transposed(dyd, "1x128_pow2", also_rowwise=True)
    y = fp.fp8_block_gemm(qx, sx, "1x128_pow2", qw, sw, "128x128_pow2")
    dx = fp.fp8_block_gemm(qdy, sdy, "1x128_pow2", qwt, swt, "128x128_pow2")
    dw = fp.fp8_block_gemm(qdyt, sdyt, "1x128_pow2", qxt, sxt, "1x128_pow2")
    torch.cuda.synchronize()
    assert fp.read_status() == 0
    xf, wf, dyf = to_f32(x), to_f32(w), to_f32(dy)
    rows, blocks = sampled(M3, I3, 20)
    a64 = p2_deq(xf[rows], "1x128_pow2")
    for nb in blocks:
        b64 = p2_deq(wf[nb * 128:(nb + 1) * 128], "128x128_pow2")
        assert_gemm_close(bf16_to_f64(y[torch.from_numpy(rows).cuda(), nb * 128:(nb + 1) * 128]),
                          OG.gemm_bf16(a64, b64))
    rows, blocks = sampled(M3, H3, 21)
    a64 = p2_deq(dyf[rows], "1x128_pow2")
    for nb in blocks:
        b64 = p2_deq(np.ascontiguousarray(wf[:, nb * 128:(nb + 1) * 128].T), "128x128_pow2")
        assert_gemm_close(bf16_to_f64(dx[torch.from_numpy(rows).cuda(), nb * 128:(nb + 1) * 128]),
                          OG.gemm_bf16(a64, b64))
    rows, blocks = sampled(I3, H3, 22)
    a64 = p2_deq(np.ascontiguousarray(dyf[:, rows].T), "1x128_pow2")
    for nb in blocks:
        b64 = p2_deq(np.ascontiguousarray(xf[:, nb * 128:(nb + 1) * 128].T), "1x128_pow2")
        assert_gemm_close(bf16_to_f64(dw[torch.from_numpy(rows).cuda(), nb * 128:(nb + 1) * 128]),
                          OG.gemm_bf16(a64, b64))
