"""GPU quantisers vs the CPU oracle: codes and scales must match bit for bit.

Cases: the tiny blockwise-linear operands, the full 8192x4096 quantise
sweep (every granularity, row-wise, transposed and dual outputs), ragged
groups and tiles, strided input rows, empty input, all-zero and extreme
magnitude tensors, and a sweep of every BF16 bit pattern.  NVFP4 runs in
four forms: one outer scale per tensor or per row, each with and without
four-over-six block scales.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import formats as OF
from oracle import quantize as OQ
from tests._util import np_f32, np_u8, to_dev_bf16, to_f32

pytestmark = pytest.mark.gpu

fp = pytest.importorskip("fp8_block_scaled_03_gb300")

ROW_ORACLE = {
    "per_tensor": OQ.quantize_per_tensor,
    "1x128": OQ.quantize_1x128,
    "128x128": OQ.quantize_128x128,
    "mxfp8": OQ.quantize_mxfp8,
    "1x128_pow2": OQ.quantize_1x128_pow2,
    "128x128_pow2": OQ.quantize_128x128_pow2,
}
BYTE_SCALES = ("mxfp8", "1x128_pow2", "128x128_pow2")


@pytest.fixture(scope="module", autouse=True)
def built():
    from fp8_block_scaled_03_gb300 import build
    build.build()
    fp.load_library()
    assert torch.cuda.is_available()


def nv_form(gran):
    """'nvfp4', 'nvfp4_row', optionally '+4o6': (library gran, flags, oracle kwargs)."""
    base, _, opt = gran.partition("+")
    fos = opt == "4o6"
    return base, (fp.FLAG_NVFP4_4OVER6 if fos else 0), {"row_scaled": base == "nvfp4_row", "four_over_six": fos}


def check_rowwise(bits, gran, x_dev=None):
    x = to_f32(bits)
    xd = x_dev if x_dev is not None else to_dev_bf16(bits)
    if gran.startswith("nvfp4"):
        base, flags, kw = nv_form(gran)
        q, s, ts = fp.fp8_quantize(xd, base, flags=flags)
        torch.cuda.synchronize()
        pq, sb, sg = OQ.quantize_nvfp4(x, **kw)
        assert np.array_equal(np_u8(q), pq), f"{gran}: {(np_u8(q) != pq).sum()} code bytes differ"
        assert np.array_equal(np_u8(s), sb), f"{gran}: {(np_u8(s) != sb).sum()} block scales differ"
        assert np.array_equal(np_f32(ts), np.atleast_1d(np.asarray(sg, dtype=np.float32)))
        return
    q, s, ts = fp.fp8_quantize(xd, gran)
    torch.cuda.synchronize()
    rq, rs = ROW_ORACLE[gran](x)
    assert np.array_equal(np_u8(q), rq), f"{gran}: {(np_u8(q) != rq).sum()} codes differ"
    if gran in BYTE_SCALES:
        assert np.array_equal(np_u8(s), rs)
    else:
        assert np.array_equal(np_f32(s).reshape(np.shape(rs)), np.asarray(rs, dtype=np.float32))


def check_transposed(bits, gran, dual):
    x = to_f32(bits)
    xd = to_dev_bf16(bits)
    qt, st, q, s = fp.fp8_quantize_transposed(xd, gran, also_rowwise=dual)
    torch.cuda.synchronize()
    rq, rs = OQ.transposed(ROW_ORACLE[gran], x)
    assert np.array_equal(np_u8(qt), rq), f"{gran}^T: {(np_u8(qt) != rq).sum()} codes differ"
    if gran in BYTE_SCALES:
        assert np.array_equal(np_u8(st), rs)
    else:
        assert np.array_equal(np_f32(st).reshape(np.shape(rs)), np.asarray(rs, dtype=np.float32))
    if dual:
        rq2, rs2 = ROW_ORACLE[gran](x)
        assert np.array_equal(np_u8(q), rq2)
        if gran in BYTE_SCALES:
            assert np.array_equal(np_u8(s), rs2)
        else:
            assert np.array_equal(np_f32(s).reshape(np.shape(rs2)), np.asarray(rs2, dtype=np.float32))


GRANS = ["per_tensor", "1x128", "128x128", "mxfp8", "1x128_pow2", "128x128_pow2"]
NV = ["nvfp4", "nvfp4_row", "nvfp4+4o6", "nvfp4_row+4o6"]


# -------------------------------------------------------------- tiny blockwise linear operands
def test_tiny_linear_operands():
    x = synth.activations((128, 256), seed=0, outlier_frac=0.01, outlier_mult=50.0)
    w = synth.weights((256, 256), seed=1, std=0.02)
    check_rowwise(x, "1x128")
    check_rowwise(w, "128x128")


# -------------------------------------------------------------- full-size quantise sweep
@pytest.fixture(scope="module")
def sweep_bits():
    return synth.activations((8192, 4096), seed=0, outlier_frac=0.001, outlier_mult=100.0)


@pytest.mark.parametrize("gran", GRANS + NV)
def test_sweep_rowwise(sweep_bits, gran):
    check_rowwise(sweep_bits, gran)


@pytest.mark.parametrize("gran", GRANS)
def test_sweep_transposed_dual(sweep_bits, gran):
    check_transposed(sweep_bits, gran, dual=True)


# -------------------------------------------------------------- shapes and edge cases
@pytest.mark.parametrize("gran", GRANS + NV)
@pytest.mark.parametrize("shape", [(1, 16), (3, 200), (130, 264), (257, 1032), (64, 4096), (5, 5136)])
def test_ragged_rowwise(gran, shape):
    if gran.startswith("nvfp4") and shape[1] % 16:
        pytest.skip("NVFP4 needs cols % 16")
    bits = synth.activations(shape, seed=sum(shape), outlier_frac=0.02, outlier_mult=80.0)
    check_rowwise(bits, gran)


@pytest.mark.parametrize("gran", GRANS)
@pytest.mark.parametrize("dual", [False, True])
@pytest.mark.parametrize("shape", [(16, 8), (144, 200), (272, 392), (128, 128)])
def test_ragged_transposed(gran, dual, shape):
    bits = synth.activations(shape, seed=3 * sum(shape), outlier_frac=0.02, outlier_mult=80.0)
    check_transposed(bits, gran, dual)


@pytest.mark.parametrize("gran", GRANS + NV)
def test_strided_rows(gran):
    bits = synth.activations((96, 384), seed=5)
    big = torch.zeros((96, 512), dtype=torch.bfloat16, device="cuda")
    big[:, :384] = to_dev_bf16(bits)
    check_rowwise(bits, gran, x_dev=big[:, :384])


@pytest.mark.parametrize("gran", GRANS + NV)
def test_zero_and_extreme_tensors(gran):
    zeros = np.zeros((64, 256), dtype=np.uint16)
    zeros[3, 7] = 0x8000                                   # a negative zero
    check_rowwise(zeros, gran)
    g = np.random.Generator(np.random.PCG64(9))
    extreme = np.where(g.random((64, 256)) < 0.5,
                       synth.f32_to_bf16_bits(g.standard_normal((64, 256)).astype(np.float32) * np.float32(3e37)),
                       synth.f32_to_bf16_bits(g.standard_normal((64, 256)).astype(np.float32) * np.float32(1e-38)))
    check_rowwise(extreme.astype(np.uint16), gran)
    tiny = synth.f32_to_bf16_bits(g.standard_normal((64, 256)).astype(np.float32) * np.float32(1e-39))
    check_rowwise(tiny, gran)


@pytest.mark.parametrize("gran", GRANS)
@pytest.mark.parametrize("dual", [False, True])
def test_zero_and_extreme_tensors_transposed(gran, dual):
    """The transposed (and dual) path on all-zero tiles with a negative zero,
    on values near float32's top and bottom, and on BF16 subnormals: the
    tiles and columns whose scale leaves the reciprocal fast path."""
    zeros = np.zeros((64, 256), dtype=np.uint16)
    zeros[3, 7] = 0x8000
    check_transposed(zeros, gran, dual)
    g = np.random.Generator(np.random.PCG64(19))
    extreme = np.where(g.random((64, 256)) < 0.5,
                       synth.f32_to_bf16_bits(g.standard_normal((64, 256)).astype(np.float32) * np.float32(3e37)),
                       synth.f32_to_bf16_bits(g.standard_normal((64, 256)).astype(np.float32) * np.float32(1e-38)))
    check_transposed(extreme.astype(np.uint16), gran, dual)
    tiny = synth.f32_to_bf16_bits(g.standard_normal((64, 256)).astype(np.float32) * np.float32(1e-39))
    check_transposed(tiny, gran, dual)
    # one tile of ordinary values beside a tile of subnormals, in the same rows and columns
    mixed = synth.activations((128, 256), seed=20).copy()
    mixed[:, 128:] = tiny[:64].repeat(2, axis=0)[:, :128]
    check_transposed(mixed, gran, dual)


def test_every_bf16_pattern_transposed():
    """All finite BF16 patterns through the transposed and dual path (rows a
    multiple of 16, as the transposed entry point requires)."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = allbits[(allbits & 0x7F80) != 0x7F80]
    g = np.random.Generator(np.random.PCG64(21))
    perm = finite[g.permutation(finite.size)]
    n = (perm.size // (16 * 256)) * 16 * 256
    parts = [perm[:n].reshape(-1, 256), np.resize(perm[n:], (16, 256))]
    for bits in parts:
        for gran in GRANS:
            check_transposed(bits, gran, dual=True)


def test_given_tensor_scale_transposed():
    """A supplied per-tensor scale divides exactly (IEEE) on the transposed
    path too, for X^T and X."""
    bits = synth.activations((64, 256), seed=22)
    x = to_f32(bits)
    xd = to_dev_bf16(bits)
    qt, st, q, s = fp.fp8_quantize_transposed(xd, "per_tensor", True,
                                              scales_t=torch.tensor([0.125], dtype=torch.float32, device="cuda"),
                                              flags=fp.FLAG_GIVEN_TENSOR_SCALE)
    assert np.array_equal(np_u8(qt), OQ.cast_e4m3(np.ascontiguousarray(x.T), np.float32(0.125)))
    assert np.array_equal(np_u8(q), OQ.cast_e4m3(x, np.float32(0.125)))
    assert fp.read_status() == 0


def test_every_bf16_pattern():
    """All 65536 BF16 bit patterns except inf/NaN, in several group contexts."""
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = allbits[(allbits & 0x7F80) != 0x7F80]
    g = np.random.Generator(np.random.PCG64(10))
    perm = finite[g.permutation(finite.size)]
    n = (perm.size // 512) * 512
    bits = perm[:n].reshape(-1, 512)
    for gran in GRANS + NV:
        check_rowwise(bits, gran)
    # every pattern with |x| <= 448 under a scale of exactly 1 (amax 448 in every group)
    small = finite[(finite & 0x7FFF) <= 0x43E0]
    small = small[g.permutation(small.size)]
    fixed = small[: (small.size // 512) * 512].reshape(-1, 512).copy()
    fixed[:, ::32] = 0x43E0                                 # 448.0
    for gran in ("1x128", "mxfp8"):
        check_rowwise(fixed, gran)


def test_empty_is_noop():
    x = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    q, s, _ = fp.fp8_quantize(x, "1x128")
    assert q.shape == (0, 128)


def test_given_tensor_scale():
    bits = synth.activations((64, 256), seed=12)
    x = to_f32(bits)
    xd = to_dev_bf16(bits)
    s_in = torch.tensor([0.125], dtype=torch.float32, device="cuda")
    q, s, _ = fp.fp8_quantize(xd, "per_tensor", scales=s_in.clone(), flags=fp.FLAG_GIVEN_TENSOR_SCALE)
    assert np.array_equal(np_u8(q), OQ.cast_e4m3(x, np.float32(0.125)))
    sg = torch.tensor([np.float32(0.01)], dtype=torch.float32, device="cuda")
    pq, sb, _ = fp.fp8_quantize(xd, "nvfp4", tensor_scale=sg, flags=fp.FLAG_GIVEN_TENSOR_SCALE)
    rq, rsb, _ = OQ.quantize_nvfp4(x, s_g=np.float32(0.01))
    assert np.array_equal(np_u8(pq), rq) and np.array_equal(np_u8(sb), rsb)


def test_given_row_scales_and_shared_gate_up_scale():
    """Per-row outer scales supplied by the caller; and gate and up weights
    quantised separately with one shared outer scale equal the quantisation
    of their concatenation (one outer weight scale for the fused GEMM)."""
    bits = synth.activations((48, 256), seed=13, outlier_frac=0.02, outlier_mult=30.0)
    x = to_f32(bits)
    xd = to_dev_bf16(bits)
    g = np.random.Generator(np.random.PCG64(14))
    rs = (g.uniform(0.5, 2.0, 48) * 0.01).astype(np.float32)
    for flags, fos in ((0, False), (fp.FLAG_NVFP4_4OVER6, True)):
        ts = torch.from_numpy(rs.copy()).cuda()
        pq, sb, _ = fp.fp8_quantize(xd, "nvfp4_row", tensor_scale=ts, flags=flags | fp.FLAG_GIVEN_TENSOR_SCALE)
        rq, rsb, _ = OQ.quantize_nvfp4(x, s_g=rs, row_scaled=True, four_over_six=fos)
        assert np.array_equal(np_u8(pq), rq) and np.array_equal(np_u8(sb), rsb)
        assert np.array_equal(np_f32(ts), rs)                      # an input: left untouched
    gate = synth.weights((96, 256), seed=15)
    up = synth.weights((96, 256), seed=16, std=0.05)
    both = np.concatenate([gate, up])
    for flags, fos in ((0, False), (fp.FLAG_NVFP4_4OVER6, True)):
        qc, sc, tc = fp.fp8_quantize(to_dev_bf16(both), "nvfp4", flags=flags)
        shared = tc.clone()
        qg, sg_, _ = fp.fp8_quantize(to_dev_bf16(gate), "nvfp4", tensor_scale=shared.clone(),
                                     flags=flags | fp.FLAG_GIVEN_TENSOR_SCALE)
        qu, su, _ = fp.fp8_quantize(to_dev_bf16(up), "nvfp4", tensor_scale=shared.clone(),
                                    flags=flags | fp.FLAG_GIVEN_TENSOR_SCALE)
        assert torch.equal(torch.cat([qg, qu]), qc) and torch.equal(torch.cat([sg_, su]), sc)
        _, _, rsg = OQ.quantize_nvfp4(to_f32(both), four_over_six=fos)
        assert np_f32(tc)[0] == rsg


def test_nvfp4_full_size_activation_rows():
    """The 16384 x 5120 NVFP4 activation of the dense FP4 linear, per-row and
    per-tensor outer scales, with and without four-over-six: every outer
    scale, and all codes of sampled rows (the oracle quantises just those
    rows; a row's result depends only on the row and the outer scale)."""
    bits = synth.activations((16384, 5120), seed=5, outlier_frac=0.01, outlier_mult=50.0)
    xd = to_dev_bf16(bits)
    rows = np.unique(np.concatenate([[0, 1, 16383], np.random.Generator(np.random.PCG64(6)).integers(0, 16384, 60)]))
    x_all = to_f32(bits)
    x_s = x_all[rows]
    for gran in NV:
        base, flags, kw = nv_form(gran)
        q, s, ts = fp.fp8_quantize(xd, base, flags=flags)
        torch.cuda.synchronize()
        if kw["row_scaled"]:
            sg_all = OQ.nvfp4_row_scales(x_all, kw["four_over_six"])
            assert np.array_equal(np_f32(ts), sg_all)
            sg_s = sg_all[rows]
        else:
            sg_s = OQ.nvfp4_tensor_scale(x_all, kw["four_over_six"])
            assert np_f32(ts)[0] == sg_s
        rq, rsb, _ = OQ.quantize_nvfp4(x_s, s_g=sg_s, **kw)
        idx = torch.from_numpy(rows).cuda()
        assert np.array_equal(np_u8(q.index_select(0, idx)), rq)
        assert np.array_equal(np_u8(s.index_select(0, idx)), rsb)


def test_fp32_scale_division_matches_ieee_codes_exhaustively():
    """The FP32-scale casts divide by a reciprocal plus one correction step
    instead of an IEEE division per element.  Over the whole domain (every
    positive BF16 amax, S = amax / 448, every BF16 x with |x| <= amax) the
    E4M3 codes must equal those of the IEEE quotient."""
    pairs, bad, fast = fp.test_quotient_sweep()
    assert bad == 0
    assert pairs > 1_000_000_000
    assert fast > 26_000          # every amax >= 2^-80 takes the fast path



def test_fp32_scales_without_ieee_operations_match_exhaustively():
    """The FP32-scale casts take S = RN(amax / 448) and RN(1/S) without
    IEEE division or reciprocal for amax >= 2^-79; for every finite BF16
    amax both must be bit-identical to the IEEE results."""
    values, bad, fast = fp.test_quotient_sweep(nvfp4=3)
    assert values == 0x7F80
    assert bad == 0
    assert fast > 26_000


def test_nvfp4_block_scale_codes_match_ieee_exhaustively():
    """The NVFP4 block scale code E4M3(RN(RN(a / 6) / S_g)) (and the
    four-over-six a / 4 form) is taken without IEEE division on the fast
    path.  Over every BF16 tensor amax, both outer divisors and every BF16
    block amax a <= amax_T the codes must equal the IEEE ones, and RN(a / 6)
    itself must be bit-exact for every BF16 a."""
    pairs, bad, fast = fp.test_quotient_sweep(nvfp4=2)
    assert bad == 0
    assert pairs > 1_000_000_000
    assert fast > 50_000          # both divisors, every amax_T down to about 2^-76


def test_nvfp4_block_division_matches_ieee_codes_exhaustively():
    """NVFP4 divides each block by S_b = E4M3value * S_g the same way; over
    every amax_T, both outer divisors, every block scale code and every BF16
    x with |x| <= amax_T the E2M1 codes must equal the IEEE quotient's."""
    pairs, bad, fast = fp.test_quotient_sweep(nvfp4=True)
    assert bad == 0
    assert pairs > 100_000_000_000
    assert fast > 1_000_000


def test_encoder_breakpoints_match_the_oracle():
    """Both casts are monotone in |x|, so they are fixed by where they change
    code.  The device finds, through the quantisers' own packed casts and for
    both signs, the smallest float32 magnitude giving each nonzero code
    magnitude (E4M3: 126, E2M1: 7); the oracle's encoder must give exactly
    that code there and the code below it one float32 step lower.  The
    device also checks that both casts are monotone and sign-symmetric over
    all 2^31 finite magnitudes; with equal breakpoints that makes them the
    oracle's casts on every finite float32."""
    out = fp.test_encoder_breakpoints()
    bp, violations = out[:266], out[266]
    assert violations == 0                       # monotone and sign-symmetric on every finite float32
    assert 0xFFFFFFFF not in bp                  # lanes agreed, signs right
    sections = ((0, 126, OF.e4m3_encode, 0x7F, 1.0), (126, 126, OF.e4m3_encode, 0x7F, -1.0),
                (252, 7, OF.e2m1_encode, 0x7, 1.0), (259, 7, OF.e2m1_encode, 0x7, -1.0))
    for start, count, enc, mask, sign in sections:
        bits = np.array(bp[start:start + count], dtype=np.uint32)
        assert np.all(np.diff(bits.astype(np.int64)) > 0)          # strictly increasing breakpoints
        at = bits.view(np.float32) * np.float32(sign)
        below = (bits - 1).view(np.float32) * np.float32(sign)
        c = np.arange(1, count + 1)
        assert np.array_equal(enc(at) & mask, c), (start, bits)
        assert np.array_equal(enc(below) & mask, c - 1), (start, bits)
    # spot values from the formats: just above 2^-10 (half of E4M3's
    # smallest subnormal, a tie to the even code 0); 432 (the midpoint of
    # 416 and 448) goes up to the even 448; E2M1 0.25 -> 0, 0.75 -> 1.0
    f = lambda b: float(np.uint32(b).view(np.float32))
    assert f(bp[0]) == float(np.nextafter(np.float32(2.0 ** -10), np.float32(1)))
    assert f(bp[125]) == 432.0
    assert f(bp[252]) == float(np.nextafter(np.float32(0.25), np.float32(1)))
    assert f(bp[253]) == 0.75
