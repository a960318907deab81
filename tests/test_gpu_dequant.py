"""GPU BF16 dequantisation vs the oracle, bit for bit.

The GPU dequantises the oracle's own codes and scales (uploaded to the
device), so these tests look at the dequantiser alone: every output must
be the exact value code x block scale (x outer scale for NVFP4) rounded
once to BF16, as the oracle computes it in float64.  Cases: every
granularity on ragged shapes, scales built so that a float32 product
would round twice to the wrong BF16 value, scales and exponents at the
bottom of the float32 range (BF16 subnormal results), strided and empty
outputs, and the full 8192x4096 sweep tensor.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import formats as OF
from oracle import gemm as OG
from oracle import quantize as OQ
from tests._util import bf16_to_f64, to_f32

pytestmark = pytest.mark.gpu
fp = pytest.importorskip("fp8_block_scaled_03_gb300")

FP8_Q = {
    "per_tensor": OQ.quantize_per_tensor,
    "1x128": OQ.quantize_1x128,
    "128x128": OQ.quantize_128x128,
    "mxfp8": OQ.quantize_mxfp8,
    "1x128_pow2": OQ.quantize_1x128_pow2,
    "128x128_pow2": OQ.quantize_128x128_pow2,
}
NV = {"nvfp4": {}, "nvfp4_row": {"row_scaled": True}, "nvfp4+4o6": {"four_over_six": True},
      "nvfp4_row+4o6": {"row_scaled": True, "four_over_six": True}}


@pytest.fixture(scope="module", autouse=True)
def built():
    from fp8_block_scaled_03_gb300 import build
    build.build()
    fp.load_library()


def dev(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(np.atleast_1d(np.asarray(a, dtype=dtype)))).cuda()


def oracle_operand(x, gran):
    """Oracle codes and scales, their device copies, and the oracle's BF16 dequantisation."""
    if gran in FP8_Q:
        c, s = FP8_Q[gran](x)
        sdt = np.uint8 if np.asarray(s).dtype == np.uint8 else np.float32
        ref = OG.dequantize_bf16(c, s, gran)
        return gran, dev(c, np.uint8), dev(s, sdt), None, ref
    kw = NV[gran]
    p, sb, sg = OQ.quantize_nvfp4(x, **kw)
    ref = OG.dequantize_bf16(p, sb, "nvfp4", s_g=sg)
    base = "nvfp4_row" if kw.get("row_scaled") else "nvfp4"
    return base, dev(p, np.uint8), dev(sb, np.uint8), dev(sg, np.float32), ref


@pytest.mark.parametrize("gran", list(FP8_Q) + list(NV))
@pytest.mark.parametrize("shape", [(1, 16), (3, 200), (130, 264), (257, 1032), (64, 4096)])
def test_dequant_matches_oracle(gran, shape):
    if gran.startswith("nvfp4") and shape[1] % 16:
        pytest.skip("NVFP4 needs cols % 16")
    x = to_f32(synth.activations(shape, seed=7 * sum(shape), outlier_frac=0.02, outlier_mult=80.0))
    g, qd, sd, td, ref = oracle_operand(x, gran)
    d = fp.fp8_dequantize(qd, sd, g, cols=shape[1], tensor_scale=td)
    torch.cuda.synchronize()
    got = bf16_to_f64(d)
    assert np.array_equal(got, ref), f"{gran}: {(got != ref).sum()} values differ"


def _all_codes_rows(n_rows):
    """Every finite E4M3 code (NaN codes 0x7F / 0xFF left out), twice padded to 256."""
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F] + [0, 0], dtype=np.uint8)
    return np.tile(codes, (n_rows, 1))


def test_dequant_single_rounding_scales():
    """1x128 scales (one per row, both groups): random scales; scales that put
    code x S just above a BF16 rounding tie by less than half a float32 ulp
    (a float32 product would round to the tie and then to even); and scales
    at the bottom of float32, subnormals included, whose results are BF16
    subnormals."""
    g = np.random.Generator(np.random.PCG64(41))
    scales = [np.float32(g.uniform(0.5, 2.0)) * np.float32(2.0 ** int(g.integers(-30, 30))) for _ in range(64)]
    for c in (1.125, 1.375, 1.625, 1.875, 3.5, 7.0, 13.0, 26.0):
        for d_ in (2.0 ** -26, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -27, -(2.0 ** -26)):
            scales.append(np.float32((1 + 2.0 ** -8 + d_) / c))
    for e in (-100, -101, -110, -118, -126, -127, -130, -135, -140, -149):
        scales += [np.float32(np.ldexp(1.0, e)), np.float32(np.ldexp(1.37, e)), np.float32(np.ldexp(1.0 + 2.0 ** -20, e))]
    s = np.array(scales, dtype=np.float32)
    s = s[s > 0]
    codes = _all_codes_rows(s.size)
    s2 = np.repeat(s[:, None], 2, axis=1)
    d = fp.fp8_dequantize(dev(codes, np.uint8), dev(s2, np.float32), "1x128")
    torch.cuda.synchronize()
    got = bf16_to_f64(d)
    ref = OG.dequantize_bf16(codes, s2, "1x128")
    assert np.array_equal(got, ref), f"{(got != ref).sum()} values differ"
    # the case set does reach values where rounding a float32 product would be wrong
    via_f32 = OF.round_to_bf16(OG.DEQUANT["1x128"](codes, s2).astype(np.float32).astype(np.float64))
    assert (via_f32 != ref).any()


def test_dequant_extreme_ue8m0_bytes():
    """MXFP8 scale bytes from 2^-127 upwards, every finite code."""
    e8 = np.array([0, 1, 2, 5, 10, 20, 60, 100, 127, 150, 200, 240, 245], dtype=np.uint8)
    codes = _all_codes_rows(e8.size)
    sc = np.repeat(e8[:, None], 8, axis=1)                 # 256 columns / 32
    d = fp.fp8_dequantize(dev(codes, np.uint8), dev(sc, np.uint8), "mxfp8")
    torch.cuda.synchronize()
    assert np.array_equal(bf16_to_f64(d), OG.dequantize_bf16(codes, sc, "mxfp8"))


def test_dequant_strided_output_and_empty():
    x = to_f32(synth.activations((96, 384), seed=3))
    g, qd, sd, td, ref = oracle_operand(x, "1x128")
    big = torch.full((96, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    fp.fp8_dequantize(qd, sd, g, cols=384, out=big[:, :384])
    torch.cuda.synchronize()
    assert np.array_equal(bf16_to_f64(big[:, :384]), ref)
    assert torch.all(big[:, 384:] == 7.0)
    e = torch.empty((0, 128), dtype=torch.uint8, device="cuda")
    out = fp.fp8_dequantize(e, torch.empty((0, 1), dtype=torch.float32, device="cuda"), "1x128", cols=128)
    assert out.shape == (0, 128)


@pytest.mark.parametrize("gran", ["1x128", "128x128", "mxfp8", "nvfp4_row+4o6"])
def test_dequant_full_sweep_tensor(gran):
    x = to_f32(synth.activations((8192, 4096), seed=0, outlier_frac=0.001, outlier_mult=100.0))
    g, qd, sd, td, ref = oracle_operand(x, gran)
    d = fp.fp8_dequantize(qd, sd, g, cols=4096, tensor_scale=td)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_to_f64(d), ref)
