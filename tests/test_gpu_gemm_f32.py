"""fp8_block_gemm with float32 output (FP8BS_OUT_F32) vs the CPU oracle.

The oracle quantises the BF16 inputs itself, dequantises exactly in float64
and multiplies in float64; that product is not rounded here, since the GPU
writes its float32 accumulator.  The bound per element follows from the
arithmetic: the accumulator is a float32 sum of the k exact products
deq(a_k) * deq(b_k), plus, on the FP32-scale path, two roundings per
128-wide K block (the scale product and the promoted partial) and, for
NVFP4, two for the outer scales.  Whatever the order of the additions, each
operation's rounding error is at most 2^-23 of its result (round to nearest
is 2^-24; 2^-23 also covers a tensor core that truncates), so

    |D - ref| <= (k + 3 k / 128 + 2) * 2^-23 * sum_k |deq(a_k) deq(b_k)|.

The float32 output rounded to BF16 must also equal the BF16 output bit for
bit: both epilogues start from the same accumulator.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import gemm as OG
from oracle import quantize as OQ
from tests._util import to_dev_bf16, to_f32

pytestmark = pytest.mark.gpu
fp = pytest.importorskip("fp8_block_scaled_03_gb300")

Q = {"per_tensor": OQ.quantize_per_tensor, "1x128": OQ.quantize_1x128, "128x128": OQ.quantize_128x128,
     "mxfp8": OQ.quantize_mxfp8, "1x128_pow2": OQ.quantize_1x128_pow2, "128x128_pow2": OQ.quantize_128x128_pow2}


@pytest.fixture(scope="module", autouse=True)
def built():
    from fp8_block_scaled_03_gb300 import build
    build.build()
    fp.load_library()
    fp.clear_status()


def deq(x_f32, gran):
    c, s = Q[gran](x_f32)
    return OG.DEQUANT[gran](c, s)


def check_f32(d32, d16, a64, b64, k):
    """The bound of the module docstring, and BF16(d32) == d16."""
    assert d32.dtype == torch.float32 and d16.dtype == torch.bfloat16
    assert torch.equal(d32.to(torch.bfloat16).view(torch.int16), d16.view(torch.int16))
    got = d32.double().cpu().numpy()
    ref = OG.gemm_f64(a64, b64)
    absprod = np.abs(a64) @ np.abs(b64).T
    bound = (k + 3 * k / 128 + 2) * 2.0 ** -23 * absprod
    err = np.abs(got - ref)
    bad = err > bound
    assert not bad.any(), (f"{int(bad.sum())} elements beyond the float32 accumulation bound; worst "
                           f"err/bound {float((err / np.maximum(bound, 1e-300)).max()):.3g}")
    return float((err / np.maximum(bound, 1e-300)).max())


@pytest.mark.parametrize("a_gran,b_gran", [("1x128", "128x128"), ("1x128", "1x128"), ("per_tensor", "128x128"),
                                           ("mxfp8", "mxfp8"), ("1x128_pow2", "128x128_pow2")])
@pytest.mark.parametrize("m,n,k", [(300, 520, 384), (1, 8, 128), (2048, 2304, 640)])
def test_f32_output(a_gran, b_gran, m, n, k):
    """Ragged row and column tiles, a single row, and several tiles per CTA."""
    ab = synth.activations((m, k), seed=m + k + 21, outlier_frac=0.01, outlier_mult=50.0)
    bb = synth.weights((n, k), seed=n + k + 22, std=0.02)
    qa, sa, _ = fp.fp8_quantize(to_dev_bf16(ab), a_gran)
    qb, sb, _ = fp.fp8_quantize(to_dev_bf16(bb), b_gran)
    d32 = fp.fp8_block_gemm(qa, sa, a_gran, qb, sb, b_gran, out_dtype=torch.float32)
    d16 = fp.fp8_block_gemm(qa, sa, a_gran, qb, sb, b_gran)
    check_f32(d32, d16, deq(to_f32(ab), a_gran), deq(to_f32(bb), b_gran), k)
    assert fp.read_status() == 0


@pytest.mark.parametrize("form", ["nvfp4", "nvfp4_row"])
@pytest.mark.parametrize("m,n,k", [(300, 520, 512), (1000, 1024, 2048)])
def test_f32_output_nvfp4(form, m, n, k):
    ab = synth.activations((m, k), seed=m + 23, outlier_frac=0.01, outlier_mult=20.0)
    bb = synth.weights((n, k), seed=n + 24)
    qa, sa, ta = fp.fp8_quantize(to_dev_bf16(ab), form)
    qb, sb, tb = fp.fp8_quantize(to_dev_bf16(bb), "nvfp4")
    d32 = fp.fp8_block_gemm(qa, sa, form, qb, sb, "nvfp4", ta, tb, k=k, out_dtype=torch.float32)
    d16 = fp.fp8_block_gemm(qa, sa, form, qb, sb, "nvfp4", ta, tb, k=k)
    pa, sba, sga = OQ.quantize_nvfp4(to_f32(ab), row_scaled=form == "nvfp4_row")
    pb, sbb, sgb = OQ.quantize_nvfp4(to_f32(bb))
    check_f32(d32, d16, OG.dequant_nvfp4(pa, sba, sga), OG.dequant_nvfp4(pb, sbb, sgb), k)
    assert fp.read_status() == 0


def test_f32_output_rejects_other_dtypes():
    q = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    s = torch.ones((128, 1), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        fp.fp8_block_gemm(q, s, "1x128", q, s, "1x128", out_dtype=torch.float16)


def test_f32_output_full_size_step_sampled():
    """The dense linear layer's three GEMMs at full size (Qwen3-4B MLP shape,
    tokens 8192, hidden 2560, intermediate 9728) with float32 output: the
    whole output rounded to BF16 equals the BF16 output, and sampled rows and
    128-column blocks meet the accumulation bound against the oracle."""
    m3, h3, i3 = 8192, 2560, 9728
    x = synth.activations((m3, h3), seed=0, outlier_frac=0.01, outlier_mult=50.0)
    w = synth.weights((i3, h3), seed=1, std=0.02)
    dy = synth.activations((m3, i3), seed=2, outlier_frac=0.01, outlier_mult=50.0)
    qxt, sxt, qx, sx = fp.fp8_quantize_transposed(to_dev_bf16(x), "1x128", also_rowwise=True)
    qwt, swt, qw, sw = fp.fp8_quantize_transposed(to_dev_bf16(w), "128x128", also_rowwise=True)
    qdyt, sdyt, qdy, sdy = fp.fp8_quantize_transposed(to_dev_bf16(dy), "1x128", also_rowwise=True)
    xf, wf, dyf = to_f32(x), to_f32(w), to_f32(dy)
    g = np.random.Generator(np.random.PCG64(31))
    cases = (
        # (A codes, scales, gran, B codes, scales, gran, k, A rows source, B rows source)
        ("fprop", (qx, sx, "1x128", qw, sw, "128x128"), h3, lambda r: xf[r], lambda c: wf[c]),
        ("dgrad", (qdy, sdy, "1x128", qwt, swt, "128x128"), i3, lambda r: dyf[r],
         lambda c: np.ascontiguousarray(wf[:, c].T)),
        ("wgrad", (qdyt, sdyt, "1x128", qxt, sxt, "1x128"), m3, lambda r: np.ascontiguousarray(dyf[:, r].T),
         lambda c: np.ascontiguousarray(xf[:, c].T)),
    )
    for name, args, k, a_src, b_src in cases:
        d32 = fp.fp8_block_gemm(*args, out_dtype=torch.float32)
        d16 = fp.fp8_block_gemm(*args)
        assert torch.equal(d32.to(torch.bfloat16).view(torch.int16), d16.view(torch.int16)), name
        m, n = d32.shape
        rows = np.sort(g.choice(m, 32, replace=False))
        rows[-1] = m - 1
        nb = int(g.integers(0, n // 128))
        cols = np.arange(nb * 128, (nb + 1) * 128)
        a64 = deq(a_src(rows), args[2])
        b64 = deq(b_src(cols), args[5])
        ref = OG.gemm_f64(a64, b64)
        bound = (k + 3 * k / 128 + 2) * 2.0 ** -23 * (np.abs(a64) @ np.abs(b64).T)
        got = d32[torch.from_numpy(rows).cuda()][:, nb * 128:(nb + 1) * 128].double().cpu().numpy()
        assert np.all(np.abs(got - ref) <= bound), name
    assert fp.read_status() == 0
