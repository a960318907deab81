"""Failure detection without a GPU fault: a GEMM whose producer withholds a
pipeline stage must give up after its bounded wait, report FP8BS_ETIMEOUT in
the workspace status word, and leave the context usable."""
import numpy as np
import pytest
import torch

import synth
from oracle import gemm as OG
from oracle import quantize as OQ
from tests._util import assert_gemm_close, bf16_to_f64, to_dev_bf16, to_f32

pytestmark = pytest.mark.gpu
fp = pytest.importorskip("fp8_block_scaled_03_gb300")


def test_stalled_pipeline_times_out_and_recovers():
    from fp8_block_scaled_03_gb300 import build
    build.build()
    fp.load_library()
    ws = torch.zeros(fp.load_library().fp8bs_workspace_size(), dtype=torch.uint8, device="cuda")
    ab = synth.activations((256, 512), seed=1)
    bb = synth.weights((256, 512), seed=2)
    qa, sa, _ = fp.fp8_quantize(to_dev_bf16(ab), "mxfp8", ws=ws)
    qb, sb, _ = fp.fp8_quantize(to_dev_bf16(bb), "mxfp8", ws=ws)
    assert fp.read_status(ws) == 0
    rc = fp.test_stalled_gemm(qa, sa, qb, sb, 50_000_000, ws=ws)   # 50 ms bound
    assert rc == 0
    assert fp.read_status(ws) == -5                                 # FP8BS_ETIMEOUT
    fp.clear_status(ws)
    assert fp.read_status(ws) == 0
    # the context is still usable and the kernel still correct
    d = fp.fp8_block_gemm(qa, sa, "mxfp8", qb, sb, "mxfp8", ws=ws)
    ca, ea = OQ.quantize_mxfp8(to_f32(ab))
    cb, eb = OQ.quantize_mxfp8(to_f32(bb))
    assert_gemm_close(bf16_to_f64(d), OG.gemm_bf16(OG.dequant_mxfp8(ca, ea), OG.dequant_mxfp8(cb, eb)))
    assert fp.read_status(ws) == 0


def test_stalled_nvfp4_pipeline_times_out_and_recovers():
    """The NVFP4 GEMM's scale loaders issue the tensor-memory copies and
    drain them before exit; a stalled stage must still end in a timeout
    status with the context usable and the next GEMM correct."""
    ws = torch.zeros(fp.load_library().fp8bs_workspace_size(), dtype=torch.uint8, device="cuda")
    ab = synth.activations((256, 512), seed=3)
    bb = synth.weights((256, 512), seed=4)
    qa, sa, ta = fp.fp8_quantize(to_dev_bf16(ab), "nvfp4", ws=ws)
    qb, sb, tb = fp.fp8_quantize(to_dev_bf16(bb), "nvfp4", ws=ws)
    assert fp.read_status(ws) == 0
    rc = fp.test_stalled_gemm_nvfp4(qa, sa, qb, sb, ta, tb, 50_000_000, ws=ws)   # 50 ms bound
    assert rc == 0
    assert fp.read_status(ws) == -5
    fp.clear_status(ws)
    d = fp.fp8_block_gemm(qa, sa, "nvfp4", qb, sb, "nvfp4", ta, tb, k=512, ws=ws)
    pa, sba, sga = OQ.quantize_nvfp4(to_f32(ab))
    pb, sbb, sgb = OQ.quantize_nvfp4(to_f32(bb))
    ref = OG.gemm_bf16(OG.dequant_nvfp4(pa, sba, sga), OG.dequant_nvfp4(pb, sbb, sgb))
    assert_gemm_close(bf16_to_f64(d), ref)
    assert fp.read_status(ws) == 0


@pytest.mark.parametrize("a_gran,b_gran", [("1x128", "128x128"), ("1x128", "1x128")])
def test_stalled_blockwise_pipeline_times_out_and_recovers(a_gran, b_gran):
    """The FP32-scale blockwise GEMM: a withheld stage must end in
    FP8BS_ETIMEOUT with the context usable (epilogue, scale loader and MMA
    issuer all give up; the CTA frees its tensor memory), and the next GEMM
    must be correct."""
    ws = torch.zeros(fp.load_library().fp8bs_workspace_size(), dtype=torch.uint8, device="cuda")
    ab = synth.activations((256, 512), seed=5)
    bb = synth.weights((256, 512), seed=6)
    qa, sa, _ = fp.fp8_quantize(to_dev_bf16(ab), a_gran, ws=ws)
    qb, sb, _ = fp.fp8_quantize(to_dev_bf16(bb), b_gran, ws=ws)
    assert fp.read_status(ws) == 0
    rc = fp.test_stalled_gemm_blockwise(qa, sa, a_gran, qb, sb, b_gran, 50_000_000, ws=ws)   # 50 ms bound
    assert rc == 0
    assert fp.read_status(ws) == -5
    fp.clear_status(ws)
    d = fp.fp8_block_gemm(qa, sa, a_gran, qb, sb, b_gran, ws=ws)
    q_fn = {"1x128": OQ.quantize_1x128, "128x128": OQ.quantize_128x128}
    dq_fn = {"1x128": OG.dequant_1x128, "128x128": OG.dequant_128x128}
    ca, ea = q_fn[a_gran](to_f32(ab))
    cb, eb = q_fn[b_gran](to_f32(bb))
    assert_gemm_close(bf16_to_f64(d), OG.gemm_bf16(dq_fn[a_gran](ca, ea), dq_fn[b_gran](cb, eb)))
    assert fp.read_status(ws) == 0
