"""The GEMM kernels' dynamic tile order.

CTAs of the blockwise kernel's 128x128-weight-scale forms, and of the
block-scaled kernel's power-of-two (UE8M0) block forms, take tiles from a
counter in the workspace as they become free.  A tile's arithmetic does not depend on which
CTA computes it, so the three GEMMs of the dense step run concurrently on
three streams (a workspace each) must give the same bits as the same calls
one after another; the counter must be back to zero after every call (the
kernel's last CTA resets it), so that the next call on that workspace starts
from tile 0.
"""
import numpy as np
import pytest
import torch

import synth
from tests._util import to_dev_bf16

pytestmark = pytest.mark.gpu
fp = pytest.importorskip("fp8_block_scaled_03_gb300")


@pytest.fixture(scope="module", autouse=True)
def built():
    from fp8_block_scaled_03_gb300 import build
    build.build()
    fp.load_library()
    fp.clear_status()


def counter_bytes(ws):
    return ws[64:80].cpu().numpy()


RECIPES = {"fp32": ("1x128", "128x128"), "pow2": ("1x128_pow2", "128x128_pow2")}


def step_operands(m, h, i, seed, recipe="fp32"):
    t, b = RECIPES[recipe]
    x = synth.activations((m, h), seed=seed, outlier_frac=0.01, outlier_mult=50.0)
    w = synth.weights((i, h), seed=seed + 1, std=0.02)
    dy = synth.activations((m, i), seed=seed + 2, outlier_frac=0.01, outlier_mult=50.0)
    qxt, sxt, qx, sx = fp.fp8_quantize_transposed(to_dev_bf16(x), t, also_rowwise=True)
    qwt, swt, qw, sw = fp.fp8_quantize_transposed(to_dev_bf16(w), b, also_rowwise=True)
    qdyt, sdyt, qdy, sdy = fp.fp8_quantize_transposed(to_dev_bf16(dy), t, also_rowwise=True)
    return ((qx, sx, t, qw, sw, b),          # fprop  [m, i]
            (qdy, sdy, t, qwt, swt, b),      # dgrad  [m, h]
            (qdyt, sdyt, t, qxt, sxt, t))    # wgrad  [i, h]


@pytest.mark.parametrize("recipe", ["fp32", "pow2"])
@pytest.mark.parametrize("m,h,i", [(1024, 640, 1152), (8192, 2560, 9728)])
def test_concurrent_step_gemms_match_sequential(m, h, i, recipe):
    ops = step_operands(m, h, i, seed=m + h, recipe=recipe)
    wss = [fp.new_workspace() for _ in range(3)]
    seq = [fp.fp8_block_gemm(*o, ws=wss[j]) for j, o in enumerate(ops)]
    torch.cuda.synchronize()
    for ws in wss:
        assert not counter_bytes(ws).any()
    outs = [torch.empty_like(t) for t in seq]
    streams = [torch.cuda.Stream() for _ in range(3)]
    ready = torch.cuda.Event()
    ready.record()
    for rep in range(3):
        for j in (2, 1, 0):                     # wgrad, dgrad, fprop, as the step launches them
            streams[j].wait_event(ready)
            with torch.cuda.stream(streams[j]):
                fp.fp8_block_gemm(*ops[j], out=outs[j], ws=wss[j])
        torch.cuda.synchronize()
        for j in range(3):
            assert torch.equal(outs[j].view(torch.int16), seq[j].view(torch.int16)), (rep, j)
    for ws in wss:
        assert fp.read_status(ws) == 0
        assert not counter_bytes(ws).any()


@pytest.mark.parametrize("recipe", ["fp32", "pow2"])
def test_counter_reset_after_every_call_and_grouped(recipe):
    """Dense and grouped calls back to back on one workspace: every call
    computes all its tiles, and the counter ends at zero."""
    t, bg = RECIPES[recipe]
    ws = fp.new_workspace()
    a = synth.activations((520, 384), seed=3, outlier_frac=0.01, outlier_mult=20.0)
    b = synth.weights((4 * 256, 384), seed=4)
    qa, sa, _ = fp.fp8_quantize(to_dev_bf16(a), t)
    qb, sb, _ = fp.fp8_quantize(to_dev_bf16(b), bg)
    ref = fp.fp8_block_gemm(qa, sa, t, qb, sb, bg, ws=ws)
    # grouped: 4 experts of 256 rows of B, ragged row counts (one empty)
    counts = [0, 130, 7, 383]
    offsets = torch.from_numpy(np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)).cuda()
    qbs, sbs = [], []
    for e in range(4):
        q_, s_, _ = fp.fp8_quantize(to_dev_bf16(b[e * 256:(e + 1) * 256]), bg)
        qbs.append(q_)
        sbs.append(s_)
    qbg, sbg = torch.stack(qbs), torch.stack(sbs)
    gref = fp.fp8_grouped_gemm(qa, sa, qbg, sbg, offsets, t, ws=fp.new_workspace())
    for _ in range(4):
        d = fp.fp8_block_gemm(qa, sa, t, qb, sb, bg, ws=ws)
        g = fp.fp8_grouped_gemm(qa, sa, qbg, sbg, offsets, t, ws=ws)
        torch.cuda.synchronize()
        assert torch.equal(d.view(torch.int16), ref.view(torch.int16))
        assert torch.equal(g.view(torch.int16), gref.view(torch.int16))
        assert not counter_bytes(ws).any()
    # the grouped rows against the dense product with each expert's B block
    for e in range(4):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi > lo:
            assert torch.equal(gref[lo:hi].view(torch.int16), ref[lo:hi, e * 256:(e + 1) * 256].view(torch.int16))
    assert fp.read_status(ws) == 0
