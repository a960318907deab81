"""The tensor-core throughput loop behind the GEMM rooflines (fp8bs_mma_peak).

With every operand and scale equal to 1.0 each accumulator element must end
at iters * 4 * K exactly (K = 32 for E4M3 and MXFP8, 64 for NVFP4), which
shows the loop really issues the instructions it claims and that the FLOP
count the bench divides by is the work done.  The random-pattern form must
run and leave the status word clean.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu
fp = pytest.importorskip("fp8_block_scaled_03_gb300")

K_PER_INSTR = {0: 32, 1: 32, 2: 64}


@pytest.fixture(scope="module", autouse=True)
def built():
    from fp8_block_scaled_03_gb300 import build
    build.build()
    fp.load_library()


@pytest.mark.parametrize("kind,n", ((0, 64), (0, 256), (1, 128), (1, 256), (2, 128), (2, 256)))
def test_peak_loop_accumulates_exactly(kind, n):
    out = torch.full((128,), -1.0, dtype=torch.float32, device="cuda")
    iters = 96
    flop = fp.mma_peak(kind, n, iters, pattern=1, out=out)
    torch.cuda.synchronize()
    expect = iters * 4 * K_PER_INSTR[kind]
    assert torch.all(out == expect), (out.min().item(), out.max().item(), expect)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert flop == sms * iters * 4 * 2 * 128 * n * K_PER_INSTR[kind]
    assert fp.read_status() == 0


@pytest.mark.parametrize("kind", (0, 1, 2))
def test_peak_loop_random_operands_runs(kind):
    fp.mma_peak(kind, 256, 512, pattern=0)
    torch.cuda.synchronize()
    assert fp.read_status() == 0


def test_peak_loop_rejects_bad_arguments():
    lib = fp.load_library()
    ws = fp.workspace()
    P = fp._ptr
    assert lib.fp8bs_mma_peak(3, 256, 1, 0, None, P(ws), ws.numel(), None) == -1
    assert lib.fp8bs_mma_peak(0, 96, 1, 0, None, P(ws), ws.numel(), None) == -1
    assert lib.fp8bs_mma_peak(1, 64, 1, 0, None, P(ws), ws.numel(), None) == -1
    assert lib.fp8bs_mma_peak(0, 256, 0, 0, None, P(ws), ws.numel(), None) == -1
    assert lib.fp8bs_mma_peak(0, 256, 1, 0, None, None, 0, None) == -6
