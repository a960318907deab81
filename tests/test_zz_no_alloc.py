"""The allocation-free per-tensor quantiser, called through the C ABI.

fp8_quantize_per_tensor_noalloc serves callers that cannot allocate device
memory (they receive input and output buffers only, e.g. from a framework
allocator or a plugin interface): it keeps the amax partials of the
per-tensor reduction in a fixed array inside the library.  Its output must
equal the workspace-based fp8_quantize(PER_TENSOR) bit for bit, on two calls
in a row (the second smaller than the first, so stale scratch contents
would show).  Named to be collected last.
"""
import ctypes

import pytest
import torch

import synth
from tests._util import to_dev_bf16

pytestmark = pytest.mark.gpu
fp = pytest.importorskip("fp8_block_scaled_03_gb300")


@pytest.fixture(scope="module")
def lib():
    from fp8_block_scaled_03_gb300 import build
    build.build()
    lib = fp.load_library()
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    lib.fp8_quantize_per_tensor_noalloc.argtypes = [P, I64, I64, I64, P, P, P]
    lib.fp8_quantize_per_tensor_noalloc.restype = ctypes.c_int
    return lib


def call_noalloc(lib, x, q, scale):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.fp8_quantize_per_tensor_noalloc(ctypes.c_void_p(x.data_ptr()), x.shape[0], x.shape[1], x.stride(0),
                                               ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(scale.data_ptr()),
                                               stream)


def test_matches_workspace_entry_point_on_two_calls(lib):
    cases = (((8192, 4096), 0, 100.0), ((300, 1032), 1, 3.0))
    for shape, seed, mult in cases:
        x = to_dev_bf16(synth.activations(shape, seed=seed, outlier_frac=0.001, outlier_mult=mult))
        q_ref, s_ref, _ = fp.fp8_quantize(x, "per_tensor")
        q = torch.full_like(q_ref, 0x55)
        s = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
        assert call_noalloc(lib, x, q, s) == 0
        torch.cuda.synchronize()
        assert torch.equal(s, s_ref), (s.item(), s_ref.item())
        assert torch.equal(q, q_ref)


def test_rejects_inputs_beyond_the_scratch(lib):
    fake = torch.empty(16, dtype=torch.uint8, device="cuda")           # never read: the size check fails first
    rows = 64 * 4096 + 1                                              # one warp task past the limit
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    p = ctypes.c_void_p(fake.data_ptr())
    assert lib.fp8_quantize_per_tensor_noalloc(p, rows, 1024, 1024, p, p, stream) == -1    # FP8BS_EINVAL


_RESET_CHILD = r"""
import ctypes, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
import synth
lib = ctypes.CDLL(sys.argv[2])
rt = ctypes.CDLL("libcudart.so.13")           # the runtime the library itself links
P, I64 = ctypes.c_void_p, ctypes.c_int64
lib.fp8_quantize_per_tensor_noalloc.argtypes = [P, I64, I64, I64, P, P, P]
lib.fp8bs_test_noalloc_scratch.argtypes = [ctypes.POINTER(P), ctypes.POINTER(P)]
rows, cols = 256, 1024
xb = np.ascontiguousarray(synth.activations((rows, cols), seed=5, outlier_frac=0.01, outlier_mult=30.0))  # BF16 bits
results = []
for attempt in range(2):
    cached, fresh = P(), P()
    assert lib.fp8bs_test_noalloc_scratch(ctypes.byref(cached), ctypes.byref(fresh)) == 0
    assert cached.value == fresh.value, (attempt, cached.value, fresh.value)   # checked before any launch
    dx, dq, ds = P(), P(), P()
    assert rt.cudaMalloc(ctypes.byref(dx), ctypes.c_size_t(xb.nbytes)) == 0
    assert rt.cudaMalloc(ctypes.byref(dq), ctypes.c_size_t(rows * cols)) == 0
    assert rt.cudaMalloc(ctypes.byref(ds), ctypes.c_size_t(4)) == 0
    assert rt.cudaMemcpy(dx, xb.ctypes.data_as(P), ctypes.c_size_t(xb.nbytes), 1) == 0
    assert lib.fp8_quantize_per_tensor_noalloc(dx, rows, cols, cols, dq, ds, None) == 0
    q = np.empty((rows, cols), np.uint8); s = np.empty(1, np.float32)
    assert rt.cudaMemcpy(q.ctypes.data_as(P), dq, ctypes.c_size_t(q.nbytes), 2) == 0
    assert rt.cudaMemcpy(s.ctypes.data_as(P), ds, ctypes.c_size_t(4), 2) == 0
    results.append((q, s))
    if attempt == 0:
        assert rt.cudaDeviceReset() == 0       # ends this process's context only
assert np.array_equal(results[0][0], results[1][0]) and results[0][1][0] == results[1][1][0]
print("ok", results[0][1][0])
"""


def test_scratch_address_follows_a_recreated_context(lib, tmp_path):
    """After cudaDeviceReset the module loads again in a new context: the
    cached partials address must be looked up afresh.  Run in a child process
    (the reset would invalidate this process's torch state); the child checks
    the cached address against a fresh lookup before it launches anything."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = tmp_path / "reset_child.py"
    script.write_text(_RESET_CHILD)
    r = subprocess.run([sys.executable, str(script), root, fp.LIB_PATH], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok")
