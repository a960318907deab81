"""The C-ABI library loads without a GPU, exports every symbol the header
declares, and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

import fp8_block_scaled_03_gb300 as fp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from fp8_block_scaled_03_gb300 import build
    build.build()
    return fp.load_library()


def header_functions():
    text = open(os.path.join(ROOT, "include", "fp8bs.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert set(fp.EXPORTS) <= set(names)
    for name in names:
        assert hasattr(lib, name), name


def test_status_strings_and_sizes(lib):
    assert lib.fp8bs_workspace_size() == 16384
    ws = lib.fp8bs_workspace_size_for
    big = 1 << 40
    assert ws(0, big, 8192, 0, 0) == 16384 and ws(0, 4, 128, 4, 0) == 16384     # per-tensor / NVFP4 amax partials
    assert ws(0, 4, 128, 0, 1) == 0 and ws(0, 4, 128, 1, 0) == 0               # given scale / 1x128: none
    assert ws(2, 4, 128, 1, 0) == 0 and ws(7, 4, 128, 3, 0) == 0               # dequantise, SwiGLU: none
    assert all(ws(op, 4, 128, 3, 0) == 16384 for op in (3, 4, 5, 6))          # GEMMs, gathers: status word
    assert ws(8, 4, 128, 1, 0) == 2 ** 64 - 1 and ws(0, -1, 128, 1, 0) == 2 ** 64 - 1
    assert lib.fp8bs_version() == 103
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        assert fp.status_string(code) != "unknown status"
    assert fp.status_string(7) == "unknown status"


FAKE = ctypes.c_void_p(0x10000)        # never dereferenced: every call below fails its host checks
MISALIGNED = ctypes.c_void_p(0x10008)


def test_quantize_rejects_bad_arguments(lib):
    q = lib.fp8_quantize
    assert q(None, 4, 128, 128, 1, FAKE, FAKE, None, 0, None, 0, None) == -1      # null x
    assert q(FAKE, 4, 120 + 4, 128, 1, FAKE, FAKE, None, 0, None, 0, None) == -1  # cols % 8
    assert q(FAKE, 4, 128, 120, 1, FAKE, FAKE, None, 0, None, 0, None) == -1      # ld < cols
    assert q(FAKE, 4, 128, 128, 9, FAKE, FAKE, None, 0, None, 0, None) == -1      # bad gran
    assert q(FAKE, -1, 128, 128, 1, FAKE, FAKE, None, 0, None, 0, None) == -1     # negative rows
    assert q(MISALIGNED, 4, 128, 128, 1, FAKE, FAKE, None, 0, None, 0, None) == -2
    assert q(FAKE, 4, 128, 128, 0, FAKE, FAKE, None, 0, None, 0, None) == -6      # per-tensor needs ws
    assert q(FAKE, 4, 128, 128, 4, FAKE, FAKE, None, 0, FAKE, 16384, None) == -1  # nvfp4 needs S_g ptr
    assert q(FAKE, 4, 120, 120, 4, FAKE, FAKE, FAKE, 0, FAKE, 16384, None) == -1  # nvfp4 cols % 16
    assert q(FAKE, 4, 128, 128, 4, FAKE, FAKE, FAKE, 0, FAKE, 1024, None) == -6   # ws too small
    assert q(FAKE, 4, 128, 128, 0, FAKE, FAKE, None, 0, MISALIGNED, 16384, None) == -2   # ws misaligned


def test_quantize_transposed_rejects_bad_arguments(lib):
    t = lib.fp8_quantize_transposed
    assert t(FAKE, 24, 128, 128, 1, FAKE, FAKE, None, None, None, 0, None, 0, None) == -1  # rows % 16
    assert t(FAKE, 32, 128, 128, 4, FAKE, FAKE, None, None, None, 0, None, 0, None) == -3  # nvfp4
    assert t(FAKE, 32, 128, 128, 1, FAKE, FAKE, FAKE, None, None, 0, None, 0, None) == -1  # q w/o scales
    assert t(FAKE, 32, 128, 128, 1, MISALIGNED, FAKE, None, None, None, 0, None, 0, None) == -2
    assert t(FAKE, 32, 2 ** 31, 2 ** 31, 1, FAKE, FAKE, None, None, None, 0, None, 0, None) == -1  # TMA range


def test_gemm_rejects_bad_arguments(lib):
    g = lib.fp8_block_gemm
    assert g(FAKE, FAKE, 1, FAKE, FAKE, 2, None, None, 128, 128, 256, FAKE, 0, None, 0, None) == -6
    assert g(FAKE, FAKE, 1, FAKE, FAKE, 2, None, None, 128, 132, 256, FAKE, 0, FAKE, 16384, None) == -1  # n % 8
    assert g(FAKE, FAKE, 1, FAKE, FAKE, 2, None, None, 0, 128, 256, FAKE, 0, FAKE, 16384, None) == -1
    assert g(FAKE, FAKE, 1, FAKE, FAKE, 2, None, None, 128, 128, 192, FAKE, 0, FAKE, 16384, None) == -1  # k % 128
    assert g(FAKE, FAKE, 3, FAKE, FAKE, 1, None, None, 128, 128, 256, FAKE, 0, FAKE, 16384, None) == -3  # mixed
    assert g(FAKE, FAKE, 4, FAKE, FAKE, 4, None, None, 128, 128, 256, FAKE, 0, FAKE, 16384, None) == -1  # nvfp4 ts
    assert g(FAKE, FAKE, 4, FAKE, FAKE, 4, FAKE, FAKE, 128, 128, 128, FAKE, 0, FAKE, 16384, None) == -1  # k % 256
    assert g(MISALIGNED, FAKE, 1, FAKE, FAKE, 2, None, None, 128, 128, 256, FAKE, 0, FAKE, 16384, None) == -2
    # TMA coordinates are 32-bit: dimensions of 2^31 and more are refused before any launch
    assert g(FAKE, FAKE, 1, FAKE, FAKE, 2, None, None, 2 ** 31, 128, 256, FAKE, 0, FAKE, 16384, None) == -1
    assert g(FAKE, FAKE, 1, FAKE, FAKE, 2, None, None, 128, 128, 2 ** 31, FAKE, 0, FAKE, 16384, None) == -1
    # the workspace holds 8-byte tile counters and the status word: 16-byte aligned
    assert g(FAKE, FAKE, 1, FAKE, FAKE, 2, None, None, 128, 128, 256, FAKE, 0, MISALIGNED, 16384, None) == -2


def test_gemm_rejects_unknown_output_dtype(lib):
    g = lib.fp8_block_gemm
    for bad in (2, -1):
        assert g(FAKE, FAKE, 1, FAKE, FAKE, 2, None, None, 128, 128, 256, FAKE, bad, FAKE, 16384, None) == -1


def test_grouped_gemm_rejects_bad_arguments(lib):
    g = lib.fp8_grouped_gemm
    assert g(FAKE, FAKE, FAKE, FAKE, None, None, None, 8, 64, 128, 256, 3, FAKE, FAKE, 16384, None) == -1  # offsets
    assert g(FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 0, 64, 128, 256, 3, FAKE, FAKE, 16384, None) == -1  # experts
    assert g(FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 8, 64, 128, 200, 3, FAKE, FAKE, 16384, None) == -1  # k
    assert g(FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 8, 64, 128, 256, 3, FAKE, None, 0, None) == -6
    assert g(FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 8, 0, 128, 256, 3, FAKE, FAKE, 16384, None) == 0  # empty
    # TMA coordinates are 32-bit: rows, and the stacked B rows (experts * n), stay below 2^31
    assert g(FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 8, 2 ** 31, 128, 256, 3, FAKE, FAKE, 16384, None) == -1
    assert g(FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 1024, 64, 2 ** 21, 256, 3, FAKE, FAKE, 16384, None) == -1
    # NVFP4: both tensor scales required, k % 256, 16-byte block scales
    assert g(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 8, 64, 128, 256, 4, FAKE, FAKE, 16384, None) == -1
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 8, 64, 128, 384, 7, FAKE, FAKE, 16384, None) == -1
    assert g(FAKE, ctypes.c_void_p(0x10004), FAKE, FAKE, FAKE, FAKE, FAKE, 8, 64, 128, 256, 4, FAKE, FAKE, 16384,
             None) == -2
    assert g(FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 8, 64, 128, 256, 9, FAKE, FAKE, 16384, None) == -1  # gran


ODD4 = ctypes.c_void_p(0x10002)        # not 4-byte aligned


def test_quantize_flags_and_row_scaled_nvfp4(lib):
    q = lib.fp8_quantize
    assert q(FAKE, 4, 128, 128, 4, FAKE, FAKE, FAKE, 4, FAKE, 16384, None) == -1   # unknown flag bit
    assert q(FAKE, 4, 128, 128, 1, FAKE, FAKE, None, 2, None, 0, None) == -1       # 4over6 on 1x128
    assert q(FAKE, 4, 128, 128, 7, FAKE, FAKE, None, 0, None, 0, None) == -1       # row S_g pointer missing
    assert q(FAKE, 4, 120, 120, 7, FAKE, FAKE, FAKE, 0, None, 0, None) == -1       # cols % 16
    assert q(FAKE, 4, 128, 128, 7, FAKE, FAKE, ODD4, 0, None, 0, None) == -2       # S_g alignment
    assert q(FAKE, 4, 128, 128, 8, FAKE, FAKE, FAKE, 0, None, 0, None) == -1       # no gran 8
    assert q(None, 0, 128, 128, 7, None, None, None, 2, None, 0, None) == 0        # empty: no-op
    t = lib.fp8_quantize_transposed
    assert t(FAKE, 32, 128, 128, 7, FAKE, FAKE, None, None, FAKE, 0, None, 0, None) == -3
    assert t(FAKE, 32, 128, 128, 1, FAKE, FAKE, None, None, None, 2, None, 0, None) == -1


def test_dequantize_rejects_bad_arguments(lib):
    d = lib.fp8_dequantize
    assert d(None, FAKE, None, 4, 128, 1, FAKE, 128, None) == -1                 # null q
    assert d(FAKE, FAKE, None, 4, 124, 1, FAKE, 128, None) == -1                 # cols % 8
    assert d(FAKE, FAKE, None, 4, 128, 1, FAKE, 120, None) == -1                 # ld_out < cols
    assert d(FAKE, FAKE, None, 4, 128, 8, FAKE, 128, None) == -1                 # bad gran
    assert d(FAKE, FAKE, None, 4, 128, 4, FAKE, 128, None) == -1                 # NVFP4 needs S_g
    assert d(FAKE, FAKE, ODD4, 4, 128, 7, FAKE, 128, None) == -2                 # S_g alignment
    assert d(ctypes.c_void_p(0x10004), FAKE, None, 4, 128, 1, FAKE, 128, None) == -2   # q 8-byte aligned
    assert d(FAKE, FAKE, None, 4, 128, 1, MISALIGNED, 128, None) == -2           # out 16-byte aligned
    assert d(None, None, None, 0, 128, 1, None, 128, None) == 0                  # empty: no-op


def test_gemm_row_scaled_nvfp4_arguments(lib):
    g = lib.fp8_block_gemm
    assert g(FAKE, FAKE, 7, FAKE, FAKE, 7, FAKE, FAKE, 128, 128, 256, FAKE, 0, FAKE, 16384, None) == -3  # B per row
    assert g(FAKE, FAKE, 7, FAKE, FAKE, 4, None, FAKE, 128, 128, 256, FAKE, 0, FAKE, 16384, None) == -1  # A S_g
    assert g(FAKE, FAKE, 7, FAKE, FAKE, 4, ODD4, FAKE, 128, 128, 256, FAKE, 0, FAKE, 16384, None) == -2
    assert g(FAKE, FAKE, 7, FAKE, FAKE, 4, FAKE, FAKE, 128, 128, 128, FAKE, 0, FAKE, 16384, None) == -1  # k % 256


def test_gathered_quantize_rejects_bad_arguments(lib):
    g = lib.fp8_quantize_gathered
    WS = 16384
    assert g(None, 8, 128, 128, FAKE, 4, 1, FAKE, FAKE, FAKE, WS, None) == -1       # null x
    assert g(FAKE, 8, 128, 128, None, 4, 1, FAKE, FAKE, FAKE, WS, None) == -1       # null index
    assert g(FAKE, 8, 124, 128, FAKE, 4, 1, FAKE, FAKE, FAKE, WS, None) == -1       # cols % 8
    assert g(FAKE, 8, 128, 120, FAKE, 4, 1, FAKE, FAKE, FAKE, WS, None) == -1       # ld < cols
    assert g(FAKE, -1, 128, 128, FAKE, 4, 1, FAKE, FAKE, FAKE, WS, None) == -1      # negative tokens
    assert g(FAKE, 8, 128, 128, FAKE, 4, 9, FAKE, FAKE, FAKE, WS, None) == -1       # bad gran
    for unsupported in (0, 2, 4, 6, 7):
        assert g(FAKE, 8, 128, 128, FAKE, 4, unsupported, FAKE, FAKE, FAKE, WS, None) == -3
    assert g(FAKE, 8, 128, 128, ODD4, 4, 3, FAKE, FAKE, FAKE, WS, None) == -2       # index 8-byte aligned
    assert g(MISALIGNED, 8, 128, 128, FAKE, 4, 3, FAKE, FAKE, FAKE, WS, None) == -2
    assert g(FAKE, 8, 128, 128, FAKE, 4, 1, FAKE, ODD4, FAKE, WS, None) == -2       # FP32 scales
    assert g(FAKE, 8, 128, 128, FAKE, 4, 3, FAKE, FAKE, None, 0, None) == -6        # status word needed
    assert g(FAKE, 8, 128, 128, FAKE, 4, 3, FAKE, FAKE, FAKE, 1024, None) == -6
    assert g(None, 0, 128, 128, None, 0, 3, None, None, None, 0, None) == 0         # empty: no-op


def test_gather_rows_rejects_bad_arguments(lib):
    # every call fails a host check before any launch (the pointers are fake)
    g = lib.fp8_gather_rows
    WS = 16384
    assert g(None, FAKE, 8, 128, 3, FAKE, 4, FAKE, FAKE, FAKE, WS, None) == -1       # null codes source
    assert g(FAKE, None, 8, 128, 3, FAKE, 4, FAKE, FAKE, FAKE, WS, None) == -1       # null scales source
    assert g(FAKE, FAKE, 8, 128, 3, None, 4, FAKE, FAKE, FAKE, WS, None) == -1       # null index
    assert g(FAKE, FAKE, 8, 128, 3, FAKE, 4, None, FAKE, FAKE, WS, None) == -1       # null output
    assert g(FAKE, FAKE, 8, 124, 3, FAKE, 4, FAKE, FAKE, FAKE, WS, None) == -1       # cols % 8
    assert g(FAKE, FAKE, -1, 128, 3, FAKE, 4, FAKE, FAKE, FAKE, WS, None) == -1      # negative tokens
    assert g(FAKE, FAKE, 8, 128, 9, FAKE, 4, FAKE, FAKE, FAKE, WS, None) == -1       # bad gran
    for unsupported in (0, 2, 4, 6, 7):
        assert g(FAKE, FAKE, 8, 128, unsupported, FAKE, 4, FAKE, FAKE, FAKE, WS, None) == -3
    assert g(FAKE, FAKE, 8, 128, 3, ODD4, 4, FAKE, FAKE, FAKE, WS, None) == -2       # index 8-byte aligned
    assert g(MISALIGNED, FAKE, 8, 128, 3, FAKE, 4, FAKE, FAKE, FAKE, WS, None) == -2
    assert g(FAKE, FAKE, 8, 128, 3, FAKE, 4, MISALIGNED, FAKE, FAKE, WS, None) == -2
    assert g(FAKE, ODD4, 8, 128, 1, FAKE, 4, FAKE, FAKE, FAKE, WS, None) == -2       # FP32 source scales
    assert g(FAKE, FAKE, 8, 128, 1, FAKE, 4, FAKE, ODD4, FAKE, WS, None) == -2       # FP32 scales
    assert g(FAKE, FAKE, 8, 128, 3, FAKE, 4, FAKE, FAKE, None, 0, None) == -6        # status word needed
    assert g(FAKE, FAKE, 8, 128, 3, FAKE, 4, FAKE, FAKE, FAKE, 1024, None) == -6
    assert g(None, None, 0, 128, 3, None, 0, None, None, None, 0, None) == 0         # empty: no-op


def test_swiglu_quantize_rejects_bad_arguments(lib):
    s = lib.fp8_swiglu_quantize
    assert s(None, 4, 128, 256, 3, FAKE, FAKE, None) == -1          # null h
    assert s(FAKE, 4, 124, 256, 3, FAKE, FAKE, None) == -1          # inter % 8
    assert s(FAKE, 4, 128, 248, 3, FAKE, FAKE, None) == -1          # ld_h < 2 * inter
    assert s(FAKE, 4, 128, 260, 3, FAKE, FAKE, None) == -1          # ld_h % 8
    assert s(FAKE, -4, 128, 256, 3, FAKE, FAKE, None) == -1
    for unsupported in (0, 2, 4, 6, 7):
        assert s(FAKE, 4, 128, 256, unsupported, FAKE, FAKE, None) == -3
    assert s(MISALIGNED, 4, 128, 256, 3, FAKE, FAKE, None) == -2
    assert s(FAKE, 4, 128, 256, 5, MISALIGNED, FAKE, None) == -2
    assert s(None, 0, 128, 256, 3, None, None, None) == 0           # empty: no-op
    assert s(None, 4, 0, 0, 3, None, None, None) == 0


def test_stalled_gemm_nvfp4_rejects_bad_arguments(lib):
    t = lib.fp8bs_test_stalled_gemm_nvfp4
    WS = 16384
    assert t(FAKE, FAKE, FAKE, FAKE, None, FAKE, 128, 128, 256, FAKE, 1000, FAKE, WS, None) == -1   # S_g A
    assert t(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 128, 128, FAKE, 1000, FAKE, WS, None) == -1   # k % 256
    assert t(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 128, 256, FAKE, 0, FAKE, WS, None) == -1      # no bound
    assert t(FAKE, ODD4, FAKE, FAKE, FAKE, FAKE, 128, 128, 256, FAKE, 1000, FAKE, WS, None) == -2   # scales
    assert t(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 128, 128, 256, FAKE, 1000, None, 0, None) == -6


def test_quotient_sweep_rejects_bad_arguments(lib):
    assert lib.fp8bs_test_quotient_sweep(None, 0, None) == -1
    assert lib.fp8bs_test_quotient_sweep(FAKE, 4, None) == -1
    assert lib.fp8bs_test_quotient_sweep(FAKE, -1, None) == -1
    assert lib.fp8bs_test_quotient_sweep(ODD4, 1, None) == -2


def test_encoder_breakpoints_and_scratch_hook_reject_bad_arguments(lib):
    assert lib.fp8bs_test_encoder_breakpoints(None, None) == -1
    assert lib.fp8bs_test_encoder_breakpoints(ctypes.c_void_p(0x1002), None) == -2
    p = ctypes.c_void_p()
    assert lib.fp8bs_test_noalloc_scratch(None, ctypes.byref(p)) == -1
    assert lib.fp8bs_test_noalloc_scratch(ctypes.byref(p), None) == -1


def test_header_compiles_as_c99_and_links(lib, tmp_path):
    """A plain C99 program (no CUDA headers) includes include/fp8bs.h, links
    libfp8bs.so and calls entry points that need no GPU."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(fp.LIB_PATH)
    exe = str(tmp_path / "abi_c99")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "abi_c99.c"), "-L", libdir, "-lfp8bs", f"-Wl,-rpath,{libdir}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and "c99 abi ok" in r.stdout, r.stdout + r.stderr
