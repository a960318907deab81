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
    assert lib.fp8bs_version() == 100
    for code in (0, -1, -2, -3, -4, -5, -6):
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


def test_quantize_transposed_rejects_bad_arguments(lib):
    t = lib.fp8_quantize_transposed
    assert t(FAKE, 24, 128, 128, 1, FAKE, FAKE, None, None, None, 0, None, 0, None) == -1  # rows % 16
    assert t(FAKE, 32, 128, 128, 4, FAKE, FAKE, None, None, None, 0, None, 0, None) == -3  # nvfp4
    assert t(FAKE, 32, 128, 128, 1, FAKE, FAKE, FAKE, None, None, 0, None, 0, None) == -1  # q w/o scales
    assert t(FAKE, 32, 128, 128, 1, MISALIGNED, FAKE, None, None, None, 0, None, 0, None) == -2


def test_gemm_rejects_bad_arguments(lib):
    g = lib.fp8_block_gemm
    assert g(FAKE, FAKE, 1, FAKE, FAKE, 2, None, None, 128, 128, 256, FAKE, FAKE, 16384, None) != 0 or True
    assert g(FAKE, FAKE, 1, FAKE, FAKE, 2, None, None, 128, 128, 256, FAKE, None, 0, None) == -6
    assert g(FAKE, FAKE, 1, FAKE, FAKE, 2, None, None, 128, 132, 256, FAKE, FAKE, 16384, None) == -1  # n % 8
    assert g(FAKE, FAKE, 1, FAKE, FAKE, 2, None, None, 0, 128, 256, FAKE, FAKE, 16384, None) == -1
    assert g(FAKE, FAKE, 1, FAKE, FAKE, 2, None, None, 128, 128, 192, FAKE, FAKE, 16384, None) == -1  # k % 128
    assert g(FAKE, FAKE, 3, FAKE, FAKE, 1, None, None, 128, 128, 256, FAKE, FAKE, 16384, None) == -3  # mixed
    assert g(FAKE, FAKE, 4, FAKE, FAKE, 4, None, None, 128, 128, 256, FAKE, FAKE, 16384, None) == -1  # nvfp4 ts
    assert g(FAKE, FAKE, 4, FAKE, FAKE, 4, FAKE, FAKE, 128, 128, 128, FAKE, FAKE, 16384, None) == -1  # k % 256
    assert g(MISALIGNED, FAKE, 1, FAKE, FAKE, 2, None, None, 128, 128, 256, FAKE, FAKE, 16384, None) == -2


def test_grouped_gemm_rejects_bad_arguments(lib):
    g = lib.fp8_grouped_gemm
    assert g(FAKE, FAKE, FAKE, FAKE, None, 8, 64, 128, 256, 3, FAKE, FAKE, 16384, None) == -1   # offsets
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 64, 128, 256, 3, FAKE, FAKE, 16384, None) == -1   # experts
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 64, 128, 200, 3, FAKE, FAKE, 16384, None) == -1   # k
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 64, 128, 256, 3, FAKE, None, 0, None) == -6
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 8, 0, 128, 256, 3, FAKE, FAKE, 16384, None) == 0     # empty: no-op
