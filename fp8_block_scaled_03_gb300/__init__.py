"""Python binding of libfp8bs.so (the block-scaled low-precision linear layer).

Argument marshalling only: every computation runs in the CUDA kernels
behind the C ABI declared in include/fp8bs.h.  PyTorch supplies device
memory and the current stream.  There is no CPU fallback: if the shared
library is missing or fails to load, every call raises.

Entry points (same names as the C ABI):
    fp8_quantize(x, gran)                 -> (q, scales, tensor_scale)
    fp8_quantize_transposed(x, gran, also_rowwise=False)
                                          -> (q_t, scales_t, q, scales)
    fp8_dequantize(q, scales, gran)       -> BF16 values (exact, rounded once)
    fp8_block_gemm(a, sa, a_gran, b, sb, b_gran, a_ts=None, b_ts=None) -> d (bf16, or float32 with
                                          out_dtype=torch.float32)
    fp8_grouped_gemm(a, sa, b, sb, offsets, gran)                      -> d (bf16)
    fp8_quantize_gathered(x, token_index, gran) -> (q, scales)   rows x[token_index]
    fp8_swiglu_quantize(h, gran)          -> (q, scales)   of BF16(silu(gate) * up)

Granularities: "per_tensor", "1x128", "128x128", "mxfp8", "nvfp4", the
block-wise recipe with power-of-two scales "1x128_pow2", "128x128_pow2", and
"nvfp4_row" (NVFP4 with one outer scale per row).  Flags:
FLAG_GIVEN_TENSOR_SCALE, FLAG_NVFP4_4OVER6.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfp8bs.so")

GRAN = {"per_tensor": 0, "1x128": 1, "128x128": 2, "mxfp8": 3, "nvfp4": 4, "1x128_pow2": 5, "128x128_pow2": 6,
        "nvfp4_row": 7}
NVFP4_GRANS = (4, 7)
FLAG_GIVEN_TENSOR_SCALE = 1
FLAG_NVFP4_4OVER6 = 2
STATUS = {0: "FP8BS_OK", -1: "FP8BS_EINVAL", -2: "FP8BS_EALIGN", -3: "FP8BS_EUNSUPPORTED",
          -4: "FP8BS_ECUDA", -5: "FP8BS_ETIMEOUT", -6: "FP8BS_EWORKSPACE", -7: "FP8BS_EINDEX", -8: "FP8BS_EOFFSETS"}
EINDEX = -7
EOFFSETS = -8
EXPORTS = ("fp8_quantize", "fp8_quantize_transposed", "fp8_dequantize", "fp8_block_gemm", "fp8_grouped_gemm",
           "fp8_quantize_gathered", "fp8_gather_rows", "fp8_swiglu_quantize", "fp8_quantize_per_tensor_noalloc",
           "fp8bs_workspace_size", "fp8bs_workspace_size_for", "fp8bs_read_status", "fp8bs_clear_status",
           "fp8bs_status_string", "fp8bs_version", "fp8bs_test_stalled_gemm", "fp8bs_test_stalled_gemm_nvfp4",
           "fp8bs_test_stalled_gemm_blockwise",
           "fp8bs_test_quotient_sweep", "fp8bs_mma_peak", "fp8bs_test_noalloc_scratch",
           "fp8bs_test_encoder_breakpoints")

_lib = None


class Fp8bsError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)} ({status_string(code)})")
        self.code = code


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libfp8bs.so and declare its signatures (no GPU needed)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libfp8bs.so not found at {path}; build it with "
                           "`python -m fp8_block_scaled_03_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    P, I64, I, U, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
    lib.fp8_quantize.argtypes = [P, I64, I64, I64, I, P, P, P, U, P, SZ, P]
    lib.fp8_quantize_transposed.argtypes = [P, I64, I64, I64, I, P, P, P, P, P, U, P, SZ, P]
    lib.fp8_dequantize.argtypes = [P, P, P, I64, I64, I, P, I64, P]
    lib.fp8_block_gemm.argtypes = [P, P, I, P, P, I, P, P, I64, I64, I64, P, I, P, SZ, P]
    lib.fp8_grouped_gemm.argtypes = [P, P, P, P, P, P, P, I, I64, I64, I64, I, P, P, SZ, P]
    lib.fp8_quantize_gathered.argtypes = [P, I64, I64, I64, P, I64, I, P, P, P, SZ, P]
    lib.fp8_gather_rows.argtypes = [P, P, I64, I64, I, P, I64, P, P, P, SZ, P]
    lib.fp8_swiglu_quantize.argtypes = [P, I64, I64, I64, I, P, P, P]
    lib.fp8bs_test_stalled_gemm.argtypes = [P, P, P, P, I64, I64, I64, P, ctypes.c_uint64, P, SZ, P]
    lib.fp8bs_test_stalled_gemm_nvfp4.argtypes = [P, P, P, P, P, P, I64, I64, I64, P, ctypes.c_uint64, P, SZ, P]
    lib.fp8bs_test_stalled_gemm_nvfp4.restype = I
    lib.fp8bs_test_stalled_gemm_blockwise.argtypes = [P, P, I, P, P, I, I64, I64, I64, P, ctypes.c_uint64, P, SZ, P]
    lib.fp8bs_test_stalled_gemm_blockwise.restype = I
    lib.fp8bs_test_quotient_sweep.argtypes = [P, I, P]
    lib.fp8bs_test_quotient_sweep.restype = I
    lib.fp8bs_mma_peak.argtypes = [I, I, I, I, P, P, SZ, P]
    lib.fp8bs_test_encoder_breakpoints.argtypes = [P, P]
    lib.fp8bs_test_encoder_breakpoints.restype = I
    lib.fp8bs_test_noalloc_scratch.argtypes = [ctypes.POINTER(P), ctypes.POINTER(P)]
    lib.fp8bs_test_noalloc_scratch.restype = I
    lib.fp8bs_mma_peak.restype = I
    lib.fp8bs_workspace_size.restype = SZ
    lib.fp8bs_workspace_size.argtypes = []
    lib.fp8bs_workspace_size_for.restype = SZ
    lib.fp8bs_workspace_size_for.argtypes = [I, I64, I64, I, U]
    lib.fp8bs_read_status.argtypes = [P, P]
    lib.fp8bs_clear_status.argtypes = [P, P]
    lib.fp8bs_status_string.restype = ctypes.c_char_p
    lib.fp8bs_status_string.argtypes = [I]
    lib.fp8bs_version.argtypes = []
    for name in ("fp8_quantize", "fp8_quantize_transposed", "fp8_dequantize", "fp8_block_gemm", "fp8_grouped_gemm",
                 "fp8_quantize_gathered", "fp8_swiglu_quantize",
                 "fp8bs_read_status", "fp8bs_clear_status", "fp8bs_version", "fp8bs_test_stalled_gemm"):
        getattr(lib, name).restype = I
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().fp8bs_status_string(int(code)).decode()


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise Fp8bsError(fn, code)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


_workspaces = {}


def workspace(device=None) -> torch.Tensor:
    """A zero-initialised workspace per device (status word + amax scratch)."""
    dev = torch.device(device if device is not None else torch.cuda.current_device())
    if dev.type == "cuda" and dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    ws = _workspaces.get(dev)
    if ws is None:
        ws = torch.zeros(load_library().fp8bs_workspace_size(), dtype=torch.uint8, device=dev)
        _workspaces[dev] = ws
    return ws


def new_workspace(device=None) -> torch.Tensor:
    """A fresh zero-initialised workspace: calls that run concurrently (on
    different streams) need one each."""
    dev = torch.device(device if device is not None else torch.cuda.current_device())
    return torch.zeros(load_library().fp8bs_workspace_size(), dtype=torch.uint8, device=dev)


def read_status(ws: Optional[torch.Tensor] = None, stream=None) -> int:
    ws = ws if ws is not None else workspace()
    return load_library().fp8bs_read_status(_ptr(ws), _stream(stream))


def clear_status(ws: Optional[torch.Tensor] = None, stream=None) -> None:
    ws = ws if ws is not None else workspace()
    _check("fp8bs_clear_status", load_library().fp8bs_clear_status(_ptr(ws), _stream(stream)))


def _gran(g) -> int:
    return GRAN[g] if isinstance(g, str) else int(g)


def _cdiv(a: int, b: int) -> int:
    return -(-a // b)


def scale_shape(gran, rows: int, cols: int):
    """Shape and dtype of the scale tensor fp8_quantize writes for [rows, cols]."""
    g = _gran(gran)
    if g == 0:
        return (1,), torch.float32
    if g == 1:
        return (rows, _cdiv(cols, 128)), torch.float32
    if g == 2:
        return (_cdiv(rows, 128), _cdiv(cols, 128)), torch.float32
    if g == 3:
        return (rows, _cdiv(cols, 32)), torch.uint8
    if g == 5:
        return (rows, _cdiv(cols, 128)), torch.uint8
    if g == 6:
        return (_cdiv(rows, 128), _cdiv(cols, 128)), torch.uint8
    return (rows, cols // 16), torch.uint8


def _as_bf16_2d(x: torch.Tensor) -> torch.Tensor:
    if x.dtype == torch.uint16:
        x = x.view(torch.bfloat16)
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_cuda:
        raise ValueError("x must be a 2-D bfloat16 CUDA tensor")
    if x.stride(1) != 1:
        raise ValueError("x must have unit column stride")
    return x


def fp8_quantize(x: torch.Tensor, gran, *, q=None, scales=None, tensor_scale=None, flags: int = 0,
                 ws=None, stream=None):
    """Row-wise quantisation of a BF16 matrix; returns (q, scales, tensor_scale)."""
    x = _as_bf16_2d(x)
    g = _gran(gran)
    rows, cols = x.shape
    dev = x.device
    if q is None:
        q = torch.empty((rows, cols // 2 if g in NVFP4_GRANS else cols), dtype=torch.uint8, device=dev)
    if scales is None:
        shp, dt = scale_shape(g, rows, cols)
        scales = torch.empty(shp, dtype=dt, device=dev)
    if g in NVFP4_GRANS and tensor_scale is None:
        tensor_scale = torch.empty((rows if g == 7 else 1,), dtype=torch.float32, device=dev)
    ws = ws if ws is not None else workspace(dev)
    rc = load_library().fp8_quantize(_ptr(x), rows, cols, x.stride(0), g, _ptr(q), _ptr(scales),
                                     _ptr(tensor_scale), flags, _ptr(ws), ws.numel(), _stream(stream))
    _check("fp8_quantize", rc)
    return q, scales, tensor_scale


def fp8_quantize_transposed(x: torch.Tensor, gran, also_rowwise: bool = False, *, q_t=None, scales_t=None,
                            q=None, scales=None, flags: int = 0, ws=None, stream=None):
    """Quantise X^T (and optionally X in the same pass); returns (q_t, scales_t, q, scales)."""
    x = _as_bf16_2d(x)
    g = _gran(gran)
    rows, cols = x.shape
    dev = x.device
    if q_t is None:
        q_t = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
    if scales_t is None:
        shp, dt = scale_shape(g, cols, rows)
        scales_t = torch.empty(shp, dtype=dt, device=dev)
    if also_rowwise:
        if q is None:
            q = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
        if scales is None:
            shp, dt = scale_shape(g, rows, cols)
            scales = torch.empty(shp, dtype=dt, device=dev)
    ws = ws if ws is not None else workspace(dev)
    rc = load_library().fp8_quantize_transposed(_ptr(x), rows, cols, x.stride(0), g, _ptr(q_t), _ptr(scales_t),
                                                _ptr(q), _ptr(scales), None, flags, _ptr(ws), ws.numel(),
                                                _stream(stream))
    _check("fp8_quantize_transposed", rc)
    return q_t, scales_t, q, scales


def fp8_dequantize(q, scales, gran, cols: Optional[int] = None, tensor_scale=None, *, out=None, stream=None):
    """BF16 values of quantised codes (exact product rounded once); returns out [rows, cols]."""
    g = _gran(gran)
    rows = q.shape[0]
    if cols is None:
        cols = q.shape[1] * (2 if g in NVFP4_GRANS else 1)
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.bfloat16, device=q.device)
    rc = load_library().fp8_dequantize(_ptr(q), _ptr(scales), _ptr(tensor_scale), rows, cols, g, _ptr(out),
                                       out.stride(0), _stream(stream))
    _check("fp8_dequantize", rc)
    return out


OUT_DTYPES = {torch.bfloat16: 0, torch.float32: 1}     # FP8BS_OUT_BF16, FP8BS_OUT_F32


def fp8_block_gemm(a, a_scales, a_gran, b, b_scales, b_gran, a_tensor_scale=None, b_tensor_scale=None, *,
                   k: Optional[int] = None, out=None, out_dtype=None, ws=None, stream=None):
    """D = deq(A) . deq(B)^T in BF16 (or float32: out_dtype=torch.float32, or
    an `out` of that dtype).  A [m, k] and B [n, k] codes (NVFP4: packed [., k/2])."""
    ga, gb = _gran(a_gran), _gran(b_gran)
    m, n = a.shape[0], b.shape[0]
    if k is None:
        k = a.shape[1] * (2 if ga in NVFP4_GRANS else 1)
    if out_dtype is None:
        out_dtype = out.dtype if out is not None else torch.bfloat16
    if out_dtype not in OUT_DTYPES:
        raise ValueError(f"fp8_block_gemm: out_dtype must be bfloat16 or float32, not {out_dtype}")
    if out is None:
        out = torch.empty((m, n), dtype=out_dtype, device=a.device)
    elif out.dtype != out_dtype:
        raise ValueError("fp8_block_gemm: out.dtype differs from out_dtype")
    ws = ws if ws is not None else workspace(a.device)
    rc = load_library().fp8_block_gemm(_ptr(a), _ptr(a_scales), ga, _ptr(b), _ptr(b_scales), gb,
                                       _ptr(a_tensor_scale), _ptr(b_tensor_scale), m, n, k, _ptr(out),
                                       OUT_DTYPES[out_dtype], _ptr(ws), ws.numel(), _stream(stream))
    _check("fp8_block_gemm", rc)
    return out


def fp8_grouped_gemm(a, a_scales, b, b_scales, offsets, gran, *, a_tensor_scale=None, b_tensor_scale=None,
                     k: Optional[int] = None, out=None, ws=None, stream=None):
    """MoE grouped GEMM: rows offsets[e]..offsets[e+1] of A times B[e]^T; D BF16 [rows, n].
    NVFP4: a, b packed codes ([rows, k/2], [experts, n, k/2]); a_tensor_scale [1] or
    [rows] ("nvfp4_row"), b_tensor_scale [experts]."""
    g = _gran(gran)
    experts, n = b.shape[0], b.shape[1]
    rows = a.shape[0]
    if k is None:
        k = a.shape[1] * (2 if g in NVFP4_GRANS else 1)
    if offsets.dtype != torch.int64 or not offsets.is_cuda or offsets.numel() != experts + 1:
        raise ValueError("offsets must be a CUDA int64 tensor of experts+1 entries")
    if out is None:
        out = torch.empty((rows, n), dtype=torch.bfloat16, device=a.device)
    ws = ws if ws is not None else workspace(a.device)
    rc = load_library().fp8_grouped_gemm(_ptr(a), _ptr(a_scales), _ptr(b), _ptr(b_scales), _ptr(a_tensor_scale),
                                         _ptr(b_tensor_scale), _ptr(offsets), experts, rows, n, k, g, _ptr(out),
                                         _ptr(ws), ws.numel(), _stream(stream))
    _check("fp8_grouped_gemm", rc)
    return out


def fp8_quantize_gathered(x: torch.Tensor, token_index: torch.Tensor, gran, *, q=None, scales=None, ws=None,
                          stream=None):
    """Quantise the rows x[token_index] (MoE dispatch into expert order); returns (q, scales).
    An index outside [0, tokens) zeroes its row and sets FP8BS_EINDEX in the workspace
    status word (read_status)."""
    x = _as_bf16_2d(x)
    g = _gran(gran)
    tokens, cols = x.shape
    if token_index.dtype != torch.int64 or not token_index.is_cuda or token_index.dim() != 1:
        raise ValueError("token_index must be a 1-D CUDA int64 tensor")
    if not token_index.is_contiguous():
        raise ValueError("token_index must be contiguous")
    rows = token_index.numel()
    dev = x.device
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    if scales is None:
        shp, dt = scale_shape(g, rows, cols)
        scales = torch.empty(shp, dtype=dt, device=dev)
    ws = ws if ws is not None else workspace(dev)
    rc = load_library().fp8_quantize_gathered(_ptr(x), tokens, cols, x.stride(0), _ptr(token_index), rows, g,
                                              _ptr(q), _ptr(scales), _ptr(ws), ws.numel(), _stream(stream))
    _check("fp8_quantize_gathered", rc)
    return q, scales


def fp8_gather_rows(q_src: torch.Tensor, scales_src: torch.Tensor, token_index: torch.Tensor, gran, *, q=None,
                    scales=None, ws=None, stream=None):
    """Rows token_index[r] of already quantised (q_src, scales_src) in expert order; returns
    (q, scales).  Equals fp8_quantize_gathered on the BF16 rows those codes came from.  An
    index outside [0, tokens) gives an all-zero row and sets FP8BS_EINDEX (read_status)."""
    g = _gran(gran)
    if q_src.dtype != torch.uint8 or q_src.dim() != 2 or not q_src.is_contiguous():
        raise ValueError("q_src must be a contiguous 2-D uint8 tensor of codes")
    tokens, cols = q_src.shape
    shp, dt = scale_shape(g, tokens, cols)
    if scales_src.dtype != dt or tuple(scales_src.shape) != tuple(shp) or not scales_src.is_contiguous():
        raise ValueError(f"scales_src must be a contiguous {dt} tensor of shape {tuple(shp)}")
    if token_index.dtype != torch.int64 or not token_index.is_cuda or token_index.dim() != 1:
        raise ValueError("token_index must be a 1-D CUDA int64 tensor")
    if not token_index.is_contiguous():
        raise ValueError("token_index must be contiguous")
    rows = token_index.numel()
    dev = q_src.device
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
    if scales is None:
        shp, dt = scale_shape(g, rows, cols)
        scales = torch.empty(shp, dtype=dt, device=dev)
    ws = ws if ws is not None else workspace(dev)
    rc = load_library().fp8_gather_rows(_ptr(q_src), _ptr(scales_src), tokens, cols, g, _ptr(token_index), rows,
                                        _ptr(q), _ptr(scales), _ptr(ws), ws.numel(), _stream(stream))
    _check("fp8_gather_rows", rc)
    return q, scales


def fp8_swiglu_quantize(h: torch.Tensor, gran, inter: Optional[int] = None, *, q=None, scales=None, stream=None):
    """Quantise y = BF16(silu(h[:, :inter]) * h[:, inter:2*inter]) row-wise; returns (q, scales)."""
    h = _as_bf16_2d(h)
    g = _gran(gran)
    rows = h.shape[0]
    if inter is None:
        if h.shape[1] % 2:
            raise ValueError("h must hold [gate | up] of equal widths")
        inter = h.shape[1] // 2
    if 2 * inter > h.shape[1]:
        raise ValueError("h is narrower than 2 * inter")
    dev = h.device
    if q is None:
        q = torch.empty((rows, inter), dtype=torch.uint8, device=dev)
    if scales is None:
        shp, dt = scale_shape(g, rows, inter)
        scales = torch.empty(shp, dtype=dt, device=dev)
    rc = load_library().fp8_swiglu_quantize(_ptr(h), rows, inter, h.stride(0), g, _ptr(q), _ptr(scales),
                                            _stream(stream))
    _check("fp8_swiglu_quantize", rc)
    return q, scales


def test_stalled_gemm(a, a_scales, b, b_scales, wait_limit_ns: int, *, out=None, ws=None, stream=None) -> int:
    """Run the MXFP8 GEMM with its producer withholding stage 0 (test hook for the
    bounded waits); returns the launch status.  The timeout shows up in the
    workspace status word (read_status)."""
    m, k = a.shape
    n = b.shape[0]
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=a.device)
    ws = ws if ws is not None else workspace(a.device)
    return load_library().fp8bs_test_stalled_gemm(_ptr(a), _ptr(a_scales), _ptr(b), _ptr(b_scales), m, n, k,
                                                  _ptr(out), int(wait_limit_ns), _ptr(ws), ws.numel(),
                                                  _stream(stream))


def test_stalled_gemm_blockwise(a, a_scales, a_gran, b, b_scales, b_gran, wait_limit_ns: int, *, out=None, ws=None,
                                stream=None) -> int:
    """As test_stalled_gemm, for the FP32-scale blockwise GEMM."""
    m, k = a.shape
    n = b.shape[0]
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=a.device)
    ws = ws if ws is not None else workspace(a.device)
    return load_library().fp8bs_test_stalled_gemm_blockwise(_ptr(a), _ptr(a_scales), _gran(a_gran), _ptr(b),
                                                            _ptr(b_scales), _gran(b_gran), m, n, k, _ptr(out),
                                                            int(wait_limit_ns), _ptr(ws), ws.numel(),
                                                            _stream(stream))


def test_stalled_gemm_nvfp4(a, a_scales, b, b_scales, a_tensor_scale, b_tensor_scale, wait_limit_ns: int, *, k=None,
                            out=None, ws=None, stream=None) -> int:
    """As test_stalled_gemm, for the NVFP4 GEMM (packed codes [rows, k/2])."""
    m, n = a.shape[0], b.shape[0]
    k = k if k is not None else 2 * a.shape[1]
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=a.device)
    ws = ws if ws is not None else workspace(a.device)
    return load_library().fp8bs_test_stalled_gemm_nvfp4(_ptr(a), _ptr(a_scales), _ptr(b), _ptr(b_scales),
                                                        _ptr(a_tensor_scale), _ptr(b_tensor_scale), m, n, k,
                                                        _ptr(out), int(wait_limit_ns), _ptr(ws), ws.numel(),
                                                        _stream(stream))


def test_quotient_sweep(nvfp4=False, stream=None):
    """Run fp8bs_test_quotient_sweep (mode 0: FP32-scale E4M3 casts, 1 or
    True: NVFP4 element casts, 2: NVFP4 block scale codes); returns (pairs,
    code mismatches, fast-path scales)."""
    counts = torch.zeros(3, dtype=torch.int64, device="cuda")
    _check("fp8bs_test_quotient_sweep",
           load_library().fp8bs_test_quotient_sweep(_ptr(counts), int(nvfp4), _stream(stream)))
    c = counts.cpu().tolist()
    return c[0], c[1], c[2]


def test_encoder_breakpoints(stream=None):
    """Run fp8bs_test_encoder_breakpoints; returns the 266 breakpoint bit
    patterns (E4M3 positive, E4M3 negative, E2M1 positive, E2M1 negative)
    followed by the count of monotonicity and symmetry violations over every
    finite float32."""
    out = torch.zeros(267, dtype=torch.int32, device="cuda")
    _check("fp8bs_test_encoder_breakpoints", load_library().fp8bs_test_encoder_breakpoints(_ptr(out), _stream(stream)))
    return [v & 0xFFFFFFFF for v in out.cpu().tolist()]


MMA_PEAK_K = {0: 32, 1: 32, 2: 64}      # K per instruction: E4M3, MXFP8, NVFP4


def mma_peak(kind: int, n: int = 256, iters: int = 1024, pattern: int = 0, *, out=None, ws=None, stream=None) -> int:
    """Launch the tensor-core throughput loop (fp8bs_mma_peak) on the current
    stream; returns the FLOPs the launch performs (time it with CUDA events)."""
    ws = ws if ws is not None else workspace()
    _check("fp8bs_mma_peak", load_library().fp8bs_mma_peak(int(kind), int(n), int(iters), int(pattern), _ptr(out),
                                                           _ptr(ws), ws.numel(), _stream(stream)))
    sms = torch.cuda.get_device_properties(ws.device).multi_processor_count
    return sms * iters * 4 * 2 * 128 * n * MMA_PEAK_K[int(kind)]
