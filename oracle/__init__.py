"""CPU oracle for the block-scaled low-precision linear layer.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously-correct
restatement of what the pages define; it exists to check the CUDA path.
Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it.  The product path
(``fp8_block_scaled_03_gb300``) never imports it and shares no code with it.

Sources (page title, section):

* "Unified FP8: Beyond Mixed Precision, Achieving Stable Accelerated MoE RL
  Training" (review page), section "FP8 Quantization": Step 1, the scale
  S = max|X| / V_max over a tensor or block; Step 2, Q(x) = round(x / S);
  the per-tensor / per-token / per-block granularities; section "FP8 Format"
  (E4M3); section "FP8 Scale Selection" (FP32 scales for training).
* "Low Precision RL" (Miles docs), table "Choose a precision": block-wise FP8
  128x128 with FP32 scales, MXFP8 1x32 with UE8M0 scales, NVFP4 E2M1 1x16 with
  two-level (E4M3 + FP32) scales; sections "3. Unified MXFP8 (Blackwell)" and
  "4. NVFP4 (Blackwell)"; the NVFP4 launcher settings that switch off 2D
  quantisation, RHT, stochastic rounding and fast math.

Modules:
  formats   -- E4M3 / E2M1 / UE8M0 / BF16 codecs (decode tables from the bit
               definitions; encode = nearest table value, ties to even)
  quantize  -- the quantisers at every granularity, row-wise and transposed
  gemm      -- dequantise in float64, multiply in float64, round to BF16

Parity-unpinned readings (the pages do not fix them; see the tests for what
is pinned): the scale used when a block is all zero (S = 1, UE8M0 2^-127,
NVFP4 S_g = 1), the NVFP4 two-level scale formula, and the all-zero code
emitted for an NVFP4 block whose E4M3 block scale rounds to zero.
"""
from . import formats, quantize, gemm  # noqa: F401
