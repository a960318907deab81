/*
 * fp8bs.h -- C ABI of the block-scaled low-precision linear layer (sm_103a).
 *
 * What is computed (page title, section):
 *   "Unified FP8: Beyond Mixed Precision, Achieving Stable Accelerated MoE RL
 *    Training", section "FP8 Quantization":
 *      Step 1  S = max|X| / V_max  over the tensor or one block,
 *      Step 2  Q(x) = round(x / S),
 *   at per-tensor, per-token and per-block granularity, FP32 scales
 *   (section "FP8 Scale Selection"), E4M3 codes (section "FP8 Format").
 *   "Low Precision RL", table "Choose a precision": block-wise FP8 128x128
 *   with FP32 scales, MXFP8 1x32 with UE8M0 scales, NVFP4 E2M1 1x16 with an
 *   E4M3 block scale and an outer FP32 scale; sections "3. Unified MXFP8
 *   (Blackwell)" (MXFP8 also for weight-gradient and data-gradient GEMMs)
 *   and "4. NVFP4 (Blackwell)".
 *
 * Arithmetic contract (bit-exact against the CPU oracle):
 *   amax is exact; FP32 scales are IEEE float32 S = amax / 448 (S = 1 when
 *   amax = 0); codes are the saturating round-to-nearest-even E4M3 cast of
 *   the IEEE float32 quotient x / S (the kernels reach the same codes by a
 *   reciprocal and one correction step, see fp8bs_test_quotient_sweep).  MXFP8: S = 2^e with e the smallest
 *   integer such that 448 * 2^e >= amax, clamped to [-127, 127], stored as
 *   the UE8M0 byte e + 127 (amax = 0 gives byte 0).  NVFP4: S_g = amax_T /
 *   2688 (1 when amax_T = 0), block byte s_b = E4M3((amax_b / 6) / S_g),
 *   S_b = E4M3value(s_b) * S_g in float32, codes E2M1(x / S_b), all-zero
 *   codes for a block whose s_b is 0.  Inputs must be finite BF16.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library never allocates or frees memory, never synchronises, and
 *     enqueues all work on `stream` (a cudaStream_t; NULL = legacy stream).
 *   - Matrices are row-major.  `ld_x` is the row pitch of the BF16 input in
 *     elements.  Outputs are densely packed (pitch = their column count).
 *   - Arguments are checked on the host before any launch; a failed check
 *     returns a negative fp8bs_status and enqueues nothing.
 *   - `workspace` is a caller-owned, 16-byte aligned device buffer of at
 *     least FP8BS_WORKSPACE_BYTES bytes, zero-filled once by the caller before its
 *     first use.  Its first 4 bytes are a sticky device status word that
 *     kernels set (never clear) when a bounded wait gives up, a gathered
 *     token index is out of range or expert offsets are malformed; read it with
 *     fp8bs_read_status and clear it with fp8bs_clear_status.  Bytes
 *     [64, 80) hold the GEMMs' tile counter (the FP32-scale forms with
 *     128x128 or per-tensor B scales and the power-of-two forms: their CTAs
 *     take tiles in index order as they become free; the kernel's last CTA
 *     puts the counter back to 0, so it is 0 between calls).  From byte 256 on it is
 *     scratch for the per-tensor / NVFP4 amax reduction.  Calls that share a
 *     workspace must be ordered on the GPU (same stream or events); calls
 *     that run concurrently need a workspace each.
 *   - Launch failures return FP8BS_ECUDA (cudaGetLastError is consumed).
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fp8bs_stream_t;   /* identical to cudaStream_t */

typedef enum {
    FP8BS_OK = 0,
    FP8BS_EINVAL = -1,        /* bad size, granularity, or NULL pointer */
    FP8BS_EALIGN = -2,        /* pointer or pitch not 16-byte aligned */
    FP8BS_EUNSUPPORTED = -3,  /* valid request this library does not implement */
    FP8BS_ECUDA = -4,         /* a CUDA runtime call or launch failed */
    FP8BS_ETIMEOUT = -5,      /* (status word) a bounded device wait gave up */
    FP8BS_EWORKSPACE = -6,    /* workspace NULL or smaller than required */
    FP8BS_EINDEX = -7,        /* (status word) a gathered token index was out of range */
    FP8BS_EOFFSETS = -8       /* (status word) grouped-GEMM expert offsets broke their contract */
} fp8bs_status;

typedef enum {
    FP8BS_PER_TENSOR = 0,     /* one float32 scale for the tensor */
    FP8BS_TOKEN_1x128 = 1,    /* float32 scale per row and 128 columns */
    FP8BS_BLOCK_128x128 = 2,  /* float32 scale per 128x128 tile */
    FP8BS_MXFP8_1x32 = 3,     /* UE8M0 byte per row and 32 columns */
    FP8BS_NVFP4_1x16 = 4,     /* E4M3 byte per row and 16 columns + float32 S_g */
    FP8BS_TOKEN_1x128_POW2 = 5,   /* UE8M0 byte per row and 128 columns */
    FP8BS_BLOCK_128x128_POW2 = 6, /* UE8M0 byte per 128x128 tile */
    FP8BS_NVFP4_ROW_1x16 = 7      /* NVFP4 with one float32 S_g per row (per token) */
} fp8bs_gran;

#define FP8BS_WORKSPACE_BYTES ((size_t)16384)

/* flags for fp8_quantize / fp8_quantize_transposed */
#define FP8BS_FLAG_GIVEN_TENSOR_SCALE 1u  /* PER_TENSOR / NVFP4: *tensor_scale is
                                             an input (S, resp. S_g); skip the amax pass */
#define FP8BS_FLAG_NVFP4_4OVER6 2u        /* NVFP4 only: four-over-six block scales */

/*
 * fp8_quantize -- row-wise quantisation of a BF16 matrix x [rows, cols].
 *
 * Steps 1-2 of "FP8 Quantization" (review) at granularity `gran`.
 * Requirements: cols % 8 == 0 (cols % 16 == 0 for NVFP4), ld_x >= cols,
 * ld_x % 8 == 0, x 16-byte aligned, q 16-byte aligned.  rows or cols == 0
 * is a no-op (pointers are then not examined and may be NULL).  A last
 * group that runs past cols (or past rows for 128x128) is ragged: its amax
 * covers only the elements that exist.
 *
 *   gran             q (uint8)             scales
 *   PER_TENSOR       E4M3 [rows, cols]     float32 [1]
 *   TOKEN_1x128      E4M3 [rows, cols]     float32 [rows, ceil(cols/128)]
 *   BLOCK_128x128    E4M3 [rows, cols]     float32 [ceil(rows/128), ceil(cols/128)]
 *   MXFP8_1x32       E4M3 [rows, cols]     uint8 UE8M0 [rows, ceil(cols/32)]
 *   NVFP4_1x16       E2M1 [rows, cols/2]   uint8 E4M3 [rows, cols/16]
 *                    (element 2j in the low nibble of byte j)
 *   NVFP4_ROW_1x16   as NVFP4_1x16
 *   TOKEN_1x128_POW2 E4M3 [rows, cols]     uint8 UE8M0 [rows, ceil(cols/128)]
 *   BLOCK_128x128_POW2 E4M3 [rows, cols]   uint8 UE8M0 [ceil(rows/128), ceil(cols/128)]
 *
 * The two _POW2 granularities are the block-wise recipe with power-of-two
 * scales ("Low Precision RL", section "2. Unified block-wise FP8": on
 * Blackwell the block-wise recipe runs through MXFP8 and needs power-of-two
 * scales): the MXFP8 scale rule applied to 1x128 groups or 128x128 tiles.
 *
 * tensor_scale: NVFP4 only, device float32[1], receives S_g (or supplies it
 * with FP8BS_FLAG_GIVEN_TENSOR_SCALE).  NVFP4_ROW_1x16: device float32[rows],
 * S_g of each row (per-token activation scaling, "4. NVFP4 (Blackwell)"):
 * S_g[r] = amax(row r) / 2688, 1 for an all-zero row; supplied by the caller
 * with FP8BS_FLAG_GIVEN_TENSOR_SCALE.  PER_TENSOR with that flag reads S
 * from scales[0].  Otherwise may be NULL.  Gate and up projections that
 * share one outer weight scale ("4. NVFP4 (Blackwell)") quantise their
 * concatenation, or pass the shared S_g with FP8BS_FLAG_GIVEN_TENSOR_SCALE.
 *
 * FP8BS_FLAG_NVFP4_4OVER6 ("Low Precision RL", "Advanced: four-over-six";
 * NVFP4_1x16 and NVFP4_ROW_1x16 only, else FP8BS_EINVAL): the outer divisor
 * becomes 256 * 6 (S_g = amax / 1536), each 1x16 block is quantised with
 * its amax mapped to 6 (s_b = E4M3((amax_b / 6) / S_g)) and to 4
 * (s_b = E4M3((amax_b / 4) / S_g)), and keeps the map-to-4 result only when
 * its squared error is strictly smaller.  The error of one choice: y =
 * E2M1value(q) * S_b, d = x - y, d * d, each an IEEE float32 operation
 * without fused multiply-add, summed in float32 over elements 0..7 and
 * 8..15 of the block in order, then the two half sums added.
 * Unknown flag bits return FP8BS_EINVAL.
 * workspace: required for PER_TENSOR and NVFP4_1x16 (amax partials); may
 * be NULL for the other granularities.
 */
int fp8_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int gran,
                 void* q, void* scales, float* tensor_scale, unsigned flags,
                 void* workspace, size_t workspace_bytes, fp8bs_stream_t stream);

/*
 * fp8_quantize_transposed -- quantise X^T [cols, rows] from the same BF16
 * source, and optionally X itself in the same pass over memory.
 *
 * Used by the backward GEMMs ("Low Precision RL", "3. Unified MXFP8
 * (Blackwell)": low-precision weight-gradient and data-gradient GEMMs),
 * which contract over the other axis of X.  The result is exactly
 * fp8_quantize applied to the transposed BF16 matrix (never a re-rounding
 * of already-quantised codes).  For BLOCK_128x128 the codes are the
 * transpose of the row-wise codes and the scales the transposed scale grid.
 *
 * gran: PER_TENSOR, TOKEN_1x128, BLOCK_128x128, MXFP8_1x32 or the two
 * _POW2 granularities (both NVFP4 granularities return FP8BS_EUNSUPPORTED).  Requirements as fp8_quantize plus rows % 16 == 0 and cols, ld_x below 2^31 - 256 (X is read by TMA).
 *   q_t      uint8 [cols, rows]           codes of X^T
 *   scales_t layout of the table above for a [cols, rows] matrix
 *   q, scales  optional (both NULL or both set): the row-wise result of
 *            fp8_quantize(x, gran), produced from the same read of x.
 */
int fp8_quantize_transposed(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int gran,
                            void* q_t, void* scales_t, void* q, void* scales,
                            float* tensor_scale, unsigned flags,
                            void* workspace, size_t workspace_bytes, fp8bs_stream_t stream);

/*
 * fp8_dequantize -- BF16 values of quantised codes: out[r, c] = BF16(code *
 * scale) (NVFP4: E2M1 code * E4M3 block scale * outer scale), the exact
 * product rounded once to nearest-even.
 *
 * The dequantized backward of "Low Precision RL" ("Advanced: dequantized
 * backward"): the BF16 backward GEMMs consume BF16 dequantisations of the
 * operands quantised for the forward pass.  q and scales as written by
 * fp8_quantize for the same gran and [rows, cols]; out BF16 [rows, cols] with
 * row pitch ld_out elements (ld_out >= cols, ld_out % 8 == 0), 16-byte
 * aligned; q 8-byte aligned.  cols % 8 == 0 (% 16 for NVFP4).  tensor_scale:
 * NVFP4 only, device float32[1] (float32[rows] for NVFP4_ROW_1x16), 4-byte
 * aligned.  rows or cols == 0 is a no-op.  UE8M0 byte 0xFF (NaN) is not
 * accepted as a scale (results unspecified).
 */
int fp8_dequantize(const void* q, const void* scales, const float* tensor_scale, int64_t rows, int64_t cols,
                   int gran, void* out, int64_t ld_out, fp8bs_stream_t stream);

/*
 * fp8_quantize_gathered -- quantise the rows x[token_index[r]] (r = 0 ..
 * rows-1) of a BF16 token matrix x [tokens, cols] in one pass: the MoE
 * dispatch that lays the routed tokens out in expert order for the grouped
 * GEMM ("Low Precision RL", section "3. Unified MXFP8 (Blackwell)": MoE
 * layers run their own GEMM backend on the routed tokens).  The pages do not
 * describe this step; it computes exactly fp8_quantize of the gathered BF16
 * matrix.
 *
 *   x            BF16 [tokens, cols], pitch ld_x (ld_x >= cols, ld_x % 8 == 0),
 *                16-byte aligned; cols % 8 == 0
 *   token_index  DEVICE int64 [rows], 8-byte aligned: the source token of
 *                each output row (repeats allowed: a token routed to k
 *                experts appears k times)
 *   gran         TOKEN_1x128, MXFP8_1x32 or TOKEN_1x128_POW2 (the other
 *                valid granularities return FP8BS_EUNSUPPORTED)
 *   q, scales    as fp8_quantize for [rows, cols] at `gran`
 *   workspace    required (FP8BS_WORKSPACE_BYTES): its status word receives
 *                FP8BS_EINDEX when an index is outside [0, tokens); such a
 *                row is quantised as an all-zero row (zero codes, scale of
 *                an all-zero group) and the other rows are unaffected.
 * rows or cols == 0 is a no-op.  tokens may be 0 (then every index is out
 * of range and x may be NULL).
 */
int fp8_quantize_gathered(const void* x, int64_t tokens, int64_t cols, int64_t ld_x,
                          const int64_t* token_index, int64_t rows, int gran, void* q, void* scales,
                          void* workspace, size_t workspace_bytes, fp8bs_stream_t stream);

/*
 * fp8_gather_rows -- the MoE dispatch of rows that are already quantised:
 * row r of (q, scales) is row token_index[r] of (q_src, scales_src).  A
 * row's codes and scales depend on that row alone, so fp8_quantize of x
 * followed by this call gives exactly what fp8_quantize_gathered gives from
 * x; the token matrix is then quantised once, not once per routed copy
 * (the same MoE step, "Low Precision RL", section "3. Unified MXFP8
 * (Blackwell)"; the pages do not describe it).
 *
 *   q_src, scales_src  codes [tokens, cols] (pitch cols) and scales of
 *                fp8_quantize at `gran`, 16-byte aligned codes, scales
 *                aligned as fp8_quantize's; cols % 8 == 0
 *   gran         TOKEN_1x128, MXFP8_1x32 or TOKEN_1x128_POW2 (the other
 *                valid granularities return FP8BS_EUNSUPPORTED)
 *   token_index  DEVICE int64 [rows], 8-byte aligned (repeats allowed)
 *   q, scales    [rows, cols] in the same layouts, written
 *   workspace    required (FP8BS_WORKSPACE_BYTES): its status word receives
 *                FP8BS_EINDEX when an index is outside [0, tokens); that row
 *                gets zero codes and the scale of an all-zero group (1.0f
 *                for TOKEN_1x128, the byte 0 otherwise), as in
 *                fp8_quantize_gathered; the other rows are unaffected.
 * rows or cols == 0 is a no-op.  tokens may be 0 (then q_src and scales_src
 * may be NULL).
 */
int fp8_gather_rows(const void* q_src, const void* scales_src, int64_t tokens, int64_t cols, int gran,
                    const int64_t* token_index, int64_t rows, void* q, void* scales, void* workspace,
                    size_t workspace_bytes, fp8bs_stream_t stream);

/*
 * fp8_swiglu_quantize -- the SwiGLU activation between the gate+up and the
 * down projection of an expert MLP, quantised row-wise for the down GEMM
 * (Qwen3 MoE experts, "Low Precision RL", section "3. Unified MXFP8
 * (Blackwell)"; the pages do not describe this step).
 *
 *   h       BF16 [rows, 2 * inter] = [gate | up] (gate in columns 0 ..
 *           inter-1, up in inter .. 2*inter-1), pitch ld_h >= 2 * inter,
 *           ld_h % 8 == 0, 16-byte aligned; inter % 8 == 0
 *   y[r,c]  = BF16(silu(g) * u), g = h[r,c], u = h[r,inter+c],
 *           silu(g) = g / (1 + e^-g): the exact value rounded once to
 *           nearest-even BF16, except where the exact value lies within 8
 *           float32 ulps (or 2^-146) of a BF16 rounding boundary, where
 *           either neighbouring BF16 value may result.  (The kernel
 *           evaluates y in float32: e^t by Cody-Waite reduction with ln 2
 *           split in two and the Taylor series of e^r to r^7, the quotient
 *           by a refined reciprocal and one correction step, within a few
 *           float32 ulps; gates below -80, where e^-g leaves the float32
 *           range, in float64.)  y must be finite.
 *   gran    TOKEN_1x128, MXFP8_1x32 or TOKEN_1x128_POW2 (other valid
 *           granularities return FP8BS_EUNSUPPORTED)
 *   q, scales  as fp8_quantize of y [rows, inter] at `gran`
 * rows or inter == 0 is a no-op.  y itself is not written.
 */
int fp8_swiglu_quantize(const void* h, int64_t rows, int64_t inter, int64_t ld_h, int gran, void* q, void* scales,
                        fp8bs_stream_t stream);

/* Output types of fp8_block_gemm's D. */
typedef enum {
    FP8BS_OUT_BF16 = 0,
    FP8BS_OUT_F32 = 1
} fp8bs_out_dtype;

/*
 * fp8_block_gemm -- D[m, n] = sum_k deq(A)[m, k] * deq(B)[n, k], D in BF16
 * or float32.
 *
 * The matching low-precision GEMM of "Low Precision RL" ("Unified training
 * recipe"), on operands quantised as above, with FP32 accumulation on the
 * tensor cores.  A is [m, k], B is [n, k]; both K-major (row-major with k
 * contiguous); D is row-major [m, n]: d_dtype FP8BS_OUT_BF16 rounds the FP32
 * accumulator to BF16 (round-to-nearest-even), FP8BS_OUT_F32 writes the
 * accumulator itself (for a caller that accumulates in float32, e.g. weight
 * gradients into float32 main gradients).  Both come from the same
 * accumulator: the BF16 output is the float32 output rounded.  Other
 * d_dtype values return FP8BS_EINVAL.
 *
 *   (a_gran, b_gran)                          scale handling
 *   {PER_TENSOR,TOKEN_1x128,BLOCK_128x128}^2  FP32 scales applied per
 *       128-wide K block to the FP32 partial sums (k % 128 == 0)
 *   (MXFP8_1x32, MXFP8_1x32)                  UE8M0 scales applied by the
 *       tensor core per 32-wide K block (k % 128 == 0)
 *   {TOKEN_1x128_POW2,BLOCK_128x128_POW2}^2   UE8M0 scales of 128-wide K
 *       blocks, each applied by the tensor core to its four 32-wide sub-blocks
 *       (k % 128 == 0)
 *   (NVFP4_1x16, NVFP4_1x16)                  E4M3 block scales applied by
 *       the tensor core per 16-wide K block, times *a_tensor_scale *
 *       *b_tensor_scale (k % 256 == 0); a, b are packed E2M1 [m|n, k/2]
 *   (NVFP4_ROW_1x16, NVFP4_1x16)              as above, row i of D times
 *       a_tensor_scale[i] * *b_tensor_scale (per-token activation scale)
 * Other pairs return FP8BS_EUNSUPPORTED.  Scale layouts are those written
 * by fp8_quantize for the operand's own [rows, k] shape.  m, n > 0,
 * n % 8 == 0, and m, n, k below 2^31 - 256 (TMA coordinates are 32-bit);
 * a, b, d 16-byte aligned.  a_tensor_scale / b_tensor_scale:
 * device float32[1], NVFP4 only (else ignored, may be NULL);
 * a_tensor_scale is float32[m] for NVFP4_ROW_1x16.
 * workspace: required (status word for the bounded pipeline waits).
 */
int fp8_block_gemm(const void* a, const void* a_scales, int a_gran,
                   const void* b, const void* b_scales, int b_gran,
                   const float* a_tensor_scale, const float* b_tensor_scale,
                   int64_t m, int64_t n, int64_t k, void* d, int d_dtype,
                   void* workspace, size_t workspace_bytes, fp8bs_stream_t stream);

/*
 * fp8_grouped_gemm -- MoE grouped (per-expert) GEMM.
 *
 * Rows offsets[e] .. offsets[e+1]-1 of A (expert-contiguous routed tokens)
 * are multiplied by expert e's weight B[e] ([n, k]):
 *   D[r, j] = sum_k deq(A)[r, k] * deq(B[e])[j, k]   for offsets[e] <= r < offsets[e+1]
 * ("Low Precision RL", "3. Unified MXFP8 (Blackwell)": the MoE GEMM backend
 * chosen separately from the dense one).  offsets: DEVICE int64 [experts+1],
 * non-decreasing, offsets[0] == 0, offsets[experts] == total_rows.  The host
 * never reads it; the kernel checks it: expert e's rows are taken as
 * [lo, hi) with lo = offsets[e] clamped to [0, total_rows] and hi =
 * offsets[e+1] clamped to [lo, total_rows], so no offsets can make the GEMM
 * read or write outside A, D or their scales, and offsets that break the
 * contract set the status word to FP8BS_EOFFSETS (the well-formed experts'
 * rows are still computed; D rows no expert covers are not written).
 * Experts with no rows cost nothing.
 *
 *   gran                 A                      B[e]                 k
 *   MXFP8_1x32           MXFP8                  MXFP8                % 128
 *   TOKEN_1x128          1x128 FP32 scales      128x128 FP32 scales  % 128
 *   TOKEN_1x128_POW2     1x128 power of two     128x128 power of two % 128
 *   NVFP4_1x16           NVFP4, S_g per tensor  NVFP4                % 256
 *   NVFP4_ROW_1x16       NVFP4, S_g per row     NVFP4                % 256
 * ("Low Precision RL", table "Choose a precision": the NVFP4 recipe on the
 * Qwen3-30B-A3B MoE; "4. NVFP4 (Blackwell)": per-token activation scales,
 * gate and up sharing one outer weight scale.)  a: [total_rows, k] codes
 * (NVFP4: packed [total_rows, k/2]), a_scales as fp8_quantize for
 * [total_rows, k]; b: [experts, n, k] codes (NVFP4: [experts, n, k/2]),
 * b_scales: the per-expert scale grids stacked along the expert axis.
 * a_tensor_scale: NVFP4 only, DEVICE float32[1] (NVFP4_1x16) or
 * float32[total_rows] (NVFP4_ROW_1x16); b_tensor_scale: NVFP4 only, DEVICE
 * float32[experts], the outer scale S_g of each expert's weight; row r of
 * expert e is multiplied by a_tensor_scale[0 or r] * b_tensor_scale[e].  Both
 * are ignored (may be NULL) for the other granularities.  NVFP4 block scales
 * 16-byte aligned.  D: BF16 [total_rows, n].  n % 8 == 0; total_rows,
 * experts * n and k below 2^31 - 256 (TMA coordinates).  workspace
 * required.
 */
int fp8_grouped_gemm(const void* a, const void* a_scales,
                     const void* b, const void* b_scales,
                     const float* a_tensor_scale, const float* b_tensor_scale,
                     const int64_t* offsets, int experts, int64_t total_rows,
                     int64_t n, int64_t k, int gran, void* d,
                     void* workspace, size_t workspace_bytes, fp8bs_stream_t stream);

/*
 * fp8bs_test_stalled_gemm -- test hook for the bounded pipeline waits.
 *
 * Runs the MXFP8 fp8_block_gemm (same arguments and requirements) with its
 * TMA producer withholding the first pipeline stage, so the MMA issuer waits
 * on a barrier that nothing will complete.  Every wait is bounded by
 * wait_limit_ns (1 .. 2e9): the kernel gives up, writes FP8BS_ETIMEOUT to
 * the workspace status word, lets its own copies in flight land, frees its
 * tensor memory and returns; the CUDA context stays usable.  No counterpart
 * on the pages: it exists to test failure detection without a GPU fault.
 * The contents of d are unspecified afterwards.
 */
int fp8bs_test_stalled_gemm(const void* a, const void* a_scales, const void* b, const void* b_scales,
                            int64_t m, int64_t n, int64_t k, void* d, uint64_t wait_limit_ns,
                            void* workspace, size_t workspace_bytes, fp8bs_stream_t stream);

/*
 * fp8bs_test_stalled_gemm_blockwise -- as fp8bs_test_stalled_gemm for the
 * FP32-scale blockwise GEMM (fp8_block_gemm with a_gran, b_gran in
 * {PER_TENSOR, TOKEN_1x128, BLOCK_128x128}; same arguments and
 * requirements, k % 128 == 0).  Its epilogue warps, which promote every
 * K block out of two TMEM buffers, and its scale-loader warp must all give
 * up on the abort, and the CTA must still free its tensor memory.  No
 * counterpart on the pages.  The contents of d are unspecified afterwards.
 */
int fp8bs_test_stalled_gemm_blockwise(const void* a, const void* a_scales, int a_gran, const void* b,
                                      const void* b_scales, int b_gran, int64_t m, int64_t n, int64_t k, void* d,
                                      uint64_t wait_limit_ns, void* workspace, size_t workspace_bytes,
                                      fp8bs_stream_t stream);

/*
 * fp8bs_test_stalled_gemm_nvfp4 -- as fp8bs_test_stalled_gemm for the
 * NVFP4 GEMM (both operands NVFP4_1x16, tensor scales as fp8_block_gemm,
 * k % 256 == 0, block scales 16-byte aligned).  Its scale loaders issue the
 * scale copies to tensor memory themselves, so this also covers their
 * drain on the abort path.  The contents of d are unspecified afterwards.
 */
int fp8bs_test_stalled_gemm_nvfp4(const void* a, const void* a_scales, const void* b, const void* b_scales,
                                  const float* a_tensor_scale, const float* b_tensor_scale, int64_t m, int64_t n,
                                  int64_t k, void* d, uint64_t wait_limit_ns, void* workspace,
                                  size_t workspace_bytes, fp8bs_stream_t stream);

/*
 * fp8bs_test_quotient_sweep -- exhaustive check of how the casts divide by
 * a scale derived from an amax.  They do not call IEEE division per
 * element: they take one correctly rounded reciprocal r = RN(1/S) per
 * group, then q = RN(y + RN(x - y S) r) with y = RN(x r) (Markstein's
 * correction step).  q can differ from RN(x / S) in its last bit but, on
 * the whole domain of the casts, never in its code; this call enumerates
 * that domain and compares the codes:
 *   nvfp4 = 0  E4M3 casts with FP32 scales: every positive finite BF16
 *              amax, S = amax / 448, every finite BF16 x with |x| <= amax
 *              (about 1.03e9 pairs);
 *   nvfp4 = 1  E2M1 casts of NVFP4: every positive finite BF16 amax_T,
 *              S_g = amax_T / 2688 and amax_T / 1536 (four-over-six), every
 *              block scale code 1..126, S = E4M3value * S_g, every finite
 *              BF16 x with |x| <= amax_T (about 1.3e11 pairs);
 *   nvfp4 = 2  NVFP4 block scale codes E4M3(RN(RN(a / 6) / S_g)), and
 *              E4M3(RN(RN(a / 4) / S_g)) for the four-over-six divisor,
 *              which the quantisers take as RN(a / 6) by the same
 *              correction step with r = RN(1/6), the exact a * 0.25, then
 *              the correction step with r = RN(1/S_g): every positive
 *              finite BF16 amax_T, both outer divisors, every BF16 block
 *              amax a <= amax_T (about 1.6e9 codes); also RN(a / 6) itself,
 *              bit for bit, for every finite BF16 a >= 0;
 *   nvfp4 = 3  FP32 scales of the casts: for every finite BF16 amax, the
 *              scale S = RN(amax / 448) and its reciprocal RN(1/S), which
 *              the quantisers take for amax >= 2^-79 by the correction step
 *              (r = RN(1/448)) and by two Newton steps from the hardware's
 *              approximate reciprocal, against IEEE division and
 *              reciprocal, bit for bit ([0] amax values, [1] mismatches,
 *              [2] values on that path).
 *   counts  DEVICE uint64[3], zero-filled by the caller, 8-byte aligned;
 *           receives [0] pairs checked, [1] pairs whose codes differ (0 is
 *           the contract; mode 2 also counts RN(a / 6) mismatches here),
 *           [2] scales on the fast path (S >= 2^-88; smaller ones divide
 *           exactly).
 * Runs for about a millisecond (nvfp4 = 0, 2, 3) or a second (nvfp4 = 1).
 * No counterpart on the pages.
 */
int fp8bs_test_quotient_sweep(unsigned long long* counts, int nvfp4, fp8bs_stream_t stream);

/*
 * fp8bs_test_encoder_breakpoints -- where the device casts change code.
 * The saturating round-to-nearest-even casts to E4M3 and E2M1 ("Low
 * Precision RL", table "Choose a precision": FP8 E4M3 and NVFP4 E2M1
 * elements) are monotone in |x|, so each is fixed by its breakpoints: for
 * every nonzero code magnitude c, the smallest float32 magnitude whose code
 * has magnitude >= c.  A one-CTA kernel finds them by binary search over
 * the float32 bit patterns, through the same packed casts the quantisers
 * use, for both signs.
 *   out  DEVICE uint32[267]: out[s*126 + c-1] (s = 0 positive, 1 negative,
 *        c = 1..126) the E4M3 breakpoints' float32 bits (magnitude);
 *        out[252 + s*7 + c-1] (c = 1..7) the E2M1 ones.  An entry is
 *        0xFFFFFFFF if the lanes of a packed cast disagreed or a code had
 *        the wrong sign.  out[266], zero-filled by the caller, receives the
 *        count of violations of monotonicity (the code magnitude of the
 *        successor of every finite positive float32 bit pattern is at least
 *        its own) and of symmetry (the code of -x is that of x with the sign
 *        bit set), for both casts over all 2^31 patterns; with the
 *        breakpoints this fixes the casts on every finite float32.
 * FP8BS_EINVAL for NULL, FP8BS_EALIGN if out is not 4-byte aligned.
 */
int fp8bs_test_encoder_breakpoints(uint32_t* out, fp8bs_stream_t stream);

/*
 * fp8bs_mma_peak -- dense tensor-core throughput loop, to measure the FP8
 * and FP4 MMA rates that the GEMM rooflines divide by.  The pages compare
 * FP8 with BF16 tensor throughput ("Unified FP8 ...", section "Tensor
 * Cores": FP8 at twice the BF16 rate on H100); this measures the rate on
 * the GPU at hand instead of assuming a ratio.
 *
 * One CTA per SM; each keeps its operands in shared memory (no memory
 * traffic) and one thread issues `iters` K blocks of four tcgen05.mma
 * instructions (M = 128 rows, N = n columns) into a TMEM accumulator:
 *   kind 0  E4M3 x E4M3, FP32 accumulate (kind::f8f6f4), K = 32 per instruction
 *   kind 1  MXFP8: E4M3 with UE8M0 scales per 32 (block_scale, scale_vec::1X), K = 32
 *   kind 2  NVFP4: E2M1 with E4M3 scales per 16 (block_scale, scale_vec::4X), K = 64
 * FLOPs per call = SMs * iters * 4 * 2 * 128 * n * K; the caller times the
 * call (CUDA events on `stream`).  n: 64 (kind 0 only), 128 or 256;
 * iters: 1 .. 2^24.
 * pattern 0: pseudo-random finite operands; pattern 1: every operand and
 * scale 1.0, so every accumulator element ends at iters * 4 * K.
 * out: NULL, or DEVICE float32[128] receiving column 0 of the first CTA's
 * accumulator (rows 0..127).  workspace: required (status word; the final
 * wait is bounded like the GEMMs').  No counterpart on the pages beyond the
 * comparison above.
 */
int fp8bs_mma_peak(int kind, int n, int iters, int pattern, float* out, void* workspace, size_t workspace_bytes,
                   fp8bs_stream_t stream);

/*
 * fp8_quantize_per_tensor_noalloc -- fp8_quantize(gran = PER_TENSOR) for
 * callers that cannot allocate device memory.  The pages have no
 * counterpart: this is an interface variant, not a different computation.
 *
 * The per-tensor scale needs the amax of the whole tensor before any code is
 * written, and the usual entry point keeps the partial maxima of that
 * reduction in a caller-provided workspace.  Callers that only receive the
 * input and output buffers (a framework allocator owns all device memory, a
 * plugin interface passes tensors but no scratch, a real-time caller forbids
 * allocation while running) use this entry point instead: the partials live
 * in a fixed array inside the library's device module
 * (FP8BS_NOALLOC_MAX_PARTIALS 32-bit words, 16 KB).  It never calls an
 * allocating routine itself, but the array is committed when the module is
 * loaded on a device, and under CUDA's default lazy module loading that
 * happens at the first call on that device (in that context).  A caller
 * with a strict no-allocation phase makes one warm-up call on each device
 * before that phase (and before any stream capture).
 *
 *   x      BF16 [rows, cols], pitch ld_x (as fp8_quantize)
 *   q      E4M3 codes [rows, cols], written
 *   scale  device float32[1], receives S = amax / 448 (1 for an all-zero tensor)
 * Results are identical to fp8_quantize(x, ..., FP8BS_PER_TENSOR, q, scale, ...).
 *
 * Limit: rows * ceil(cols / 1024) <= 64 * FP8BS_NOALLOC_MAX_PARTIALS
 * (262144; e.g. 268,435,456 elements when cols is a multiple of 1024);
 * larger inputs return FP8BS_EINVAL and launch nothing.  Other checks and
 * codes as fp8_quantize.  The first call in each context looks up the
 * array's device address (cudaGetSymbolAddress) and caches it under the
 * context's unique id, so a context destroyed and created again
 * (cudaDeviceReset) is looked up afresh rather than served a stale address.
 * Every call uses the same array: calls that overlap on the GPU (different
 * streams without ordering) race and give wrong scales.
 */
#define FP8BS_NOALLOC_MAX_PARTIALS 4096
int fp8_quantize_per_tensor_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld_x, void* q,
                                    float* scale, fp8bs_stream_t stream);

/*
 * fp8bs_test_noalloc_scratch -- test hook for the entry point above.
 * Writes to *cached the device address of its partials array that the
 * entry point would use in the calling thread's current context (through
 * its per-context cache, looking it up if needed) and to *looked_up the
 * address a fresh cudaGetSymbolAddress returns.  They are equal unless the
 * cache is stale.  Launches nothing.  FP8BS_EINVAL for NULL arguments,
 * FP8BS_ECUDA if a lookup fails.
 */
int fp8bs_test_noalloc_scratch(void** cached, void** looked_up);

/* Bytes of workspace every entry point accepts (FP8BS_WORKSPACE_BYTES). */
size_t fp8bs_workspace_size(void);

/* Operations, for fp8bs_workspace_size_for. */
typedef enum {
    FP8BS_OP_QUANTIZE = 0,
    FP8BS_OP_QUANTIZE_TRANSPOSED = 1,
    FP8BS_OP_DEQUANTIZE = 2,
    FP8BS_OP_BLOCK_GEMM = 3,
    FP8BS_OP_GROUPED_GEMM = 4,
    FP8BS_OP_QUANTIZE_GATHERED = 5,
    FP8BS_OP_GATHER_ROWS = 6,
    FP8BS_OP_SWIGLU_QUANTIZE = 7
} fp8bs_op;

/* Bytes of workspace one call of `op` on a [rows, cols] operand at
 * granularity `gran` (and `flags`, as passed to the quantisers) requires:
 * 0 when the call takes none (it may then be NULL), else
 * FP8BS_WORKSPACE_BYTES.  The size does not grow with the operand: the
 * status word is 4 bytes, and the tensor-amax reduction of PER_TENSOR and
 * NVFP4_1x16 quantisation uses at most 4032 partial maxima whatever the
 * size.  Returns (size_t)-1 for an unknown op or granularity or negative
 * sizes. */
size_t fp8bs_workspace_size_for(int op, int64_t rows, int64_t cols, int gran, unsigned flags);

/* Synchronises `stream`, then returns the sticky device status word of
 * `workspace` (FP8BS_OK, FP8BS_ETIMEOUT if a bounded wait gave up,
 * FP8BS_EINDEX if a gathered token index was out of range, or
 * FP8BS_EOFFSETS if grouped-GEMM offsets broke their contract), or
 * FP8BS_ECUDA if the copy failed. */
int fp8bs_read_status(const void* workspace, fp8bs_stream_t stream);

/* Enqueues a reset of the status word to FP8BS_OK on `stream`. */
int fp8bs_clear_status(void* workspace, fp8bs_stream_t stream);

/* Static English text for a status code. */
const char* fp8bs_status_string(int status);

/* ABI version: 100 * major + minor. */
int fp8bs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
