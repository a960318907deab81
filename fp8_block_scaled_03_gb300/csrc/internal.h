// internal.h -- launchers behind the C ABI (host side, not exported).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace fp8bs {

// Workspace layout: [0, 4) sticky status word; [256, ...) amax partials.
constexpr size_t kWorkspaceBytes = 16384;
constexpr size_t kPartialsOffset = 256;
// Blockwise GEMM tile counter in the workspace: bytes [64, 72) the next tile
// past the first wave, [72, 76) the CTAs finished; the kernel's last CTA
// puts both back to 0, so they are 0 between calls.
constexpr size_t kTileCounterOffset = 64;
constexpr int kMaxPartials = (int)((kWorkspaceBytes - kPartialsOffset) / 4);

int sm_count();  // of the current device, cached per device

// ---- quantisers (quant.cu); return a cudaError_t as int
struct QuantJob {
    const uint16_t* x;  // BF16 bits
    int64_t rows, cols, ldx;
    int gran;
    uint8_t* q;         // row-wise codes (may be null in transposed mode)
    void* s;            // row-wise scales
    uint8_t* qt;        // transposed codes (transposed mode)
    void* st;           // transposed scales
    float* tensor_scale;
    bool given_scale;
    bool four_over_six; // NVFP4: four-over-six block scales
    uint32_t* partials; // amax partials (per-tensor / NVFP4)
    int* status;        // sticky status word of the workspace, or null
};
int launch_quantize(const QuantJob& j, cudaStream_t s);
int launch_quantize_transposed(const QuantJob& j, cudaStream_t s);
// Row-wise quantisation (1x128, MXFP8, 1x128 power-of-two) of rows that
// are not a plain matrix: gathered rows (token_index != null: row r is row
// token_index[r] of x, x has `tokens` rows) or the SwiGLU activation (up > 0:
// row r is silu(x[r, 0:cols]) * x[r, up:up+cols]).
int launch_quantize_rows_src(const QuantJob& j, const int64_t* token_index, int64_t tokens, int64_t up,
                             cudaStream_t s);
// Gather of already quantised rows (1x128, MXFP8, 1x128 power-of-two):
// row r of q / s is row idx[r] of q_src / s_src ([tokens, cols] layouts).
struct GatherJob {
    const uint8_t* q_src;
    const void* s_src;
    int64_t tokens, cols, rows;
    const int64_t* idx;
    uint8_t* q;
    void* s;
    int gran;
    int* status;
};
int launch_gather_rows(const GatherJob& j, cudaStream_t s);
// Exhaustive check of the FP32-scale division used by the casts (test hook).
int launch_encoder_breakpoints(uint32_t* out, cudaStream_t st);
int launch_quotient_sweep(unsigned long long* counts, int nvfp4, cudaStream_t s);
int launch_quantize_per_tensor_scratch(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q,
                                       float* scale, uint32_t* partials, int nparts, cudaStream_t s);

// ---- dequantisation to BF16 (dequant.cu)
int launch_dequantize(const uint8_t* q, const void* scales, const float* tensor_scale, int64_t rows, int64_t cols,
                      int gran, void* out, int64_t ld_out, cudaStream_t s);

// ---- GEMMs (gemm_blockwise.cu, gemm_mx.cu)
struct GemmJob {
    const void* a; const void* sa; int a_gran;
    const void* b; const void* sb; int b_gran;
    const float* a_ts; const float* b_ts;
    bool a_ts_rows = false;               // NVFP4: a_ts holds one outer scale per row of A
    int64_t m, n, k;
    void* d;
    bool d_f32 = false;                   // D is float32 (fp8_block_gemm's FP8BS_OUT_F32), else BF16
    int* status;
    // grouped
    const int64_t* offsets; int experts;  // experts == 0 -> dense
    uint64_t wait_ns = 0;                 // 0 -> default bound (1 s)
    int stall_stage0 = 0;                 // test hook (fp8bs_test_stalled_gemm)
};
int launch_gemm_blockwise(const GemmJob& j, cudaStream_t s);
int launch_gemm_mx(const GemmJob& j, cudaStream_t s);

// ---- tensor-core throughput loop (peak.cu)
int launch_mma_peak(int kind, int ctas, int iters, int n, int pattern, float* out, int* status, cudaStream_t s);

}  // namespace fp8bs
