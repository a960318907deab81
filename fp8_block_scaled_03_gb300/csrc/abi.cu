// abi.cu -- the extern "C" entry points declared in include/fp8bs.h.
//
// Host-side argument checks, then a launch on the caller's stream.  Nothing
// here allocates device memory or synchronises (except fp8bs_read_status,
// whose job is to read the status word back).
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "../../include/fp8bs.h"
#include "common.cuh"
#include "internal.h"

namespace fp8bs {

int sm_count() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace fp8bs

using namespace fp8bs;

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Scale pointers: FP32 scales and UE8M0 words are read 4 bytes at a time,
// NVFP4 block scales 16 bytes at a time.
inline bool is_nvfp4(int gran) { return gran == FP8BS_NVFP4_1x16 || gran == FP8BS_NVFP4_ROW_1x16; }
inline bool scales_aligned(const void* s, int gran) {
    if (is_nvfp4(gran)) return aligned16(s);
    if (gran == FP8BS_TOKEN_1x128_POW2 || gran == FP8BS_BLOCK_128x128_POW2) return true;   // read bytewise
    return aligned4(s);
}
inline bool is_pow2_block(int gran) { return gran == FP8BS_TOKEN_1x128_POW2 || gran == FP8BS_BLOCK_128x128_POW2; }

// Launchers return 0, a cudaError_t (> 0) or a negative fp8bs_status.
inline int cuda_status(int err) {
    if (err < 0) return err;
    if (err != 0) {
        (void)cudaGetLastError();
        return FP8BS_ECUDA;
    }
    return FP8BS_OK;
}

// Size and granularity checks shared by both quantisers.  Returns 1 (not an
// error) for an empty matrix, which the callers turn into a no-op before any
// pointer is looked at (allocators may hand out NULL for empty tensors).
int check_quant_common(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int gran) {
    if (rows < 0 || cols < 0) return FP8BS_EINVAL;
    if (gran < FP8BS_PER_TENSOR || gran > FP8BS_NVFP4_ROW_1x16) return FP8BS_EINVAL;
    if (cols % 8 != 0 || ld_x < cols || ld_x % 8 != 0) return FP8BS_EINVAL;
    if (is_nvfp4(gran) && cols % 16 != 0) return FP8BS_EINVAL;
    if (ceil_div(rows, 128) > 65535 || ceil_div(cols, 128) > 0x7FFFFFFF) return FP8BS_EINVAL;
    if (rows == 0 || cols == 0) return 1;
    if (x == nullptr) return FP8BS_EINVAL;
    if (!aligned16(x)) return FP8BS_EALIGN;
    return FP8BS_OK;
}

// Sizes that TMA addresses: tensor-map coordinates are 32-bit signed, so a
// dimension a kernel walks by TMA stays below 2^31 (less one 256-wide box).
constexpr int64_t kMaxTmaDim = 0x7FFFFF00;
inline bool tma_dims_ok(int64_t a, int64_t b = 0, int64_t c = 0) {
    return a <= kMaxTmaDim && b <= kMaxTmaDim && c <= kMaxTmaDim;
}

// Unknown flag bits, or four-over-six on a non-NVFP4 granularity.
bool bad_flags(int gran, unsigned flags) {
    if (flags & ~(FP8BS_FLAG_GIVEN_TENSOR_SCALE | FP8BS_FLAG_NVFP4_4OVER6)) return true;
    return (flags & FP8BS_FLAG_NVFP4_4OVER6) && !is_nvfp4(gran);
}

// The row-wise granularities the MoE entry points produce (those a grouped
// or dense GEMM consumes along K with one scale per row and group).
inline bool is_moe_rowwise(int gran) {
    return gran == FP8BS_TOKEN_1x128 || gran == FP8BS_MXFP8_1x32 || gran == FP8BS_TOKEN_1x128_POW2;
}

bool needs_partials(int gran, unsigned flags) {
    return (gran == FP8BS_PER_TENSOR || gran == FP8BS_NVFP4_1x16) && !(flags & FP8BS_FLAG_GIVEN_TENSOR_SCALE);
}

}  // namespace

extern "C" {

int fp8_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int gran,
                 void* q, void* scales, float* tensor_scale, unsigned flags,
                 void* workspace, size_t workspace_bytes, fp8bs_stream_t stream) {
    if (bad_flags(gran, flags)) return FP8BS_EINVAL;
    int rc = check_quant_common(x, rows, cols, ld_x, gran);
    if (rc) return rc > 0 ? FP8BS_OK : rc;
    if (q == nullptr || scales == nullptr) return FP8BS_EINVAL;
    if (is_nvfp4(gran) && tensor_scale == nullptr) return FP8BS_EINVAL;
    if (is_nvfp4(gran) && !aligned4(tensor_scale)) return FP8BS_EALIGN;
    if (!aligned16(q)) return FP8BS_EALIGN;
    if (needs_partials(gran, flags) && (workspace == nullptr || workspace_bytes < kWorkspaceBytes))
        return FP8BS_EWORKSPACE;
    if (workspace != nullptr && !aligned16(workspace)) return FP8BS_EALIGN;
    QuantJob j{};
    j.x = static_cast<const uint16_t*>(x);
    j.rows = rows; j.cols = cols; j.ldx = ld_x; j.gran = gran;
    j.q = static_cast<uint8_t*>(q); j.s = scales;
    j.tensor_scale = tensor_scale;
    j.given_scale = (flags & FP8BS_FLAG_GIVEN_TENSOR_SCALE) != 0;
    j.four_over_six = (flags & FP8BS_FLAG_NVFP4_4OVER6) != 0;
    j.partials = workspace ? reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + kPartialsOffset) : nullptr;
    return cuda_status(launch_quantize(j, reinterpret_cast<cudaStream_t>(stream)));
}

int fp8_quantize_transposed(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int gran,
                            void* q_t, void* scales_t, void* q, void* scales,
                            float* tensor_scale, unsigned flags,
                            void* workspace, size_t workspace_bytes, fp8bs_stream_t stream) {
    (void)tensor_scale;
    if (is_nvfp4(gran)) return FP8BS_EUNSUPPORTED;
    if (bad_flags(gran, flags)) return FP8BS_EINVAL;
    if (rows % 16 != 0) return FP8BS_EINVAL;
    if (!tma_dims_ok(rows, cols, ld_x)) return FP8BS_EINVAL;
    int rc = check_quant_common(x, rows, cols, ld_x, gran);
    if (rc) return rc > 0 ? FP8BS_OK : rc;
    if (q_t == nullptr || scales_t == nullptr) return FP8BS_EINVAL;
    if ((q == nullptr) != (scales == nullptr)) return FP8BS_EINVAL;
    if (!aligned16(q_t) || (q != nullptr && !aligned16(q))) return FP8BS_EALIGN;
    if (needs_partials(gran, flags) && (workspace == nullptr || workspace_bytes < kWorkspaceBytes))
        return FP8BS_EWORKSPACE;
    if (workspace != nullptr && !aligned16(workspace)) return FP8BS_EALIGN;
    QuantJob j{};
    j.x = static_cast<const uint16_t*>(x);
    j.rows = rows; j.cols = cols; j.ldx = ld_x; j.gran = gran;
    j.qt = static_cast<uint8_t*>(q_t); j.st = scales_t;
    j.q = static_cast<uint8_t*>(q); j.s = scales;
    j.given_scale = (flags & FP8BS_FLAG_GIVEN_TENSOR_SCALE) != 0;
    j.partials = workspace ? reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + kPartialsOffset) : nullptr;
    j.status = (workspace != nullptr && workspace_bytes >= kWorkspaceBytes) ? static_cast<int*>(workspace) : nullptr;
    return cuda_status(launch_quantize_transposed(j, reinterpret_cast<cudaStream_t>(stream)));
}

int fp8_dequantize(const void* q, const void* scales, const float* tensor_scale, int64_t rows, int64_t cols,
                   int gran, void* out, int64_t ld_out, fp8bs_stream_t stream) {
    if (rows < 0 || cols < 0 || gran < FP8BS_PER_TENSOR || gran > FP8BS_NVFP4_ROW_1x16) return FP8BS_EINVAL;
    if (cols % 8 != 0 || ld_out < cols || ld_out % 8 != 0) return FP8BS_EINVAL;
    if (is_nvfp4(gran) && cols % 16 != 0) return FP8BS_EINVAL;
    if (rows == 0 || cols == 0) return FP8BS_OK;
    if (q == nullptr || scales == nullptr || out == nullptr) return FP8BS_EINVAL;
    if (is_nvfp4(gran) && tensor_scale == nullptr) return FP8BS_EINVAL;
    if ((reinterpret_cast<uintptr_t>(q) & 7u) || !aligned16(out) || !scales_aligned(scales, gran) ||
        (is_nvfp4(gran) && !aligned4(tensor_scale)))
        return FP8BS_EALIGN;
    return cuda_status(launch_dequantize(static_cast<const uint8_t*>(q), scales, tensor_scale, rows, cols, gran, out,
                                         ld_out, reinterpret_cast<cudaStream_t>(stream)));
}

int fp8_quantize_gathered(const void* x, int64_t tokens, int64_t cols, int64_t ld_x,
                          const int64_t* token_index, int64_t rows, int gran, void* q, void* scales,
                          void* workspace, size_t workspace_bytes, fp8bs_stream_t stream) {
    if (tokens < 0 || rows < 0 || cols < 0) return FP8BS_EINVAL;
    if (gran < FP8BS_PER_TENSOR || gran > FP8BS_NVFP4_ROW_1x16) return FP8BS_EINVAL;
    if (!is_moe_rowwise(gran)) return FP8BS_EUNSUPPORTED;
    if (cols % 8 != 0 || ld_x < cols || ld_x % 8 != 0) return FP8BS_EINVAL;
    if (rows == 0 || cols == 0) return FP8BS_OK;
    // with no tokens x is never read (every index is out of range) and may be NULL
    if ((x == nullptr && tokens > 0) || token_index == nullptr || q == nullptr || scales == nullptr)
        return FP8BS_EINVAL;
    if (!aligned16(x) || !aligned16(q) || !scales_aligned(scales, gran) ||
        (reinterpret_cast<uintptr_t>(token_index) & 7u))
        return FP8BS_EALIGN;
    if (workspace == nullptr || workspace_bytes < kWorkspaceBytes) return FP8BS_EWORKSPACE;
    if (!aligned16(workspace)) return FP8BS_EALIGN;
    QuantJob j{};
    j.x = static_cast<const uint16_t*>(x);
    j.rows = rows; j.cols = cols; j.ldx = ld_x; j.gran = gran;
    j.q = static_cast<uint8_t*>(q); j.s = scales;
    j.status = static_cast<int*>(workspace);
    return cuda_status(launch_quantize_rows_src(j, token_index, tokens, 0, reinterpret_cast<cudaStream_t>(stream)));
}

int fp8_gather_rows(const void* q_src, const void* scales_src, int64_t tokens, int64_t cols, int gran,
                    const int64_t* token_index, int64_t rows, void* q, void* scales, void* workspace,
                    size_t workspace_bytes, fp8bs_stream_t stream) {
    if (tokens < 0 || rows < 0 || cols < 0) return FP8BS_EINVAL;
    if (gran < FP8BS_PER_TENSOR || gran > FP8BS_NVFP4_ROW_1x16) return FP8BS_EINVAL;
    if (!is_moe_rowwise(gran)) return FP8BS_EUNSUPPORTED;
    if (cols % 8 != 0) return FP8BS_EINVAL;
    if (rows == 0 || cols == 0) return FP8BS_OK;
    // with no tokens the sources are never read (every index is out of range) and may be NULL
    if (((q_src == nullptr || scales_src == nullptr) && tokens > 0) || token_index == nullptr || q == nullptr ||
        scales == nullptr)
        return FP8BS_EINVAL;
    if (!aligned16(q_src) || !aligned16(q) || !scales_aligned(scales, gran) || !scales_aligned(scales_src, gran) ||
        (reinterpret_cast<uintptr_t>(token_index) & 7u))
        return FP8BS_EALIGN;
    if (workspace == nullptr || workspace_bytes < kWorkspaceBytes) return FP8BS_EWORKSPACE;
    if (!aligned16(workspace)) return FP8BS_EALIGN;
    GatherJob j{};
    j.q_src = static_cast<const uint8_t*>(q_src);
    j.s_src = scales_src;
    j.tokens = tokens; j.cols = cols; j.rows = rows;
    j.idx = token_index;
    j.q = static_cast<uint8_t*>(q); j.s = scales;
    j.gran = gran;
    j.status = static_cast<int*>(workspace);
    return cuda_status(launch_gather_rows(j, reinterpret_cast<cudaStream_t>(stream)));
}

int fp8_swiglu_quantize(const void* h, int64_t rows, int64_t inter, int64_t ld_h, int gran, void* q, void* scales,
                        fp8bs_stream_t stream) {
    if (rows < 0 || inter < 0) return FP8BS_EINVAL;
    if (gran < FP8BS_PER_TENSOR || gran > FP8BS_NVFP4_ROW_1x16) return FP8BS_EINVAL;
    if (!is_moe_rowwise(gran)) return FP8BS_EUNSUPPORTED;
    if (inter % 8 != 0 || ld_h < 2 * inter || ld_h % 8 != 0) return FP8BS_EINVAL;
    if (rows == 0 || inter == 0) return FP8BS_OK;
    if (h == nullptr || q == nullptr || scales == nullptr) return FP8BS_EINVAL;
    if (!aligned16(h) || !aligned16(q) || !scales_aligned(scales, gran)) return FP8BS_EALIGN;
    QuantJob j{};
    j.x = static_cast<const uint16_t*>(h);
    j.rows = rows; j.cols = inter; j.ldx = ld_h; j.gran = gran;
    j.q = static_cast<uint8_t*>(q); j.s = scales;
    return cuda_status(launch_quantize_rows_src(j, nullptr, 0, inter, reinterpret_cast<cudaStream_t>(stream)));
}

int fp8_block_gemm(const void* a, const void* a_scales, int a_gran,
                   const void* b, const void* b_scales, int b_gran,
                   const float* a_tensor_scale, const float* b_tensor_scale,
                   int64_t m, int64_t n, int64_t k, void* d, int d_dtype,
                   void* workspace, size_t workspace_bytes, fp8bs_stream_t stream) {
    if (a == nullptr || b == nullptr || d == nullptr || a_scales == nullptr || b_scales == nullptr)
        return FP8BS_EINVAL;
    if (m <= 0 || n <= 0 || k <= 0 || n % 8 != 0) return FP8BS_EINVAL;
    if (!tma_dims_ok(m, n, k)) return FP8BS_EINVAL;
    if (d_dtype != FP8BS_OUT_BF16 && d_dtype != FP8BS_OUT_F32) return FP8BS_EINVAL;
    if (a_gran < 0 || a_gran > FP8BS_NVFP4_ROW_1x16 || b_gran < 0 || b_gran > FP8BS_NVFP4_ROW_1x16)
        return FP8BS_EINVAL;
    if (!aligned16(a) || !aligned16(b) || !aligned16(d)) return FP8BS_EALIGN;
    if (!scales_aligned(a_scales, a_gran) || !scales_aligned(b_scales, b_gran)) return FP8BS_EALIGN;
    if (workspace == nullptr || workspace_bytes < kWorkspaceBytes) return FP8BS_EWORKSPACE;
    if (!aligned16(workspace)) return FP8BS_EALIGN;
    const bool fp32_a = a_gran <= FP8BS_BLOCK_128x128, fp32_b = b_gran <= FP8BS_BLOCK_128x128;
    GemmJob j{};
    j.a = a; j.sa = a_scales; j.a_gran = a_gran;
    j.b = b; j.sb = b_scales; j.b_gran = b_gran;
    j.a_ts = a_tensor_scale; j.b_ts = b_tensor_scale;
    j.m = m; j.n = n; j.k = k; j.d = d;
    j.d_f32 = d_dtype == FP8BS_OUT_F32;
    j.status = static_cast<int*>(workspace);
    j.offsets = nullptr; j.experts = 0;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (fp32_a && fp32_b) {
        if (k % 128 != 0) return FP8BS_EINVAL;
        return cuda_status(launch_gemm_blockwise(j, st));
    }
    if (a_gran == FP8BS_MXFP8_1x32 && b_gran == FP8BS_MXFP8_1x32) {
        if (k % 128 != 0) return FP8BS_EINVAL;
        return cuda_status(launch_gemm_mx(j, st));
    }
    if (is_pow2_block(a_gran) && is_pow2_block(b_gran)) {
        if (k % 128 != 0) return FP8BS_EINVAL;
        return cuda_status(launch_gemm_mx(j, st));
    }
    if (is_nvfp4(a_gran) && b_gran == FP8BS_NVFP4_1x16) {
        if (k % 256 != 0) return FP8BS_EINVAL;
        if (a_tensor_scale == nullptr || b_tensor_scale == nullptr) return FP8BS_EINVAL;
        if (!aligned4(a_tensor_scale) || !aligned4(b_tensor_scale)) return FP8BS_EALIGN;
        j.a_ts_rows = a_gran == FP8BS_NVFP4_ROW_1x16;
        j.a_gran = FP8BS_NVFP4_1x16;
        return cuda_status(launch_gemm_mx(j, st));
    }
    return FP8BS_EUNSUPPORTED;
}

int fp8_grouped_gemm(const void* a, const void* a_scales,
                     const void* b, const void* b_scales,
                     const float* a_tensor_scale, const float* b_tensor_scale,
                     const int64_t* offsets, int experts, int64_t total_rows,
                     int64_t n, int64_t k, int gran, void* d,
                     void* workspace, size_t workspace_bytes, fp8bs_stream_t stream) {
    if (a == nullptr || b == nullptr || d == nullptr || a_scales == nullptr || b_scales == nullptr ||
        offsets == nullptr)
        return FP8BS_EINVAL;
    if (gran < 0 || gran > FP8BS_NVFP4_ROW_1x16) return FP8BS_EINVAL;
    const bool nv = is_nvfp4(gran);
    if (experts <= 0 || experts > 1024 || total_rows < 0 || n <= 0 || k <= 0 || n % 8 != 0 ||
        k % (nv ? 256 : 128) != 0)
        return FP8BS_EINVAL;
    if (!tma_dims_ok(total_rows, n * experts, k)) return FP8BS_EINVAL;
    if (nv && (a_tensor_scale == nullptr || b_tensor_scale == nullptr)) return FP8BS_EINVAL;
    if (!aligned16(a) || !aligned16(b) || !aligned16(d)) return FP8BS_EALIGN;
    if (!aligned4(a_scales) || !aligned4(b_scales) || (reinterpret_cast<uintptr_t>(offsets) & 7u)) return FP8BS_EALIGN;
    if (nv && (!aligned16(a_scales) || !aligned16(b_scales) || !aligned4(a_tensor_scale) ||
               !aligned4(b_tensor_scale)))
        return FP8BS_EALIGN;
    if (workspace == nullptr || workspace_bytes < kWorkspaceBytes) return FP8BS_EWORKSPACE;
    if (!aligned16(workspace)) return FP8BS_EALIGN;
    if (total_rows == 0) return FP8BS_OK;
    GemmJob j{};
    j.a = a; j.sa = a_scales; j.b = b; j.sb = b_scales;
    j.m = total_rows; j.n = n; j.k = k; j.d = d;
    j.status = static_cast<int*>(workspace);
    j.offsets = offsets; j.experts = experts;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (gran == FP8BS_MXFP8_1x32) {
        j.a_gran = j.b_gran = FP8BS_MXFP8_1x32;
        return cuda_status(launch_gemm_mx(j, st));
    }
    if (gran == FP8BS_TOKEN_1x128) {
        j.a_gran = FP8BS_TOKEN_1x128; j.b_gran = FP8BS_BLOCK_128x128;
        return cuda_status(launch_gemm_blockwise(j, st));
    }
    if (gran == FP8BS_TOKEN_1x128_POW2) {
        j.a_gran = FP8BS_TOKEN_1x128_POW2; j.b_gran = FP8BS_BLOCK_128x128_POW2;
        return cuda_status(launch_gemm_mx(j, st));
    }
    if (nv) {
        j.a_gran = j.b_gran = FP8BS_NVFP4_1x16;
        j.a_ts = a_tensor_scale; j.b_ts = b_tensor_scale;
        j.a_ts_rows = gran == FP8BS_NVFP4_ROW_1x16;
        return cuda_status(launch_gemm_mx(j, st));
    }
    return FP8BS_EUNSUPPORTED;
}

int fp8bs_test_stalled_gemm(const void* a, const void* a_scales, const void* b, const void* b_scales,
                            int64_t m, int64_t n, int64_t k, void* d, uint64_t wait_limit_ns,
                            void* workspace, size_t workspace_bytes, fp8bs_stream_t stream) {
    if (a == nullptr || b == nullptr || d == nullptr || a_scales == nullptr || b_scales == nullptr)
        return FP8BS_EINVAL;
    if (m <= 0 || n <= 0 || k <= 0 || n % 8 != 0 || k % 128 != 0) return FP8BS_EINVAL;
    if (!tma_dims_ok(m, n, k)) return FP8BS_EINVAL;
    if (wait_limit_ns == 0 || wait_limit_ns > 2000000000ull) return FP8BS_EINVAL;
    if (!aligned16(a) || !aligned16(b) || !aligned16(d) || !aligned4(a_scales) || !aligned4(b_scales))
        return FP8BS_EALIGN;
    if (workspace == nullptr || workspace_bytes < kWorkspaceBytes) return FP8BS_EWORKSPACE;
    if (!aligned16(workspace)) return FP8BS_EALIGN;
    GemmJob j{};
    j.a = a; j.sa = a_scales; j.a_gran = FP8BS_MXFP8_1x32;
    j.b = b; j.sb = b_scales; j.b_gran = FP8BS_MXFP8_1x32;
    j.m = m; j.n = n; j.k = k; j.d = d;
    j.status = static_cast<int*>(workspace);
    j.offsets = nullptr; j.experts = 0;
    j.wait_ns = wait_limit_ns;
    j.stall_stage0 = 1;
    return cuda_status(launch_gemm_mx(j, reinterpret_cast<cudaStream_t>(stream)));
}

int fp8bs_test_stalled_gemm_blockwise(const void* a, const void* a_scales, int a_gran, const void* b,
                                      const void* b_scales, int b_gran, int64_t m, int64_t n, int64_t k, void* d,
                                      uint64_t wait_limit_ns, void* workspace, size_t workspace_bytes,
                                      fp8bs_stream_t stream) {
    if (a == nullptr || b == nullptr || d == nullptr || a_scales == nullptr || b_scales == nullptr)
        return FP8BS_EINVAL;
    if (a_gran < FP8BS_PER_TENSOR || a_gran > FP8BS_BLOCK_128x128 || b_gran < FP8BS_PER_TENSOR ||
        b_gran > FP8BS_BLOCK_128x128)
        return FP8BS_EINVAL;
    if (m <= 0 || n <= 0 || k <= 0 || n % 8 != 0 || k % 128 != 0) return FP8BS_EINVAL;
    if (!tma_dims_ok(m, n, k)) return FP8BS_EINVAL;
    if (wait_limit_ns == 0 || wait_limit_ns > 2000000000ull) return FP8BS_EINVAL;
    if (!aligned16(a) || !aligned16(b) || !aligned16(d) || !aligned4(a_scales) || !aligned4(b_scales))
        return FP8BS_EALIGN;
    if (workspace == nullptr || workspace_bytes < kWorkspaceBytes) return FP8BS_EWORKSPACE;
    if (!aligned16(workspace)) return FP8BS_EALIGN;
    GemmJob j{};
    j.a = a; j.sa = a_scales; j.a_gran = a_gran;
    j.b = b; j.sb = b_scales; j.b_gran = b_gran;
    j.m = m; j.n = n; j.k = k; j.d = d;
    j.status = static_cast<int*>(workspace);
    j.offsets = nullptr; j.experts = 0;
    j.wait_ns = wait_limit_ns;
    j.stall_stage0 = 1;
    return cuda_status(launch_gemm_blockwise(j, reinterpret_cast<cudaStream_t>(stream)));
}

int fp8bs_test_stalled_gemm_nvfp4(const void* a, const void* a_scales, const void* b, const void* b_scales,
                                  const float* a_tensor_scale, const float* b_tensor_scale, int64_t m, int64_t n,
                                  int64_t k, void* d, uint64_t wait_limit_ns, void* workspace,
                                  size_t workspace_bytes, fp8bs_stream_t stream) {
    if (a == nullptr || b == nullptr || d == nullptr || a_scales == nullptr || b_scales == nullptr ||
        a_tensor_scale == nullptr || b_tensor_scale == nullptr)
        return FP8BS_EINVAL;
    if (m <= 0 || n <= 0 || k <= 0 || n % 8 != 0 || k % 256 != 0) return FP8BS_EINVAL;
    if (!tma_dims_ok(m, n, k)) return FP8BS_EINVAL;
    if (wait_limit_ns == 0 || wait_limit_ns > 2000000000ull) return FP8BS_EINVAL;
    if (!aligned16(a) || !aligned16(b) || !aligned16(d) || !aligned16(a_scales) || !aligned16(b_scales) ||
        !aligned4(a_tensor_scale) || !aligned4(b_tensor_scale))
        return FP8BS_EALIGN;
    if (workspace == nullptr || workspace_bytes < kWorkspaceBytes) return FP8BS_EWORKSPACE;
    if (!aligned16(workspace)) return FP8BS_EALIGN;
    GemmJob j{};
    j.a = a; j.sa = a_scales; j.a_gran = FP8BS_NVFP4_1x16;
    j.b = b; j.sb = b_scales; j.b_gran = FP8BS_NVFP4_1x16;
    j.a_ts = a_tensor_scale; j.b_ts = b_tensor_scale;
    j.m = m; j.n = n; j.k = k; j.d = d;
    j.status = static_cast<int*>(workspace);
    j.offsets = nullptr; j.experts = 0;
    j.wait_ns = wait_limit_ns;
    j.stall_stage0 = 1;
    return cuda_status(launch_gemm_mx(j, reinterpret_cast<cudaStream_t>(stream)));
}

int fp8bs_test_quotient_sweep(unsigned long long* counts, int nvfp4, fp8bs_stream_t stream) {
    if (counts == nullptr || nvfp4 < 0 || nvfp4 > 3) return FP8BS_EINVAL;
    if (reinterpret_cast<uintptr_t>(counts) & 7u) return FP8BS_EALIGN;
    return cuda_status(launch_quotient_sweep(counts, nvfp4, reinterpret_cast<cudaStream_t>(stream)));
}

int fp8bs_test_encoder_breakpoints(uint32_t* out, fp8bs_stream_t stream) {
    if (out == nullptr) return FP8BS_EINVAL;
    if (reinterpret_cast<uintptr_t>(out) & 3u) return FP8BS_EALIGN;
    return cuda_status(launch_encoder_breakpoints(out, reinterpret_cast<cudaStream_t>(stream)));
}

int fp8bs_mma_peak(int kind, int n, int iters, int pattern, float* out, void* workspace, size_t workspace_bytes,
                   fp8bs_stream_t stream) {
    if (kind < 0 || kind > 2 || (n != 64 && n != 128 && n != 256) || (kind != 0 && n == 64) || iters < 1 ||
        iters > (1 << 24) ||
        (pattern != 0 && pattern != 1))
        return FP8BS_EINVAL;
    if (out != nullptr && !aligned4(out)) return FP8BS_EALIGN;
    if (workspace == nullptr || workspace_bytes < kWorkspaceBytes) return FP8BS_EWORKSPACE;
    if (!aligned16(workspace)) return FP8BS_EALIGN;
    return cuda_status(launch_mma_peak(kind, sm_count(), iters, n, pattern, out, static_cast<int*>(workspace),
                                       reinterpret_cast<cudaStream_t>(stream)));
}

size_t fp8bs_workspace_size(void) { return kWorkspaceBytes; }

size_t fp8bs_workspace_size_for(int op, int64_t rows, int64_t cols, int gran, unsigned flags) {
    if (rows < 0 || cols < 0 || gran < FP8BS_PER_TENSOR || gran > FP8BS_NVFP4_ROW_1x16) return (size_t)-1;
    switch (op) {
    case FP8BS_OP_QUANTIZE:
    case FP8BS_OP_QUANTIZE_TRANSPOSED:
        return needs_partials(gran, flags) ? kWorkspaceBytes : 0;
    case FP8BS_OP_DEQUANTIZE:
    case FP8BS_OP_SWIGLU_QUANTIZE:
        return 0;
    case FP8BS_OP_BLOCK_GEMM:
    case FP8BS_OP_GROUPED_GEMM:
    case FP8BS_OP_QUANTIZE_GATHERED:
    case FP8BS_OP_GATHER_ROWS:
        return kWorkspaceBytes;
    default:
        return (size_t)-1;
    }
}

int fp8bs_read_status(const void* workspace, fp8bs_stream_t stream) {
    if (workspace == nullptr) return FP8BS_EINVAL;
    int v = 0;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return cuda_status(1);
    if (cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return cuda_status(1);
    return v;
}

int fp8bs_clear_status(void* workspace, fp8bs_stream_t stream) {
    if (workspace == nullptr) return FP8BS_EINVAL;
    return cuda_status((int)cudaMemsetAsync(workspace, 0, sizeof(int), reinterpret_cast<cudaStream_t>(stream)));
}

const char* fp8bs_status_string(int status) {
    switch (status) {
    case FP8BS_OK: return "ok";
    case FP8BS_EINVAL: return "invalid argument (size, granularity or null pointer)";
    case FP8BS_EALIGN: return "pointer or pitch not 16-byte aligned";
    case FP8BS_EUNSUPPORTED: return "combination not implemented";
    case FP8BS_ECUDA: return "CUDA runtime error or launch failure";
    case FP8BS_ETIMEOUT: return "a bounded device wait timed out";
    case FP8BS_EWORKSPACE: return "workspace missing or too small";
    case FP8BS_EINDEX: return "a token index was out of range (its row was zeroed)";
    case FP8BS_EOFFSETS: return "expert offsets out of range or decreasing (clamped; malformed experts skipped)";
    default: return "unknown status";
    }
}

int fp8bs_version(void) { return 103; }

}  // extern "C"
