// quant.cu -- fused amax / scale / cast quantisers (BF16 -> E4M3 / E2M1).
//
// Steps 1 and 2 of "FP8 Quantization" (Unified FP8 review): S = max|X| / V_max
// over the group, Q(x) = round(x / S), at the granularities of the
// "Choose a precision" table of the "Low Precision RL" page.  All of them
// are HBM-bound streaming kernels: every BF16 element is read once (twice
// for the per-tensor / NVFP4 tensor amax), every code written once.
//
// Row-wise kernels: one warp task is one row segment of 1024 columns; a lane
// owns 4 x 8 consecutive BF16 (four 16-byte loads in flight per lane).  A
// 1x128 group is 16 lanes, a 1x32 group 4 lanes, a 1x16 group 2 lanes, so
// every group amax is a handful of xor-shuffles; no shared memory.
// 128x128 and transposed kernels: one CTA per 128x128 tile, the tile held
// in registers (16 rows x 4 columns per thread), per-column partial amaxes
// combined through shared memory.
#include "common.cuh"
#include "internal.h"

namespace fp8bs {

enum { kGranPT = 0, kGranTok = 1, kGranBlk = 2, kGranMx = 3, kGranNv = 4, kGranTokP2 = 5, kGranBlkP2 = 6,
       kGranNvRow = 7 };

// Granularities whose scale is a power of two (UE8M0 byte): the division by
// the scale is an exact multiplication by 2^-e.
template <int G> constexpr bool kPow2 = (G == kGranMx || G == kGranTokP2 || G == kGranBlkP2);

constexpr int kSeg = 1024;       // columns per row-wise warp task
constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t absmax_v4(const uint4& v) {
    return max(max(bf16x2_absmax_bits(v.x), bf16x2_absmax_bits(v.y)),
               max(bf16x2_absmax_bits(v.z), bf16x2_absmax_bits(v.w)));
}

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Eight elements x / S -> eight E4M3 bytes.
__device__ __forceinline__ uint2 cast8_div(const float* f, float s) {
    uint2 o;
    o.x = e4m3x4(__fdiv_rn(f[0], s), __fdiv_rn(f[1], s), __fdiv_rn(f[2], s), __fdiv_rn(f[3], s));
    o.y = e4m3x4(__fdiv_rn(f[4], s), __fdiv_rn(f[5], s), __fdiv_rn(f[6], s), __fdiv_rn(f[7], s));
    return o;
}

// Eight elements x * 2^-e (exact power-of-two division) -> eight E4M3 bytes.
__device__ __forceinline__ uint2 cast8_mul(const float* f, float m) {
    uint2 o;
    o.x = e4m3x4(__fmul_rn(f[0], m), __fmul_rn(f[1], m), __fmul_rn(f[2], m), __fmul_rn(f[3], m));
    o.y = e4m3x4(__fmul_rn(f[4], m), __fmul_rn(f[5], m), __fmul_rn(f[6], m), __fmul_rn(f[7], m));
    return o;
}

// Block-wide max of a u32; every thread gets the result.
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v) {
    __shared__ uint32_t red[32];
    v = warp_max_u32(v, 32);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    uint32_t r = 0;
    const int nw = (blockDim.x + 31) >> 5;
    for (int i = 0; i < nw; ++i) r = max(r, red[i]);
    return r;
}

// Tensor amax (BF16 bits) from the per-CTA partials of amax_partials_kernel.
__device__ __forceinline__ float tensor_amax(const uint32_t* __restrict__ partials, int nparts) {
    uint32_t m = 0;
    for (int i = threadIdx.x; i < nparts; i += blockDim.x) m = max(m, partials[i]);
    return amax_bits_to_f32(block_max_u32(m));
}

// ---------------------------------------------------------------- pass 1: amax partials
__global__ void __launch_bounds__(kThreads)
amax_partials_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
                     uint32_t* __restrict__ partials) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t segs = ceil_div(cols, kSeg);
    const int64_t total = rows * segs;
    uint32_t m = 0;
    for (int64_t t = gw; t < total; t += nw) {
        const int64_t r = t / segs;
        const int64_t cb = (t - r * segs) * kSeg;
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t c = cb + j * 256 + lane * 8;
            v[j] = (c < cols) ? ldg_v4(x + r * ldx + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) m = max(m, absmax_v4(v[j]));
    }
    m = block_max_u32(m);
    if (threadIdx.x == 0) partials[blockIdx.x] = m;
}

// ---------------------------------------------------------------- row-wise 1x128 / 1x32 / per-tensor
template <int GRAN>
__global__ void __launch_bounds__(kThreads)
quant_rows_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
                  uint8_t* __restrict__ q, void* __restrict__ sout,
                  const uint32_t* __restrict__ partials, int nparts, const float* __restrict__ given) {
    const int lane = threadIdx.x & 31;
    float s_uniform = 1.0f;
    if constexpr (GRAN == kGranPT) {
        if (given != nullptr) {
            s_uniform = *given;
        } else {
            s_uniform = fp32_scale_from_amax(tensor_amax(partials, nparts));
            if (blockIdx.x == 0 && threadIdx.x == 0) static_cast<float*>(sout)[0] = s_uniform;
        }
    }
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t segs = ceil_div(cols, kSeg);
    const int64_t total = rows * segs;
    const int64_t ng = ceil_div(cols, GRAN == kGranMx ? 32 : 128);
    for (int64_t t = gw; t < total; t += nw) {
        const int64_t r = t / segs;
        const int64_t cb = (t - r * segs) * kSeg;
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t c = cb + j * 256 + lane * 8;
            v[j] = (c < cols) ? ldg_v4(x + r * ldx + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t c = cb + j * 256 + lane * 8;
            const bool ok = c < cols;
            float f[8];
            unpack8(v[j], f);
            uint2 o;
            if constexpr (GRAN == kGranTok) {
                const uint32_t m = warp_max_u32(absmax_v4(v[j]), 16);
                const float s = fp32_scale_from_amax(amax_bits_to_f32(m));
                o = cast8_div(f, s);
                if (ok && (lane & 15) == 0) static_cast<float*>(sout)[r * ng + (c >> 7)] = s;
            } else if constexpr (GRAN == kGranMx) {
                const uint32_t m = warp_max_u32(absmax_v4(v[j]), 4);
                const int e = mx_exponent_from_amax_bits(m << 16);
                o = cast8_mul(f, exp2_neg(e));
                if (ok && (lane & 3) == 0) static_cast<uint8_t*>(sout)[r * ng + (c >> 5)] = (uint8_t)(e + 127);
            } else if constexpr (GRAN == kGranTokP2) {
                const uint32_t m = warp_max_u32(absmax_v4(v[j]), 16);
                const int e = mx_exponent_from_amax_bits(m << 16);
                o = cast8_mul(f, exp2_neg(e));
                if (ok && (lane & 15) == 0) static_cast<uint8_t*>(sout)[r * ng + (c >> 7)] = (uint8_t)(e + 127);
            } else {
                o = cast8_div(f, s_uniform);
            }
            if (ok) *reinterpret_cast<uint2*>(q + r * cols + c) = o;
        }
    }
}

// ---------------------------------------------------------------- NVFP4 1x16 (row-wise)
// "4. NVFP4 (Blackwell)": E2M1 codes in 1x16 blocks, an E4M3 block scale
// s_b = E4M3((amax_b / 6) / S_g) and an outer float32 S_g (per tensor, or per
// row for per-token activation scaling).  A lane owns 8 elements, so a block
// is a lane pair (2j, 2j+1).
//
// Four-over-six ("Advanced: four-over-six"): each block is also quantised
// with its amax mapped to 4 (s_b from amax_b / 4) and keeps that result only
// when its squared error is strictly smaller.  The error of 8 elements is
// summed in order in float32 (no fused multiply-add); the two lanes' half
// sums are then added, which is the same sum on both lanes (IEEE addition
// commutes).  S_g is amax / (256 * 6) in that mode.

__device__ __forceinline__ uint32_t e2m1_quant8(const float* f, float big_s) {
    if (big_s == 0.0f) return 0u;
    float t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) t[i] = __fdiv_rn(f[i], big_s);
    return e2m1x8(t);
}

// sum_i (x_i - E2M1(q_i) * S_b)^2 over this lane's 8 elements, in order.
__device__ __forceinline__ float half_sq_err(const float* f, uint32_t packed, float big_s) {
    float acc = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 e = e2m1x2_to_float2((packed >> (8 * k)) & 0xFFu);
        const float d0 = __fsub_rn(f[2 * k], __fmul_rn(e.x, big_s));
        const float d1 = __fsub_rn(f[2 * k + 1], __fmul_rn(e.y, big_s));
        acc = (k == 0) ? __fmul_rn(d0, d0) : __fadd_rn(acc, __fmul_rn(d0, d0));
        acc = __fadd_rn(acc, __fmul_rn(d1, d1));
    }
    return acc;
}

// One lane's half block: packed E2M1 codes and the block's scale byte.  Every
// lane of the warp must call this (shuffles).
template <bool FOS>
__device__ __forceinline__ void nvfp4_half_block(const uint4& v, float s_g, uint32_t& packed, uint32_t& code) {
    const uint32_t m = warp_max_u32(absmax_v4(v), 2);
    const float amax_b = amax_bits_to_f32(m);
    float f[8];
    unpack8(v, f);
    code = e4m3_byte(__fdiv_rn(__fdiv_rn(amax_b, kE2M1Max), s_g));
    const float s6 = __fmul_rn(e4m3_value(code), s_g);
    packed = e2m1_quant8(f, s6);
    if constexpr (FOS) {
        const uint32_t code4 = e4m3_byte(__fdiv_rn(__fdiv_rn(amax_b, 4.0f), s_g));
        const float s4 = __fmul_rn(e4m3_value(code4), s_g);
        const uint32_t p4 = e2m1_quant8(f, s4);
        float e6 = half_sq_err(f, packed, s6);
        float e4 = half_sq_err(f, p4, s4);
        e6 = __fadd_rn(e6, __shfl_xor_sync(0xFFFFFFFFu, e6, 1));
        e4 = __fadd_rn(e4, __shfl_xor_sync(0xFFFFFFFFu, e4, 1));
        if (e4 < e6) {
            packed = p4;
            code = code4;
        }
    }
}

// Quantise columns [cb, cb + 1024) of row r with outer scale s_g.
template <bool FOS>
__device__ __forceinline__ void nvfp4_segment(const uint16_t* __restrict__ x, int64_t r, int64_t cb, int64_t cols,
                                              int64_t ldx, uint8_t* __restrict__ q, uint8_t* __restrict__ sb,
                                              float s_g, int lane) {
    const int64_t nb = cols >> 4;
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t c = cb + j * 256 + lane * 8;
        v[j] = (c < cols) ? ldg_v4(x + r * ldx + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int64_t c = cb + j * 256 + lane * 8;
        uint32_t packed, code;
        nvfp4_half_block<FOS>(v[j], s_g, packed, code);
        if (c < cols) {
            *reinterpret_cast<uint32_t*>(q + r * (cols >> 1) + (c >> 1)) = packed;
            if ((lane & 1) == 0) sb[r * nb + (c >> 4)] = (uint8_t)code;
        }
    }
}

// One outer scale for the tensor (from the amax partials, or given).
template <bool FOS>
__global__ void __launch_bounds__(kThreads)
quant_nvfp4_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
                   uint8_t* __restrict__ q, uint8_t* __restrict__ sb, float* __restrict__ tensor_scale,
                   const uint32_t* __restrict__ partials, int nparts, bool given) {
    const int lane = threadIdx.x & 31;
    float s_g;
    if (given) {
        s_g = *tensor_scale;
    } else {
        const float amax = tensor_amax(partials, nparts);
        s_g = amax == 0.0f ? 1.0f : __fdiv_rn(amax, FOS ? kNvfp4GlobalDiv4over6 : kNvfp4GlobalDiv);
        if (blockIdx.x == 0 && threadIdx.x == 0) *tensor_scale = s_g;
    }
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t segs = ceil_div(cols, kSeg);
    const int64_t total = rows * segs;
    for (int64_t t = gw; t < total; t += nw) {
        const int64_t r = t / segs;
        nvfp4_segment<FOS>(x, r, (t - r * segs) * kSeg, cols, ldx, q, sb, s_g, lane);
    }
}

// One outer scale per row (per token): a warp owns a row, reads it once for
// its amax and again (from L2) to quantise it.
template <bool FOS>
__global__ void __launch_bounds__(kThreads)
quant_nvfp4_row_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
                       uint8_t* __restrict__ q, uint8_t* __restrict__ sb, float* __restrict__ row_scale, bool given) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = gw; r < rows; r += nw) {
        float s_g;
        if (given) {
            s_g = row_scale[r];
        } else {
            uint32_t m = 0;
            for (int64_t cb = 0; cb < cols; cb += kSeg) {
                uint4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int64_t c = cb + j * 256 + lane * 8;
                    v[j] = (c < cols) ? ldg_v4(x + r * ldx + c) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) m = max(m, absmax_v4(v[j]));
            }
            const float amax = amax_bits_to_f32(warp_max_u32(m, 32));
            s_g = amax == 0.0f ? 1.0f : __fdiv_rn(amax, FOS ? kNvfp4GlobalDiv4over6 : kNvfp4GlobalDiv);
            if (lane == 0) row_scale[r] = s_g;
        }
        for (int64_t cb = 0; cb < cols; cb += kSeg) nvfp4_segment<FOS>(x, r, cb, cols, ldx, q, sb, s_g, lane);
    }
}

// ---------------------------------------------------------------- 128x128 (row-wise)
template <bool P2>
__global__ void __launch_bounds__(kThreads)
quant_block_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
                   uint8_t* __restrict__ q, void* __restrict__ s) {
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = (int64_t)blockIdx.y * 128, c0 = (int64_t)blockIdx.x * 128;
    const int64_t c = c0 + (lane & 15) * 8;
    const bool cok = c < cols;
    uint4 v[8];
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = r0 + 16 * w + 2 * i + (lane >> 4);
        v[i] = (cok && r < rows) ? ldg_v4(x + r * ldx + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) m = max(m, absmax_v4(v[i]));
    const uint32_t bm = block_max_u32(m);
    float sc = 1.0f;
    if constexpr (P2) {
        const int e = mx_exponent_from_amax_bits(bm << 16);
        sc = exp2_neg(e);
        if (threadIdx.x == 0) static_cast<uint8_t*>(s)[(int64_t)blockIdx.y * gridDim.x + blockIdx.x] = (uint8_t)(e + 127);
    } else {
        sc = fp32_scale_from_amax(amax_bits_to_f32(bm));
        if (threadIdx.x == 0) static_cast<float*>(s)[(int64_t)blockIdx.y * gridDim.x + blockIdx.x] = sc;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = r0 + 16 * w + 2 * i + (lane >> 4);
        if (cok && r < rows) {
            float f[8];
            unpack8(v[i], f);
            *reinterpret_cast<uint2*>(q + r * cols + c) = P2 ? cast8_mul(f, sc) : cast8_div(f, sc);
        }
    }
}

// ---------------------------------------------------------------- transposed (+ optional row-wise)
// CTA tile: 128 rows x 128 columns of X, 512 threads.  Warp w owns rows
// 8w..8w+7, lane l owns columns 4l..4l+3 (8-byte loads, 256 bytes per warp
// and row).  Column amaxes are combined through shared memory.  The codes
// of X^T are staged in shared memory as a [column][row] byte tile (row pitch
// 136 bytes, so the 8-byte stores of one warp spread over all banks) and
// leave as whole 128-byte rows of X^T; the optional row-wise codes of X
// leave straight from registers as 4-byte runs (128 bytes per warp and row).
constexpr int kTileThreads = 512;
constexpr int kTPitch = 136;

template <int GRAN, bool DUAL>
__global__ void __launch_bounds__(kTileThreads, 2)
quant_tile_t_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
                    uint8_t* __restrict__ qt, void* __restrict__ st,
                    uint8_t* __restrict__ q, void* __restrict__ s,
                    const uint32_t* __restrict__ partials, int nparts, const float* __restrict__ given) {
    __shared__ uint32_t red[16][128];
    __shared__ __align__(16) uint8_t tq[128 * kTPitch];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t rt = blockIdx.y, ct = blockIdx.x;
    const int64_t r0 = rt * 128, c0 = ct * 128;
    const int64_t cc = c0 + lane * 4;
    const bool cok = cc < cols;
    const int64_t rw = r0 + 8 * w;           // first row of this warp
    const bool wok = rw < rows;              // rows % 16 == 0: 8 rows all valid or all not

    float s_uniform = 1.0f;
    if constexpr (GRAN == kGranPT) {
        if (given != nullptr) {
            s_uniform = *given;
        } else {
            s_uniform = fp32_scale_from_amax(tensor_amax(partials, nparts));
            if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
                static_cast<float*>(st)[0] = s_uniform;
                if (DUAL) static_cast<float*>(s)[0] = s_uniform;
            }
        }
    }

    uint2 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v[i] = (cok && wok) ? ldg_v2(x + (rw + i) * ldx + cc) : make_uint2(0, 0);

    uint32_t cm[4] = {0, 0, 0, 0};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        cm[0] = max(cm[0], v[i].x & 0x7FFFu);
        cm[1] = max(cm[1], (v[i].x >> 16) & 0x7FFFu);
        cm[2] = max(cm[2], v[i].y & 0x7FFFu);
        cm[3] = max(cm[3], (v[i].y >> 16) & 0x7FFFu);
    }

    float col_s[4] = {1.0f, 1.0f, 1.0f, 1.0f};   // divisor (FP32 grans) or multiplier (power-of-two grans)
    int col_e[4] = {0, 0, 0, 0};
    float s_blk = 1.0f;
    int e_blk = 0;
    if constexpr (GRAN == kGranTok || GRAN == kGranMx || GRAN == kGranTokP2) {
#pragma unroll
        for (int j = 0; j < 4; ++j) red[w][lane * 4 + j] = cm[j];
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t m = 0;
            if constexpr (GRAN == kGranTok || GRAN == kGranTokP2) {
#pragma unroll
                for (int k = 0; k < 16; ++k) m = max(m, red[k][lane * 4 + j]);
                if constexpr (GRAN == kGranTok) {
                    col_s[j] = fp32_scale_from_amax(amax_bits_to_f32(m));
                } else {
                    col_e[j] = mx_exponent_from_amax_bits(m << 16);
                    col_s[j] = exp2_neg(col_e[j]);
                }
            } else {
                const int g = w & ~3;            // 32 rows = 4 warps
#pragma unroll
                for (int k = 0; k < 4; ++k) m = max(m, red[g + k][lane * 4 + j]);
                col_e[j] = mx_exponent_from_amax_bits(m << 16);
                col_s[j] = exp2_neg(col_e[j]);
            }
        }
    } else if constexpr (GRAN == kGranBlk || GRAN == kGranBlkP2) {
        const uint32_t bm = block_max_u32(max(max(cm[0], cm[1]), max(cm[2], cm[3])));
        if constexpr (GRAN == kGranBlk) {
            s_blk = fp32_scale_from_amax(amax_bits_to_f32(bm));
        } else {
            e_blk = mx_exponent_from_amax_bits(bm << 16);
            s_blk = exp2_neg(e_blk);
        }
    }

    // ---- transposed codes: column cc + j, rows rw .. rw+7 -> shared tile
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float f[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t word = (j < 2) ? v[i].x : v[i].y;
            f[i] = (j & 1) ? bf16_hi(word) : bf16_lo(word);
        }
        const float d = (GRAN == kGranPT) ? s_uniform : ((GRAN == kGranBlk || GRAN == kGranBlkP2) ? s_blk : col_s[j]);
        uint2 o;
        if constexpr (kPow2<GRAN>) {
            o.x = e4m3x4(__fmul_rn(f[0], d), __fmul_rn(f[1], d), __fmul_rn(f[2], d), __fmul_rn(f[3], d));
            o.y = e4m3x4(__fmul_rn(f[4], d), __fmul_rn(f[5], d), __fmul_rn(f[6], d), __fmul_rn(f[7], d));
        } else {
            o.x = e4m3x4(__fdiv_rn(f[0], d), __fdiv_rn(f[1], d), __fdiv_rn(f[2], d), __fdiv_rn(f[3], d));
            o.y = e4m3x4(__fdiv_rn(f[4], d), __fdiv_rn(f[5], d), __fdiv_rn(f[6], d), __fdiv_rn(f[7], d));
        }
        *reinterpret_cast<uint2*>(tq + (lane * 4 + j) * kTPitch + 8 * w) = o;
    }
    __syncthreads();
    // ---- whole rows of X^T: 128 columns x 128 bytes, 16 bytes per thread and pass
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        const int t = threadIdx.x + pass * kTileThreads;
        const int qc = t >> 3, k = t & 7;    // column of X (row of X^T), 16-byte chunk
        const int64_t c = c0 + qc;
        if (c < cols && r0 + 16 * k < rows) {
            const uint8_t* src = tq + qc * kTPitch + 16 * k;
            const uint2 lo = *reinterpret_cast<const uint2*>(src);
            const uint2 hi = *reinterpret_cast<const uint2*>(src + 8);
            *reinterpret_cast<uint4*>(qt + c * rows + r0 + 16 * k) = make_uint4(lo.x, lo.y, hi.x, hi.y);
        }
    }
    // ---- scales of X^T ([cols, *] grid)
    if constexpr (GRAN == kGranTok) {
        if (w == 0 && cok) {
            const int64_t nrb = ceil_div(rows, 128);
#pragma unroll
            for (int j = 0; j < 4; ++j) static_cast<float*>(st)[(cc + j) * nrb + rt] = col_s[j];
        }
    } else if constexpr (GRAN == kGranMx) {
        if ((w & 3) == 0 && cok && wok) {
            const int64_t nrb = ceil_div(rows, 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) static_cast<uint8_t*>(st)[(cc + j) * nrb + (rw >> 5)] = (uint8_t)(col_e[j] + 127);
        }
    } else if constexpr (GRAN == kGranTokP2) {
        if (w == 0 && cok) {
            const int64_t nrb = ceil_div(rows, 128);
#pragma unroll
            for (int j = 0; j < 4; ++j) static_cast<uint8_t*>(st)[(cc + j) * nrb + rt] = (uint8_t)(col_e[j] + 127);
        }
    } else if constexpr (GRAN == kGranBlk) {
        if (threadIdx.x == 0) static_cast<float*>(st)[ct * gridDim.y + rt] = s_blk;
    } else if constexpr (GRAN == kGranBlkP2) {
        if (threadIdx.x == 0) static_cast<uint8_t*>(st)[ct * gridDim.y + rt] = (uint8_t)(e_blk + 127);
    }

    // ---- row-wise codes of X from the same registers
    if constexpr (DUAL) {
        const int64_t ncb = ceil_div(cols, GRAN == kGranMx ? 32 : 128);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float f[4] = {bf16_lo(v[i].x), bf16_hi(v[i].x), bf16_lo(v[i].y), bf16_hi(v[i].y)};
            const uint32_t m4 = max(bf16x2_absmax_bits(v[i].x), bf16x2_absmax_bits(v[i].y));
            uint32_t o;
            if constexpr (GRAN == kGranTok) {
                const float sr = fp32_scale_from_amax(amax_bits_to_f32(warp_max_u32(m4, 32)));
                o = e4m3x4(__fdiv_rn(f[0], sr), __fdiv_rn(f[1], sr), __fdiv_rn(f[2], sr), __fdiv_rn(f[3], sr));
                if (lane == 0 && wok) static_cast<float*>(s)[(rw + i) * ncb + ct] = sr;
            } else if constexpr (GRAN == kGranMx) {
                const int e = mx_exponent_from_amax_bits(warp_max_u32(m4, 8) << 16);
                const float mm = exp2_neg(e);
                o = e4m3x4(__fmul_rn(f[0], mm), __fmul_rn(f[1], mm), __fmul_rn(f[2], mm), __fmul_rn(f[3], mm));
                if ((lane & 7) == 0 && cok && wok) static_cast<uint8_t*>(s)[(rw + i) * ncb + (cc >> 5)] = (uint8_t)(e + 127);
            } else if constexpr (GRAN == kGranTokP2) {
                const int e = mx_exponent_from_amax_bits(warp_max_u32(m4, 32) << 16);
                const float mm = exp2_neg(e);
                o = e4m3x4(__fmul_rn(f[0], mm), __fmul_rn(f[1], mm), __fmul_rn(f[2], mm), __fmul_rn(f[3], mm));
                if (lane == 0 && wok) static_cast<uint8_t*>(s)[(rw + i) * ncb + ct] = (uint8_t)(e + 127);
            } else if constexpr (GRAN == kGranBlkP2) {
                o = e4m3x4(__fmul_rn(f[0], s_blk), __fmul_rn(f[1], s_blk), __fmul_rn(f[2], s_blk), __fmul_rn(f[3], s_blk));
            } else {
                const float d = (GRAN == kGranPT) ? s_uniform : s_blk;
                o = e4m3x4(__fdiv_rn(f[0], d), __fdiv_rn(f[1], d), __fdiv_rn(f[2], d), __fdiv_rn(f[3], d));
            }
            if (cok && wok) *reinterpret_cast<uint32_t*>(q + (rw + i) * cols + cc) = o;
        }
        if constexpr (GRAN == kGranBlk) {
            if (threadIdx.x == 0) static_cast<float*>(s)[rt * gridDim.x + ct] = s_blk;
        } else if constexpr (GRAN == kGranBlkP2) {
            if (threadIdx.x == 0) static_cast<uint8_t*>(s)[rt * gridDim.x + ct] = (uint8_t)(e_blk + 127);
        }
    }
}

// ---------------------------------------------------------------- launchers
static int rowwise_blocks(int64_t rows, int64_t cols, int cap) {
    const int64_t tasks = rows * ceil_div(cols, kSeg);
    const int64_t want = ceil_div(tasks, kThreads / 32);
    return (int)std::max<int64_t>(1, std::min<int64_t>(want, cap));
}

static int launch_amax(const QuantJob& j, cudaStream_t st, int* nparts) {
    const int n = rowwise_blocks(j.rows, j.cols, std::min(kMaxPartials, sm_count() * 4));
    amax_partials_kernel<<<n, kThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.partials);
    *nparts = n;
    return (int)cudaGetLastError();
}

int launch_quantize(const QuantJob& j, cudaStream_t st) {
    const int cap = sm_count() * 8;
    const int nb = rowwise_blocks(j.rows, j.cols, cap);
    int nparts = 0;
    switch (j.gran) {
    case kGranTok:
        quant_rows_kernel<kGranTok><<<nb, kThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.q, j.s, nullptr, 0, nullptr);
        break;
    case kGranMx:
        quant_rows_kernel<kGranMx><<<nb, kThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.q, j.s, nullptr, 0, nullptr);
        break;
    case kGranPT: {
        if (!j.given_scale) {
            const int e = launch_amax(j, st, &nparts);
            if (e) return e;
        }
        quant_rows_kernel<kGranPT><<<nb, kThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.q, j.s, j.partials, nparts,
                                                             j.given_scale ? static_cast<const float*>(j.s) : nullptr);
        break;
    }
    case kGranBlk:
    case kGranBlkP2: {
        dim3 grid((unsigned)ceil_div(j.cols, 128), (unsigned)ceil_div(j.rows, 128));
        if (j.gran == kGranBlk)
            quant_block_kernel<false><<<grid, kThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.q, j.s);
        else
            quant_block_kernel<true><<<grid, kThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.q, j.s);
        break;
    }
    case kGranTokP2:
        quant_rows_kernel<kGranTokP2><<<nb, kThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.q, j.s, nullptr, 0, nullptr);
        break;
    case kGranNv: {
        if (!j.given_scale) {
            const int e = launch_amax(j, st, &nparts);
            if (e) return e;
        }
        auto* sb = static_cast<uint8_t*>(j.s);
        if (j.four_over_six)
            quant_nvfp4_kernel<true><<<nb, kThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.q, sb, j.tensor_scale,
                                                              j.partials, nparts, j.given_scale);
        else
            quant_nvfp4_kernel<false><<<nb, kThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.q, sb, j.tensor_scale,
                                                               j.partials, nparts, j.given_scale);
        break;
    }
    case kGranNvRow: {
        const int rb = (int)std::max<int64_t>(1, std::min<int64_t>(ceil_div(j.rows, kThreads / 32), cap));
        auto* sb = static_cast<uint8_t*>(j.s);
        if (j.four_over_six)
            quant_nvfp4_row_kernel<true><<<rb, kThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.q, sb, j.tensor_scale,
                                                                  j.given_scale);
        else
            quant_nvfp4_row_kernel<false><<<rb, kThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.q, sb,
                                                                   j.tensor_scale, j.given_scale);
        break;
    }
    default:
        return (int)cudaErrorInvalidValue;
    }
    return (int)cudaGetLastError();
}

template <int GRAN>
static void launch_tile(const QuantJob& j, cudaStream_t st, int nparts, const float* given) {
    dim3 grid((unsigned)ceil_div(j.cols, 128), (unsigned)ceil_div(j.rows, 128));
    if (j.q != nullptr)
        quant_tile_t_kernel<GRAN, true><<<grid, kTileThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.qt, j.st, j.q, j.s,
                                                                   j.partials, nparts, given);
    else
        quant_tile_t_kernel<GRAN, false><<<grid, kTileThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.qt, j.st, nullptr,
                                                                    nullptr, j.partials, nparts, given);
}

int launch_quantize_transposed(const QuantJob& j, cudaStream_t st) {
    int nparts = 0;
    switch (j.gran) {
    case kGranTok: launch_tile<kGranTok>(j, st, 0, nullptr); break;
    case kGranMx: launch_tile<kGranMx>(j, st, 0, nullptr); break;
    case kGranBlk: launch_tile<kGranBlk>(j, st, 0, nullptr); break;
    case kGranTokP2: launch_tile<kGranTokP2>(j, st, 0, nullptr); break;
    case kGranBlkP2: launch_tile<kGranBlkP2>(j, st, 0, nullptr); break;
    case kGranPT: {
        if (!j.given_scale) {
            const int e = launch_amax(j, st, &nparts);
            if (e) return e;
        }
        launch_tile<kGranPT>(j, st, nparts, j.given_scale ? static_cast<const float*>(j.st) : nullptr);
        break;
    }
    default:
        return (int)cudaErrorInvalidValue;
    }
    return (int)cudaGetLastError();
}

}  // namespace fp8bs

namespace fp8bs {

// Per-tensor quantisation with the amax partials in scratch the caller
// names: pass 1 runs exactly `nparts` CTAs, each writing one partial, and
// pass 2 reduces those `nparts` partials, so no slot needs clearing first.
int launch_quantize_per_tensor_scratch(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q,
                                       float* scale, uint32_t* partials, int nparts, cudaStream_t st) {
    amax_partials_kernel<<<nparts, kThreads, 0, st>>>(x, rows, cols, ldx, partials);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    const int nb = rowwise_blocks(rows, cols, sm_count() * 8);
    quant_rows_kernel<kGranPT><<<nb, kThreads, 0, st>>>(x, rows, cols, ldx, q, scale, partials, nparts, nullptr);
    return (int)cudaGetLastError();
}

}  // namespace fp8bs
