// dequant.cu -- BF16 dequantisation of quantised operands.
//
// "Low Precision RL", section "Advanced: dequantized backward": the BF16
// backward GEMMs consume BF16 dequantisations of the low-precision forward
// operands.  The value of an element is code * block scale (* outer scale
// for NVFP4); it is rounded once to BF16 (nearest, ties to even).
//
// Single rounding without wide arithmetic uses rounding to odd (Boldo and
// Melquiond, "Emulation of FMA and correctly rounded sums: proved algorithms
// using rounding to odd", IEEE TC 2008): the float32 product is rounded
// toward zero and its last bit set when inexact (exactness from an FMA
// residual); rounding that odd-rounded value to BF16 (8 significant bits,
// 16 fewer than float32) gives the correctly rounded result.  Below 2^-100
// the FMA residual itself could underflow, so those rare elements take an
// exact double-precision product instead, odd-rounded to float32 the same way.
//
// HBM-bound: a thread turns 8 codes into 8 BF16 values (one 16-byte store).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace fp8bs {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float round_odd_mul(float a, float b) {
    const float p = __fmul_rz(a, b);
    if (fabsf(p) < 0x1p-100f && p != 0.0f) {
        const double d = (double)a * (double)b;                  // exact: 24 + 24 bits
        const float f = __double2float_rz(d);
        return ((double)f != d) ? __uint_as_float(__float_as_uint(f) | 1u) : f;
    }
    const float err = __fmaf_rn(a, b, -p);
    return err != 0.0f ? __uint_as_float(__float_as_uint(p) | 1u) : p;
}

__device__ __forceinline__ uint32_t bf16x2_of(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// One thread: 8 consecutive elements of one row.  GRAN is the fp8bs_gran
// value: 4 NVFP4 (one outer scale), 7 NVFP4 with one outer scale per row.
template <int GRAN>
__global__ void __launch_bounds__(kThreads)
dequant_kernel(const uint8_t* __restrict__ q, const void* __restrict__ scales, const float* __restrict__ tensor_scale,
               int64_t rows, int64_t cols, __nv_bfloat16* __restrict__ out, int64_t ld_out) {
    const int64_t per_row = cols >> 3;
    const int64_t total = rows * per_row;
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = t / per_row;
        const int64_t c = (t - r * per_row) << 3;
        float v[8];
        if constexpr (GRAN == 4 || GRAN == 7) {   // NVFP4: packed E2M1, E4M3 block scale per 16, S_g
            const uint32_t w = *reinterpret_cast<const uint32_t*>(q + r * (cols >> 1) + (c >> 1));
            const float sb = e4m3_value(static_cast<const uint8_t*>(scales)[r * (cols >> 4) + (c >> 4)]);
            const float sg = (GRAN == 7) ? tensor_scale[r] : *tensor_scale;
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = round_odd_mul(e2m1_value((w >> (4 * i)) & 0xFu) * sb, sg);
        } else {
            const uint2 w = *reinterpret_cast<const uint2*>(q + r * cols + c);
            float s;
            if constexpr (GRAN == 0) {
                s = *static_cast<const float*>(scales);
            } else if constexpr (GRAN == 1) {
                s = static_cast<const float*>(scales)[r * ((cols + 127) >> 7) + (c >> 7)];
            } else if constexpr (GRAN == 2) {
                s = static_cast<const float*>(scales)[(r >> 7) * ((cols + 127) >> 7) + (c >> 7)];
            } else if constexpr (GRAN == 3) {
                s = exp2_neg(127 - (int)static_cast<const uint8_t*>(scales)[r * ((cols + 31) >> 5) + (c >> 5)]);
            } else if constexpr (GRAN == 5) {
                s = exp2_neg(127 - (int)static_cast<const uint8_t*>(scales)[r * ((cols + 127) >> 7) + (c >> 7)]);
            } else {
                s = exp2_neg(127 - (int)static_cast<const uint8_t*>(scales)[(r >> 7) * ((cols + 127) >> 7) + (c >> 7)]);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t code = ((i < 4 ? w.x : w.y) >> (8 * (i & 3))) & 0xFFu;
                v[i] = round_odd_mul(e4m3_value(code), s);
            }
        }
        uint4 o;
        o.x = bf16x2_of(v[0], v[1]);
        o.y = bf16x2_of(v[2], v[3]);
        o.z = bf16x2_of(v[4], v[5]);
        o.w = bf16x2_of(v[6], v[7]);
        *reinterpret_cast<uint4*>(out + r * ld_out + c) = o;
    }
}

}  // namespace

int launch_dequantize(const uint8_t* q, const void* scales, const float* tensor_scale, int64_t rows, int64_t cols,
                      int gran, void* out, int64_t ld_out, cudaStream_t st) {
    const int64_t total = rows * (cols >> 3);
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>(ceil_div(total, kThreads), sm_count() * 8));
    auto* o = static_cast<__nv_bfloat16*>(out);
    switch (gran) {
    case 0: dequant_kernel<0><<<blocks, kThreads, 0, st>>>(q, scales, tensor_scale, rows, cols, o, ld_out); break;
    case 1: dequant_kernel<1><<<blocks, kThreads, 0, st>>>(q, scales, tensor_scale, rows, cols, o, ld_out); break;
    case 2: dequant_kernel<2><<<blocks, kThreads, 0, st>>>(q, scales, tensor_scale, rows, cols, o, ld_out); break;
    case 3: dequant_kernel<3><<<blocks, kThreads, 0, st>>>(q, scales, tensor_scale, rows, cols, o, ld_out); break;
    case 4: dequant_kernel<4><<<blocks, kThreads, 0, st>>>(q, scales, tensor_scale, rows, cols, o, ld_out); break;
    case 5: dequant_kernel<5><<<blocks, kThreads, 0, st>>>(q, scales, tensor_scale, rows, cols, o, ld_out); break;
    case 6: dequant_kernel<6><<<blocks, kThreads, 0, st>>>(q, scales, tensor_scale, rows, cols, o, ld_out); break;
    case 7: dequant_kernel<7><<<blocks, kThreads, 0, st>>>(q, scales, tensor_scale, rows, cols, o, ld_out); break;
    default: return (int)cudaErrorInvalidValue;
    }
    return (int)cudaGetLastError();
}

}  // namespace fp8bs
