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
// HBM-bound: a thread turns 16 codes into 16 BF16 values (two 16-byte stores).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace fp8bs {
namespace {

// a * b rounded to odd, for |a * b| >= 2^-100 or a * b == 0 (callers check
// the scale once per chunk: every nonzero code value is at least 2^-10).
__device__ __forceinline__ float round_odd_mul_normal(float a, float b) {
    const float p = __fmul_rz(a, b);
    const float err = __fmaf_rn(a, b, -p);
    return err != 0.0f ? __uint_as_float(__float_as_uint(p) | 1u) : p;
}

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

// Block of 32 x 8 threads: threadIdx.x walks 16-element column chunks (a
// warp covers 512 columns of one row), threadIdx.y and the grid's y walk
// rows.  A chunk lies inside one scale group at every granularity (groups are
// 16, 32 or 128 columns wide and chunks start at multiples of 16).  When
// cols % 16 == 8 the row's last chunk holds 8 elements.  VEC16: the codes of
// a chunk are read with one 16-byte load (q 16-byte aligned, cols % 16 == 0),
// else with two 8-byte loads.
template <int GRAN, bool VEC16>
__global__ void __launch_bounds__(256)
dequant_kernel(const uint8_t* __restrict__ q, const void* __restrict__ scales, const float* __restrict__ tensor_scale,
               int64_t rows, int64_t cols, __nv_bfloat16* __restrict__ out, int64_t ld_out) {
    const int64_t c = ((int64_t)blockIdx.x * 32 + threadIdx.x) * 16;
    if (c >= cols) return;
    const bool full = c + 16 <= cols;
    for (int64_t r = (int64_t)blockIdx.y * 8 + threadIdx.y; r < rows; r += (int64_t)gridDim.y * 8) {
        float v[16];
        if constexpr (GRAN == 4 || GRAN == 7) {   // NVFP4: packed E2M1, one E4M3 block scale per chunk, S_g
            const uint2 w = *reinterpret_cast<const uint2*>(q + r * (cols >> 1) + (c >> 1));
            const float sb = e4m3_value(static_cast<const uint8_t*>(scales)[r * (cols >> 4) + (c >> 4)]);
            const float sg = (GRAN == 7) ? tensor_scale[r] : *tensor_scale;
            // E2M1 x E4M3 is exact in float32 and at least 2^-10 when nonzero
            if (fabsf(sg) >= 0x1p-90f) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 f = e2m1x2_to_float2(((i < 4 ? w.x : w.y) >> (8 * (i & 3))) & 0xFFu);
                    v[2 * i] = round_odd_mul_normal(f.x * sb, sg);
                    v[2 * i + 1] = round_odd_mul_normal(f.y * sb, sg);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 f = e2m1x2_to_float2(((i < 4 ? w.x : w.y) >> (8 * (i & 3))) & 0xFFu);
                    v[2 * i] = round_odd_mul(f.x * sb, sg);
                    v[2 * i + 1] = round_odd_mul(f.y * sb, sg);
                }
            }
        } else {
            uint4 w;
            const uint8_t* src = q + r * cols + c;
            if (VEC16) {
                w = *reinterpret_cast<const uint4*>(src);
            } else {
                const uint2 lo = *reinterpret_cast<const uint2*>(src);
                const uint2 hi = full ? *reinterpret_cast<const uint2*>(src + 8) : make_uint2(0u, 0u);
                w = make_uint4(lo.x, lo.y, hi.x, hi.y);
            }
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
            const uint32_t words[4] = {w.x, w.y, w.z, w.w};
            if (GRAN == 3 || GRAN == 5 || GRAN == 6) {
                // power-of-two scale: code * 2^-e is exact (at worst a float32
                // subnormal with room for the code's 4 significant bits)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 f = e4m3x2_to_float2(words[i >> 1] >> (16 * (i & 1)));
                    v[2 * i] = __fmul_rn(f.x, s);
                    v[2 * i + 1] = __fmul_rn(f.y, s);
                }
            } else if (fabsf(s) >= 0x1p-90f) {   // every nonzero E4M3 value is at least 2^-9
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 f = e4m3x2_to_float2(words[i >> 1] >> (16 * (i & 1)));
                    v[2 * i] = round_odd_mul_normal(f.x, s);
                    v[2 * i + 1] = round_odd_mul_normal(f.y, s);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 f = e4m3x2_to_float2(words[i >> 1] >> (16 * (i & 1)));
                    v[2 * i] = round_odd_mul(f.x, s);
                    v[2 * i + 1] = round_odd_mul(f.y, s);
                }
            }
        }
        __nv_bfloat16* dst = out + r * ld_out + c;
        uint4 o;
        o.x = bf16x2_of(v[0], v[1]);
        o.y = bf16x2_of(v[2], v[3]);
        o.z = bf16x2_of(v[4], v[5]);
        o.w = bf16x2_of(v[6], v[7]);
        *reinterpret_cast<uint4*>(dst) = o;
        if (full) {
            o.x = bf16x2_of(v[8], v[9]);
            o.y = bf16x2_of(v[10], v[11]);
            o.z = bf16x2_of(v[12], v[13]);
            o.w = bf16x2_of(v[14], v[15]);
            *reinterpret_cast<uint4*>(dst + 8) = o;
        }
    }
}

template <int GRAN>
void launch_g(dim3 grid, bool vec16, const uint8_t* q, const void* scales, const float* ts, int64_t rows,
              int64_t cols, __nv_bfloat16* o, int64_t ld_out, cudaStream_t st) {
    const dim3 block(32, 8);
    if (vec16)
        dequant_kernel<GRAN, true><<<grid, block, 0, st>>>(q, scales, ts, rows, cols, o, ld_out);
    else
        dequant_kernel<GRAN, false><<<grid, block, 0, st>>>(q, scales, ts, rows, cols, o, ld_out);
}

}  // namespace

int launch_dequantize(const uint8_t* q, const void* scales, const float* tensor_scale, int64_t rows, int64_t cols,
                      int gran, void* out, int64_t ld_out, cudaStream_t st) {
    const dim3 grid((unsigned)ceil_div(cols, 512), (unsigned)std::min<int64_t>(ceil_div(rows, 8), 65535));
    const bool vec16 = (cols % 16 == 0) && ((reinterpret_cast<uintptr_t>(q) & 15u) == 0);
    auto* o = static_cast<__nv_bfloat16*>(out);
    switch (gran) {
    case 0: launch_g<0>(grid, vec16, q, scales, tensor_scale, rows, cols, o, ld_out, st); break;
    case 1: launch_g<1>(grid, vec16, q, scales, tensor_scale, rows, cols, o, ld_out, st); break;
    case 2: launch_g<2>(grid, vec16, q, scales, tensor_scale, rows, cols, o, ld_out, st); break;
    case 3: launch_g<3>(grid, vec16, q, scales, tensor_scale, rows, cols, o, ld_out, st); break;
    case 4: launch_g<4>(grid, vec16, q, scales, tensor_scale, rows, cols, o, ld_out, st); break;
    case 5: launch_g<5>(grid, vec16, q, scales, tensor_scale, rows, cols, o, ld_out, st); break;
    case 6: launch_g<6>(grid, vec16, q, scales, tensor_scale, rows, cols, o, ld_out, st); break;
    case 7: launch_g<7>(grid, vec16, q, scales, tensor_scale, rows, cols, o, ld_out, st); break;
    default: return (int)cudaErrorInvalidValue;
    }
    return (int)cudaGetLastError();
}

}  // namespace fp8bs
