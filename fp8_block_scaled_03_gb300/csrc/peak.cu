// peak.cu -- dense tensor-core throughput loop (measures the FP8 / FP4 MMA peak).
//
// The GEMM rooflines need the dense FP8 and FP4 tensor rates of this part.
// A cuBLAS BF16 GEMM gives the BF16 rate only, and the FP8/FP4 rates are
// not a fixed multiple of it on every part, so this loop measures them with
// the same instructions the GEMM kernels issue: one CTA per SM, operands
// resident in shared memory (no memory traffic at all), one thread issuing
// tcgen05.mma back to back into a TMEM accumulator, M = 128 rows per CTA.
//   kind 0  kind::f8f6f4, E4M3 x E4M3, K = 32 per instruction
//   kind 1  kind::mxf8f6f4.block_scale.scale_vec::1X, E4M3 with UE8M0 scales, K = 32
//   kind 2  kind::mxf4nvf4.block_scale.scale_vec::4X, E2M1 with E4M3 scales, K = 64
// Each K block is four instructions (one 128-byte row of operand bytes).
// The caller times the launch; FLOPs per launch = ctas * iters * 4 * 2 *
// 128 * n * K.  pattern 1 fills every operand with 1.0 and every scale with
// 1.0, so each accumulator element ends at iters * 4 * K (the check the
// tests make); pattern 0 fills them with pseudo-random finite values, as
// real operands would toggle.  The tensor cores see the same instruction
// stream either way.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace {

constexpr int A_BYTES = 128 * 128, B_BYTES = 256 * 128, SF_BYTES = 12 * 512;
// more than half of an SM's shared memory, so that no two CTAs share an SM (and its TMEM)
constexpr size_t PEAK_SMEM = 120 * 1024;
static_assert(PEAK_SMEM >= 1024 + A_BYTES + B_BYTES + SF_BYTES, "peak loop shared memory");

__device__ __forceinline__ uint32_t hash32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352dU;
    x ^= x >> 15;
    x *= 0x846ca68bU;
    x ^= x >> 16;
    return x;
}

template <int KIND>
__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int iters, int n, int pattern, float* out, int* status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t done;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    // operands: E4M3 codes with the lowest exponent bit cleared (never NaN),
    // or E2M1 nibbles; 1.0 is 0x38 in E4M3 and 0x2 per nibble in E2M1
    const uint32_t one_word = (KIND == 2) ? 0x22222222u : 0x38383838u;
    uint32_t* w = reinterpret_cast<uint32_t*>(base);
    for (int i = threadIdx.x; i < (A_BYTES + B_BYTES) / 4; i += blockDim.x) {
        uint32_t v = one_word;
        if (pattern == 0) {
            v = hash32((uint32_t)i * 2654435761u + blockIdx.x);
            if (KIND != 2) v &= 0xF7F7F7F7u;
        }
        w[i] = v;
    }
    // scale atoms: UE8M0 1.0 = 127, E4M3 1.0 = 0x38
    const uint32_t sf_word = (KIND == 2) ? 0x38383838u : 0x7F7F7F7Fu;
    uint32_t* sf = reinterpret_cast<uint32_t*>(base + A_BYTES + B_BYTES);
    for (int i = threadIdx.x; i < SF_BYTES / 4; i += blockDim.x) sf[i] = sf_word;
    fence_proxy_async_smem();   // generic-proxy writes, read by the tensor core (async proxy)

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&done), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (threadIdx.x < 32) {
        tmem_alloc(smem_u32(&tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (threadIdx.x == 0) {
        const uint32_t a_addr = smem_u32(base);
        const uint64_t adesc = kmajor_sw128_desc(a_addr);
        const uint64_t bdesc = kmajor_sw128_desc(a_addr + A_BYTES);
        const uint32_t sfa = tmem + 256, sfb = sfa + 16;
        if (KIND != 0) {
            // A scale atoms then B scale atoms (4 + 8 for NVFP4, 1 + 2 for MXFP8)
            const int atoms = (KIND == 2) ? 12 : 3;
            const uint32_t sf_smem = smem_u32(sf);
            for (int j = 0; j < atoms; ++j) {
                const uint32_t col = (KIND == 2) ? (j < 4 ? sfa + 4 * j : sfb + 4 * (j - 4))
                                                 : (j < 1 ? sfa : sfb + 4 * (j - 1));
                tmem_cp_32x128b_x4(col, smem_desc(sf_smem + 512 * j, 0, 128, 0));
            }
        }
        const uint32_t idesc_f8 = idesc_f8f6f4_e4m3(128, (uint32_t)n);
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
                if (KIND == 0) {
                    mma_f8f6f4(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc_f8, acc);
                } else if (KIND == 1) {
                    mma_mxf8(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc_block_scaled(128, n, 0, 0, 1, kk, kk), sfa,
                             sfb, acc);
                } else {
                    mma_nvf4(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc_block_scaled(128, n, 1, 1, 0, 0, 0),
                             sfa + 4 * kk, sfb + 8 * kk, acc);
                }
            }
        }
        mma_commit(smem_u32(&done));
    }
    __syncwarp();
    // every thread waits for the MMAs (bounded), then warp q reads its 32
    // rows of accumulator column 0
    const bool ok = mbar_wait(smem_u32(&done), 0, &abort_flag, status);
    tc_fence_after();
    if (__all_sync(0xFFFFFFFFu, ok) && out != nullptr && blockIdx.x == 0) {
        uint32_t r[16];
        const int q = threadIdx.x >> 5;
        tmem_ld_32x32b_x16(tmem + ((uint32_t)(32 * q) << 16), r);
        tmem_ld_wait16(r);
        out[threadIdx.x] = __uint_as_float(r[0]);
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x < 32) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int KIND>
int launch_peak(int ctas, int iters, int n, int pattern, float* out, int* status, cudaStream_t st) {
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(mma_peak_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)PEAK_SMEM);
        if (e != cudaSuccess) return (int)e;
        attr_set[dev] = true;
    }
    mma_peak_kernel<KIND><<<ctas, 128, PEAK_SMEM, st>>>(iters, n, pattern, out, status);
    return (int)cudaGetLastError();
}

}  // namespace

int launch_mma_peak(int kind, int ctas, int iters, int n, int pattern, float* out, int* status, cudaStream_t st) {
    if (kind == 0) return launch_peak<0>(ctas, iters, n, pattern, out, status, st);
    if (kind == 1) return launch_peak<1>(ctas, iters, n, pattern, out, status, st);
    return launch_peak<2>(ctas, iters, n, pattern, out, status, st);
}

}  // namespace fp8bs
