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
#include <algorithm>
#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "tmap.h"

namespace fp8bs {

enum { kGranPT = 0, kGranTok = 1, kGranBlk = 2, kGranMx = 3, kGranNv = 4, kGranTokP2 = 5, kGranBlkP2 = 6,
       kGranNvRow = 7 };

// Granularities whose scale is a power of two (UE8M0 byte): the division by
// the scale is an exact multiplication by 2^-e.
template <int G> constexpr bool kPow2 = (G == kGranMx || G == kGranTokP2 || G == kGranBlkP2);

constexpr int kSeg = 1024;       // columns per row-wise warp task
constexpr int kThreads = 256;

// max |x| of eight BF16 values as BF16 bits: packed 16-bit maxima of the
// magnitude bits first (non-negative BF16 patterns order like their values),
// then the larger half.
__device__ __forceinline__ uint32_t absmax_v4(const uint4& v) {
    const uint32_t m = __vmaxu2(__vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu),
                                __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu));
    return max(m & 0xFFFFu, m >> 16);
}

// The same maximum pair by pair (the plain MXFP8 row kernel measured faster
// with it: 23.3 against 25.3 us for [8192, 4096]; its MoE gather and SwiGLU
// forms were faster with the packed one).
__device__ __forceinline__ uint32_t absmax_v4_pairs(const uint4& v) {
    return max(max(bf16x2_absmax_bits(v.x), bf16x2_absmax_bits(v.y)),
               max(bf16x2_absmax_bits(v.z), bf16x2_absmax_bits(v.w)));
}

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Eight elements x / S -> eight E4M3 bytes.
__device__ __forceinline__ uint2 cast8_div(const float* f, const ScaleDiv& d) {
    uint2 o;
    if (d.fast) {   // one test per group, not per element
        const ScaleDiv2 d2 = scale_div2(d);
        o.x = e4m3x4_div_fast2(pair_f32(f[0], f[1]), pair_f32(f[2], f[3]), d2);
        o.y = e4m3x4_div_fast2(pair_f32(f[4], f[5]), pair_f32(f[6], f[7]), d2);
    } else {
        o.x = e4m3x4(__fdiv_rn(f[0], d.s), __fdiv_rn(f[1], d.s), __fdiv_rn(f[2], d.s), __fdiv_rn(f[3], d.s));
        o.y = e4m3x4(__fdiv_rn(f[4], d.s), __fdiv_rn(f[5], d.s), __fdiv_rn(f[6], d.s), __fdiv_rn(f[7], d.s));
    }
    return o;
}

// Eight elements x * 2^-e (exact power-of-two division) -> eight E4M3 bytes.
__device__ __forceinline__ uint2 cast8_mul(const float* f, float m) {
    const uint64_t m2 = pair_f32(m, m);
    uint2 o;
    o.x = e4m3x4_mul2(pair_f32(f[0], f[1]), pair_f32(f[2], f[3]), m2);
    o.y = e4m3x4_mul2(pair_f32(f[4], f[5]), pair_f32(f[6], f[7]), m2);
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

// ---------------------------------------------------------------- warp task cursor
// A warp's tasks are t = gw, gw + nw, ...; task t is segment t % segs of row
// t / segs.  Both parts advance by a constant per stride, so a task loop
// divides once, not once per task.
struct TaskCursor {
    int64_t r, si;               // current row and segment
    int64_t dr, ds, segs;
    __device__ __forceinline__ TaskCursor(int64_t gw, int64_t nw, int64_t segs_) : segs(segs_) {
        r = gw / segs;
        si = gw - r * segs;
        dr = nw / segs;
        ds = nw - dr * segs;
    }
    __device__ __forceinline__ int64_t next_row() const { return r + dr + (si + ds >= segs ? 1 : 0); }
    __device__ __forceinline__ void advance() {
        si += ds;
        r += dr;
        if (si >= segs) {
            si -= segs;
            ++r;
        }
    }
};

// ---------------------------------------------------------------- pass 1: amax partials
// The cast pass that follows reads X again.  When X fits in L2 (the host
// decides: `keep`), the pass's loads of X mark their lines evict-last, and
// the cast pass then finds X in L2 instead of HBM.  Without the mark the
// second pass over a tensor of about L2's size found little of it: the
// lines it wants first are the ones the first pass evicted first.  For a
// larger X, marking a share of it only crowded the cast pass's own traffic
// out of L2, so X is then loaded plainly.
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint4 ldg_v4_policy(const void* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

__global__ void __launch_bounds__(kThreads)
amax_partials_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
                     uint32_t* __restrict__ partials, bool keep) {
    const uint64_t pol = l2_policy_evict_last();
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
            v[j] = (c < cols) ? (keep ? ldg_v4_policy(x + r * ldx + c, pol) : ldg_v4(x + r * ldx + c))
                              : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) m = max(m, absmax_v4(v[j]));
    }
    m = block_max_u32(m);
    if (threadIdx.x == 0) partials[blockIdx.x] = m;
}

// ---------------------------------------------------------------- row sources
// Where a row-wise quantiser's row r comes from: row r of x (plain); row
// idx[r] of x (the MoE gather, rows in expert order); or the SwiGLU of row r
// of the gate+up output, y = BF16(silu(gate) * up) with gate at columns
// 0.. and up at columns `up`.. of that row.
enum { kSrcPlain = 0, kSrcGather = 1, kSrcSwiglu = 2 };
struct RowSrc {
    const int64_t* idx;   // gather: source token of each row
    int64_t tokens;       // gather: rows of x
    int64_t up;           // SwiGLU: column where up starts
    int* status;          // gather: sticky status word for an index out of range
    bool keep_x;          // gather: load x with an L2 evict-last policy (x fits in L2)
};

// Float32 pair arithmetic, each half rounded on its own (round to nearest).
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fsub2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ void unpair(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t splat2(float c) { return pair_f32(c, c); }

// e^x of two elements in float32, two elements per instruction where the
// operation allows: Cody and Waite's reduction x = n ln2 + r ("Software
// Manual for the Elementary Functions", 1980) with ln 2 split into a 16-bit
// head and a tail, the Taylor series of e^r to r^7 in Horner form, and the
// scaling by 2^(n-1) * 2.  The compiler may fuse a pair multiplication with
// the pair addition that follows it (it does so for mul/sub.rn.f32x2), which
// only removes a rounding; the SwiGLU contract allows for a few float32 ulps.  +inf above 89, 0 below -87 (where 1 + e^x is 1 in
// float32 already).  Within 2 float32 ulps of e^x.  The sequence runs on x
// clamped to [-87, 89] (which keeps n in [-126, 128]); the out-of-range
// results are selected at the end, with no branch per element.
__device__ __forceinline__ uint64_t exp_seq2(float x0, float x1) {
    const uint64_t xc = pair_f32(fminf(fmaxf(x0, -0x1.5cp+6f), 0x1.64p+6f), fminf(fmaxf(x1, -0x1.5cp+6f), 0x1.64p+6f));
    float t0, t1;
    unpair(fmul2(xc, splat2(0x1.715476p+0f)), t0, t1);
    const float n0 = rintf(t0), n1 = rintf(t1);
    const uint64_t n = pair_f32(n0, n1);
    const uint64_t r = fsub2(fsub2(xc, fmul2(n, splat2(0x1.62e4p-1f))), fmul2(n, splat2(0x1.7f7d1cp-20f)));
    uint64_t p = splat2(0x1.a01a02p-13f);
    p = fadd2(fmul2(p, r), splat2(0x1.6c16c2p-10f));
    p = fadd2(fmul2(p, r), splat2(0x1.111112p-7f));
    p = fadd2(fmul2(p, r), splat2(0x1.555556p-5f));
    p = fadd2(fmul2(p, r), splat2(0x1.555556p-3f));
    p = fadd2(fmul2(p, r), splat2(0.5f));
    p = fadd2(fmul2(p, r), splat2(1.0f));
    p = fadd2(fmul2(p, r), splat2(1.0f));
    const int ni0 = (int)n0 - 1, ni1 = (int)n1 - 1;
    const float h0 = ni0 >= -126 ? __int_as_float((ni0 + 127) << 23) : __int_as_float(0x00400000);
    const float h1 = ni1 >= -126 ? __int_as_float((ni1 + 127) << 23) : __int_as_float(0x00400000);
    float e0, e1;
    unpair(fmul2(fmul2(p, pair_f32(h0, h1)), splat2(2.0f)), e0, e1);
    e0 = x0 > 0x1.64p+6f ? __int_as_float(0x7F800000) : e0;
    e0 = x0 < -0x1.5cp+6f ? 0.0f : e0;
    e1 = x1 > 0x1.64p+6f ? __int_as_float(0x7F800000) : e1;
    e1 = x1 < -0x1.5cp+6f ? 0.0f : e1;
    return pair_f32(e0, e1);
}

// Round a float64 value once to nearest-even BF16 (bits).  The value is
// scaled by a power of two so that its BF16 quantum becomes 1 (2^-133 below
// the normal range), rounded to an integer, and scaled back: every step but
// the rounding is exact.
__device__ __forceinline__ uint32_t bf16_bits_rne_f64(double v) {
    int e = 0;
    (void)frexp(v, &e);
    const int qe = max(e - 8, -133);
    const float f = (float)ldexp(rint(ldexp(v, -qe)), qe);   // a BF16 value, or +-inf past the largest
    return __float_as_uint(f) >> 16;
}

// Eight SwiGLU outputs as BF16: silu(g) = g / (1 + e^-g), times up, in
// float32 on element pairs (a few float32 ulps from the exact value before
// the BF16 rounding).  The quotient g / d, d = 1 + e^-g in [1, e^80 + 1],
// takes the correction step of div_fast with r from the hardware's
// approximate reciprocal refined by Newton steps (rcp_newton): within about
// one float32 ulp of the IEEE quotient, at a quarter of its instructions.
// As in neg_quotient2, the pair steps run negated: q' = -g/d, and the
// product with -up gives y.
__device__ __forceinline__ uint4 swiglu8_f32(const float* g, const uint4& uv) {
    float u[8], y[8];
    unpack8(uv, u);
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
        float d0, d1;
        const uint64_t d2 = fadd2(splat2(1.0f), exp_seq2(-g[i], -g[i + 1]));
        unpair(d2, d0, d1);
        const uint64_t n2 = pair_f32(-rcp_newton(d0), -rcp_newton(d1));
        const uint64_t g2 = pair_f32(g[i], g[i + 1]);
        uint64_t yq, t, q;
        asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(yq) : "l"(g2), "l"(n2));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(t) : "l"(yq), "l"(d2), "l"(g2));
        asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(q) : "l"(t), "l"(n2), "l"(yq));
        unpair(fmul2(q, pair_f32(-u[i], -u[i + 1])), y[i], y[i + 1]);
    }
    uint4 o;
    uint32_t* ow = &o.x;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 b = __floats2bfloat162_rn(y[2 * i], y[2 * i + 1]);
        ow[i] = *reinterpret_cast<uint32_t*>(&b);
    }
    return o;
}

// The eight outputs when some gate is below -80: the float32 form for the
// others, the float64 form for those (a separate function, so that the
// common path keeps its registers).
__device__ __noinline__ uint4 swiglu8_with_far_negative(uint4 gv, uint4 uv) {
    float g[8], u[8];
    unpack8(gv, g);
    unpack8(uv, u);
    uint4 o = swiglu8_f32(g, uv);
    uint32_t* ow = &o.x;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (g[i] < -80.0f) {
            const uint32_t b = bf16_bits_rne_f64((double)g[i] * exp((double)g[i]) * (double)u[i]);
            ow[i >> 1] = (i & 1) ? ((ow[i >> 1] & 0xFFFFu) | (b << 16)) : ((ow[i >> 1] & 0xFFFF0000u) | b);
        }
    }
    return o;
}

// SwiGLU of eight elements.  Gates below -80 never occur in activations of
// ordinary size; for them e^-g is at or beyond the float32 range (it
// overflows above 88.7), while y = silu(g) * up = g e^g up / (1 + e^g) can
// still be a small normal or subnormal BF16 number.  1 + e^g equals 1 there
// to far below float64 precision, so such an element is evaluated as
// g e^g up in float64 and rounded once.
__device__ __forceinline__ uint4 swiglu8(const uint4& gv, const uint4& uv) {
    float g[8];
    unpack8(gv, g);
    bool far = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) far |= g[i] < -80.0f;
    if (far) return swiglu8_with_far_negative(gv, uv);
    return swiglu8_f32(g, uv);
}

// ---------------------------------------------------------------- row-wise 1x128 / 1x32 / per-tensor
// Plain and SwiGLU rows are held to 64 registers, four CTAs (32 warps) per
// SM: the 1x128 form measured 26.6 -> 23.5 us on [8192, 4096] against its
// unconstrained 66 registers (three CTAs), with the same codes; the MXFP8 and
// per-tensor forms did not move, and five or more CTAs per SM were slower.
// The SwiGLU source's rare float64 path would otherwise raise its count too.
// The gathered source keeps its own count (capped, its MXFP8 form spills).
template <int GRAN, int SRC = kSrcPlain>
__global__ void __launch_bounds__(kThreads, SRC == kSrcGather ? 1 : 4)
quant_rows_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
                  uint8_t* __restrict__ q, void* __restrict__ sout,
                  const uint32_t* __restrict__ partials, int nparts, const float* __restrict__ given,
                  RowSrc src = RowSrc{}) {
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
    const ScaleDiv sd_uniform = scale_div(s_uniform, given == nullptr);
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t segs = ceil_div(cols, kSeg);
    const int64_t total = rows * segs;
    const int64_t ng = ceil_div(cols, GRAN == kGranMx ? 32 : 128);
    TaskCursor tc(gw, nw, segs);
    int64_t tok_next = 0;     // gather: the next task's token, loaded one task ahead
    if constexpr (SRC == kSrcGather) {
        if (gw < total) tok_next = __ldg(src.idx + tc.r);
    }
    for (int64_t t = gw; t < total; t += nw, tc.advance()) {
        const int64_t r = tc.r;
        const int64_t cb = tc.si * kSeg;
        const uint16_t* xr = x + r * ldx;
        bool valid = true;
        if constexpr (SRC == kSrcGather) {
            const int64_t tok = tok_next;
            if (t + nw < total) tok_next = __ldg(src.idx + tc.next_row());
            valid = tok >= 0 && tok < src.tokens;
            xr = x + (valid ? tok : 0) * ldx;
            if (!valid && lane == 0 && cb == 0 && src.status != nullptr) atomicExch(src.status, kStatusIndex);
        }
        uint4 v[4];
        uint4 uv[SRC == kSrcSwiglu ? 4 : 1];   // SwiGLU: v holds gate, uv up, until group j is formed
        if constexpr (SRC == kSrcSwiglu) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t c = cb + j * 256 + lane * 8;
                v[j] = (c < cols) ? ldg_v4(xr + c) : make_uint4(0, 0, 0, 0);
                uv[j] = (c < cols) ? ldg_v4(xr + src.up + c) : make_uint4(0, 0, 0, 0);
            }
        } else if (SRC == kSrcGather && src.keep_x) {
            // Each token is gathered once per expert it is routed to, rows
            // apart; the evict-last mark keeps x in L2 between those copies
            // while the codes stream out.
            const uint64_t pol = l2_policy_evict_last();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t c = cb + j * 256 + lane * 8;
                v[j] = (c < cols && valid) ? ldg_v4_policy(xr + c, pol) : make_uint4(0, 0, 0, 0);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int64_t c = cb + j * 256 + lane * 8;
                v[j] = (c < cols && valid) ? ldg_v4(xr + c) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t c = cb + j * 256 + lane * 8;
            const bool ok = c < cols;
            if constexpr (SRC == kSrcSwiglu) {
                if (ok) v[j] = swiglu8(v[j], uv[j]);
            }
            float f[8];
            unpack8(v[j], f);
            uint2 o;
            if constexpr (GRAN == kGranTok) {
                const uint32_t m = warp_max_u32(absmax_v4(v[j]), 16);
                const ScaleDiv sd = scale_div_from_amax(amax_bits_to_f32(m));
                o = cast8_div(f, sd);
                if (ok && (lane & 15) == 0) static_cast<float*>(sout)[r * ng + (c >> 7)] = sd.s;
            } else if constexpr (GRAN == kGranMx) {
                const uint32_t m = warp_max_u32(SRC == kSrcPlain ? absmax_v4_pairs(v[j]) : absmax_v4(v[j]), 4);
                const int e = mx_exponent_from_amax_bits(m << 16);
                o = cast8_mul(f, exp2_neg(e));
                if (ok && (lane & 3) == 0) static_cast<uint8_t*>(sout)[r * ng + (c >> 5)] = (uint8_t)(e + 127);
            } else if constexpr (GRAN == kGranTokP2) {
                const uint32_t m = warp_max_u32(absmax_v4(v[j]), 16);
                const int e = mx_exponent_from_amax_bits(m << 16);
                o = cast8_mul(f, exp2_neg(e));
                if (ok && (lane & 15) == 0) static_cast<uint8_t*>(sout)[r * ng + (c >> 7)] = (uint8_t)(e + 127);
            } else {
                o = cast8_div(f, sd_uniform);
            }
            if (ok) {
                if constexpr (SRC == kSrcGather)
                    stg_cs_v2(q + r * cols + c, o);
                else
                    *reinterpret_cast<uint2*>(q + r * cols + c) = o;
            }
        }
    }
}

// ---------------------------------------------------------------- NVFP4 1x16 (row-wise)
// "4. NVFP4 (Blackwell)": E2M1 codes in 1x16 blocks, an E4M3 block scale
// s_b = E4M3((amax_b / 6) / S_g) and an outer float32 S_g (per tensor, or per
// row for per-token activation scaling).  A lane owns whole blocks (two
// 16-byte loads each), so a block's scale is computed once, with no
// shuffle.
//
// Four-over-six ("Advanced: four-over-six"): each block is also quantised
// with its amax mapped to 4 (s_b from amax_b / 4) and keeps that result only
// when its squared error is strictly smaller.  The error of each half block
// (8 elements) is summed in order in float32 (no fused multiply-add), and
// the two half sums are then added.  S_g is amax / (256 * 6) in that mode.

// tab[c] = RN(1/S_b) for S_b = RN(E4M3value(c) * S_g), c = 0..127 (entries
// for c = 0 and the NaN code 127 are never read), written by `n` threads
// starting at thread `t`: the reciprocal each block would otherwise take,
// computed once per outer scale.
__device__ __forceinline__ void nvfp4_fill_rcp(float* tab, float s_g, int t, int n) {
    for (int c = t; c < 128; c += n) tab[c] = __frcp_rn(__fmul_rn(e4m3_value((uint32_t)c), s_g));
}

// E2M1(x / S_b) for 8 elements.  S_b = E4M3value(s_b) * S_g: with S_g from
// the tensor (or row) amax the quotient is the reciprocal-and-correction one
// (div_fast, the test hoisted out of the loop); every E2M1 code on that
// domain matches the IEEE quotient's, checked by enumeration
// (fp8bs_test_quotient_sweep with nvfp4 = 1).  A supplied S_g divides exactly.
// r is RN(1/S_b), read from the kernel's table of the 127 possible S_b of
// its S_g (nvfp4_fill_rcp) instead of one reciprocal per block and lane.
__device__ __forceinline__ uint32_t e2m1_quant8(const float* f, float big_s, float r, bool from_amax) {
    if (big_s == 0.0f) return 0u;
    ScaleDiv d;
    d.s = big_s;
    d.fast = from_amax && big_s >= kFastDivMinScale;
    d.r = r;
    if (d.fast) return e2m1x8_div_fast2(f, scale_div2(d));
    float t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) t[i] = __fdiv_rn(f[i], big_s);
    return e2m1x8(t);
}

// sum_i (x_i - E2M1(q_i) * S_b)^2 over this lane's 8 elements, in order.
// Scalar on purpose: written with mul.rn.f32x2 and sub.rn.f32x2 on element
// pairs, the difference came out as one fused multiply-add (x - e S rounded
// once), which changed 2627 code bytes of a [8192, 4096] four-over-six
// quantisation; the scalar intrinsics keep the product rounded on its own.
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

// The block scale code E4M3(RN(RN(a / 6) / S_g)) of a block amax a (a
// BF16 value), and with four = true the four-over-six alternative
// E4M3(RN(RN(a / 4) / S_g)).  On the fast path (S_g derived from a tensor
// or row amax, S_g >= 2^-88) both divisions take the correction step of
// div_fast: RN(a / 6) with r = RN(1/6), which equals the IEEE quotient for
// every BF16 a; RN(a / 4) is the exact product a * 0.25; the division by
// S_g with dg's reciprocal, whose E4M3 code equals that of the IEEE
// quotient for every BF16 amax_T and every BF16 a <= amax_T, for both outer
// divisors.  Both facts were checked by enumeration on the device
// (fp8bs_test_quotient_sweep with mode 2).  Otherwise: IEEE division.
constexpr float kRecip6 = 0x1.555556p-3f;   // RN(1/6)

__device__ __forceinline__ float div6_fast(float a) {
    const float y = __fmul_rn(a, kRecip6);
    const float e = __fmaf_rn(-y, kE2M1Max, a);
    return __fmaf_rn(e, kRecip6, y);
}

__device__ __forceinline__ uint32_t nvfp4_block_code(float amax_b, float s_g, const ScaleDiv& dg, bool four) {
    if (dg.fast) return e4m3_byte(div_fast(four ? __fmul_rn(amax_b, 0.25f) : div6_fast(amax_b), dg));
    return e4m3_byte(__fdiv_rn(__fdiv_rn(amax_b, four ? 4.0f : kE2M1Max), s_g));
}

// One lane's whole block of 16 elements (v0: elements 0..7, v1: 8..15):
// packed E2M1 codes (element i in bits 4i..4i+3 of the 64-bit result) and
// the block's scale byte.  With four-over-six the squared error of each half
// of the block is summed in element order and the two halves are then added.
template <bool FOS>
__device__ __forceinline__ void nvfp4_block(const uint4& v0, const uint4& v1, float s_g, const ScaleDiv& dg,
                                            const float* rcp, bool from_amax, uint2& packed, uint32_t& code) {
    const float amax_b = amax_bits_to_f32(max(absmax_v4(v0), absmax_v4(v1)));
    float f[16];
    unpack8(v0, f);
    unpack8(v1, f + 8);
    code = nvfp4_block_code(amax_b, s_g, dg, false);
    const float s6 = __fmul_rn(e4m3_value(code), s_g), r6 = rcp[code];
    packed = make_uint2(e2m1_quant8(f, s6, r6, from_amax), e2m1_quant8(f + 8, s6, r6, from_amax));
    if constexpr (FOS) {
        const uint32_t code4 = nvfp4_block_code(amax_b, s_g, dg, true);
        const float s4 = __fmul_rn(e4m3_value(code4), s_g), r4 = rcp[code4];
        const uint2 p4 = make_uint2(e2m1_quant8(f, s4, r4, from_amax), e2m1_quant8(f + 8, s4, r4, from_amax));
        const float e6 = __fadd_rn(half_sq_err(f, packed.x, s6), half_sq_err(f + 8, packed.y, s6));
        const float e4 = __fadd_rn(half_sq_err(f, p4.x, s4), half_sq_err(f + 8, p4.y, s4));
        if (e4 < e6) {
            packed = p4;
            code = code4;
        }
    }
}

// 16 bytes of BF16 through L1 (the lane's block is one 32-byte sector read
// by two such loads: the second finds it in L1).
__device__ __forceinline__ uint4 ldg_v4_l1(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Quantise columns [cb, cb + 1024) of row r with outer scale s_g: lane l owns
// the blocks at columns cb + 16 l and cb + 512 + 16 l (cols % 16 == 0, so a
// block lies wholly inside the row or wholly past its end).
template <bool FOS>
__device__ __forceinline__ void nvfp4_segment(const uint16_t* __restrict__ x, int64_t r, int64_t cb, int64_t cols,
                                              int64_t ldx, uint8_t* __restrict__ q, uint8_t* __restrict__ sb,
                                              float s_g, const ScaleDiv& dg, const float* rcp, bool from_amax,
                                              int lane) {
    const int64_t nb = cols >> 4;
    const uint16_t* xr = x + r * ldx;
    uint4 v[4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int64_t c = cb + 512 * h + 16 * lane;
        const bool in = c < cols;
        v[2 * h] = in ? ldg_v4_l1(xr + c) : make_uint4(0, 0, 0, 0);
        v[2 * h + 1] = in ? ldg_v4_l1(xr + c + 8) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int64_t c = cb + 512 * h + 16 * lane;
        uint2 packed;
        uint32_t code;
        nvfp4_block<FOS>(v[2 * h], v[2 * h + 1], s_g, dg, rcp, from_amax, packed, code);
        if (c < cols) {
            *reinterpret_cast<uint2*>(q + r * (cols >> 1) + (c >> 1)) = packed;
            sb[r * nb + (c >> 4)] = (uint8_t)code;
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
    TaskCursor tc(gw, nw, segs);
    const ScaleDiv dg = scale_div(s_g, !given);
    __shared__ float rcp[128];
    nvfp4_fill_rcp(rcp, s_g, threadIdx.x, blockDim.x);
    __syncthreads();
    for (int64_t t = gw; t < total; t += nw, tc.advance())
        nvfp4_segment<FOS>(x, tc.r, tc.si * kSeg, cols, ldx, q, sb, s_g, dg, rcp, !given, lane);
}

// One outer scale per row (per token): a warp owns a row, reads it once for
// its amax and again (from L2) to quantise it.
template <bool FOS>
__global__ void __launch_bounds__(kThreads)
quant_nvfp4_row_kernel(const uint16_t* __restrict__ x, int64_t rows, int64_t cols, int64_t ldx,
                       uint8_t* __restrict__ q, uint8_t* __restrict__ sb, float* __restrict__ row_scale, bool given) {
    __shared__ float rcp_rows[kThreads / 32][128];   // per warp: RN(1/S_b) of its row's S_g
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
        const ScaleDiv dg = scale_div(s_g, !given);
        float* rcp = rcp_rows[threadIdx.x >> 5];
        __syncwarp();                       // the previous row's table is no longer read
        nvfp4_fill_rcp(rcp, s_g, lane, 32);
        __syncwarp();
        for (int64_t cb = 0; cb < cols; cb += kSeg)
            nvfp4_segment<FOS>(x, r, cb, cols, ldx, q, sb, s_g, dg, rcp, !given, lane);
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
            *reinterpret_cast<uint2*>(q + r * cols + c) = P2 ? cast8_mul(f, sc) : cast8_div(f, scale_div(sc, true));
        }
    }
}

// ---------------------------------------------------------------- transposed (+ optional row-wise), TMA-fed
// 1x128, 1x128 with power-of-two scales, and MXFP8: a scale per column of X
// (per row of X^T) and, in dual mode, another per row of X.  Per-tensor,
// 128x128 and 128x128 with power-of-two scales: one scale covers the whole
// 128x128 tile, so the codes of X and of X^T are the same bytes; each thread
// casts its block once (by rows) and transposes the 8 x 8 bytes in registers.
// Persistent CTAs of 256 threads, three per SM (two for the dual
// power-of-two forms, kTileCtas).  A 2-stage ring of 128x128
// BF16 tiles (32 KB each) per CTA is filled by TMA ahead of the compute, so
// the load of the next tile is in flight while a tile is quantised.
// Thread t holds an 8 x 8 block of the tile in registers, read as eight
// 16-byte shared-memory loads: columns 8*(t%16) .. +7 of rows 8*(t/16) ..
// +7, so a warp holds 16 whole rows and a half-warp 8.  From the registers:
//   column pass (codes of X^T): column maxima over the thread's 8 rows,
//     over the warp's 16 by one shuffle, then over the tile's 128 rows
//     (1x128: the eight warps' maxima meet in shared memory and each
//     column's scale is computed once) or over a 32-row group (MXFP8: two
//     warps).  Codes of two rows of a column per float32-pair instruction;
//     a column's 8 codes go into the consumed stage as 8 bytes of a
//     [column][row] byte tile (16-byte chunks XOR-swizzled by column/8, so
//     a warp's stores spread over all banks) and leave as whole 128-byte
//     rows of X^T.
//   row pass (row-wise codes of X, dual mode): a row's 128 columns lie in
//     the 16 lanes of a half-warp.  A transposing butterfly of shuffles
//     leaves each lane pair with the maximum of one of the half-warp's 8
//     rows (1x128), or each lane with two rows of its 32-column group
//     (MXFP8); the scales come back through shared memory (1x128) or
//     shuffles (MXFP8).  Codes of two adjacent columns per float32-pair
//     instruction; a half-warp stores whole 128-byte row segments.
// Every thread fences its generic accesses to a stage at the end of the
// tile; the stage is refilled once every thread has passed the barrier that
// opens the next tile.
constexpr int kTileThreads = 256;
constexpr int kTileStages = 2;
// CTAs per SM: three, except for the dual power-of-two forms (MXFP8, 1x128
// power of two), which spill at three CTAs' register share (80) and run
// faster at two (MXFP8 dual [8192, 4096]: 32.8 against 30.7 us).
template <int GRAN, bool DUAL> constexpr int kTileCtas = (kPow2<GRAN> && DUAL) ? 2 : 3;
constexpr uint32_t kTileBytes = 128 * 128 * 2;

struct TileShared {
    uint32_t tile[kTileStages][128 * 64];   // BF16 pairs, row pitch 64 words
    uint4 red[8][16];          // per warp and 8-column group: |x| maxima (BF16 bit pairs) over the warp's 16 rows
    float2 csr[128];           // per column of the tile: S (or 2^-e) and RN(1/S), 0 off the fast path
    float2 rsr[8][16];         // per warp and row (1x128 rows, dual): the same
    uint32_t tmax[8];          // one scale per tile: each warp's |x| maximum (BF16 bits)
    uint64_t full[kTileStages];
};
constexpr size_t kTileSmem = sizeof(TileShared) + 1024;


__device__ __forceinline__ bool tile_wait(uint32_t bar, uint32_t parity, int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0 && globaltimer() - t0 > kWaitLimitNs) {
            if (status != nullptr) atomicExch(status, kStatusTimeout);
            return false;
        }
    }
}

// 4 x 4 byte transpose: a_k holds bytes (k, 0..3), c_j receives bytes (0..3, j).
__device__ __forceinline__ void transpose4x4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t& c0,
                                             uint32_t& c1, uint32_t& c2, uint32_t& c3) {
    const uint32_t t0 = __byte_perm(a0, a1, 0x5140), t1 = __byte_perm(a0, a1, 0x7362);   // (0,0) (1,0) (0,1) (1,1); (0,2) ..
    const uint32_t t2 = __byte_perm(a2, a3, 0x5140), t3 = __byte_perm(a2, a3, 0x7362);
    c0 = __byte_perm(t0, t2, 0x5410);
    c1 = __byte_perm(t0, t2, 0x7632);
    c2 = __byte_perm(t1, t3, 0x5410);
    c3 = __byte_perm(t1, t3, 0x7632);
}

// Eight E4M3 codes of two float32 pairs each of two values: x / S by the
// correction step (FP32 scale S, r = RN(1/S)) or x * m (power of two, m in s).
template <bool P2>
__device__ __forceinline__ uint2 codes8_fast(uint64_t x01, uint64_t x23, uint64_t x45, uint64_t x67, float s, float r) {
    if constexpr (P2) {
        const uint64_t m2 = pair_f32(s, s);
        return make_uint2(e4m3x4_mul2(x01, x23, m2), e4m3x4_mul2(x45, x67, m2));
    } else {
        const ScaleDiv2 d = scale_div2(ScaleDiv{s, r, true});
        return make_uint2(e4m3x4_div_fast2(x01, x23, d), e4m3x4_div_fast2(x45, x67, d));
    }
}

// The same eight codes of x / S for a group off the fast path (r = 0: IEEE
// division; an all-zero or tiny group), out of line: such groups are rare.
__device__ __noinline__ uint2 codes8_slow(uint64_t x01, uint64_t x23, uint64_t x45, uint64_t x67, float s, float r) {
    const ScaleDiv d{s, r, r != 0.0f};
    float f[8];
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f[0]), "=f"(f[1]) : "l"(x01));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f[2]), "=f"(f[3]) : "l"(x23));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f[4]), "=f"(f[5]) : "l"(x45));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f[6]), "=f"(f[7]) : "l"(x67));
    return make_uint2(e4m3x4(div_scale(f[0], d), div_scale(f[1], d), div_scale(f[2], d), div_scale(f[3], d)),
                      e4m3x4(div_scale(f[4], d), div_scale(f[5], d), div_scale(f[6], d), div_scale(f[7], d)));
}

template <int GRAN, bool DUAL>
__global__ void __launch_bounds__(kTileThreads, kTileCtas<GRAN, DUAL>)
quant_tile_tma_kernel(const __grid_constant__ CUtensorMap tm_x, int64_t rows, int64_t cols,
                      uint8_t* __restrict__ qt, void* __restrict__ st,
                      uint8_t* __restrict__ q, void* __restrict__ s, int* status,
                      const uint32_t* __restrict__ partials, int nparts, const float* __restrict__ given) {
    constexpr bool kOne = GRAN == kGranPT || GRAN == kGranBlk || GRAN == kGranBlkP2;   // one scale per tile
    static_assert(kOne || GRAN == kGranTok || GRAN == kGranTokP2 || GRAN == kGranMx, "transposed granularities");
    constexpr bool kMxG = GRAN == kGranMx;
    constexpr bool kP2 = kPow2<GRAN>;     // MXFP8 and 1x128 power of two: codes by multiplication
    constexpr uint32_t kFull = 0xFFFFFFFFu;
    extern __shared__ uint8_t tile_smem_raw[];
    TileShared& sh = *reinterpret_cast<TileShared*>((reinterpret_cast<uintptr_t>(tile_smem_raw) + 1023) &
                                                    ~uintptr_t(1023));
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int cg = lane & 15, half = lane >> 4, rg = 2 * w + half;   // the thread's 8-column and 8-row groups
    // rows < 2^23 (at most 65535 row tiles); column tiles < 2^31
    const int tiles_c = (int)ceil_div(cols, 128), tiles_r = (int)ceil_div(rows, 128);
    const int nrows = (int)rows;
    const int64_t ntiles = (int64_t)tiles_c * tiles_r;
    // The CTA's tiles are t = blockIdx.x + i * gridDim.x, walked as (row tile,
    // column tile) cursors: one for the loads (thread 0), one for the compute.
    const int step_r = (int)(gridDim.x / (unsigned)tiles_c), step_c = (int)(gridDim.x % (unsigned)tiles_c);
    auto advance = [&](int& rt_, int& ct_) {
        ct_ += step_c;
        rt_ += step_r;
        if (ct_ >= tiles_c) {
            ct_ -= tiles_c;
            ++rt_;
        }
    };
    int rt = (int)(blockIdx.x / (unsigned)tiles_c), ct = (int)(blockIdx.x % (unsigned)tiles_c);
    int lrt = rt, lct = ct;

    if (tid == 0) {
        for (int k = 0; k < kTileStages; ++k) mbar_init(smem_u32(&sh.full[k]), 1);
        fence_barrier_init();
        tma_prefetch_desc(&tm_x);
    }
    __syncthreads();
    int64_t issued = 0;     // tiles whose load thread 0 has issued
    auto issue = [&](int64_t i) {  // the next tile of this CTA into stage i % kTileStages
        const uint32_t bar = smem_u32(&sh.full[i % kTileStages]);
        mbar_arrive_expect_tx(bar, kTileBytes);
        tma_load_2d(smem_u32(sh.tile[i % kTileStages]), &tm_x, bar, lct * 128, lrt * 128);
        advance(lrt, lct);
    };
    const int64_t mine = (ntiles > blockIdx.x) ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    if (tid == 0) {
        for (; issued < mine && issued < kTileStages; ++issued) issue(issued);
    }

    // Per-tensor: S from the amax partials (written out by one thread), or
    // supplied (then divided by exactly, IEEE).
    float pt_s = 1.0f, pt_r = 0.0f;
    if constexpr (GRAN == kGranPT) {
        ScaleDiv sd;
        if (given != nullptr) {
            sd = scale_div(*given, false);
        } else {
            sd = scale_div(fp32_scale_from_amax(tensor_amax(partials, nparts)), true);
            if (blockIdx.x == 0 && tid == 0) {
                static_cast<float*>(st)[0] = sd.s;
                if constexpr (DUAL) static_cast<float*>(s)[0] = sd.s;
            }
        }
        pt_s = sd.s;
        pt_r = sd.fast ? sd.r : 0.0f;
    }

    int64_t consumed = 0;   // tiles whose load has been waited for
    for (int64_t i = 0; i < mine; ++i) {
        const int stg = (int)(i % kTileStages);
        const bool got = tile_wait(smem_u32(&sh.full[stg]), (uint32_t)((i / kTileStages) & 1), status);
        if (!__syncthreads_and(got)) break;
        consumed = i + 1;
        // every thread is done with the previous tile's stage: refill it
        if (tid == 0 && i > 0 && issued < mine) {
            issue(issued);
            ++issued;
        }
        const int r0 = rt * 128, rbase = r0 + 8 * rg;                           // the thread's first row
        const int64_t c0 = (int64_t)ct * 128, cbase = c0 + 8 * cg;             // and first column
        uint32_t* tile = sh.tile[stg];

        // ---------------- the thread's 8 x 8 block: x[k][j] = columns 2j, 2j+1 of row k
        uint32_t x[8][4];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint4 v = *reinterpret_cast<const uint4*>(tile + (8 * rg + k) * 64 + 4 * cg);
            x[k][0] = v.x;
            x[k][1] = v.y;
            x[k][2] = v.z;
            x[k][3] = v.w;
        }
        uint8_t* ct8 = reinterpret_cast<uint8_t*>(tile);   // the consumed stage, later the [column][row] byte tile
        const int sw = cg & 7;   // its 16-byte chunk swizzle: (column / 8) % 8, the same for the thread's 8 columns
        if constexpr (kOne) {
            // ---------------- one scale for the tile: the codes of X and of X^T are the same bytes
            float sv = pt_s, rv = pt_r;
            if constexpr (GRAN != kGranPT) {
                uint32_t m2 = 0;
#pragma unroll
                for (int k = 0; k < 8; ++k)
#pragma unroll
                    for (int j = 0; j < 4; ++j) m2 = __vmaxu2(m2, x[k][j] & 0x7FFF7FFFu);
                const uint32_t m = warp_max_u32(max(m2 & 0xFFFFu, m2 >> 16), 32);
                if (lane == 0) sh.tmax[w] = m;
            }
            __syncthreads();   // every thread holds its block (the stage's BF16 data is dead); tmax is complete
            if constexpr (GRAN != kGranPT) {
                const uint4 t0 = *reinterpret_cast<const uint4*>(&sh.tmax[0]);
                const uint4 t1 = *reinterpret_cast<const uint4*>(&sh.tmax[4]);
                const uint32_t m = max(max(max(t0.x, t0.y), max(t0.z, t0.w)), max(max(t1.x, t1.y), max(t1.z, t1.w)));
                if constexpr (GRAN == kGranBlk) {
                    const ScaleDiv sd = scale_div_from_amax(amax_bits_to_f32(m));
                    sv = sd.s;
                    rv = sd.fast ? sd.r : 0.0f;
                    if (tid == 0) {
                        static_cast<float*>(st)[(int64_t)ct * tiles_r + rt] = sv;
                        if constexpr (DUAL) static_cast<float*>(s)[(int64_t)rt * tiles_c + ct] = sv;
                    }
                } else {
                    const int e = mx_exponent_from_amax_bits(m << 16);
                    sv = exp2_neg(e);
                    if (tid == 0) {
                        static_cast<uint8_t*>(st)[(int64_t)ct * tiles_r + rt] = (uint8_t)(e + 127);
                        if constexpr (DUAL) static_cast<uint8_t*>(s)[(int64_t)rt * tiles_c + ct] = (uint8_t)(e + 127);
                    }
                }
            }
            // codes of the thread's 8 rows (bytes 0..7 = its 8 columns)
            uint2 rc[8];
            auto rows_cast = [&](auto fast) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t p0 = pair_bf16(x[k][0]), p1 = pair_bf16(x[k][1]);
                    const uint64_t p2 = pair_bf16(x[k][2]), p3 = pair_bf16(x[k][3]);
                    if constexpr (kP2 || decltype(fast)::value) rc[k] = codes8_fast<kP2>(p0, p1, p2, p3, sv, rv);
                    else rc[k] = codes8_slow(p0, p1, p2, p3, sv, rv);
                }
            };
            if (kP2 || rv != 0.0f) rows_cast(std::true_type{});
            else rows_cast(std::false_type{});
            if constexpr (DUAL) {
                if (cbase < cols) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        if (rbase + k < nrows) *reinterpret_cast<uint2*>(q + (int64_t)(rbase + k) * cols + cbase) = rc[k];
                }
            }
            // the same bytes as 8 columns of 8 rows: an 8 x 8 byte transpose in four 4 x 4 blocks
            uint32_t cl[8], chh[8];   // column j: rows 0..3, rows 4..7
            transpose4x4(rc[0].x, rc[1].x, rc[2].x, rc[3].x, cl[0], cl[1], cl[2], cl[3]);
            transpose4x4(rc[4].x, rc[5].x, rc[6].x, rc[7].x, chh[0], chh[1], chh[2], chh[3]);
            transpose4x4(rc[0].y, rc[1].y, rc[2].y, rc[3].y, cl[4], cl[5], cl[6], cl[7]);
            transpose4x4(rc[4].y, rc[5].y, rc[6].y, rc[7].y, chh[4], chh[5], chh[6], chh[7]);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<uint2*>(ct8 + (8 * cg + j) * 128 + 16 * (w ^ sw) + 8 * half) = make_uint2(cl[j], chh[j]);
        } else {
        // |x| maxima as BF16 bit pairs (non-negative patterns order like their
        // values): per column pair over the 8 rows, per row over the 8 columns
        uint32_t cm[4] = {0u, 0u, 0u, 0u}, rm[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t a0 = x[k][0] & 0x7FFF7FFFu, a1 = x[k][1] & 0x7FFF7FFFu;
            const uint32_t a2 = x[k][2] & 0x7FFF7FFFu, a3 = x[k][3] & 0x7FFF7FFFu;
            cm[0] = __vmaxu2(cm[0], a0);
            cm[1] = __vmaxu2(cm[1], a1);
            cm[2] = __vmaxu2(cm[2], a2);
            cm[3] = __vmaxu2(cm[3], a3);
            rm[k] = __vmaxu2(__vmaxu2(a0, a1), __vmaxu2(a2, a3));
        }
        // column maxima over the warp's 16 rows (both halves end with them)
#pragma unroll
        for (int j = 0; j < 4; ++j) cm[j] = __vmaxu2(cm[j], __shfl_xor_sync(kFull, cm[j], 16));
        if (half == 0) sh.red[w][cg] = make_uint4(cm[0], cm[1], cm[2], cm[3]);

        // ---------------- row pass: row-wise codes of X
        if constexpr (DUAL) {
            // row k's 8 values as float32 pairs (columns 2j, 2j+1)
            auto row_codes = [&](int k, float sv, float rv, bool fast) -> uint2 {
                if (kP2 || fast) return codes8_fast<kP2>(pair_bf16(x[k][0]), pair_bf16(x[k][1]), pair_bf16(x[k][2]),
                                                          pair_bf16(x[k][3]), sv, rv);
                return codes8_slow(pair_bf16(x[k][0]), pair_bf16(x[k][1]), pair_bf16(x[k][2]), pair_bf16(x[k][3]), sv, rv);
            };
            const bool cols_in = cbase < cols;
            if constexpr (!kMxG) {
                // Transposing butterfly over the half-warp: each step halves the
                // rows a lane keeps and doubles the lanes they are reduced over.
                // At the end lanes 2p and 2p + 1 hold row p, p = 4 b3 + 2 b2 + b1.
                const bool b3 = (lane & 8) != 0, b2 = (lane & 4) != 0, b1 = (lane & 2) != 0;
                uint32_t m4[4], m2[2];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t send = b3 ? rm[k] : rm[4 + k], keep = b3 ? rm[4 + k] : rm[k];
                    m4[k] = __vmaxu2(keep, __shfl_xor_sync(kFull, send, 8));
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const uint32_t send = b2 ? m4[k] : m4[2 + k], keep = b2 ? m4[2 + k] : m4[k];
                    m2[k] = __vmaxu2(keep, __shfl_xor_sync(kFull, send, 4));
                }
                uint32_t m1 = __vmaxu2(b1 ? m2[1] : m2[0], __shfl_xor_sync(kFull, b1 ? m2[0] : m2[1], 2));
                m1 = __vmaxu2(m1, __shfl_xor_sync(kFull, m1, 1));
                const uint32_t m = max(m1 & 0xFFFFu, m1 >> 16);
                const int p = (b3 ? 4 : 0) + (b2 ? 2 : 0) + (b1 ? 1 : 0);
                const int r = rbase + p;
                float sv, rv = 0.0f;
                if constexpr (GRAN == kGranTok) {
                    const ScaleDiv sd = scale_div_from_amax(amax_bits_to_f32(m));
                    sv = sd.s;
                    rv = sd.fast ? sd.r : 0.0f;
                    if ((lane & 1) == 0 && r < nrows) static_cast<float*>(s)[(int64_t)r * tiles_c + ct] = sv;
                } else {
                    const int e = mx_exponent_from_amax_bits(m << 16);
                    sv = exp2_neg(e);
                    if ((lane & 1) == 0 && r < nrows) static_cast<uint8_t*>(s)[(int64_t)r * tiles_c + ct] = (uint8_t)(e + 127);
                }
                if ((lane & 1) == 0) sh.rsr[w][8 * half + p] = make_float2(sv, rv);
                const bool warp_fast = __all_sync(kFull, kP2 || rv != 0.0f);   // the warp's 16 rows
                __syncwarp();
                auto rows_out = [&](auto fast) {
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const float2 sr = sh.rsr[w][8 * half + k];
                        const int r = rbase + k;
                        const uint2 o = row_codes(k, sr.x, sr.y, decltype(fast)::value || sr.y != 0.0f);
                        if (r < nrows && cols_in) *reinterpret_cast<uint2*>(q + (int64_t)r * cols + cbase) = o;
                    }
                };
                if (warp_fast) rows_out(std::true_type{});
                else rows_out(std::false_type{});
            } else {
                // MXFP8: a 32-column group is 4 lanes (lane bits 0 and 1).  After
                // the butterfly lane j of the group holds rows 2j and 2j + 1.
                const bool b1 = (lane & 2) != 0, b0 = (lane & 1) != 0;
                uint32_t m4[4], m2[2];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t send = b1 ? rm[k] : rm[4 + k], keep = b1 ? rm[4 + k] : rm[k];
                    m4[k] = __vmaxu2(keep, __shfl_xor_sync(kFull, send, 2));
                }
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const uint32_t send = b0 ? m4[k] : m4[2 + k], keep = b0 ? m4[2 + k] : m4[k];
                    m2[k] = __vmaxu2(keep, __shfl_xor_sync(kFull, send, 1));
                }
                const int p0 = (b1 ? 4 : 0) + (b0 ? 2 : 0);
                const int64_t ncb = ceil_div(cols, 32);
                const int64_t gcol = c0 + 32 * (cg >> 2);   // the group's first column
                uint32_t packed = 0;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int e = mx_exponent_from_amax_bits(max(m2[k] & 0xFFFFu, m2[k] >> 16) << 16);
                    packed |= (uint32_t)(e + 127) << (8 * k);
                    const int r = rbase + p0 + k;
                    if (r < nrows && gcol < cols) static_cast<uint8_t*>(s)[(int64_t)r * ncb + (gcol >> 5)] = (uint8_t)(e + 127);
                }
                uint32_t pk[4];   // biased exponents of rows 2j (bits 0..7) and 2j + 1 (bits 8..15)
#pragma unroll
                for (int j = 0; j < 4; ++j) pk[j] = __shfl_sync(kFull, packed, (lane & ~3) | j);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int r = rbase + k;
                    const float mk = exp2_neg((int)((pk[k >> 1] >> (8 * (k & 1))) & 0xFFu) - 127);
                    const uint2 o = row_codes(k, mk, 0.0f, true);
                    if (r < nrows && cols_in) *reinterpret_cast<uint2*>(q + (int64_t)r * cols + cbase) = o;
                }
            }
        }

        // ---------------- column scales
        __syncthreads();   // red is complete, and every thread holds its block: the stage's BF16 data is dead
        // MXFP8: column j's exponent from the group's maxima in cm
        auto mx_col_exp = [&](int j) {
            return mx_exponent_from_amax_bits(((j & 1) ? (cm[j >> 1] >> 16) : (cm[j >> 1] & 0xFFFFu)) << 16);
        };
        bool tile_fast = true;
        if constexpr (kMxG) {
            // this warp's and the other warp's maxima of the 32-row group (read
            // back rather than kept in registers through the row pass)
            const uint4 o0 = sh.red[w][cg], o1 = sh.red[w ^ 1][cg];
            cm[0] = __vmaxu2(o0.x, o1.x);
            cm[1] = __vmaxu2(o0.y, o1.y);
            cm[2] = __vmaxu2(o0.z, o1.z);
            cm[3] = __vmaxu2(o0.w, o1.w);
            // X^T scales: one byte per column and 32-row group, from the group's first warp
            if ((w & 1) == 0 && half == 0 && r0 + 16 * w < nrows) {
                const int64_t nrb = ceil_div(rows, 32), rb = (r0 >> 5) + (w >> 1);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (cbase + j < cols) static_cast<uint8_t*>(st)[(cbase + j) * nrb + rb] = (uint8_t)(mx_col_exp(j) + 127);
            }
        } else {
            bool mine_fast = true;
            if (tid < 64) {
                // columns 2 tid and 2 tid + 1: word tid % 4 of 8-column group tid / 4
                uint32_t mm = 0;
#pragma unroll
                for (int ww = 0; ww < 8; ++ww) mm = __vmaxu2(mm, reinterpret_cast<const uint32_t*>(&sh.red[ww][tid >> 2])[tid & 3]);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t mb = h ? (mm >> 16) : (mm & 0xFFFFu);
                    const int cl = 2 * tid + h;
                    const int64_t c = c0 + cl;
                    if constexpr (GRAN == kGranTok) {
                        const ScaleDiv sd = scale_div_from_amax(amax_bits_to_f32(mb));
                        sh.csr[cl] = make_float2(sd.s, sd.fast ? sd.r : 0.0f);
                        mine_fast = mine_fast && sd.fast;
                        if (c < cols) static_cast<float*>(st)[c * tiles_r + rt] = sd.s;
                    } else {
                        const int e = mx_exponent_from_amax_bits(mb << 16);
                        sh.csr[cl] = make_float2(exp2_neg(e), 0.0f);
                        if (c < cols) static_cast<uint8_t*>(st)[c * tiles_r + rt] = (uint8_t)(e + 127);
                    }
                }
            }
            tile_fast = __syncthreads_and(mine_fast);   // the tile's column scales are in csr
        }

        // ---------------- X^T codes: the thread's 8 rows of each of its 8 columns,
        // as 8 bytes of the [column][row] byte tile in the consumed stage
        auto cols_out = [&](auto fast) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int jw = j >> 1;
                float v[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) v[k] = (j & 1) ? bf16_hi(x[k][jw]) : bf16_lo(x[k][jw]);
                float sv, rv = 0.0f;
                if constexpr (kMxG) {
                    sv = exp2_neg(mx_col_exp(j));
                } else {
                    const float2 sr = sh.csr[8 * cg + j];
                    sv = sr.x;
                    rv = sr.y;
                }
                const uint64_t p01 = pair_f32(v[0], v[1]), p23 = pair_f32(v[2], v[3]);
                const uint64_t p45 = pair_f32(v[4], v[5]), p67 = pair_f32(v[6], v[7]);
                uint2 o;
                if (kP2 || decltype(fast)::value || rv != 0.0f) o = codes8_fast<kP2>(p01, p23, p45, p67, sv, rv);
                else o = codes8_slow(p01, p23, p45, p67, sv, rv);
                *reinterpret_cast<uint2*>(ct8 + (8 * cg + j) * 128 + 16 * (w ^ sw) + 8 * half) = o;
            }
        };
        if (kP2 || tile_fast) cols_out(std::true_type{});
        else cols_out(std::false_type{});
        }
        __syncthreads();   // the byte tile is complete
#pragma unroll
        for (int pass = 0; pass < 4; ++pass) {
            const int xr = (tid >> 3) + 32 * pass, k = tid & 7;   // row of X^T within the tile, 16-byte chunk
            const int64_t c = c0 + xr;
            if (c < cols && r0 + 16 * k < nrows)
                *reinterpret_cast<uint4*>(qt + c * rows + r0 + 16 * k) =
                    *reinterpret_cast<const uint4*>(ct8 + xr * 128 + 16 * (k ^ ((xr >> 3) & 7)));
        }
        fence_proxy_async_smem();   // this thread's generic accesses to the stage come before its refill
        advance(rt, ct);
    }
    // After an abort, copies issued but not yet waited for must land before
    // the CTA exits (each stage has at most one such copy).
    if (tid == 0) {
        for (int64_t i = consumed; i < issued; ++i)
            mbar_wait_drain(smem_u32(&sh.full[i % kTileStages]), (uint32_t)((i / kTileStages) & 1), kWaitLimitNs);
    }
}

// ---------------------------------------------------------------- launchers
static int rowwise_blocks(int64_t rows, int64_t cols, int cap) {
    const int64_t tasks = rows * ceil_div(cols, kSeg);
    const int64_t want = ceil_div(tasks, kThreads / 32);
    return (int)std::max<int64_t>(1, std::min<int64_t>(want, cap));
}

// Whether the amax pass keeps X in L2 for the cast pass: X up to 96 MB,
// three quarters of GB300's 126 MB L2.
static bool l2_keep_x(int64_t rows, int64_t ldx) {
    return 2.0 * (double)rows * (double)ldx <= 96.0 * 1024 * 1024;
}

static int launch_amax(const QuantJob& j, cudaStream_t st, int* nparts) {
    const int n = rowwise_blocks(j.rows, j.cols, std::min(kMaxPartials, sm_count() * 4));
    amax_partials_kernel<<<n, kThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.partials,
                                                 l2_keep_x(j.rows, j.ldx));
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

// Every (amax, x) pair of the FP32-scale casts: amax a positive finite BF16
// value, x a finite BF16 value with |x| <= amax, S = fp32_scale_from_amax(amax).
// Counts the pairs, the pairs whose E4M3 code through div_scale differs from
// the code of the IEEE quotient, and the amax values that take the fast path.
__global__ void __launch_bounds__(256) quotient_sweep_kernel(unsigned long long* __restrict__ counts) {
    const uint32_t ai = blockIdx.x * blockDim.x + threadIdx.x;
    if (ai == 0 || ai > 0x7F7Fu) return;
    const float amax = __uint_as_float(ai << 16);
    const float sc = fp32_scale_from_amax(amax);
    const ScaleDiv d = scale_div(sc, true);
    const ScaleDiv2 d2 = scale_div2(d);
    unsigned long long n = 0, bad = 0;
    for (uint32_t xb = 0; xb < 0x10000u; ++xb) {
        if (((xb >> 7) & 0xFFu) == 0xFFu) continue;
        const float x = __uint_as_float(xb << 16);
        if (fabsf(x) > amax) continue;
        ++n;
        // the code as the quantisers take it: packed pairs on the fast path
        // (both byte positions of a pair checked), IEEE division otherwise
        const uint32_t want = e4m3_byte(__fdiv_rn(x, sc));
        if (d.fast) {
            const uint32_t c4 = e4m3x4_div_fast2(pair_f32(x, x), pair_f32(x, x), d2);
            bad += ((c4 & 0xFFu) != want || (c4 >> 24) != want) ? 1 : 0;
        } else {
            bad += (e4m3_byte(__fdiv_rn(x, d.s)) != want) ? 1 : 0;
        }
    }
    atomicAdd(&counts[0], n);
    atomicAdd(&counts[1], bad);
    if (d.fast) atomicAdd(&counts[2], 1ull);
}

// NVFP4: every positive BF16 amax_T, S_g = amax_T / D (D = 2688, or 1536
// for four-over-six), every nonzero block scale code s_b (1..126),
// S_b = E4M3value(s_b) * S_g, every finite BF16 x with |x| <= amax_T; E2M1
// code through div_scale against the IEEE quotient's.  One thread per
// (amax_T, s_b, D).
__global__ void __launch_bounds__(256) quotient_sweep_nvfp4_kernel(unsigned long long* __restrict__ counts) {
    const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
    const uint32_t ai = t / 252u, rest = t - ai * 252u;      // 126 codes x 2 divisors
    const uint32_t code = 1u + (rest >> 1);
    if (ai == 0 || ai > 0x7F7Fu) return;
    const float amax = __uint_as_float(ai << 16);
    const float s_g = __fdiv_rn(amax, (rest & 1u) ? kNvfp4GlobalDiv4over6 : kNvfp4GlobalDiv);
    const float big_s = __fmul_rn(e4m3_value(code), s_g);
    if (big_s == 0.0f) return;                                // both paths give code 0
    const ScaleDiv d = scale_div(big_s, true);
    const ScaleDiv2 d2 = scale_div2(d);
    unsigned long long n = 0, bad = 0;
    for (uint32_t xb = 0; xb < 0x10000u; ++xb) {
        if (((xb >> 7) & 0xFFu) == 0xFFu) continue;
        const float x = __uint_as_float(xb << 16);
        if (fabsf(x) > amax) continue;
        ++n;
        // the codes as the quantisers take them (packed pairs on the fast
        // path; the first and last positions checked) against IEEE division
        const float b[8] = {__fdiv_rn(x, big_s), 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const uint32_t want = e2m1x8(b) & 0xFu;
        if (d.fast) {
            const float a[8] = {x, x, x, x, x, x, x, x};
            const uint32_t c8 = e2m1x8_div_fast2(a, d2);
            bad += ((c8 & 0xFu) != want || (c8 >> 28) != want) ? 1 : 0;
        } else {
            const float a[8] = {__fdiv_rn(x, d.s), 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            bad += ((e2m1x8(a) & 0xFu) != want) ? 1 : 0;
        }
    }
    atomicAdd(&counts[0], n);
    atomicAdd(&counts[1], bad);
    if (d.fast) atomicAdd(&counts[2], 1ull);
}

// Breakpoints of the product's casts.  Both casts are monotone in the
// magnitude of their float32 input, so for each nonzero code magnitude c
// there is a smallest float32 magnitude whose code has magnitude >= c; a
// binary search over the (ordered) bit patterns of the positive floats finds
// it.  Thread t < 252: E4M3, sign t / 126, c = 1 + t % 126, through the
// packed pair cast the quantisers use (all four bytes must agree); thread
// 252 <= t < 266: E2M1, sign (t - 252) / 7, c = 1 + (t - 252) % 7, through
// the eight-wide cast (all eight nibbles must agree).  out[t] receives the
// breakpoint's bits; a disagreement between lanes, or a code of the wrong
// sign, writes 0xFFFFFFFF instead.
__global__ void __launch_bounds__(288) encoder_breakpoints_kernel(uint32_t* __restrict__ out) {
    const int t = threadIdx.x;
    if (t >= 266) return;
    const bool fp4 = t >= 252;
    const int u = fp4 ? t - 252 : t;
    const int per_sign = fp4 ? 7 : 126;
    const bool neg = u >= per_sign;
    const uint32_t c = 1u + (uint32_t)(u % per_sign);
    bool ok = true;
    // magnitude of the code of (sign) * bits, checking every lane agrees
    auto mag = [&](uint32_t bits) -> uint32_t {
        const float x = __uint_as_float(bits | (neg ? 0x80000000u : 0u));
        if (!fp4) {
            const uint32_t r = e4m3x4_pairs(pair_f32(x, x), pair_f32(x, x));
            const uint32_t b = r & 0xFFu;
            if (r != b * 0x01010101u) ok = false;
            if (neg && b != 0u && (b & 0x80u) == 0u) ok = false;
            if (!neg && (b & 0x80u) != 0u) ok = false;
            return b & 0x7Fu;
        }
        const float a[8] = {x, x, x, x, x, x, x, x};
        const uint32_t r = e2m1x8(a);
        const uint32_t b = r & 0xFu;
        if (r != b * 0x11111111u) ok = false;
        if (neg && b != 0u && (b & 0x8u) == 0u) ok = false;
        if (!neg && (b & 0x8u) != 0u) ok = false;
        return b & 0x7u;
    };
    uint32_t lo = 0u, hi = 0x7F7FFFFFu;          // mag(0) = 0 < c; FLT_MAX saturates to the largest code
    if (mag(hi) < c) ok = false;
    while (lo + 1u < hi) {                       // invariant: mag(lo) < c <= mag(hi)
        const uint32_t mid = lo + ((hi - lo) >> 1);
        if (mag(mid) >= c) hi = mid; else lo = mid;
    }
    out[t] = ok ? hi : 0xFFFFFFFFu;
}

// Every finite positive float32 bit pattern b in [0, 0x7F7FFFFE]: the
// packed E4M3 and E2M1 casts of b+1 give a code magnitude at least that of
// b (monotone), and the cast of -b is the cast of b with its sign bit set
// (symmetric).  Violations are counted into *bad.  With the breakpoints
// above this fixes both casts on every finite float32.
__global__ void __launch_bounds__(256) encoder_monotone_kernel(unsigned int* __restrict__ bad) {
    const uint32_t stride = gridDim.x * blockDim.x;
    unsigned int n = 0;
    for (uint32_t b = blockIdx.x * blockDim.x + threadIdx.x; b < 0x7F7FFFFFu; b += stride) {
        const float x0 = __uint_as_float(b), x1 = __uint_as_float(b + 1);
        const uint32_t e = e4m3x4_pairs(pair_f32(x0, x1), pair_f32(-x0, -x1));
        const uint32_t c0 = e & 0xFFu, c1 = (e >> 8) & 0xFFu, n0 = (e >> 16) & 0xFFu, n1 = e >> 24;
        n += (c1 < c0) ? 1u : 0u;
        n += (n0 != (c0 | 0x80u) || n1 != (c1 | 0x80u)) ? 1u : 0u;
        const float a[8] = {x0, x1, -x0, -x1, 0.f, 0.f, 0.f, 0.f};
        const uint32_t f = e2m1x8(a);
        const uint32_t d0 = f & 0xFu, d1 = (f >> 4) & 0xFu, m0 = (f >> 8) & 0xFu, m1 = (f >> 12) & 0xFu;
        n += (d1 < d0) ? 1u : 0u;
        n += (m0 != (d0 | 0x8u) || m1 != (d1 | 0x8u)) ? 1u : 0u;
    }
    if (n) atomicAdd(bad, n);
}

int launch_encoder_breakpoints(uint32_t* out, cudaStream_t st) {
    encoder_breakpoints_kernel<<<1, 288, 0, st>>>(out);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    encoder_monotone_kernel<<<sm_count() * 8, 256, 0, st>>>(out + 266);
    return (int)cudaGetLastError();
}

// NVFP4 block scale codes: every positive BF16 amax_T with S_g =
// RN(amax_T / D) on the fast path, for D = 2688 and D = 1536, and every BF16
// a <= amax_T: the code through nvfp4_block_code against
// E4M3(RN(RN(a / 6) / S_g)) by IEEE division, and for D = 1536 (the
// four-over-six divisor) also the a / 4 form.  Each thread also compares
// div6_fast(amax_T) with RN(amax_T / 6), bit for bit, for every BF16
// amax_T including zero and the subnormals.  One thread per amax_T.
__global__ void __launch_bounds__(256) quotient_sweep_block_code_kernel(unsigned long long* __restrict__ counts) {
    const uint32_t ai = blockIdx.x * blockDim.x + threadIdx.x;
    if (ai > 0x7F7Fu) return;
    const float amax = __uint_as_float(ai << 16);
    unsigned long long n = 1, bad = 0, fast = 0;
    bad += __float_as_uint(div6_fast(amax)) != __float_as_uint(__fdiv_rn(amax, kE2M1Max)) ? 1 : 0;
    if (ai != 0) {
        for (int v = 0; v < 2; ++v) {
            const float s_g = __fdiv_rn(amax, v ? kNvfp4GlobalDiv4over6 : kNvfp4GlobalDiv);
            const ScaleDiv dg = scale_div(s_g, true);
            if (!dg.fast) continue;
            ++fast;
            for (uint32_t bi = 0; bi <= ai; ++bi) {
                const float a = __uint_as_float(bi << 16);
                ++n;
                bad += nvfp4_block_code(a, s_g, dg, false) != e4m3_byte(__fdiv_rn(__fdiv_rn(a, kE2M1Max), s_g)) ? 1 : 0;
                if (v) {
                    ++n;
                    bad += nvfp4_block_code(a, s_g, dg, true) != e4m3_byte(__fdiv_rn(__fdiv_rn(a, 4.0f), s_g)) ? 1 : 0;
                }
            }
        }
    }
    atomicAdd(&counts[0], n);
    atomicAdd(&counts[1], bad);
    atomicAdd(&counts[2], fast);
}

// FP32 scales without IEEE operations: for every finite BF16 amax (zero
// and subnormals included), the S and RN(1/S) that scale_div_from_amax
// gives against __fdiv_rn(amax, 448) and __frcp_rn(S), bit for bit.
// counts[0] amax values, [1] mismatches, [2] values on the fast path.
__global__ void __launch_bounds__(256) quotient_sweep_scale_kernel(unsigned long long* __restrict__ counts) {
    const uint32_t ai = blockIdx.x * blockDim.x + threadIdx.x;
    if (ai > 0x7F7Fu) return;
    const float amax = __uint_as_float(ai << 16);
    const ScaleDiv got = scale_div_from_amax(amax);
    const ScaleDiv want = scale_div(fp32_scale_from_amax(amax), true);
    const bool same = __float_as_uint(got.s) == __float_as_uint(want.s) && got.fast == want.fast &&
                      (!want.fast || __float_as_uint(got.r) == __float_as_uint(want.r));
    atomicAdd(&counts[0], 1ull);
    if (!same) atomicAdd(&counts[1], 1ull);
    if (amax >= kFastScaleMinAmax) atomicAdd(&counts[2], 1ull);
}

int launch_quotient_sweep(unsigned long long* counts, int nvfp4, cudaStream_t st) {
    if (nvfp4 == 3)
        quotient_sweep_scale_kernel<<<(0x7F80u + 255u) / 256u, 256, 0, st>>>(counts);
    else if (nvfp4 == 2)
        quotient_sweep_block_code_kernel<<<(0x7F80u + 255u) / 256u, 256, 0, st>>>(counts);
    else if (nvfp4)
        quotient_sweep_nvfp4_kernel<<<(0x7F80u * 252u + 255u) / 256u, 256, 0, st>>>(counts);
    else
        quotient_sweep_kernel<<<(0x7F80 + 255) / 256, 256, 0, st>>>(counts);
    return (int)cudaGetLastError();
}

// ---------------------------------------------------------------- gather of quantised rows
// q[r] = q_src[idx[r]] and the scale row likewise, for the row-wise layouts
// of 1x128 (FP32 scales), MXFP8 and 1x128 power-of-two (byte scales).  The
// codes and scales of a row depend on that row alone, so this equals the
// gathered quantiser on the same tokens.  An index outside [0, tokens)
// gives the all-zero row (zero codes, the scale of an all-zero group: 1.0,
// or the byte 0 of exponent -127) and sets kStatusIndex.  One warp per row;
// V16: 16-byte code chunks (cols % 16 == 0), else 8-byte ones.
template <int GRAN, bool V16>
__global__ void __launch_bounds__(kThreads)
gather_rows_kernel(const uint8_t* __restrict__ q_src, const void* __restrict__ s_src, int64_t tokens, int64_t cols,
                   const int64_t* __restrict__ idx, int64_t rows, uint8_t* __restrict__ q, void* __restrict__ s,
                   int* status) {
    constexpr int CH = V16 ? 16 : 8;
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t ng = ceil_div(cols, GRAN == kGranMx ? 32 : 128);
    for (int64_t r = gw; r < rows; r += nw) {
        const int64_t t = __ldg(idx + r);
        const bool valid = t >= 0 && t < tokens;
        if (!valid && lane == 0 && status != nullptr) atomicExch(status, kStatusIndex);
        const uint8_t* src = q_src + (valid ? t : 0) * cols;
        uint8_t* dst = q + r * cols;
        for (int64_t c = (int64_t)CH * lane; c < cols; c += 32 * CH) {
            if constexpr (V16) stg_cs_v4(dst + c, valid ? ldg_v4(src + c) : make_uint4(0, 0, 0, 0));
            else stg_cs_v2(dst + c, valid ? ldg_v2(src + c) : make_uint2(0, 0));
        }
        for (int64_t g = lane; g < ng; g += 32) {
            if constexpr (GRAN == kGranTok)
                static_cast<float*>(s)[r * ng + g] = valid ? __ldg(static_cast<const float*>(s_src) + t * ng + g) : 1.0f;
            else
                static_cast<uint8_t*>(s)[r * ng + g] = valid ? __ldg(static_cast<const uint8_t*>(s_src) + t * ng + g)
                                                             : (uint8_t)0;
        }
    }
}

template <int GRAN>
static int launch_gather_g(const GatherJob& j, cudaStream_t st) {
    const int nb = (int)std::max<int64_t>(1, std::min<int64_t>(ceil_div(j.rows, kThreads / 32), sm_count() * 8));
    if (j.cols % 16 == 0)
        gather_rows_kernel<GRAN, true><<<nb, kThreads, 0, st>>>(j.q_src, j.s_src, j.tokens, j.cols, j.idx, j.rows,
                                                               j.q, j.s, j.status);
    else
        gather_rows_kernel<GRAN, false><<<nb, kThreads, 0, st>>>(j.q_src, j.s_src, j.tokens, j.cols, j.idx, j.rows,
                                                                j.q, j.s, j.status);
    return (int)cudaGetLastError();
}

int launch_gather_rows(const GatherJob& j, cudaStream_t st) {
    switch (j.gran) {
    case kGranTok: return launch_gather_g<kGranTok>(j, st);
    case kGranMx: return launch_gather_g<kGranMx>(j, st);
    case kGranTokP2: return launch_gather_g<kGranTokP2>(j, st);
    default: return (int)cudaErrorInvalidValue;
    }
}

template <int SRC>
static int launch_rows_src(const QuantJob& j, const RowSrc& src, int nb, cudaStream_t st) {
    switch (j.gran) {
    case kGranTok:
        quant_rows_kernel<kGranTok, SRC><<<nb, kThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.q, j.s, nullptr, 0,
                                                                  nullptr, src);
        break;
    case kGranMx:
        quant_rows_kernel<kGranMx, SRC><<<nb, kThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.q, j.s, nullptr, 0,
                                                                 nullptr, src);
        break;
    case kGranTokP2:
        quant_rows_kernel<kGranTokP2, SRC><<<nb, kThreads, 0, st>>>(j.x, j.rows, j.cols, j.ldx, j.q, j.s, nullptr, 0,
                                                                    nullptr, src);
        break;
    default:
        return (int)cudaErrorInvalidValue;
    }
    return (int)cudaGetLastError();
}

int launch_quantize_rows_src(const QuantJob& j, const int64_t* token_index, int64_t tokens, int64_t up,
                             cudaStream_t st) {
    const int nb = rowwise_blocks(j.rows, j.cols, sm_count() * 8);
    RowSrc src{token_index, tokens, up, j.status, token_index != nullptr && l2_keep_x(tokens, j.ldx)};
    if (token_index != nullptr) return launch_rows_src<kSrcGather>(j, src, nb, st);
    return launch_rows_src<kSrcSwiglu>(j, src, nb, st);
}

template <int GRAN, bool DUAL>
static int launch_tile_k(const CUtensorMap& tm, const QuantJob& j, int64_t tiles, cudaStream_t st,
                         const uint32_t* partials, int nparts, const float* given) {
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, kTileCtas<GRAN, DUAL> * (int64_t)sm_count()));
    static bool attr_set[64] = {false};   // one flag per kernel instantiation and device
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(quant_tile_tma_kernel<GRAN, DUAL>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTileSmem);
        if (e != cudaSuccess) return (int)e;
        attr_set[dev] = true;
    }
    quant_tile_tma_kernel<GRAN, DUAL><<<grid, kTileThreads, kTileSmem, st>>>(
        tm, j.rows, j.cols, j.qt, j.st, DUAL ? j.q : nullptr, DUAL ? j.s : nullptr, j.status, partials, nparts, given);
    return (int)cudaGetLastError();
}

template <int GRAN>
static int launch_tile(const QuantJob& j, cudaStream_t st, const uint32_t* partials = nullptr, int nparts = 0,
                       const float* given = nullptr) {
    CUtensorMap tm;
    if (!make_tmap_b16(&tm, j.x, (uint64_t)j.cols, (uint64_t)j.rows, (uint64_t)j.ldx, 128, 128))
        return (int)cudaErrorInvalidValue;
    const int64_t tiles = ceil_div(j.cols, 128) * ceil_div(j.rows, 128);
    if (j.q != nullptr) return launch_tile_k<GRAN, true>(tm, j, tiles, st, partials, nparts, given);
    return launch_tile_k<GRAN, false>(tm, j, tiles, st, partials, nparts, given);
}


// Granularities with a scale per column of X (1x128, 1x32 groups of X^T's
// rows) take the TMA-fed kernel; those with one scale per tile the
// register-resident one (each the faster of the two on GB300).
int launch_quantize_transposed(const QuantJob& j, cudaStream_t st) {
    int nparts = 0;
    switch (j.gran) {
    case kGranTok: return launch_tile<kGranTok>(j, st);
    case kGranMx: return launch_tile<kGranMx>(j, st);
    case kGranTokP2: return launch_tile<kGranTokP2>(j, st);
    case kGranBlk: return launch_tile<kGranBlk>(j, st);
    case kGranBlkP2: return launch_tile<kGranBlkP2>(j, st);
    case kGranPT: {
        if (!j.given_scale) {
            const int e = launch_amax(j, st, &nparts);
            if (e) return e;
        }
        return launch_tile<kGranPT>(j, st, j.partials, nparts, j.given_scale ? static_cast<const float*>(j.st) : nullptr);
    }
    default:
        return (int)cudaErrorInvalidValue;
    }
}

}  // namespace fp8bs

namespace fp8bs {

// Per-tensor quantisation with the amax partials in scratch the caller
// names: pass 1 runs exactly `nparts` CTAs, each writing one partial, and
// pass 2 reduces those `nparts` partials, so no slot needs clearing first.
int launch_quantize_per_tensor_scratch(const uint16_t* x, int64_t rows, int64_t cols, int64_t ldx, uint8_t* q,
                                       float* scale, uint32_t* partials, int nparts, cudaStream_t st) {
    amax_partials_kernel<<<nparts, kThreads, 0, st>>>(x, rows, cols, ldx, partials, l2_keep_x(rows, ldx));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
    const int nb = rowwise_blocks(rows, cols, sm_count() * 8);
    quant_rows_kernel<kGranPT><<<nb, kThreads, 0, st>>>(x, rows, cols, ldx, q, scale, partials, nparts, nullptr);
    return (int)cudaGetLastError();
}

}  // namespace fp8bs
