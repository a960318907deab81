// gemm_blockwise.cu -- FP8 E4M3 GEMM with FP32 block scales (tcgen05 + TMA + TMEM).
//
//   D[m, n] = sum_kb  sa(m, kb) * sb(n, kb) * sum_{k in kb} qa[m, k] * qb[n, k]
//
// the block-wise ("DeepSeek-style") recipe of the "Low Precision RL" page
// (table "Choose a precision": 128x128 blocks, FP32 scales; section
// "2. Unified block-wise FP8") with per-token 1x128 activation scales (the
// review's "FP8 Quantization": per-token for activations and gradients).
// FP32 scales cannot ride on the tensor core's power-of-two block-scale
// path, so each 128-wide K block is accumulated on its own in TMEM and the
// epilogue warps fold it into FP32 registers with the scale product
// ("promotion").  Two TMEM partial buffers alternate, so the MMAs of block
// kb+1 run while block kb is being promoted.
//
// CTA: 384 threads (3 warpgroups), one CTA per SM (persistent), tile
// 128 x 256, K block 128.  Launched at 168 registers per thread; the
// producer warpgroup gives registers back (72) and the two epilogue
// warpgroups take them (216): 128*72 + 256*216 = 384*168.
//   warp 0      TMA producer (one lane): A 128x128 and B 256x128 boxes,
//               128-byte swizzle, 3-stage ring.
//   warp 1      TMEM owner + MMA issuer (one lane): 4 x tcgen05.mma
//               kind::f8f6f4 (M128 N256 K32) per K block into partial
//               buffer kb & 1, then tcgen05.commit to free the stage and to
//               publish the partial.
//   warp 2      scale loader: for each group of 4 K blocks of a tile, the
//               128 row scales of A and the 256 column scales of B, read as
//               16-byte runs (4 K blocks of one row / column) and stored
//               transposed ([K block][row], [K block][column]) into a 2-slot
//               shared-memory ring.  The per-column B scales of the 1x128
//               mode would otherwise cost every epilogue warp one scattered
//               load per column per K block.
//   warp 3      tile fetcher (one lane): the CTA's first tile is blockIdx.x,
//               each later one the next index of a tile counter in the
//               workspace (atomicAdd), published to the other roles through
//               a shared-memory ring.  Tiles go in index order to whichever
//               CTA is free, so a launch that starts on SMs as an earlier
//               kernel leaves them evens out its own tail.  The last CTA to
//               finish puts the counter back to 0 for the next launch.
//   warps 4..11 epilogue: warp w reads TMEM lanes 32*(w%4).. (one D row per
//               thread) and columns 128*((w-4)/4).. (one 128-column half);
//               acc += partial * sa * sb with both scales read from the
//               ring.  At the end of the tile each warp writes its 32 rows as
//               BF16 into a 4 KB staging buffer, 64 columns at a time (float32
//               output: 32 at a time), and a TMA store takes them out, so the
//               warp is back to promoting while the store drains (its stores
//               used to hold the MMA up).
// Scale modes (template): 0 per-tensor, 1 per row (1x128), 2 per 128-row block.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"
#include "tmap.h"

namespace fp8bs {
namespace {

constexpr int BM = 128, BN = 256, BK = 128, STAGES = 3;
constexpr int OSTAGE_BYTES = 32 * 128;   // per epilogue warp: 32 rows x 64 BF16 columns
constexpr int SG = 4;          // K blocks per scale group
constexpr int SRING = 2;       // scale groups in flight
constexpr int A_BYTES = BM * BK, B_BYTES = BN * BK, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 384;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC = idesc_f8f6f4_e4m3(BM, BN);
// Tile indices in flight.  One: a CTA claims its next tile when its
// epilogue starts the current one, so claims keep pace with the work (a
// deeper ring let every CTA claim several tiles at launch, in arbitrary
// order: the tiles spread unevenly over the CTAs and wgrad took 0.38 ms
// instead of 0.29).
constexpr int TQ = 1;
constexpr int TQ_READERS = 11; // producer, MMA thread, scale loader, 8 epilogue warps
// Dynamic tile order for B with one scale per 128 x 128 block (or per
// tensor).  The per-column-scale form (the weight gradient's 1 x 128 B)
// keeps the static order: a tile index that arrives at run time stays live
// through its epilogue's K loop, and that form is already at the register
// limit there (its spills grew and it ran 6 % slower).
template <int SB> constexpr bool kDynamicTiles = SB != 1;

struct Params {
    int64_t m, n, k;
    const float* sa;
    const float* sb;
    __nv_bfloat16* d;
    int* status;
    const int64_t* offsets;
    int experts;
    uint64_t wait_ns;     // bound of every pipeline wait
    int stall_stage0;     // test hook: the producer withholds stage 0
    int out_f32;          // D is float32 (tm_d then maps float32 32 x 32 boxes)
    unsigned long long* tile_next;   // tiles handed out past the first wave (nullptr: static order)
    unsigned int* tile_done;         // CTAs finished
};

struct alignas(16) Shared {
    float sa[SRING][SG][BM];   // A scale of each tile row, per K block of the group
    float sb[SRING][SG][BN];   // B scale of each tile column (modes 0 / 2: entries 0 and 128 only)
    uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], sfull[SRING], sempty[SRING], drain;
    uint64_t tq_full[TQ], tq_empty[TQ];
    int64_t tq[TQ];            // tile index ring (an index >= total ends the CTA's work)
    uint32_t tmem_base;
    int abort;
    SchedShared sched;
};

constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 8 * OSTAGE_BYTES + sizeof(Shared);

// Four consecutive K-block scales starting at kb0 from a row of `nkb` FP32
// scales (zero past the row's end); one 16-byte load when `vec`.
__device__ __forceinline__ float4 scales4(const float* __restrict__ src, int64_t kb0, int64_t nkb, bool vec) {
    if (vec) return __ldg(reinterpret_cast<const float4*>(src + kb0));
    float4 v;
    v.x = __ldg(src + kb0);
    v.y = (kb0 + 1 < nkb) ? __ldg(src + kb0 + 1) : 0.0f;
    v.z = (kb0 + 2 < nkb) ? __ldg(src + kb0 + 2) : 0.0f;
    v.w = (kb0 + 3 < nkb) ? __ldg(src + kb0 + 3) : 0.0f;
    return v;
}

__device__ __forceinline__ void put4(float (*dst)[BN], int idx, float4 v) {
    dst[0][idx] = v.x;
    dst[1][idx] = v.y;
    dst[2][idx] = v.z;
    dst[3][idx] = v.w;
}
__device__ __forceinline__ void put4a(float (*dst)[BM], int idx, float4 v) {
    dst[0][idx] = v.x;
    dst[1][idx] = v.y;
    dst[2][idx] = v.z;
    dst[3][idx] = v.w;
}

template <int SA_MODE, int SB_MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
gemm_blockwise_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                      const __grid_constant__ CUtensorMap tm_d, Params p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ostage = stages + (size_t)STAGES * STAGE_BYTES;   // 1024-byte aligned
    Shared* sh = reinterpret_cast<Shared*>(ostage + 8 * OSTAGE_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nkb = p.k / BK;
    const int64_t n_tiles = (p.n + BN - 1) / BN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&sh->full[s]), 1);
            mbar_init(smem_u32(&sh->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&sh->tfull[b]), 1);
            mbar_init(smem_u32(&sh->tempty[b]), 8);
        }
        for (int g = 0; g < SRING; ++g) {
            mbar_init(smem_u32(&sh->sfull[g]), 32);    // every loader lane arrives
            mbar_init(smem_u32(&sh->sempty[g]), 8);    // every epilogue warp arrives
        }
        mbar_init(smem_u32(&sh->drain), 1);
        for (int i = 0; i < TQ; ++i) {
            mbar_init(smem_u32(&sh->tq_full[i]), 1);
            mbar_init(smem_u32(&sh->tq_empty[i]), TQ_READERS);
        }
        sh->abort = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&sh->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    const int64_t total = sched_setup<BM>(&sh->sched, p.offsets, p.experts, p.m, n_tiles, p.status);  // has __syncthreads
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    volatile int* abort = &sh->abort;
    // The i-th tile of this CTA: from the ring (dynamic order), or
    // blockIdx.x + i * gridDim.x.  `t` >= total ends the work.  The caller
    // releases the ring slot once it has read it.
    auto next_tile = [&](uint32_t i, int64_t& t) -> bool {
        if constexpr (!kDynamicTiles<SB_MODE>) {
            t = (int64_t)blockIdx.x + (int64_t)i * gridDim.x;
            return true;
        }
        const uint32_t slot = i % TQ;
        if (!mbar_wait(smem_u32(&sh->tq_full[slot]), (i / TQ) & 1, abort, p.status, p.wait_ns)) return false;
        t = sh->tq[slot];
        return true;
    };
    auto release_tile = [&](uint32_t i) {
        if constexpr (kDynamicTiles<SB_MODE>) mbar_arrive(smem_u32(&sh->tq_empty[i % TQ]));
    };

    if (warp < 4) {
    setmaxnreg_dec<72>();
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            for (uint32_t ti_i = 0; ok; ++ti_i) {
                int64_t t;
                if (!next_tile(ti_i, t)) { ok = false; break; }
                release_tile(ti_i);
                if (t >= total) break;
                const TileInfo ti = sched_tile<BM, BN>(&sh->sched, p.offsets, p.experts, p.m, n_tiles, t);
                const int32_t brow = (int32_t)(ti.expert * p.n + ti.n0);
                for (int64_t kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    if (!mbar_wait(smem_u32(&sh->empty[s]), ph ^ 1, abort, p.status, p.wait_ns)) { ok = false; break; }
                    if (p.stall_stage0 && it == 0) continue;   // test hook: never fill stage 0
                    const uint32_t fb = smem_u32(&sh->full[s]);
                    uint8_t* sa_ptr = stages + (size_t)s * STAGE_BYTES;
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    tma_load_2d(smem_u32(sa_ptr), &tm_a, fb, (int32_t)(kb * BK), (int32_t)ti.row0);
                    tma_load_2d(smem_u32(sa_ptr + A_BYTES), &tm_b, fb, (int32_t)(kb * BK), brow);
                }
            }
            // Copies issued to the last STAGES stages must have landed before
            // the CTA exits (on the normal path they already have).
            for (uint32_t j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
                if (!(p.stall_stage0 && j == 0))
                    mbar_wait_drain(smem_u32(&sh->full[j % STAGES]), (j / STAGES) & 1, p.wait_ns);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t it = 0, kbg = 0;
            bool ok = true;
            for (uint32_t ti_i = 0; ok; ++ti_i) {
                int64_t t;
                if (!next_tile(ti_i, t)) { ok = false; break; }
                release_tile(ti_i);
                if (t >= total) break;
                for (int64_t kb = 0; kb < nkb; ++kb, ++it, ++kbg) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    const uint32_t b = kbg & 1, tph = (kbg >> 1) & 1;
                    if (!mbar_wait(smem_u32(&sh->full[s]), ph, abort, p.status, p.wait_ns)) { ok = false; break; }
                    if (!mbar_wait(smem_u32(&sh->tempty[b]), tph ^ 1, abort, p.status, p.wait_ns)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(stages + (size_t)s * STAGE_BYTES);
                    const uint64_t adesc = kmajor_sw128_desc(a_addr);
                    const uint64_t bdesc = kmajor_sw128_desc(a_addr + A_BYTES);
                    const uint32_t d_tmem = tmem + b * BN;
#pragma unroll
                    for (int kk = 0; kk < BK / 32; ++kk)
                        mma_f8f6f4(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, IDESC, kk > 0 ? 1u : 0u);
                    mma_commit(smem_u32(&sh->empty[s]));
                    mma_commit(smem_u32(&sh->tfull[b]));
                }
            }
            mma_commit(smem_u32(&sh->drain));
            mbar_wait(smem_u32(&sh->drain), 0, abort, p.status);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------ scale loader
        const bool vec_a = SA_MODE == 1 && (nkb & 3) == 0 && (reinterpret_cast<uintptr_t>(p.sa) & 15u) == 0;
        const bool vec_b = SB_MODE == 1 && (nkb & 3) == 0 && (reinterpret_cast<uintptr_t>(p.sb) & 15u) == 0;
        const float sa0 = (SA_MODE == 0) ? __ldg(p.sa) : 0.0f;
        uint32_t gg = 0;
        bool ok = true;
        // one tile's scale groups, under the dynamic or the static loop (the
        // body written out in each, as in the epilogue)
        if constexpr (kDynamicTiles<SB_MODE>) {
        for (uint32_t ti_i = 0; ok; ++ti_i) {
            int64_t t = 0;
            bool got = true;
            if (lane == 0) {
                got = next_tile(ti_i, t);
                if (got) release_tile(ti_i);
            }
            if (!__shfl_sync(0xFFFFFFFFu, got, 0)) { ok = false; break; }
            t = __shfl_sync(0xFFFFFFFFu, t, 0);
            if (t >= total) break;
            const TileInfo ti = sched_tile<BM, BN>(&sh->sched, p.offsets, p.experts, p.m, n_tiles, t);
            const float* sb_e = p.sb;
            if (p.experts) {
                const int64_t per = (SB_MODE == 2) ? ((p.n + 127) / 128) * nkb : p.n * nkb;
                sb_e = p.sb + (int64_t)ti.expert * per;
            }
            for (int64_t kb0 = 0; kb0 < nkb; kb0 += SG, ++gg) {
                const uint32_t g = gg % SRING, ph = (gg / SRING) & 1;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&sh->sempty[g]), ph ^ 1, abort, p.status, p.wait_ns))) {
                    ok = false;
                    break;
                }
                float4 va[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int64_t row = ti.row0 + lane + 32 * i;
                    if (SA_MODE == 0) va[i] = make_float4(sa0, sa0, sa0, sa0);
                    else if (row >= ti.row_end) va[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                    else if (SA_MODE == 1) va[i] = scales4(p.sa + row * nkb, kb0, nkb, vec_a);
                    else va[i] = scales4(p.sa + (row >> 7) * nkb, kb0, nkb, false);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) put4a(sh->sa[g], lane + 32 * i, va[i]);
                if (SB_MODE == 1) {
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float4 vb[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int64_t col = ti.n0 + lane + 32 * (4 * half + i);
                            vb[i] = (col < p.n) ? scales4(sb_e + col * nkb, kb0, nkb, vec_b) : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) put4(sh->sb[g], lane + 32 * (4 * half + i), vb[i]);
                    }
                } else if (lane < 2) {
                    const int64_t col = ti.n0 + 128 * lane;
                    float4 vb = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (col < p.n) {
                        if (SB_MODE == 0) {
                            const float s0 = __ldg(sb_e);
                            vb = make_float4(s0, s0, s0, s0);
                        } else {
                            vb = scales4(sb_e + (col >> 7) * nkb, kb0, nkb, false);
                        }
                    }
                    put4(sh->sb[g], 128 * lane, vb);
                }
                mbar_arrive(smem_u32(&sh->sfull[g]));
            }
        }
        } else {
        for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const TileInfo ti = sched_tile<BM, BN>(&sh->sched, p.offsets, p.experts, p.m, n_tiles, t);
            const float* sb_e = p.sb;
            if (p.experts) {
                const int64_t per = (SB_MODE == 2) ? ((p.n + 127) / 128) * nkb : p.n * nkb;
                sb_e = p.sb + (int64_t)ti.expert * per;
            }
            for (int64_t kb0 = 0; kb0 < nkb; kb0 += SG, ++gg) {
                const uint32_t g = gg % SRING, ph = (gg / SRING) & 1;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&sh->sempty[g]), ph ^ 1, abort, p.status, p.wait_ns))) {
                    ok = false;
                    break;
                }
                float4 va[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int64_t row = ti.row0 + lane + 32 * i;
                    if (SA_MODE == 0) va[i] = make_float4(sa0, sa0, sa0, sa0);
                    else if (row >= ti.row_end) va[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                    else if (SA_MODE == 1) va[i] = scales4(p.sa + row * nkb, kb0, nkb, vec_a);
                    else va[i] = scales4(p.sa + (row >> 7) * nkb, kb0, nkb, false);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) put4a(sh->sa[g], lane + 32 * i, va[i]);
                if (SB_MODE == 1) {
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        float4 vb[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int64_t col = ti.n0 + lane + 32 * (4 * half + i);
                            vb[i] = (col < p.n) ? scales4(sb_e + col * nkb, kb0, nkb, vec_b) : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
#pragma unroll
                        for (int i = 0; i < 4; ++i) put4(sh->sb[g], lane + 32 * (4 * half + i), vb[i]);
                    }
                } else if (lane < 2) {
                    const int64_t col = ti.n0 + 128 * lane;
                    float4 vb = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (col < p.n) {
                        if (SB_MODE == 0) {
                            const float s0 = __ldg(sb_e);
                            vb = make_float4(s0, s0, s0, s0);
                        } else {
                            vb = scales4(sb_e + (col >> 7) * nkb, kb0, nkb, false);
                        }
                    }
                    put4(sh->sb[g], 128 * lane, vb);
                }
                mbar_arrive(smem_u32(&sh->sfull[g]));
            }
        }
        }
        __syncwarp();
    } else if (warp == 3) {
        // ------------------------------------------------------------ tile fetcher
        if (kDynamicTiles<SB_MODE> && lane == 0) {
            for (uint32_t i = 0;; ++i) {
                const uint32_t slot = i % TQ;
                if (!mbar_wait(smem_u32(&sh->tq_empty[slot]), ((i / TQ) & 1) ^ 1, abort, p.status, p.wait_ns)) break;
                int64_t t = (int64_t)blockIdx.x + (int64_t)i * gridDim.x;   // static order
                if (p.tile_next != nullptr && i > 0)
                    t = (int64_t)gridDim.x + (int64_t)atomicAdd(p.tile_next, 1ull);
                sh->tq[slot] = t < total ? t : total;
                mbar_arrive(smem_u32(&sh->tq_full[slot]));   // release: the index is visible to the waiters
                if (t >= total) break;
            }
        }
        __syncwarp();
    }
    } else {
        setmaxnreg_inc<216>();
        // ------------------------------------------------------------ epilogue (8 warps)
        const int ew = warp - 4;
        const int q = warp & 3;          // TMEM lane quarter this warp may access
        const int h = ew >> 2;           // 128-column half of the tile
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        uint32_t kbg = 0, gg = 0;
        bool ok = true;
        // The same tile body under two loops (written out twice: wrapped in a
        // lambda, the body compiled to code 2-3 % slower): the dynamic order
        // takes each index from the ring (lane 0, then a shuffle), the static
        // one computes it.
        if constexpr (kDynamicTiles<SB_MODE>) {
        for (uint32_t ti_i = 0; ok; ++ti_i) {
            int64_t t = 0;
            bool got = true;
            if (lane == 0) {
                got = next_tile(ti_i, t);
                if (got) release_tile(ti_i);
            }
            if (!__shfl_sync(0xFFFFFFFFu, got, 0)) { ok = false; break; }
            t = __shfl_sync(0xFFFFFFFFu, t, 0);
            if (t >= total) break;
            const TileInfo ti = sched_tile<BM, BN>(&sh->sched, p.offsets, p.experts, p.m, n_tiles, t);
            const int64_t row = ti.row0 + 32 * q + lane;
            const int64_t col0 = ti.n0 + 128 * h;
            uint64_t acc[64];   // FP32 pairs: columns (2j, 2j+1) of this thread's 128-column half
#pragma unroll
            for (int j = 0; j < 64; ++j) acc[j] = 0ull;

            for (int64_t kb = 0; kb < nkb; ++kb, ++kbg) {
                const uint32_t g = gg % SRING, kk = (uint32_t)(kb & (SG - 1));
                if (kk == 0) {
                    const bool got_s = mbar_wait(smem_u32(&sh->sfull[g]), (gg / SRING) & 1, abort, p.status, p.wait_ns);
                    if (!__all_sync(0xFFFFFFFFu, got_s)) { ok = false; break; }
                }
                const float fa = sh->sa[g][kk][32 * q + lane];
                const float* sbk = &sh->sb[g][kk][128 * h];
                const uint32_t b = kbg & 1, tph = (kbg >> 1) & 1;
                const bool got = mbar_wait(smem_u32(&sh->tfull[b]), tph, abort, p.status);
                if (!__all_sync(0xFFFFFFFFu, got)) { ok = false; break; }   // tcgen05.ld is .sync.aligned
                tc_fence_after();
                const float fb = (SB_MODE == 1) ? 0.0f : sbk[0];
                const uint64_t f2 = f2_pack(fa * fb, fa * fb);
                const uint64_t fa2 = f2_pack(fa, fa);
                const float4* buf4 = reinterpret_cast<const float4*>(sbk);
                const uint32_t taddr = tmem + lane_base + b * BN + 128 * h;
                // Promote one 16-column chunk held in r: acc += partial * scale.
                auto promote = [&](const uint32_t* r, int c) {
                    if (SB_MODE == 1) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4) {
                            const float4 s4 = buf4[(16 * c + j) >> 2];
                            f2_fma(acc[(16 * c + j) / 2], f2_pack_bits(r[j], r[j + 1]), f2_mul(fa2, f2_pack(s4.x, s4.y)));
                            f2_fma(acc[(16 * c + j) / 2 + 1], f2_pack_bits(r[j + 2], r[j + 3]),
                                   f2_mul(fa2, f2_pack(s4.z, s4.w)));
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 8; ++j) f2_fma(acc[8 * c + j], f2_pack_bits(r[2 * j], r[2 * j + 1]), f2);
                    }
                };
                // Two 16-register staging buffers: the TMEM load of chunk c+1 is
                // in flight while chunk c is promoted.
                uint32_t ra[16], rb[16];
                tmem_ld_32x32b_x16(taddr, ra);
                tmem_ld_wait16(ra);
#pragma unroll
                for (int c = 0; c < 8; c += 2) {
                    tmem_ld_32x32b_x16(taddr + 16 * (c + 1), rb);
                    promote(ra, c);
                    tmem_ld_wait16(rb);
                    if (c + 2 < 8) {
                        tmem_ld_32x32b_x16(taddr + 16 * (c + 2), ra);
                        promote(rb, c + 1);
                        tmem_ld_wait16(ra);
                    } else {
                        // every read of this partial buffer is complete: hand it back to the MMA warp
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[b]));
                        promote(rb, c + 1);
                    }
                }
                if (kk == SG - 1 || kb + 1 == nkb) {
                    // this warp's last read of the scale group: hand the slot back to the loader
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sh->sempty[g]));
                    ++gg;
                }
            }
            if (!ok) break;
            // This warp's 32 rows leave by TMA when they all belong to the
            // tile's row group (always for a dense GEMM; an expert's last,
            // partial row block may end inside them, and the rows after it
            // belong to the next expert).
            if ((p.experts == 0 || ti.row0 + 32 * q + 32 <= ti.row_end) && p.out_f32) {
                // float32 output: the same staging buffer holds 32 rows x 32
                // floats (128-byte rows, same swizzle); four boxes per warp
                uint8_t* ob = ostage + (size_t)ew * OSTAGE_BYTES;
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        float a0, a1, a2, a3;
                        f2_unpack(acc[16 * qq + 2 * c], a0, a1);
                        f2_unpack(acc[16 * qq + 2 * c + 1], a2, a3);
                        *reinterpret_cast<float4*>(ob + lane * 128 + 16 * (c ^ (lane & 7))) = make_float4(a0, a1, a2, a3);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tm_d, smem_u32(ob), (int32_t)(col0 + 32 * qq), (int32_t)(ti.row0 + 32 * q));
                        bulk_commit();
                    }
                }
            } else if (p.experts == 0 || ti.row0 + 32 * q + 32 <= ti.row_end) {
                // BF16 tile rows through this warp's staging buffer (128-byte
                // swizzle: 16-byte chunk j of row r at chunk j ^ (r % 8)), then a
                // TMA store of the 32 x 64 box; the TMA clips rows and columns
                // past the matrix
                uint8_t* ob = ostage + (size_t)ew * OSTAGE_BYTES;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint32_t o[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            float lo, hi;
                            f2_unpack(acc[32 * half + 4 * c + u], lo, hi);
                            __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
                            o[u] = *reinterpret_cast<uint32_t*>(&v);
                        }
                        *reinterpret_cast<uint4*>(ob + lane * 128 + 16 * (c ^ (lane & 7))) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tm_d, smem_u32(ob), (int32_t)(col0 + 64 * half), (int32_t)(ti.row0 + 32 * q));
                        bulk_commit();
                    }
                }
            } else if (row < ti.row_end && p.out_f32) {
                float* drow = reinterpret_cast<float*>(p.d) + row * p.n + col0;
#pragma unroll
                for (int j = 0; j < 128; j += 4) {
                    if (col0 + j < p.n) {
                        float a0, a1, a2, a3;
                        f2_unpack(acc[j / 2], a0, a1);
                        f2_unpack(acc[j / 2 + 1], a2, a3);
                        *reinterpret_cast<float4*>(drow + j) = make_float4(a0, a1, a2, a3);
                    }
                }
            } else if (row < ti.row_end) {
                __nv_bfloat16* drow = p.d + row * p.n + col0;
#pragma unroll
                for (int j = 0; j < 128; j += 8) {
                    if (col0 + j < p.n) {
                        uint4 o;
                        float a0, a1, a2, a3, a4, a5, a6, a7;
                        f2_unpack(acc[j / 2 + 0], a0, a1);
                        f2_unpack(acc[j / 2 + 1], a2, a3);
                        f2_unpack(acc[j / 2 + 2], a4, a5);
                        f2_unpack(acc[j / 2 + 3], a6, a7);
                        __nv_bfloat162 v0 = __floats2bfloat162_rn(a0, a1);
                        __nv_bfloat162 v1 = __floats2bfloat162_rn(a2, a3);
                        __nv_bfloat162 v2 = __floats2bfloat162_rn(a4, a5);
                        __nv_bfloat162 v3 = __floats2bfloat162_rn(a6, a7);
                        o.x = *reinterpret_cast<uint32_t*>(&v0);
                        o.y = *reinterpret_cast<uint32_t*>(&v1);
                        o.z = *reinterpret_cast<uint32_t*>(&v2);
                        o.w = *reinterpret_cast<uint32_t*>(&v3);
                        *reinterpret_cast<uint4*>(drow + j) = o;
                    }
                }
            }
        }
        } else {
        // Static order: the per-column-scale form only (kDynamicTiles).  Its B
        // carries one scale per column and K block, so TMEM is read in the
        // .16x256b shape: thread t holds rows rq, rq + 8, rq + 16, rq + 24 of
        // the warp's 32 (rq = t / 4) and, in each 8-column group of its half,
        // columns cq and cq + 1 (cq = 2 (t % 4)).  It then needs 32 column
        // scales a K block instead of the 128 of a whole row: with one row
        // per thread, the shared loads of the column scales (16 bytes to all
        // 32 lanes per 4 columns) kept the LSU write-back 61 % busy and
        // bounded the K block.
        static_assert(SB_MODE == 1, "the static loop serves the per-column-scale form");
        const int rq = lane >> 2, cq = 2 * (lane & 3);
        for (int64_t t = blockIdx.x; t < total && ok; t += gridDim.x) {
            const TileInfo ti = sched_tile<BM, BN>(&sh->sched, p.offsets, p.experts, p.m, n_tiles, t);
            const int64_t col0 = ti.n0 + 128 * h;
            uint64_t acc[64];   // FP32 pairs: acc[16 ri + g] = row rq + 8 ri, columns 8g + cq, 8g + cq + 1
#pragma unroll
            for (int j = 0; j < 64; ++j) acc[j] = 0ull;

            for (int64_t kb = 0; kb < nkb; ++kb, ++kbg) {
                const uint32_t g = gg % SRING, kk = (uint32_t)(kb & (SG - 1));
                if (kk == 0) {
                    const bool got_s = mbar_wait(smem_u32(&sh->sfull[g]), (gg / SRING) & 1, abort, p.status, p.wait_ns);
                    if (!__all_sync(0xFFFFFFFFu, got_s)) { ok = false; break; }
                }
                uint64_t fa2[4];   // the four rows' A scales, as pairs
#pragma unroll
                for (int ri = 0; ri < 4; ++ri) {
                    const float fa = sh->sa[g][kk][32 * q + rq + 8 * ri];
                    fa2[ri] = f2_pack(fa, fa);
                }
                const float* sbk = &sh->sb[g][kk][128 * h + cq];
                const uint32_t b = kbg & 1, tph = (kbg >> 1) & 1;
                const bool got = mbar_wait(smem_u32(&sh->tfull[b]), tph, abort, p.status);
                if (!__all_sync(0xFFFFFFFFu, got)) { ok = false; break; }   // tcgen05.ld is .sync.aligned
                tc_fence_after();
                const uint32_t taddr = tmem + lane_base + b * BN + 128 * h;
                // chunk k: column groups 4(k/2) .. +3 of lanes 16 (k%2) .. +15 of the quarter
                auto load_chunk = [&](int k, uint32_t* r) {
                    tmem_ld_16x256b_x4(taddr + ((uint32_t)(16 * (k & 1)) << 16) + 32 * (k >> 1), r);
                };
                float2 sc[4];      // column scales of the chunk's four groups
                // acc += partial * s_a * s_b for one chunk held in r
                auto promote = [&](const uint32_t* r, int k) {
                    const int c = k >> 1, hb = k & 1;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint64_t sb2 = f2_pack(sc[j].x, sc[j].y);
#pragma unroll
                        for (int rr = 0; rr < 2; ++rr) {
                            const int ri = 2 * hb + rr;
                            f2_fma(acc[16 * ri + 4 * c + j], f2_pack_bits(r[4 * j + 2 * rr], r[4 * j + 2 * rr + 1]),
                                   f2_mul(fa2[ri], sb2));
                        }
                    }
                };
                uint32_t ra[16], rb[16];
                load_chunk(0, ra);
                tmem_ld_wait16(ra);
#pragma unroll
                for (int k = 0; k < 8; k += 2) {
                    load_chunk(k + 1, rb);
#pragma unroll
                    for (int j = 0; j < 4; ++j) sc[j] = *reinterpret_cast<const float2*>(sbk + 8 * (2 * k + j));
                    promote(ra, k);
                    tmem_ld_wait16(rb);
                    if (k + 2 < 8) {
                        load_chunk(k + 2, ra);
                        promote(rb, k + 1);
                        tmem_ld_wait16(ra);
                    } else {
                        // every read of this partial buffer is complete: hand it back to the MMA warp
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&sh->tempty[b]));
                        promote(rb, k + 1);
                    }
                }
                if (kk == SG - 1 || kb + 1 == nkb) {
                    // this warp's last read of the scale group: hand the slot back to the loader
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sh->sempty[g]));
                    ++gg;
                }
            }
            if (!ok) break;
            if ((p.experts == 0 || ti.row0 + 32 * q + 32 <= ti.row_end) && p.out_f32) {
                // float32 boxes of 32 rows x 32 columns (128-byte rows, 128-byte swizzle)
                uint8_t* ob = ostage + (size_t)ew * OSTAGE_BYTES;
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
#pragma unroll
                    for (int ri = 0; ri < 4; ++ri) {
                        const int lr = rq + 8 * ri;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {   // group 4 qq + j: bytes 32 j + 4 cq of the row
                            float lo, hi;
                            f2_unpack(acc[16 * ri + 4 * qq + j], lo, hi);
                            *reinterpret_cast<float2*>(ob + lr * 128 + 16 * ((2 * j + (cq >> 2)) ^ (lr & 7)) +
                                                       ((4 * cq) & 15)) = make_float2(lo, hi);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tm_d, smem_u32(ob), (int32_t)(col0 + 32 * qq), (int32_t)(ti.row0 + 32 * q));
                        bulk_commit();
                    }
                }
            } else if (p.experts == 0 || ti.row0 + 32 * q + 32 <= ti.row_end) {
                // BF16 boxes of 32 rows x 64 columns (16-byte chunk j of row r at j ^ (r % 8))
                uint8_t* ob = ostage + (size_t)ew * OSTAGE_BYTES;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
#pragma unroll
                    for (int ri = 0; ri < 4; ++ri) {
                        const int lr = rq + 8 * ri;
#pragma unroll
                        for (int j = 0; j < 8; ++j) {   // group 8 half + j: bytes 16 j + 2 cq of the row
                            float lo, hi;
                            f2_unpack(acc[16 * ri + 8 * half + j], lo, hi);
                            __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
                            *reinterpret_cast<uint32_t*>(ob + lr * 128 + 16 * (j ^ (lr & 7)) + 2 * cq) =
                                *reinterpret_cast<uint32_t*>(&v);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tm_d, smem_u32(ob), (int32_t)(col0 + 64 * half), (int32_t)(ti.row0 + 32 * q));
                        bulk_commit();
                    }
                }
            } else {
                // rows of an expert's last, partial row block: direct stores, row by row
#pragma unroll
                for (int ri = 0; ri < 4; ++ri) {
                    const int64_t row = ti.row0 + 32 * q + rq + 8 * ri;
                    if (row >= ti.row_end) continue;
#pragma unroll
                    for (int gq = 0; gq < 16; ++gq) {
                        const int64_t col = col0 + 8 * gq + cq;
                        if (col >= p.n) continue;
                        float lo, hi;
                        f2_unpack(acc[16 * ri + gq], lo, hi);
                        if (p.out_f32) {
                            *reinterpret_cast<float2*>(reinterpret_cast<float*>(p.d) + row * p.n + col) = make_float2(lo, hi);
                        } else {
                            __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
                            *reinterpret_cast<__nv_bfloat162*>(p.d + row * p.n + col) = v;
                        }
                    }
                }
            }
        }
        }
        if (lane == 0) bulk_wait0();   // this warp's output stores are complete
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    // Every fetch of this CTA has returned (the fetcher used its value before
    // the barrier above); the last CTA to get here puts the counter back to 0.
    if (kDynamicTiles<SB_MODE> && p.tile_next != nullptr && threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.tile_done, 1u) == gridDim.x - 1) {
            atomicExch(p.tile_next, 0ull);
            atomicExch(p.tile_done, 0u);
        }
    }
}

template <int SA, int SB>
int launch_typed(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td, const Params& p, int grid,
                 cudaStream_t st) {
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_blockwise_kernel<SA, SB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SMEM_BYTES);
        if (e != cudaSuccess) return (int)e;
        attr_set[dev] = true;
    }
    gemm_blockwise_kernel<SA, SB><<<grid, NUM_THREADS, SMEM_BYTES, st>>>(ta, tb, td, p);
    return (int)cudaGetLastError();
}

int mode_of(int gran) { return gran == 0 ? 0 : (gran == 1 ? 1 : 2); }

}  // namespace

int launch_gemm_blockwise(const GemmJob& j, cudaStream_t st) {
    if (j.experts > kMaxExperts) return -3;
    CUtensorMap ta, tb;
    const uint64_t b_rows = (uint64_t)j.n * (uint64_t)(j.experts > 0 ? j.experts : 1);
    if (!make_tmap_u8(&ta, j.a, (uint64_t)j.k, (uint64_t)j.m, (uint64_t)j.k, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_u8(&tb, j.b, (uint64_t)j.k, b_rows, (uint64_t)j.k, BK, BN, CU_TENSOR_MAP_SWIZZLE_128B))
        return (int)cudaErrorInvalidValue;
    CUtensorMap td;
    const bool td_ok = j.d_f32 ? make_tmap_out_f32(&td, j.d, (uint64_t)j.n, (uint64_t)j.m, (uint64_t)j.n, 32,
                                                   CU_TENSOR_MAP_SWIZZLE_128B)
                               : make_tmap_out_bf16(&td, j.d, (uint64_t)j.n, (uint64_t)j.m, (uint64_t)j.n);
    if (!td_ok) return (int)cudaErrorInvalidValue;
    Params p{};
    p.m = j.m; p.n = j.n; p.k = j.k;
    p.sa = static_cast<const float*>(j.sa);
    p.sb = static_cast<const float*>(j.sb);
    p.d = static_cast<__nv_bfloat16*>(j.d);
    p.status = j.status;
    p.offsets = j.offsets;
    p.experts = j.experts;
    p.wait_ns = j.wait_ns ? j.wait_ns : kWaitLimitNs;
    p.stall_stage0 = j.stall_stage0;
    p.out_f32 = j.d_f32 ? 1 : 0;
    if (j.status != nullptr) {   // the workspace: its tile counter
        char* ws = reinterpret_cast<char*>(j.status);
        p.tile_next = reinterpret_cast<unsigned long long*>(ws + kTileCounterOffset);
        p.tile_done = reinterpret_cast<unsigned int*>(ws + kTileCounterOffset + 8);
    }
    const int sms = sm_count();
    int grid = sms;
    if (j.experts == 0) {
        const int64_t tiles = ceil_div(j.m, BM) * ceil_div(j.n, BN);
        grid = (int)std::min<int64_t>(tiles, sms);
    }
    const int sa = mode_of(j.a_gran), sb = mode_of(j.b_gran);
#define FP8BS_BW_CASE(A, B) \
    if (sa == A && sb == B) return launch_typed<A, B>(ta, tb, td, p, grid, st);
    FP8BS_BW_CASE(1, 2) FP8BS_BW_CASE(1, 1) FP8BS_BW_CASE(1, 0)
    FP8BS_BW_CASE(2, 2) FP8BS_BW_CASE(2, 1) FP8BS_BW_CASE(2, 0)
    FP8BS_BW_CASE(0, 2) FP8BS_BW_CASE(0, 1) FP8BS_BW_CASE(0, 0)
#undef FP8BS_BW_CASE
    return (int)cudaErrorInvalidValue;
}

}  // namespace fp8bs
