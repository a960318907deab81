// gemm_mx.cu -- block-scaled GEMMs on the tensor core's own scale path:
// MXFP8 (E4M3, UE8M0 scale per 32 K-elements) and NVFP4 (E2M1, E4M3 scale
// per 16 K-elements, times the two FP32 tensor scales), dense and MoE
// grouped.
//
// "Low Precision RL", table "Choose a precision": MXFP8 1x32 with UE8M0
// scales and NVFP4 1x16 with two-level (E4M3 + FP32) scales, both Blackwell
// formats; section "2. Unified block-wise FP8": on Blackwell the block-wise
// recipe runs on this path with power-of-two scales (one UE8M0 byte per
// 128-wide K block, replicated over its four 32-wide sub-blocks); section
// "3. Unified MXFP8 (Blackwell)": the MoE GEMM backend is chosen separately
// from the dense one.  Here both are one kernel: a dense
// GEMM is the grouped GEMM with one group.
//
// CTA: 384 threads, one CTA per SM (persistent), tile 128 x 256.
//   warp 0      TMA producer: A 128 x 128 B and B 256 x 128 B boxes per stage
//               (128 FP8 or 256 FP4 K-elements), 128-byte swizzle.
//   warp 1      TMEM owner + MMA issuer: per stage 4 block-scaled MMAs
//               (M128 N256; K32 for MXFP8, K64 for NVFP4), accumulating the
//               whole K range in TMEM; before them the tcgen05.cp of the
//               stage's A scale atoms (NVFP4) or of all its atoms (power of
//               two).
//   warps 2-3   scale loaders: read the row-major scale bytes of a stage's
//               rows and write them in the 32 x 16-byte atom layout that
//               tcgen05.cp 32x128b.warpx4 replicates into all TMEM lane
//               quarters (row r0 + 32*r1 at byte r0*16 + r1*4).  MXFP8 and
//               NVFP4: the two warps take turns by stage and issue the
//               stage's copies themselves (all of them for MXFP8, the B
//               atoms for NVFP4).  Power of two: both warps serve every
//               stage, split by rows, four stages per load.
//   warps 4-11  epilogue: drain the 128 x 256 FP32 accumulator (one row and
//               128 columns per thread) with one TMEM wait, release it,
//               convert to BF16 and store 32 x 32 boxes by TMA through a
//               2 KB staging buffer per warp (float32 output: 32 x 16 boxes).
// TMEM: columns 0..255 accumulator, 256.. scale factors per stage.  Dense
// tiles are walked in groups of row tiles (sched_tile's GM).  One pass per
// tile order and stage ring is shared by the dense and grouped forms.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"
#include "tmap.h"

namespace fp8bs {
namespace {

constexpr int BM = 128, BN = 256, BKB = 128;  // BKB: K bytes per stage and row
constexpr int A_BYTES = BM * BKB, B_BYTES = BN * BKB;
constexpr int NUM_THREADS = 384;
constexpr uint32_t TMEM_COLS = 512;

enum { kMx = 0, kNv = 1, kP2 = 2 };   // MXFP8, NVFP4, block-wise with power-of-two scales

template <int KIND> struct Cfg;
template <> struct Cfg<kMx> {
    static constexpr int STAGES = 4;
    static constexpr int K_PER_STAGE = 128;           // elements
    static constexpr int A_ATOMS = 1, B_ATOMS = 2;    // 512-byte scale atoms per stage
    static constexpr int SF_BYTES_PER_ROW = 4;        // scale bytes per row per stage
};
template <> struct Cfg<kP2> {                     // one UE8M0 byte per 128-wide K block,
    static constexpr int STAGES = 4;              // replicated over its four 32-wide sub-blocks
    static constexpr int K_PER_STAGE = 128;
    static constexpr int A_ATOMS = 1, B_ATOMS = 2;
    static constexpr int SF_BYTES_PER_ROW = 4;
};
template <> struct Cfg<kNv> {
    static constexpr int STAGES = 3;
    static constexpr int K_PER_STAGE = 256;
    static constexpr int A_ATOMS = 4, B_ATOMS = 8;
    static constexpr int SF_BYTES_PER_ROW = 16;
};

// Tile order.  The power-of-two form (the block-wise recipe's fast path,
// whose dense GEMMs the step runs concurrently) takes its tiles dynamically:
// the producer claims each next tile from a counter in the workspace
// (atomicAdd, one tile ahead) and publishes the indices through a small
// shared-memory ring that the MMA thread, the scale loaders and the
// epilogue read; the last CTA to finish puts the counter back to 0.  The
// MXFP8 and NVFP4 forms keep the static order blockIdx.x + i * gridDim.x.
template <int KIND> constexpr bool kDynMx = KIND == kP2;
constexpr int MX_TQ = 4;           // tile indices in flight (how far the producer may run ahead)
constexpr int MX_TQ_READERS = 11;  // MMA thread, two scale loaders, eight epilogue warps

struct Params {
    int64_t m, n, k;
    const uint8_t* sa;   // row-major scale bytes [m, k / vec]
    const uint8_t* sb;   // [experts * n, k / vec]
    const float* a_ts;   // NVFP4 outer scales: [1], or [m] when a_ts_rows
    const float* b_ts;   // [1], or [experts] for a grouped GEMM
    int a_ts_rows;
    __nv_bfloat16* d;
    int* status;
    const int64_t* offsets;
    int experts;
    uint64_t wait_ns;     // bound of every pipeline wait
    int stall_stage0;     // test hook: the producer withholds stage 0
    unsigned long long* tile_next;   // tiles handed out past the first wave (dynamic order)
    unsigned int* tile_done;         // CTAs finished
};

// Dense tile order: groups of row tiles, row tile fastest inside a group.
// NVFP4 takes 16 (its 906 MB of D otherwise pushes W out of L2 between
// waves: 1.049 -> 0.979 ms), the FP8 kinds 8 (power-of-two fprop
// 0.169 -> 0.157 ms).  The blockwise kernel measured slower with it.
template <int KIND> constexpr int kTileGroupM = (KIND == kNv) ? 16 : 8;

template <int STAGES>
struct alignas(16) Shared {
    uint64_t full[STAGES], empty[STAGES], tfull, tempty, drain;
    uint64_t ldrain[2];    // per scale loader: its scale copies have landed (exit path)
    uint64_t tq_full[MX_TQ], tq_empty[MX_TQ];
    int64_t tq[MX_TQ];     // tile index ring (dynamic order; an index >= total ends the work)
    uint32_t tmem_base;
    int abort;
    SchedShared sched;
};

// Stage = A tile | B tile | scale atoms, rounded up to 1024 bytes so that
// every tile starts on a 128-byte-swizzle atom boundary.
template <int KIND>
constexpr size_t stage_bytes() {
    return ((size_t)A_BYTES + B_BYTES + 512u * (Cfg<KIND>::A_ATOMS + Cfg<KIND>::B_ATOMS) + 1023) & ~size_t(1023);
}
// Per epilogue warp: 32 rows x 32 BF16 columns for a TMA store (64-byte swizzle).
constexpr int OSTAGE_BYTES = 32 * 64;
template <int STAGES>
constexpr size_t shared_bytes_aligned() { return (sizeof(Shared<STAGES>) + 1023) & ~size_t(1023); }
template <int KIND>
constexpr size_t smem_bytes() {
    return 1024 + Cfg<KIND>::STAGES * stage_bytes<KIND>() + shared_bytes_aligned<Cfg<KIND>::STAGES>() +
           8 * OSTAGE_BYTES;
}
static_assert(smem_bytes<kMx>() <= 232448 && smem_bytes<kP2>() <= 232448 && smem_bytes<kNv>() <= 232448,
              "shared memory per CTA");

// Scale words of one stage for one lane: A rows r0 + 32*r1 (r1 < 4) and B rows
// r0 + 32*r1 (r1 < 8); MXFP8 one 32-bit word per row, NVFP4 four.
template <int KIND>
struct ScaleRegs {
    static constexpr int W = Cfg<KIND>::SF_BYTES_PER_ROW / 4;
    uint32_t a[4][W];
    uint32_t b[8][W];
};

template <int KIND, int SA, int SB>
__device__ __forceinline__ void load_scales(ScaleRegs<KIND>& r, const Params& p, const TileInfo& ti, int64_t kb,
                                            int lane, int64_t sf_pitch) {
    constexpr int W = ScaleRegs<KIND>::W;
    static_assert(KIND != kP2, "power-of-two scales use load_scales_group");
    const int64_t koff = kb * Cfg<KIND>::SF_BYTES_PER_ROW;
#pragma unroll
    for (int r1 = 0; r1 < 4; ++r1) {
        const int64_t row = ti.row0 + lane + 32 * r1;
        const bool ok = row < p.m;
        const uint8_t* src = p.sa + row * sf_pitch + koff;
        if (W == 1) {
            r.a[r1][0] = ok ? __ldg(reinterpret_cast<const uint32_t*>(src)) : 0u;
        } else {
            const uint4 v = ok ? __ldg(reinterpret_cast<const uint4*>(src)) : make_uint4(0, 0, 0, 0);
            r.a[r1][0] = v.x; r.a[r1][1 % W] = v.y; r.a[r1][2 % W] = v.z; r.a[r1][3 % W] = v.w;
        }
    }
    const int64_t brow0 = (int64_t)ti.expert * p.n + ti.n0;
#pragma unroll
    for (int r1 = 0; r1 < 8; ++r1) {
        const int64_t n = ti.n0 + lane + 32 * r1;
        const bool ok = n < p.n;
        const uint8_t* src = p.sb + (brow0 + lane + 32 * r1) * sf_pitch + koff;
        if (W == 1) {
            r.b[r1][0] = ok ? __ldg(reinterpret_cast<const uint32_t*>(src)) : 0u;
        } else {
            const uint4 v = ok ? __ldg(reinterpret_cast<const uint4*>(src)) : make_uint4(0, 0, 0, 0);
            r.b[r1][0] = v.x; r.b[r1][1 % W] = v.y; r.b[r1][2 % W] = v.z; r.b[r1][3 % W] = v.w;
        }
    }
}

// Write one stage's scales into the tcgen05.cp atom layout.  Atom j of A
// holds the j-th scale word of every row (MXFP8: j = 0 only); B atoms are
// ordered (j, 128-row chunk).
template <int KIND>
__device__ __forceinline__ void store_scales(const ScaleRegs<KIND>& r, uint8_t* sf, int lane) {
    constexpr int W = ScaleRegs<KIND>::W;
#pragma unroll
    for (int j = 0; j < W; ++j) {
        *reinterpret_cast<uint4*>(sf + j * 512 + lane * 16) = make_uint4(r.a[0][j], r.a[1][j], r.a[2][j], r.a[3][j]);
    }
    uint8_t* sfb = sf + Cfg<KIND>::A_ATOMS * 512;
#pragma unroll
    for (int j = 0; j < W; ++j) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            *reinterpret_cast<uint4*>(sfb + (j * 2 + c) * 512 + lane * 16) =
                make_uint4(r.b[4 * c + 0][j], r.b[4 * c + 1][j], r.b[4 * c + 2][j], r.b[4 * c + 3][j]);
        }
    }
}

// Power-of-two scales, four stages at a time: word g of a row slot holds
// the byte of stage kb0 + g, replicated to the four 32-wide sub-blocks.  One
// 4-byte load per row covers the four stages when the row pitch and base
// allow it; per-stage byte loads would cost one 32-sector request per row
// slot and stage (the rows of a stage are 32 apart).  (MXFP8 keeps the
// per-stage loader: 16-byte groups measured slower there, partly because
// the MoE down projection's 24-byte rows rule them out.)
constexpr int kSfGroup = 4;
struct WideRegs {
    uint32_t a[4][kSfGroup];
    uint32_t b[8][kSfGroup];
};

__device__ __forceinline__ void load_row_group(uint32_t* w, const uint8_t* __restrict__ src, int64_t kb0, int64_t nkb,
                                               bool ok, bool vec) {
    if (!ok) {
#pragma unroll
        for (int g = 0; g < kSfGroup; ++g) w[g] = 0u;
        return;
    }
    const uint8_t* p = src + kb0;
    if (kb0 + kSfGroup <= nkb) {
        uint32_t v;
        if (vec) {
            v = __ldg(reinterpret_cast<const uint32_t*>(p));
        } else {
            // row pitch not a multiple of 4: the aligned word holding p, and
            // the next one only when p is not aligned (it then holds p[3], a
            // byte of this group, so the read stays inside the words that
            // hold the tensor)
            const uintptr_t ap = reinterpret_cast<uintptr_t>(p);
            const uint32_t* q = reinterpret_cast<const uint32_t*>(ap & ~static_cast<uintptr_t>(3));
            const uint32_t sh = 8u * static_cast<uint32_t>(ap & 3u);
            const uint32_t w0 = __ldg(q);
            v = sh != 0u ? __funnelshift_r(w0, __ldg(q + 1), sh) : w0;
        }
#pragma unroll
        for (int g = 0; g < kSfGroup; ++g) w[g] = ((v >> (8 * g)) & 0xFFu) * 0x01010101u;
    } else {
#pragma unroll
        for (int g = 0; g < kSfGroup; ++g) w[g] = (kb0 + g < nkb) ? (uint32_t)__ldg(p + g) * 0x01010101u : 0u;
    }
}

// SA / SB: 1 = one byte per row, 2 = one byte per 128-row block.
// part: which of the two loaders (the split of the rows is store_scales_p2's).
template <int SA, int SB>
__device__ __forceinline__ void load_scales_group(WideRegs& w, const Params& p, const TileInfo& ti, int64_t kb0,
                                                  int64_t nkb, int lane, int64_t sf_pitch, bool vec, int part) {
    const int64_t nb_e = (p.n + 127) / 128;
    auto brow = [&](int r1) {
        const int64_t n = ti.n0 + lane + 32 * r1;
        const int64_t srow = (SB == 2) ? (int64_t)ti.expert * nb_e + (n >> 7) : (int64_t)ti.expert * p.n + n;
        load_row_group(w.b[r1], p.sb + srow * sf_pitch, kb0, nkb, n < p.n, vec);
    };
    // 128x128 blocks of B: a tile (256 rows from a multiple of 256) covers two
    // blocks, rows 0..127 and 128..255, so one load per block serves its four
    // row slots (rows past n read 0, and a block that starts past n is not read)
    auto bblock = [&](int c) {
        const int64_t nb = ti.n0 + 128 * c;
        load_row_group(w.b[4 * c], p.sb + ((int64_t)ti.expert * nb_e + (nb >> 7)) * sf_pitch, kb0, nkb, nb < p.n, vec);
#pragma unroll
        for (int r1 = 1; r1 < 4; ++r1) {
            const bool in = ti.n0 + 128 * c + lane + 32 * r1 < p.n;
#pragma unroll
            for (int g = 0; g < kSfGroup; ++g) w.b[4 * c + r1][g] = in ? w.b[4 * c][g] : 0u;
        }
        if (ti.n0 + 128 * c + lane >= p.n) {
#pragma unroll
            for (int g = 0; g < kSfGroup; ++g) w.b[4 * c][g] = 0u;
        }
    };
    auto arow = [&](int r1) {
        const int64_t row = ti.row0 + lane + 32 * r1;
        const int64_t srow = (SA == 2) ? (row >> 7) : row;
        load_row_group(w.a[r1], p.sa + srow * sf_pitch, kb0, nkb, row < p.m, vec);
    };
    // The two loaders take six row words each (per-row B scales) or two A
    // rows and one B block each (128x128 B blocks): see store_scales_p2.
    // (every register index a constant: a run-time index would put the
    // register buffers in local memory)
    if constexpr (SB == 2) {
        if (part == 0) {
            arow(0);
            arow(1);
            bblock(0);
        } else {
            arow(2);
            arow(3);
            bblock(1);
        }
    } else if (part == 0) {
#pragma unroll
        for (int r1 = 0; r1 < 4; ++r1) arow(r1);
        brow(0);
        brow(1);
    } else {
#pragma unroll
        for (int r1 = 2; r1 < 8; ++r1) brow(r1);
    }
}

// One loader's share of a stage's atoms (power-of-two scales: one word per
// row; lane l's 16 bytes of an atom hold rows l, l+32, l+64, l+96).  With
// per-row B scales part 0 writes the A atom and rows l, l+32 of the first B
// atom, part 1 the rest of the B atoms; with 128x128 B blocks each part
// writes half of the A atom and one B atom.  Six loads or three a lane each.
template <int KIND, int SB>
__device__ __forceinline__ void store_scales_p2(const ScaleRegs<KIND>& r, uint8_t* sf, int lane, int part) {
    uint8_t* sfb = sf + Cfg<KIND>::A_ATOMS * 512;
    if constexpr (SB == 2) {
        if (part == 0) {
            *reinterpret_cast<uint2*>(sf + lane * 16) = make_uint2(r.a[0][0], r.a[1][0]);
            *reinterpret_cast<uint4*>(sfb + lane * 16) = make_uint4(r.b[0][0], r.b[1][0], r.b[2][0], r.b[3][0]);
        } else {
            *reinterpret_cast<uint2*>(sf + lane * 16 + 8) = make_uint2(r.a[2][0], r.a[3][0]);
            *reinterpret_cast<uint4*>(sfb + 512 + lane * 16) = make_uint4(r.b[4][0], r.b[5][0], r.b[6][0], r.b[7][0]);
        }
    } else if (part == 0) {
        *reinterpret_cast<uint4*>(sf + lane * 16) = make_uint4(r.a[0][0], r.a[1][0], r.a[2][0], r.a[3][0]);
        *reinterpret_cast<uint2*>(sfb + lane * 16) = make_uint2(r.b[0][0], r.b[1][0]);
    } else {
        *reinterpret_cast<uint2*>(sfb + lane * 16 + 8) = make_uint2(r.b[2][0], r.b[3][0]);
        *reinterpret_cast<uint4*>(sfb + 512 + lane * 16) = make_uint4(r.b[4][0], r.b[5][0], r.b[6][0], r.b[7][0]);
    }
}

template <int KIND>
__device__ __forceinline__ void group_stage(ScaleRegs<KIND>& r, const WideRegs& w, int g) {
#pragma unroll
    for (int r1 = 0; r1 < 4; ++r1) r.a[r1][0] = w.a[r1][g];
#pragma unroll
    for (int r1 = 0; r1 < 8; ++r1) r.b[r1][0] = w.b[r1][g];
}

// Copy a stage's scale atoms from shared memory into its TMEM columns
// (tcgen05.cp 32x128b.warpx4, one per 512-byte atom: A atoms first, then B).
// One copy takes about 60 cycles to issue, and the serial work of the MMA
// thread and of the loaders per stage bounds these kernels, so the copies
// are split where there is slack.  The loader that wrote a stage's atoms
// issues its share and commits it to the stage's full barrier (arrives once
// they have landed); the MMA thread issues the rest just before its MMAs.
//   MXFP8 (3 copies a stage): all by the loaders (idle half the time);
//   NVFP4 (12): the 8 B atoms by the loaders, the 4 A atoms by the MMA
//   thread (both were near saturation with all 12 on one side);
//   power of two (3): all by the MMA thread (its row-split loaders are busy).
template <int KIND> constexpr int kLoaderCopyFirst = (KIND == kMx) ? 0 : (KIND == kNv ? Cfg<KIND>::A_ATOMS
                                                                                      : Cfg<KIND>::A_ATOMS + Cfg<KIND>::B_ATOMS);
template <int KIND> constexpr bool kLoaderCopies = kLoaderCopyFirst<KIND> < Cfg<KIND>::A_ATOMS + Cfg<KIND>::B_ATOMS;

// Atoms [J0, J1) of a stage.
template <int KIND, int J0, int J1>
__device__ __forceinline__ void copy_scales_to_tmem(uint32_t sf_tmem, uint32_t sf_smem) {
#pragma unroll
    for (int j = J0; j < J1; ++j) tmem_cp_32x128b_x4(sf_tmem + 4 * j, smem_desc(sf_smem + 512 * j, 0, 128, 0));
}

// Before a loader warp exits, its last scale copies must have landed (on an
// aborted run the MMA thread may not have waited for them).
__device__ __forceinline__ void drain_scale_copies(uint32_t bar, int lane, uint64_t limit_ns) {
    if (lane == 0) {
        mma_commit(bar);
        mbar_wait_drain(bar, 0, limit_ns);
    }
    __syncwarp();
}

// F32: D is float32 (tm_d then maps float32 32 x 16 boxes); a template
// parameter rather than a run-time flag, since the extra epilogue branch
// cost the short-K grouped GEMMs a few per cent.
template <int KIND, int SA, int SB, bool F32>
__global__ void __launch_bounds__(NUM_THREADS, 1)
gemm_mx_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ CUtensorMap tm_d, Params p) {
    constexpr int STAGES = Cfg<KIND>::STAGES;
    constexpr size_t STAGE_B = stage_bytes<KIND>();
    constexpr uint32_t SF_COLS = 4 * (Cfg<KIND>::A_ATOMS + Cfg<KIND>::B_ATOMS);  // TMEM columns per stage
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Shared<STAGES>* sh = reinterpret_cast<Shared<STAGES>*>(stages + STAGES * STAGE_B);
    uint8_t* ostage = stages + STAGES * STAGE_B + shared_bytes_aligned<STAGES>();   // 1024-aligned

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nkb = p.k / Cfg<KIND>::K_PER_STAGE;
    const int64_t n_tiles = (p.n + BN - 1) / BN;
    const int64_t sf_pitch = p.k / (KIND == kMx ? 32 : (KIND == kNv ? 16 : 128));

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // TMA bytes + scale loader(s); NVFP4: the loader's plain arrive (it releases the
            // atoms the MMA thread copies) and its commit of the copies it issues
            mbar_init(smem_u32(&sh->full[s]), (KIND == kP2 || KIND == kNv) ? 3 : 2);
            mbar_init(smem_u32(&sh->empty[s]), 1);
        }
        mbar_init(smem_u32(&sh->tfull), 1);
        mbar_init(smem_u32(&sh->tempty), 8);
        mbar_init(smem_u32(&sh->drain), 1);
        mbar_init(smem_u32(&sh->ldrain[0]), 1);
        mbar_init(smem_u32(&sh->ldrain[1]), 1);
        for (int i = 0; i < MX_TQ; ++i) {
            mbar_init(smem_u32(&sh->tq_full[i]), 1);
            mbar_init(smem_u32(&sh->tq_empty[i]), MX_TQ_READERS);
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
    const int64_t total = sched_setup<BM>(&sh->sched, p.offsets, p.experts, p.m, n_tiles, p.status);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh->tmem_base;
    volatile int* abort = &sh->abort;
    // The i-th tile of this CTA: the static order, or the ring's i-th index,
    // read and released by the calling thread (tile_one) or by lane 0 and
    // handed to the whole warp (tile_of).  false: a wait gave up.
    auto tile_one = [&](uint32_t i, int64_t& t) -> bool {
        if constexpr (!kDynMx<KIND>) {
            t = (int64_t)blockIdx.x + (int64_t)i * gridDim.x;
            return true;
        }
        const uint32_t slot = i % MX_TQ;
        if (!mbar_wait(smem_u32(&sh->tq_full[slot]), (i / MX_TQ) & 1, abort, p.status, p.wait_ns)) return false;
        t = sh->tq[slot];
        mbar_arrive(smem_u32(&sh->tq_empty[slot]));
        return true;
    };
    auto tile_of = [&](uint32_t i, int64_t& t) -> bool {
        if constexpr (!kDynMx<KIND>) {
            t = (int64_t)blockIdx.x + (int64_t)i * gridDim.x;
            return true;
        }
        bool got = true;
        int64_t v = 0;
        if (lane == 0) got = tile_one(i, v);
        t = __shfl_sync(0xFFFFFFFFu, v, 0);
        return __shfl_sync(0xFFFFFFFFu, got, 0);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t it = 0;
            bool ok = true;
            // Dynamic order: round i's index is published while round i-1's
            // tile is being loaded, right after it was claimed, so every reader
            // finds it there before it needs it.  The index past the last tile
            // (total) is published once and ends every role's loop.
            auto publish = [&](uint32_t i, int64_t v) -> bool {
                const uint32_t slot = i % MX_TQ;
                if (!mbar_wait(smem_u32(&sh->tq_empty[slot]), ((i / MX_TQ) & 1) ^ 1, abort, p.status, p.wait_ns))
                    return false;
                sh->tq[slot] = v < total ? v : total;
                mbar_arrive(smem_u32(&sh->tq_full[slot]));
                return true;
            };
            int64_t cur = blockIdx.x;
            if constexpr (kDynMx<KIND>) ok = publish(0, cur);
            for (uint32_t ti_i = 0; ok; ++ti_i) {
                const int64_t t = cur;
                if (t >= total) break;
                cur = t + gridDim.x;
                if constexpr (kDynMx<KIND>) {
                    if (p.tile_next != nullptr) cur = (int64_t)gridDim.x + (int64_t)atomicAdd(p.tile_next, 1ull);
                    if (!publish(ti_i + 1, cur)) { ok = false; break; }
                }
                const TileInfo ti = sched_tile<BM, BN, kTileGroupM<KIND>>(&sh->sched, p.offsets, p.experts, p.m, n_tiles, t);
                const int32_t brow = (int32_t)(ti.expert * p.n + ti.n0);
                for (int64_t kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    if (!mbar_wait(smem_u32(&sh->empty[s]), ph ^ 1, abort, p.status, p.wait_ns)) { ok = false; break; }
                    if (p.stall_stage0 && it == 0) continue;   // test hook: never fill stage 0
                    const uint32_t fb = smem_u32(&sh->full[s]);
                    uint8_t* st = stages + s * STAGE_B;
                    mbar_arrive_expect_tx(fb, A_BYTES + B_BYTES);
                    tma_load_2d(smem_u32(st), &tm_a, fb, (int32_t)(kb * BKB), (int32_t)ti.row0);
                    tma_load_2d(smem_u32(st + A_BYTES), &tm_b, fb, (int32_t)(kb * BKB), brow);
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
            uint32_t it = 0, tcount = 0;
            bool ok = true;
            for (uint32_t ti_i = 0; ok; ++ti_i, ++tcount) {
                int64_t t;
                if (!tile_one(ti_i, t)) { ok = false; break; }
                if (t >= total) break;
                if (!mbar_wait(smem_u32(&sh->tempty), (tcount & 1) ^ 1, abort, p.status, p.wait_ns)) { ok = false; break; }
                tc_fence_after();
                for (int64_t kb = 0; kb < nkb; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    if (!mbar_wait(smem_u32(&sh->full[s]), ph, abort, p.status, p.wait_ns)) { ok = false; break; }
                    tc_fence_after();
                    uint8_t* st = stages + s * STAGE_B;
                    const uint32_t a_addr = smem_u32(st);
                    const uint64_t adesc = kmajor_sw128_desc(a_addr);
                    const uint64_t bdesc = kmajor_sw128_desc(a_addr + A_BYTES);
                    const uint32_t sfa = tmem + 256 + s * SF_COLS;
                    const uint32_t sfb = sfa + 4 * Cfg<KIND>::A_ATOMS;
                    copy_scales_to_tmem<KIND, 0, kLoaderCopyFirst<KIND>>(sfa, a_addr + A_BYTES + B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint32_t acc = (kb > 0 || kk > 0) ? 1u : 0u;
                        if constexpr (KIND != kNv) {
                            const uint32_t idesc = idesc_block_scaled(BM, BN, 0, 0, 1, kk, kk);
                            mma_mxf8(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, sfa, sfb, acc);
                        } else {
                            const uint32_t idesc = idesc_block_scaled(BM, BN, 1, 1, 0, 0, 0);
                            mma_nvf4(tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc, sfa + 4 * kk, sfb + 8 * kk, acc);
                        }
                    }
                    mma_commit(smem_u32(&sh->empty[s]));
                }
                if (!ok) break;
                mma_commit(smem_u32(&sh->tfull));
            }
            mma_commit(smem_u32(&sh->drain));
            mbar_wait(smem_u32(&sh->drain), 0, abort, p.status);
        }
        __syncwarp();
    } else if ((warp == 2 || warp == 3) && KIND == kP2) {
        // ------------------------------------------------------------ scale loaders (power of two)
        // Both warps walk every stage in order and split the rows evenly
        // (store_scales_p2; the stage's full barrier counts both).  Groups of four stages are
        // loaded one group ahead of the one being written out (two register
        // buffers, the loop unrolled by two so both names are constants).
        const int part = warp - 2;
        const bool vec = (sf_pitch & 3) == 0 && ((reinterpret_cast<uintptr_t>(p.sa) | reinterpret_cast<uintptr_t>(p.sb)) & 3u) == 0;
        // Load cursor: the tile's round, index and layout, and the first
        // stage of the group.  A tile's index is read when its first group is
        // loaded, not when the previous tile's last one is (the groups of that
        // tile still to be written out must not wait on the next index).
        uint32_t lt_i = 0;
        int64_t lt = 0, lkb0 = 0;
        bool lneed = true;
        TileInfo lti{};
        auto load_next = [&](WideRegs& w, int64_t& kb0_out) -> bool {
            if (lneed) {
                lneed = false;
                if (!tile_of(lt_i, lt)) lt = total;       // a wait gave up: the abort flag ends the rest
                if (lt < total) lti = sched_tile<BM, BN, kTileGroupM<KIND>>(&sh->sched, p.offsets, p.experts, p.m, n_tiles, lt);
            }
            if (lt >= total) return false;
            load_scales_group<SA, SB>(w, p, lti, lkb0, nkb, lane, sf_pitch, vec, part);
            kb0_out = lkb0;
            lkb0 += kSfGroup;
            if (lkb0 >= nkb) {
                lkb0 = 0;
                ++lt_i;
                lneed = true;
            }
            return true;
        };
        uint32_t it = 0;
        bool ok = true;
        auto store_group = [&](const WideRegs& w, int64_t kb0) {
#pragma unroll
            for (int g = 0; g < kSfGroup; ++g) {
                if (!ok || kb0 + g >= nkb) break;
                const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                if (!mbar_wait(smem_u32(&sh->empty[s]), ph ^ 1, abort, p.status, p.wait_ns)) { ok = false; break; }
                ScaleRegs<KIND> r;
                group_stage<KIND>(r, w, g);
                store_scales_p2<KIND, SB>(r, stages + s * STAGE_B + A_BYTES + B_BYTES, lane, part);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh->full[s]));
                ++it;
            }
        };
        WideRegs w0, w1;
        int64_t k0 = 0, k1 = 0;
        bool h0 = load_next(w0, k0), h1 = load_next(w1, k1);
        while (h0 && ok) {
            store_group(w0, k0);
            h0 = load_next(w0, k0);
            if (!h1 || !ok) break;
            store_group(w1, k1);
            h1 = load_next(w1, k1);
            if (!h0) break;
        }
    } else if (warp == 2 || warp == 3) {
        // ------------------------------------------------------------ scale loaders (MXFP8, NVFP4)
        if constexpr (KIND != kP2) {
            // Two warps take turns by stage (warp 2 the even stages, warp 3 the
            // odd ones).  Each keeps a load cursor SF_PD of its stages ahead of
            // its store cursor; the loaded words wait in a register ring (slot
            // = stage mod SF_PD, the loop unrolled so every slot index is a
            // constant), which keeps the L2 latency of the scale loads off the
            // per-stage path.
            constexpr int SF_PD = (KIND == kNv) ? 2 : 4;   // NVFP4 stages carry 4x the scale words
            ScaleRegs<KIND> ring[SF_PD];
            int64_t lt = blockIdx.x, lkb = 0;                 // load cursor
            TileInfo lti{};
            if (lt < total) lti = sched_tile<BM, BN, kTileGroupM<KIND>>(&sh->sched, p.offsets, p.experts, p.m, n_tiles, lt);
            auto step_load = [&]() {
                if (++lkb == nkb) {
                    lkb = 0;
                    lt += gridDim.x;
                    if (lt < total) lti = sched_tile<BM, BN, kTileGroupM<KIND>>(&sh->sched, p.offsets, p.experts, p.m, n_tiles, lt);
                }
            };
            int64_t st_t = blockIdx.x, st_kb = 0;           // store cursor
            auto step_store = [&]() {
                if (++st_kb == nkb) {
                    st_kb = 0;
                    st_t += gridDim.x;
                }
            };
            uint32_t it = (uint32_t)(warp - 2);
            if (warp == 3) {
                step_load();
                step_store();
            }
#pragma unroll
            for (int d = 0; d < SF_PD; ++d) {
                if (lt < total) {
                    load_scales<KIND, SA, SB>(ring[d], p, lti, lkb, lane, sf_pitch);
                    step_load();
                    if (lt < total) step_load();
                }
            }
            bool ok = true;
            while (st_t < total && ok) {
#pragma unroll
                for (int d = 0; d < SF_PD; ++d) {
                    if (st_t >= total || !ok) break;
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
                    if (!mbar_wait(smem_u32(&sh->empty[s]), ph ^ 1, abort, p.status, p.wait_ns)) { ok = false; break; }
                    uint8_t* sf = stages + s * STAGE_B + A_BYTES + B_BYTES;
                    store_scales<KIND>(ring[d], sf, lane);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if constexpr (kLoaderCopies<KIND>) {
                            if constexpr (kLoaderCopyFirst<KIND> > 0) mbar_arrive(smem_u32(&sh->full[s]));
                            copy_scales_to_tmem<KIND, kLoaderCopyFirst<KIND>, Cfg<KIND>::A_ATOMS + Cfg<KIND>::B_ATOMS>(
                                tmem + 256 + s * SF_COLS, smem_u32(sf));
                            mma_commit(smem_u32(&sh->full[s]));
                        } else {
                            mbar_arrive(smem_u32(&sh->full[s]));
                        }
                    }
                    it += 2;
                    if (lt < total) {
                        load_scales<KIND, SA, SB>(ring[d], p, lti, lkb, lane, sf_pitch);
                        step_load();
                        if (lt < total) step_load();
                    }
                    step_store();
                    if (st_t < total) step_store();
                }
            }
            if constexpr (kLoaderCopies<KIND>) drain_scale_copies(smem_u32(&sh->ldrain[warp - 2]), lane, p.wait_ns);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue (8 warps)
        const int q = warp & 3, h = (warp - 4) >> 2;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        // NVFP4: D = acc * S_g(A) * S_g(B), with S_g(A) per tensor or per row and
        // S_g(B) per expert (one value for a dense GEMM)
        float g = 1.0f;
        uint32_t tcount = 0;
        for (uint32_t ti_i = 0;; ++ti_i, ++tcount) {
            int64_t t;
            if (!tile_of(ti_i, t)) break;
            if (t >= total) break;
            const TileInfo ti = sched_tile<BM, BN, kTileGroupM<KIND>>(&sh->sched, p.offsets, p.experts, p.m, n_tiles, t);
            const int64_t row = ti.row0 + 32 * q + lane;
            if (KIND == kNv) {
                const float gb = __ldg(p.b_ts + ti.expert);
                if (p.a_ts_rows) g = (row < ti.row_end) ? __ldg(p.a_ts + row) * gb : 0.0f;
                else g = __ldg(p.a_ts) * gb;
            }
            const bool got = mbar_wait(smem_u32(&sh->tfull), tcount & 1, abort, p.status);
            if (!__all_sync(0xFFFFFFFFu, got)) break;   // warp-uniform: tcgen05.ld is .sync.aligned
            tc_fence_after();
            // All four loads in flight, one wait, then the accumulator goes back
            // to the MMA thread before any conversion: with one accumulator
            // buffer the next tile's MMAs start only after this drain.
            uint32_t r[128];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(tmem + lane_base + 128 * h + 32 * c, r + 32 * c);
            tmem_ld_wait(r);
            tmem_ld_wait(r + 32);
            tmem_ld_wait(r + 64);
            tmem_ld_wait(r + 96);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh->tempty));
            const int64_t col0 = ti.n0 + 128 * h;
            if constexpr (F32) {
                // float32 output: 32 rows x 16 floats per box (64-byte rows,
                // the same swizzle and staging buffer as the BF16 boxes)
#pragma unroll
                for (int j = 0; j < 128; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * g);
                if (p.experts == 0 || ti.row0 + 32 * q + 32 <= ti.row_end) {
                    uint8_t* ob = ostage + (warp - 4) * OSTAGE_BYTES;
#pragma unroll
                    for (int qb = 0; qb < 8; ++qb) {
                        if (lane == 0) bulk_wait_read0();
                        __syncwarp();
#pragma unroll
                        for (int c = 0; c < 4; ++c)
                            *reinterpret_cast<uint4*>(ob + lane * 64 + 16 * (c ^ ((lane >> 1) & 3))) =
                                make_uint4(r[16 * qb + 4 * c], r[16 * qb + 4 * c + 1], r[16 * qb + 4 * c + 2],
                                           r[16 * qb + 4 * c + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tm_d, smem_u32(ob), (int32_t)(col0 + 16 * qb), (int32_t)(ti.row0 + 32 * q));
                            bulk_commit();
                        }
                    }
                } else if (row < ti.row_end) {
                    float* drow = reinterpret_cast<float*>(p.d) + row * p.n + col0;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (col0 + 4 * j < p.n)
                            *reinterpret_cast<uint4*>(drow + 4 * j) =
                                make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                    }
                }
                continue;
            }
            uint32_t packed[64];
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(r[2 * j]) * g, __uint_as_float(r[2 * j + 1]) * g);
                packed[j] = *reinterpret_cast<uint32_t*>(&v);
            }
            if (p.experts == 0 || ti.row0 + 32 * q + 32 <= ti.row_end) {
                // The warp's 32 rows all belong to the tile's row group: out by
                // TMA, 32 columns at a time through the warp's staging buffer
                // (64-byte swizzle: 16-byte chunk c of row r at c ^ ((r >> 1) & 3));
                // the TMA clips rows and columns past the matrix.
                uint8_t* ob = ostage + (warp - 4) * OSTAGE_BYTES;
#pragma unroll
                for (int qb = 0; qb < 4; ++qb) {
                    if (lane == 0) bulk_wait_read0();
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        *reinterpret_cast<uint4*>(ob + lane * 64 + 16 * (c ^ ((lane >> 1) & 3))) =
                            make_uint4(packed[16 * qb + 4 * c], packed[16 * qb + 4 * c + 1],
                                       packed[16 * qb + 4 * c + 2], packed[16 * qb + 4 * c + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tm_d, smem_u32(ob), (int32_t)(col0 + 32 * qb), (int32_t)(ti.row0 + 32 * q));
                        bulk_commit();
                    }
                }
            } else if (row < ti.row_end) {
                // an expert's last row block ends inside this warp's rows
                __nv_bfloat16* drow = p.d + row * p.n + col0;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    if (col0 + 8 * j < p.n)
                        *reinterpret_cast<uint4*>(drow + 8 * j) =
                            make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
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
    // Every claim of this CTA has returned (the producer used its value
    // before the barrier above); the last CTA to get here resets the counter.
    if (kDynMx<KIND> && p.tile_next != nullptr && threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.tile_done, 1u) == gridDim.x - 1) {
            atomicExch(p.tile_next, 0ull);
            atomicExch(p.tile_done, 0u);
        }
    }
}

template <int KIND, int SA, int SB, bool F32>
int launch_typed(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td, const Params& p, int grid,
                 cudaStream_t st) {
    static bool attr_set[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(gemm_mx_kernel<KIND, SA, SB, F32>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<KIND>());
        if (e != cudaSuccess) return (int)e;
        attr_set[dev] = true;
    }
    gemm_mx_kernel<KIND, SA, SB, F32><<<grid, NUM_THREADS, smem_bytes<KIND>(), st>>>(ta, tb, td, p);
    return (int)cudaGetLastError();
}

template <int KIND, int SA = 0, int SB = 0>
int launch_kind(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td, const Params& p, int grid,
                bool f32, cudaStream_t st) {
    return f32 ? launch_typed<KIND, SA, SB, true>(ta, tb, td, p, grid, st)
               : launch_typed<KIND, SA, SB, false>(ta, tb, td, p, grid, st);
}

}  // namespace

int launch_gemm_mx(const GemmJob& j, cudaStream_t st) {
    if (j.experts > kMaxExperts) return -3;
    const bool nv = j.a_gran == 4;
    const uint64_t kbytes = nv ? (uint64_t)j.k / 2 : (uint64_t)j.k;
    const uint64_t b_rows = (uint64_t)j.n * (uint64_t)(j.experts > 0 ? j.experts : 1);
    CUtensorMap ta, tb, td;
    const bool td_ok = j.d_f32 ? make_tmap_out_f32(&td, j.d, (uint64_t)j.n, (uint64_t)j.m, (uint64_t)j.n, 16,
                                                   CU_TENSOR_MAP_SWIZZLE_64B)
                               : make_tmap_out_bf16(&td, j.d, (uint64_t)j.n, (uint64_t)j.m, (uint64_t)j.n, 32,
                                                    CU_TENSOR_MAP_SWIZZLE_64B);
    if (!make_tmap_u8(&ta, j.a, kbytes, (uint64_t)j.m, kbytes, BKB, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_u8(&tb, j.b, kbytes, b_rows, kbytes, BKB, BN, CU_TENSOR_MAP_SWIZZLE_128B) || !td_ok)
        return (int)cudaErrorInvalidValue;
    Params p{};
    p.m = j.m; p.n = j.n; p.k = j.k;
    p.sa = static_cast<const uint8_t*>(j.sa);
    p.sb = static_cast<const uint8_t*>(j.sb);
    p.a_ts = j.a_ts; p.b_ts = j.b_ts;
    p.a_ts_rows = j.a_ts_rows ? 1 : 0;
    p.d = static_cast<__nv_bfloat16*>(j.d);
    p.status = j.status;
    p.offsets = j.offsets;
    p.experts = j.experts;
    p.wait_ns = j.wait_ns ? j.wait_ns : kWaitLimitNs;
    p.stall_stage0 = j.stall_stage0;
    if (j.status != nullptr) {
        p.tile_next = reinterpret_cast<unsigned long long*>(reinterpret_cast<uint8_t*>(j.status) + kTileCounterOffset);
        p.tile_done = reinterpret_cast<unsigned int*>(reinterpret_cast<uint8_t*>(j.status) + kTileCounterOffset + 8);
    }
    const bool f32 = j.d_f32;
    const int sms = sm_count();
    int grid = sms;
    if (j.experts == 0) grid = (int)std::min<int64_t>(ceil_div(j.m, BM) * ceil_div(j.n, BN), sms);
    if (nv) return launch_kind<kNv>(ta, tb, td, p, grid, f32, st);
    if (j.a_gran == 3) return launch_kind<kMx>(ta, tb, td, p, grid, f32, st);
    // power-of-two block-wise: 5 = one byte per row and 128 K, 6 = per 128x128 block
    const int sa = j.a_gran == 5 ? 1 : 2, sb = j.b_gran == 5 ? 1 : 2;
    if (sa == 1 && sb == 2) return launch_kind<kP2, 1, 2>(ta, tb, td, p, grid, f32, st);
    if (sa == 1 && sb == 1) return launch_kind<kP2, 1, 1>(ta, tb, td, p, grid, f32, st);
    if (sa == 2 && sb == 2) return launch_kind<kP2, 2, 2>(ta, tb, td, p, grid, f32, st);
    return launch_kind<kP2, 2, 1>(ta, tb, td, p, grid, f32, st);
}

}  // namespace fp8bs
