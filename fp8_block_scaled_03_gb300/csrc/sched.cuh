// sched.cuh -- persistent tile scheduler for the dense and MoE grouped GEMMs.
//
// Dense: tiles of BM x BN over D[m, n], numbered with the n-tile fastest.
// Grouped: expert e owns rows offsets[e] .. offsets[e+1]-1 of A and D; it
// contributes ceil(rows_e / BM) * n_tiles tiles, experts in order, so an
// expert with no rows contributes none.  Every CTA builds the tile prefix
// sum in shared memory itself (one warp scan over the device offsets);
// tile t is then found by a binary search over the prefix, and its
// expert's row range read from the offsets (L1/L2).  The host never reads
// the offsets.
//
// Offsets are checked on the device: expert e's rows are taken as
// [lo_e, hi_e) with lo_e = offsets[e] clamped to [0, m] and hi_e =
// offsets[e+1] clamped to [lo_e, m], so no tile ever addresses a row of A, D
// or their scales outside [0, m), whatever the offsets hold.  Offsets that
// break the contract (offsets[0] == 0, non-decreasing, offsets[E] == m) set
// the sticky status FP8BS_EOFFSETS; the rows of the well-formed experts are
// still computed.
#pragma once

#include <cstdint>

namespace fp8bs {

constexpr int kMaxExperts = 1024;
constexpr int kStatusOffsets = -8;   // FP8BS_EOFFSETS

// Row range of expert e, clamped as described above.
__device__ __forceinline__ void expert_rows(const int64_t* __restrict__ offsets, int e, int64_t m, int64_t& lo,
                                            int64_t& hi) {
    lo = min(max(__ldg(offsets + e), (int64_t)0), m);
    hi = min(max(__ldg(offsets + e + 1), lo), m);
}

struct TileInfo {
    int64_t row0;     // first row of A / D
    int64_t row_end;  // one past the last valid row of this tile's group
    int64_t n0;       // first column of D (row of B within the expert)
    int expert;       // 0 for dense
};

struct SchedShared {
    int64_t prefix[kMaxExperts + 1];
};

// Called by every thread of the CTA (contains __syncthreads).  Returns the
// total number of tiles.
template <int BM>
__device__ __forceinline__ int64_t sched_setup(SchedShared* sh, const int64_t* __restrict__ offsets, int experts,
                                               int64_t m, int64_t n_tiles, int* status) {
    if (experts == 0) return ((m + BM - 1) / BM) * n_tiles;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int per = (experts + 31) / 32;
        const int lo_e = min(experts, lane * per), hi_e = min(experts, lo_e + per);
        int64_t local = 0;
        bool bad = false;
        for (int e = lo_e; e < hi_e; ++e) {
            int64_t lo, hi;
            expert_rows(offsets, e, m, lo, hi);
            bad |= lo != __ldg(offsets + e) || hi != __ldg(offsets + e + 1);
            local += ((hi - lo + BM - 1) / BM) * n_tiles;
        }
        if (lane == 0) bad |= __ldg(offsets) != 0;
        if (lane == 31) bad |= __ldg(offsets + experts) != m;
        int64_t incl = local;
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        int64_t run = incl - local;
        for (int e = lo_e; e < hi_e; ++e) {
            sh->prefix[e] = run;
            int64_t lo, hi;
            expert_rows(offsets, e, m, lo, hi);
            run += ((hi - lo + BM - 1) / BM) * n_tiles;
        }
        if (lane == 31) sh->prefix[experts] = incl;
        if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && blockIdx.x == 0 && status != nullptr)
            atomicExch(status, kStatusOffsets);
    }
    __syncthreads();
    return sh->prefix[experts];
}

// GM (dense only): 0 numbers the tiles with the column tile fastest; GM > 0
// walks groups of GM row tiles with the row tile fastest inside a group, so
// the tiles in flight together share a few row blocks of A and column
// blocks of B.
template <int BM, int BN, int GM = 0>
__device__ __forceinline__ TileInfo sched_tile(const SchedShared* sh, const int64_t* __restrict__ offsets,
                                               int experts, int64_t m, int64_t n_tiles, int64_t t) {
    TileInfo ti;
    if (experts == 0) {
        int64_t mt, nt;
        if constexpr (GM > 0) {
            const int64_t m_tiles = (m + BM - 1) / BM;
            const int64_t per_group = (int64_t)GM * n_tiles;
            const int64_t g = t / per_group, r = t - g * per_group;
            const int64_t gm = min((int64_t)GM, m_tiles - g * GM);
            nt = r / gm;
            mt = g * GM + (r - nt * gm);
        } else {
            mt = t / n_tiles;
            nt = t - mt * n_tiles;
        }
        ti.row0 = mt * BM;
        ti.row_end = m;
        ti.n0 = nt * BN;
        ti.expert = 0;
        return ti;
    }
    int lo = 0, hi = experts;  // find e with prefix[e] <= t < prefix[e+1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sh->prefix[mid] <= t) lo = mid; else hi = mid;
    }
    // skip experts without tiles (prefix[e] == prefix[e+1])
    while (lo + 1 < experts && sh->prefix[lo + 1] <= t) ++lo;
    const int64_t local = t - sh->prefix[lo];
    const int64_t mt = local / n_tiles, nt = local - mt * n_tiles;
    int64_t r_lo, r_hi;
    expert_rows(offsets, lo, m, r_lo, r_hi);
    ti.row0 = r_lo + mt * BM;
    ti.row_end = r_hi;
    ti.n0 = nt * BN;
    ti.expert = lo;
    return ti;
}

}  // namespace fp8bs
