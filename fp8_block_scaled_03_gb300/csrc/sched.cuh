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
#pragma once

#include <cstdint>

namespace fp8bs {

constexpr int kMaxExperts = 1024;

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
                                               int64_t m, int64_t n_tiles) {
    if (experts == 0) return ((m + BM - 1) / BM) * n_tiles;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int per = (experts + 31) / 32;
        const int lo = min(experts, lane * per), hi = min(experts, lo + per);
        int64_t local = 0;
        for (int e = lo; e < hi; ++e) local += ((__ldg(offsets + e + 1) - __ldg(offsets + e) + BM - 1) / BM) * n_tiles;
        int64_t incl = local;
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        int64_t run = incl - local;
        for (int e = lo; e < hi; ++e) {
            sh->prefix[e] = run;
            run += ((__ldg(offsets + e + 1) - __ldg(offsets + e) + BM - 1) / BM) * n_tiles;
        }
        if (lane == 31) sh->prefix[experts] = incl;
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
    ti.row0 = __ldg(offsets + lo) + mt * BM;
    ti.row_end = __ldg(offsets + lo + 1);
    ti.n0 = nt * BN;
    ti.expert = lo;
    return ti;
}

}  // namespace fp8bs
