// Static work partition shared by the streaming decode kernels.
//
// The work of a call is a list of tiles (a slot's tokens, up to a fixed number
// per tile), each cut into P pieces of equal weight (bytes moved).  pref[] is
// the exclusive prefix of the tiles' weights (pref[NT] = total W).  CTA b of G
// takes the pieces whose weight start lies in [ceil(W b / G), ceil(W (b+1) / G)):
// contiguous, disjoint, covering every piece once, and within one piece of an
// equal share of the bytes.  Consecutive pieces of a CTA that share a tile (and
// whatever else the caller groups by) form one unit of work.
#pragma once

#include <cstdint>

namespace lora {

// Last index i in [0, N) with pref[i] <= v (pref ascending).
__device__ __forceinline__ int32_t last_le(const int32_t *pref, int32_t N, int64_t v) {
    int32_t lo = 0, hi = N;
    while (lo < hi) {
        const int32_t mid = (lo + hi) >> 1;
        if (pref[mid] <= v) lo = mid + 1;
        else hi = mid;
    }
    return lo - 1;
}

// A CTA's share of a list of weighted work pieces: the pieces whose weight
// start lies in [lo, hi), CTA b of G taking lo = ceil(W b / G).  Every tile
// holds P pieces of equal weight (its weight / P).
struct Range {
    int32_t tile, idx;  // current piece: tile and index within the tile
    int64_t hi;
};

__device__ __forceinline__ Range first_piece(const int32_t *pref, int32_t NT, int32_t P) {
    Range r;
    const int64_t W = pref[NT];
    const int64_t G = gridDim.x, b = blockIdx.x;
    const int64_t lo = (W * b + G - 1) / G;
    r.hi = (W * (b + 1) + G - 1) / G;
    r.tile = NT;
    r.idx = 0;
    if (lo >= W) return r;
    int32_t t = last_le(pref, NT, lo);
    const int32_t w = (pref[t + 1] - pref[t]) / P;
    int32_t i = static_cast<int32_t>((lo - pref[t] + w - 1) / w);
    if (i >= P) {
        ++t;
        i = 0;
    }
    r.tile = t;
    r.idx = i;
    return r;
}

// True while the current piece starts below this CTA's bound.
__device__ __forceinline__ bool piece_valid(const Range &r, const int32_t *pref, int32_t NT, int32_t P) {
    if (r.tile >= NT) return false;
    const int32_t w = (pref[r.tile + 1] - pref[r.tile]) / P;
    return static_cast<int64_t>(pref[r.tile]) + static_cast<int64_t>(r.idx) * w < r.hi;
}

// Number of this CTA's pieces in tile r.tile from r.idx on.
__device__ __forceinline__ int32_t pieces_left_in_tile(const Range &r, const int32_t *pref, int32_t P) {
    const int32_t w = (pref[r.tile + 1] - pref[r.tile]) / P;
    const int64_t room = r.hi - pref[r.tile] - static_cast<int64_t>(r.idx) * w;  // > 0
    const int32_t fit = static_cast<int32_t>((room + w - 1) / w);
    return min(P - r.idx, fit);
}

// The same partition when the number of pieces differs between tiles: P(t)
// gives tile t's count (every piece of a tile still has the same weight).
template <class PF>
__device__ __forceinline__ Range first_piece_var(const int32_t *pref, int32_t NT, PF P) {
    Range r;
    const int64_t W = pref[NT];
    const int64_t G = gridDim.x, b = blockIdx.x;
    const int64_t lo = (W * b + G - 1) / G;
    r.hi = (W * (b + 1) + G - 1) / G;
    r.tile = NT;
    r.idx = 0;
    if (lo >= W) return r;
    int32_t t = last_le(pref, NT, lo);
    const int32_t w = (pref[t + 1] - pref[t]) / P(t);
    int32_t i = static_cast<int32_t>((lo - pref[t] + w - 1) / w);
    if (i >= P(t)) {
        ++t;
        i = 0;
    }
    r.tile = t;
    r.idx = i;
    return r;
}

template <class PF>
__device__ __forceinline__ bool piece_valid_var(const Range &r, const int32_t *pref, int32_t NT, PF P) {
    if (r.tile >= NT) return false;
    const int32_t w = (pref[r.tile + 1] - pref[r.tile]) / P(r.tile);
    return static_cast<int64_t>(pref[r.tile]) + static_cast<int64_t>(r.idx) * w < r.hi;
}

template <class PF>
__device__ __forceinline__ int32_t pieces_left_var(const Range &r, const int32_t *pref, PF P) {
    const int32_t p = P(r.tile);
    const int32_t w = (pref[r.tile + 1] - pref[r.tile]) / p;
    const int64_t room = r.hi - pref[r.tile] - static_cast<int64_t>(r.idx) * w;  // > 0
    const int32_t fit = static_cast<int32_t>((room + w - 1) / w);
    return min(p - r.idx, fit);
}

}  // namespace lora
