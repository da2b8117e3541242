// One side of a BlockMask read as 128 x 128 compute tiles.
//
// The BlockMask tuple of the flex_attention op ("[Inductor][Flex Attention]
// Add Subtiling Option for Alpha Scaling", PyTorch PR #167356, test diffs)
// carries a Q block size and a KV block size; the kernels here compute on
// 128 x 128 tiles.  A list side has one row per block of its "own" dimension
// (q blocks for the kv side, kv blocks for the q side) listing blocks of the
// "walked" dimension, partial ones in (num, idx) and full ones in
// (fnum, fidx).  For one 128-row own tile:
//   * the rows covering it are the own blocks that overlap it (one block
//     when own blocks are 128 or larger, 128 / size of them when smaller);
//   * a walked 128-tile is listed when any covering row lists any walked
//     block overlapping it, partial or full;
//   * it is full when every (covering row, covering walked block) pair is
//     listed full, i.e. when the count of full pairs reaches
//     (rows per tile) x (walked blocks per tile).  A coarser block that is
//     full makes every 128-tile inside it full; a partial one makes them
//     partial (mask_mod then decides every element).  A tile that reaches
//     past a length has covering blocks that do not exist, so it never
//     reaches the count: tail tiles stay partial, as at 128.
#pragma once

#include "flex_internal.h"

namespace flex {

struct TileLists {
    const int32_t *num, *idx, *fnum, *fidx;
    int own_nb;    // list rows per (b, h): blocks of the own dimension
    int walk_nb;   // list row length: blocks of the walked dimension
    int own_bs;    // own block size (a power of two, 16 .. 1024)
    int walk_bs;   // walked block size
    int walk_nt;   // 128-tiles of the walked dimension
};

// One 32-bit word per walked tile holds up to two own tiles u = 0, 1:
// bit 16 u: listed; bits 8 + 16 u .. 15 + 16 u: count of full pairs.
__device__ __forceinline__ uint32_t tl_listed_bit(int u) { return u ? (1u << 16) : 1u; }
__device__ __forceinline__ uint32_t tl_full_one(int u) { return u ? (1u << 24) : (1u << 8); }
__device__ __forceinline__ bool tl_listed(uint32_t w, int u) { return (w & tl_listed_bit(u)) != 0u; }
// Full pairs that make a walked tile full: (rows per own tile) x (walked blocks per tile).
__device__ __forceinline__ uint32_t tl_expect(const TileLists &L) {
    return (uint32_t)(L.own_bs >= 128 ? 1 : 128 / L.own_bs) * (uint32_t)(L.walk_bs >= 128 ? 1 : 128 / L.walk_bs);
}
__device__ __forceinline__ bool tl_full(uint32_t expect, uint32_t w, int u) {
    return ((w >> (u ? 24 : 8)) & 0xFFu) == expect;
}

// List rows [r0, r1) covering own tile `ot`.
__device__ __forceinline__ void tl_rows(const TileLists &L, int ot, int &r0, int &r1) {
    if (L.own_bs >= 128) {
        r0 = (int)(((int64_t)ot * 128) / L.own_bs);
        r1 = min(r0 + 1, L.own_nb);
    } else {
        const int k = 128 / L.own_bs;
        r0 = ot * k;
        r1 = min(r0 + k, L.own_nb);
    }
}

// Walked tiles [t0, t1) overlapping walked block `wb`.
__device__ __forceinline__ void tl_tiles(const TileLists &L, int wb, int &t0, int &t1) {
    if (L.walk_bs >= 128) {
        const int k = L.walk_bs / 128;
        t0 = wb * k;
        t1 = min(t0 + k, L.walk_nt);
    } else {
        t0 = wb / (128 / L.walk_bs);
        t1 = t0 + 1;
    }
}

__device__ __forceinline__ void tl_mark_entry(const TileLists &L, int wb, bool full, int u, uint32_t *words,
                                              int tlo, int thi) {
    if ((unsigned)wb >= (unsigned)L.walk_nb) return;  // malformed entry: dropped, nothing written
    int t0, t1;
    tl_tiles(L, wb, t0, t1);
    t0 = max(t0, tlo);
    t1 = min(t1, thi);
    for (int t = t0; t < t1; ++t) {
        atomicOr(&words[t - tlo], tl_listed_bit(u));
        if (full) atomicAdd(&words[t - tlo], tl_full_one(u));
    }
}

// Mark, with the 32 lanes of one warp, the walked tiles in [tlo, thi) of own
// tile `ot` of (b, h) pair `bh` as own slot u into words[t - tlo] (zeroed by
// the caller).  Counts are clamped to [0, walk_nb] and entries outside
// [0, walk_nb) are dropped, so a malformed BlockMask never writes outside
// words.  The index loads of a chunk are all issued before any is used, and
// those of a row's first chunk together with its counts (every entry below
// walk_nb lies in the row; entries past a count are dropped), so a short list
// costs one memory latency.
__device__ __forceinline__ void tl_mark_warp(const TileLists &L, int64_t bh, int ot, int u, uint32_t *words,
                                             int tlo, int thi, int lane) {
    int r0, r1;
    tl_rows(L, ot, r0, r1);
    constexpr int kUnroll = 2;
    for (int r = r0; r < r1; ++r) {
        const int64_t row = bh * L.own_nb + r;
        const int32_t *pi = L.idx + row * L.walk_nb, *fi = L.fidx + row * L.walk_nb;
        int jp[kUnroll], jf[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const int x = 32 * k + lane;
            jp[k] = x < L.walk_nb ? __ldg(pi + x) : -1;
            jf[k] = x < L.walk_nb ? __ldg(fi + x) : -1;
        }
        const int np = min(max(__ldg(L.num + row), 0), L.walk_nb);
        const int nf = min(max(__ldg(L.fnum + row), 0), L.walk_nb);
        for (int base = 0; base < max(np, nf); base += 32 * kUnroll) {
            if (base > 0) {
#pragma unroll
                for (int k = 0; k < kUnroll; ++k) {
                    const int x = base + 32 * k + lane;
                    jp[k] = x < np ? __ldg(pi + x) : -1;
                    jf[k] = x < nf ? __ldg(fi + x) : -1;
                }
            }
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int x = base + 32 * k + lane;
                tl_mark_entry(L, x < np ? jp[k] : -1, false, u, words, tlo, thi);
                tl_mark_entry(L, x < nf ? jf[k] : -1, true, u, words, tlo, thi);
            }
        }
    }
}

}  // namespace flex
