// BlockMask build: classify every Q_BLOCK x KV_BLOCK tile of mask_mod as
// full, partial or empty and write the kv-side BlockMask tensors of the
// flex_attention op ("[Inductor][Flex Attention] Add Subtiling Option for
// Alpha Scaling", PyTorch PR #167356, the BlockMask tuple: kv_num_blocks,
// kv_indices, full_kv_num_blocks, full_kv_indices and its Q_BLOCK and
// KV_BLOCK sizes).
//
// One CTA per (batch b, q block qb); each warp classifies whole tiles.
//  * causal, sliding window, causal + prefix, all: for a fixed row q the kept
//    kv form exactly the interval [lo(q), hi(q)] (mask_row_interval), so a
//    tile is full when every row's interval covers the tile's columns and
//    empty when no row's interval meets them: Q_BLOCK row tests instead of
//    Q_BLOCK x KV_BLOCK predicate evaluations.
//  * document: exact quick decisions first (a tile above the diagonal is
//    empty; a tile on or below it whose row and column ids are one id is
//    full; disjoint id ranges are empty), otherwise mask_mod is evaluated on
//    every pair of the tile, so arbitrary ids stay exact.
// Lengths need not be multiples of the block sizes: positions past Q_LEN or
// KV_LEN are padding and count as masked, so a tile reaching past either is
// never full.  None of the enumerated mask_mods depends on the head, so a
// row is classified once and written for every head.  Index rows hold the
// selected kv blocks in ascending order followed by the remaining kv blocks
// ascending.
#include <climits>

#include "flex_internal.h"

namespace flex {
namespace {

constexpr int kBmThreads = 256;
constexpr int kBmWarps = kBmThreads / 32;

enum : uint8_t { kEmpty = 0, kPartial = 1, kFull = 2 };

// Interval kinds: lane `lane` tests rows lane + 32 j of the qbs x kvbs tile
// at (q0, kv0); a row's interval ends at KV_LEN - 1, and rows past Q_LEN
// keep nothing.
__device__ __forceinline__ uint8_t classify_interval_tile(const MaskDesc &m, int q0, int kv0, int qbs, int kvbs,
                                                          int lane) {
    bool any = false, all = true;
    for (int r = lane; r < qbs; r += 32) {
        const int q = q0 + r;
        int lo, hi;
        mask_row_interval(m, q, lo, hi);
        hi = min(hi, m.kv_len - 1);
        const bool row = q < m.q_len;
        const int a = max(lo, kv0), e = min(hi, kv0 + kvbs - 1);
        any |= row && a <= e;
        all &= row && lo <= kv0 && hi >= kv0 + kvbs - 1;
    }
    any = __any_sync(0xffffffffu, any);
    all = __all_sync(0xffffffffu, all);
    return all ? kFull : (any ? kPartial : kEmpty);
}

// Document kind: quick exact decisions, else every (q, kv) pair of the tile.
// Ids are read only inside the lengths; padding rows and columns keep nothing.
__device__ __forceinline__ uint8_t classify_document_tile(const MaskDesc &m, int b, int q0, int kv0, int qbs,
                                                          int kvbs, int lane, const int32_t *row_doc, int row_min,
                                                          int row_max) {
    if (kv0 > q0 + qbs - 1) return kEmpty;  // every kv of the tile is above every q: kv > q
    const int32_t *ids = m.doc_ids + (int64_t)b * m.doc_len;
    int cmin = INT_MAX, cmax = INT_MIN;
    for (int c = lane; c < kvbs; c += 32) {
        const int kv = kv0 + c;
        if (kv < m.kv_len) {
            const int d = ids[kv];
            cmin = min(cmin, d);
            cmax = max(cmax, d);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        cmin = min(cmin, __shfl_xor_sync(0xffffffffu, cmin, o));
        cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
    }
    if (cmax < row_min || cmin > row_max) return kEmpty;  // no id in common
    const bool whole = q0 + qbs <= m.q_len && kv0 + kvbs <= m.kv_len;
    if (whole && kv0 + kvbs - 1 <= q0 && cmin == cmax && row_min == row_max && cmin == row_min) return kFull;
    bool any = false, all = true;
    for (int c0 = 0; c0 < kvbs; c0 += 32) {  // every lane runs every group: the votes below need all 32
        const int c = c0 + lane;
        const int kv = kv0 + c;
        const bool col = c < kvbs;
        const int cd = col && kv < m.kv_len ? ids[kv] : 0;
        for (int r = 0; r < qbs; ++r) {
            const int q = q0 + r;
            const bool keep = q < m.q_len && kv < m.kv_len && q >= kv && row_doc[r] == cd;
            if (col) {
                any |= keep;
                all &= keep;
            }
        }
    }
    any = __any_sync(0xffffffffu, any);
    all = __all_sync(0xffffffffu, all);
    return all ? kFull : (any ? kPartial : kEmpty);
}

// Selected indices (status == want) ascending, then the rest ascending.
__device__ __forceinline__ int compact_row(const uint8_t *status, int nkvb, uint8_t want, int32_t *list,
                                           int lane) {
    const unsigned lt = (1u << lane) - 1u;
    int count = 0;
    for (int base = 0; base < nkvb; base += 32) {
        const int c = base + lane;
        const bool sel = c < nkvb && status[c] == want;
        const unsigned bal = __ballot_sync(0xffffffffu, sel);
        if (sel) list[count + __popc(bal & lt)] = c;
        count += __popc(bal);
    }
    const int nsel = count;
    for (int base = 0; base < nkvb; base += 32) {
        const int c = base + lane;
        const bool sel = c < nkvb && status[c] != want;
        const unsigned bal = __ballot_sync(0xffffffffu, sel);
        if (sel) list[count + __popc(bal & lt)] = c;
        count += __popc(bal);
    }
    return nsel;
}

// Dynamic shared memory of one CTA: the row's tile classes, its two compacted
// lists, and the document ids of its rows.
__host__ __device__ constexpr size_t block_mask_smem(int nkvb, int qbs) {
    return (size_t)nkvb * 2 * sizeof(int32_t) + (size_t)qbs * sizeof(int32_t) + (size_t)nkvb;
}

template <int KIND>
__global__ void __launch_bounds__(kBmThreads) block_mask_kernel(MaskDesc m, int H, int nqb, int nkvb, int qbs,
                                                                int kvbs, int32_t *kv_num, int32_t *kv_idx,
                                                                int32_t *full_num, int32_t *full_idx) {
    extern __shared__ int32_t bm_smem[];
    int32_t *part_list = bm_smem;
    int32_t *full_list = part_list + nkvb;
    int32_t *row_doc = full_list + nkvb;
    uint8_t *status = reinterpret_cast<uint8_t *>(row_doc + qbs);
    __shared__ int32_t row_range[2];
    __shared__ int32_t counts[2];

    const int qb = blockIdx.x, b = blockIdx.y;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int q0 = qb * qbs;

    if constexpr (KIND == FLEX_MASK_DOCUMENT) {
        if (threadIdx.x == 0) {
            row_range[0] = INT_MAX;
            row_range[1] = INT_MIN;
        }
        __syncthreads();
        for (int r = threadIdx.x; r < qbs; r += kBmThreads) {
            if (q0 + r >= m.q_len) {  // padding row
                row_doc[r] = 0;
                continue;
            }
            const int d = m.doc_ids[(int64_t)b * m.doc_len + q0 + r];
            row_doc[r] = d;
            atomicMin(&row_range[0], d);
            atomicMax(&row_range[1], d);
        }
        __syncthreads();
    }
    for (int kvb = warp; kvb < nkvb; kvb += kBmWarps) {
        uint8_t st;
        if constexpr (KIND == FLEX_MASK_DOCUMENT)
            st = classify_document_tile(m, b, q0, kvb * kvbs, qbs, kvbs, lane, row_doc, row_range[0], row_range[1]);
        else
            st = classify_interval_tile(m, q0, kvb * kvbs, qbs, kvbs, lane);
        if (lane == 0) status[kvb] = st;
    }
    __syncthreads();
    if (warp == 0) {
        const int n = compact_row(status, nkvb, kPartial, part_list, lane);
        if (lane == 0) counts[0] = n;
    } else if (warp == 1) {
        const int n = compact_row(status, nkvb, kFull, full_list, lane);
        if (lane == 0) counts[1] = n;
    }
    __syncthreads();
    for (int h = 0; h < H; ++h) {
        const int64_t row = ((int64_t)b * H + h) * nqb + qb;
        int32_t *pi = kv_idx + row * nkvb;
        int32_t *fi = full_idx + row * nkvb;
        for (int i = threadIdx.x; i < nkvb; i += kBmThreads) {
            pi[i] = part_list[i];
            fi[i] = full_list[i];
        }
        if (threadIdx.x == 0) {
            kv_num[row] = counts[0];
            full_num[row] = counts[1];
        }
    }
}

template <int KIND>
cudaError_t launch_kind(const MaskDesc &mask, int B, int H, int nqb, int nkvb, int qbs, int kvbs, int32_t *kv_num,
                        int32_t *kv_idx, int32_t *full_num, int32_t *full_idx, cudaStream_t stream) {
    const size_t smem = block_mask_smem(nkvb, qbs);
    cudaError_t e = cudaFuncSetAttribute(block_mask_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    block_mask_kernel<KIND><<<dim3(nqb, B), kBmThreads, smem, stream>>>(mask, H, nqb, nkvb, qbs, kvbs, kv_num,
                                                                      kv_idx, full_num, full_idx);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_block_mask(const MaskDesc &mask, int B, int H, int q_len, int kv_len, int q_block, int kv_block,
                              int32_t *kv_num, int32_t *kv_idx, int32_t *full_num, int32_t *full_idx,
                              cudaStream_t stream) {
    const int nqb = ceil_div(q_len, q_block), nkvb = ceil_div(kv_len, kv_block);
    switch (mask.kind) {
        case FLEX_MASK_CAUSAL:
            return launch_kind<FLEX_MASK_CAUSAL>(mask, B, H, nqb, nkvb, q_block, kv_block, kv_num, kv_idx,
                                                 full_num, full_idx, stream);
        case FLEX_MASK_SLIDING_WINDOW:
            return launch_kind<FLEX_MASK_SLIDING_WINDOW>(mask, B, H, nqb, nkvb, q_block, kv_block, kv_num, kv_idx,
                                                         full_num, full_idx, stream);
        case FLEX_MASK_CAUSAL_PREFIX:
            return launch_kind<FLEX_MASK_CAUSAL_PREFIX>(mask, B, H, nqb, nkvb, q_block, kv_block, kv_num, kv_idx,
                                                        full_num, full_idx, stream);
        case FLEX_MASK_DOCUMENT:
            return launch_kind<FLEX_MASK_DOCUMENT>(mask, B, H, nqb, nkvb, q_block, kv_block, kv_num, kv_idx,
                                                   full_num, full_idx, stream);
        default:
            return launch_kind<FLEX_MASK_ALL>(mask, B, H, nqb, nkvb, q_block, kv_block, kv_num, kv_idx, full_num,
                                              full_idx, stream);
    }
}

}  // namespace flex
