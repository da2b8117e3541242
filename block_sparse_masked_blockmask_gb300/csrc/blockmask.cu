// BlockMask build: classify every 128 x 128 tile of mask_mod as full, partial
// or empty and write the kv-side BlockMask tensors of the flex_attention op
// ("[Inductor][Flex Attention] Add Subtiling Option for Alpha Scaling",
// PyTorch PR #167356, the BlockMask tuple: kv_num_blocks, kv_indices,
// full_kv_num_blocks, full_kv_indices at Q_BLOCK = KV_BLOCK = 128).
//
// One CTA per (batch b, q block qb); each warp classifies whole tiles.
//  * causal, sliding window, causal + prefix, all: for a fixed row q the kept
//    kv form exactly the interval [lo(q), hi(q)] (mask_row_interval), so a
//    tile is full when every row's interval covers the tile's 128 columns and
//    empty when no row's interval meets them: 128 row tests instead of 16384
//    predicate evaluations.
//  * document: exact quick decisions first (a tile above the diagonal is
//    empty; a tile below it whose 256 row and column ids are one id is full;
//    disjoint id ranges are empty), otherwise mask_mod is evaluated on all
//    16384 pairs, so arbitrary ids stay exact.
// Lengths need not be multiples of 128: positions past Q_LEN or KV_LEN are
// padding and count as masked, so a tile reaching past either is never full.
// None of the enumerated mask_mods depends on the head, so a row is
// classified once and written for every head.  Index rows hold the selected kv
// blocks in ascending order followed by the remaining kv blocks ascending.
#include <climits>

#include "flex_internal.h"

namespace flex {
namespace {

constexpr int kBmThreads = 256;
constexpr int kBmWarps = kBmThreads / 32;

enum : uint8_t { kEmpty = 0, kPartial = 1, kFull = 2 };

// Interval kinds: lane `lane` tests rows lane + 32 j of the tile; a row's
// interval ends at KV_LEN - 1, and rows past Q_LEN keep nothing.
__device__ __forceinline__ uint8_t classify_interval_tile(const MaskDesc &m, int q0, int kv0, int lane) {
    bool any = false, all = true;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int q = q0 + lane + 32 * j;
        int lo, hi;
        mask_row_interval(m, q, lo, hi);
        hi = min(hi, m.kv_len - 1);
        const bool row = q < m.q_len;
        const int a = max(lo, kv0), e = min(hi, kv0 + kBlock - 1);
        any |= row && a <= e;
        all &= row && lo <= kv0 && hi >= kv0 + kBlock - 1;
    }
    any = __any_sync(0xffffffffu, any);
    all = __all_sync(0xffffffffu, all);
    return all ? kFull : (any ? kPartial : kEmpty);
}

// Document kind: quick exact decisions, else every (q, kv) pair of the tile.
// Ids are read only inside the lengths; padding rows and columns keep nothing.
__device__ __forceinline__ uint8_t classify_document_tile(const MaskDesc &m, int b, int qb, int kvb, int lane,
                                                          const int32_t *row_doc, int row_min, int row_max) {
    if (kvb > qb) return kEmpty;  // every kv of the tile is above every q: kv > q
    const int kv0 = kvb * kBlock;
    const int q0 = qb * kBlock;
    int col_doc[4];
    int cmin = INT_MAX, cmax = INT_MIN;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int kv = kv0 + lane + 32 * j;
        col_doc[j] = kv < m.kv_len ? m.doc_ids[(int64_t)b * m.doc_len + kv] : 0;
        if (kv < m.kv_len) {
            cmin = min(cmin, col_doc[j]);
            cmax = max(cmax, col_doc[j]);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        cmin = min(cmin, __shfl_xor_sync(0xffffffffu, cmin, o));
        cmax = max(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
    }
    if (cmax < row_min || cmin > row_max) return kEmpty;  // no id in common
    const bool whole = q0 + kBlock <= m.q_len && kv0 + kBlock <= m.kv_len;
    if (whole && kvb < qb && cmin == cmax && row_min == row_max && cmin == row_min) return kFull;
    bool any = false, all = true;
    for (int r = 0; r < kBlock; ++r) {
        const int q = q0 + r;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int kv = kv0 + lane + 32 * j;
            const bool keep = q < m.q_len && kv < m.kv_len && q >= kv && row_doc[r] == col_doc[j];
            any |= keep;
            all &= keep;
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

template <int KIND>
__global__ void __launch_bounds__(kBmThreads) block_mask_kernel(MaskDesc m, int H, int nqb, int nkvb,
                                                                int32_t *kv_num, int32_t *kv_idx,
                                                                int32_t *full_num, int32_t *full_idx) {
    __shared__ uint8_t status[kMaxKvBlocks];
    __shared__ int32_t part_list[kMaxKvBlocks];
    __shared__ int32_t full_list[kMaxKvBlocks];
    __shared__ int32_t row_doc[kBlock];
    __shared__ int32_t row_range[2];
    __shared__ int32_t counts[2];

    const int qb = blockIdx.x, b = blockIdx.y;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int q0 = qb * kBlock;

    if constexpr (KIND == FLEX_MASK_DOCUMENT) {
        if (threadIdx.x == 0) {
            row_range[0] = INT_MAX;
            row_range[1] = INT_MIN;
        }
        __syncthreads();
        for (int r = threadIdx.x; r < kBlock; r += kBmThreads) {
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
            st = classify_document_tile(m, b, qb, kvb, lane, row_doc, row_range[0], row_range[1]);
        else
            st = classify_interval_tile(m, q0, kvb * kBlock, lane);
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

}  // namespace

cudaError_t launch_block_mask(const MaskDesc &mask, int B, int H, int q_len, int kv_len, int32_t *kv_num,
                              int32_t *kv_idx, int32_t *full_num, int32_t *full_idx, cudaStream_t stream) {
    const int nqb = ceil_blocks(q_len), nkvb = ceil_blocks(kv_len);
    const dim3 grid(nqb, B), block(kBmThreads);
    switch (mask.kind) {
        case FLEX_MASK_CAUSAL:
            block_mask_kernel<FLEX_MASK_CAUSAL><<<grid, block, 0, stream>>>(mask, H, nqb, nkvb, kv_num, kv_idx,
                                                                            full_num, full_idx);
            break;
        case FLEX_MASK_SLIDING_WINDOW:
            block_mask_kernel<FLEX_MASK_SLIDING_WINDOW><<<grid, block, 0, stream>>>(mask, H, nqb, nkvb, kv_num,
                                                                                    kv_idx, full_num, full_idx);
            break;
        case FLEX_MASK_CAUSAL_PREFIX:
            block_mask_kernel<FLEX_MASK_CAUSAL_PREFIX><<<grid, block, 0, stream>>>(mask, H, nqb, nkvb, kv_num,
                                                                                   kv_idx, full_num, full_idx);
            break;
        case FLEX_MASK_DOCUMENT:
            block_mask_kernel<FLEX_MASK_DOCUMENT><<<grid, block, 0, stream>>>(mask, H, nqb, nkvb, kv_num,
                                                                              kv_idx, full_num, full_idx);
            break;
        default:
            block_mask_kernel<FLEX_MASK_ALL><<<grid, block, 0, stream>>>(mask, H, nqb, nkvb, kv_num, kv_idx,
                                                                         full_num, full_idx);
            break;
    }
    return cudaGetLastError();
}

}  // namespace flex
