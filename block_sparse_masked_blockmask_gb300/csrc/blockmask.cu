// BlockMask build: classify every 128 x 128 tile of mask_mod as full, partial
// or empty and write the kv-side BlockMask tensors of the flex_attention op
// ("[Inductor][Flex Attention] Add Subtiling Option for Alpha Scaling",
// PyTorch PR #167356, the BlockMask tuple: kv_num_blocks, kv_indices,
// full_kv_num_blocks, full_kv_indices at Q_BLOCK = KV_BLOCK = 128).
//
// One CTA per (batch b, q block qb).  Each warp classifies whole tiles by
// evaluating mask_mod on all 16384 (q, kv) pairs of the tile (no closed-form
// shortcut, so document masks with arbitrary ids are exact).  None of the
// enumerated mask_mods depends on the head, so a row is classified once and
// written for every head.  Index rows hold the selected kv blocks in
// ascending order followed by the remaining kv blocks in ascending order.
#include "flex_internal.h"

namespace flex {
namespace {

constexpr int kBmThreads = 256;
constexpr int kBmWarps = kBmThreads / 32;

enum : uint8_t { kEmpty = 0, kPartial = 1, kFull = 2 };

// Lane `lane` tests the four columns lane + 32 j of the tile against all 128
// rows; the warp then reduces "any true" and "all true".
template <int KIND>
__device__ __forceinline__ uint8_t classify_tile(const MaskDesc &m, int b, int q0, int kv0, int lane,
                                                 const int32_t *row_doc) {
    bool any = false, all = true;
    int col_doc[4];
    if constexpr (KIND == FLEX_MASK_DOCUMENT) {
#pragma unroll
        for (int j = 0; j < 4; ++j) col_doc[j] = m.doc_ids[(int64_t)b * m.doc_len + kv0 + lane + 32 * j];
    }
    for (int r = 0; r < kBlock; ++r) {
        const int q = q0 + r;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int kv = kv0 + lane + 32 * j;
            bool keep;
            if constexpr (KIND == FLEX_MASK_CAUSAL) {
                keep = q >= kv;
            } else if constexpr (KIND == FLEX_MASK_SLIDING_WINDOW) {
                keep = q >= kv && q - kv < m.window;
            } else if constexpr (KIND == FLEX_MASK_CAUSAL_PREFIX) {
                keep = (q <= m.prefix && kv <= m.prefix) || q >= kv;
            } else if constexpr (KIND == FLEX_MASK_DOCUMENT) {
                keep = q >= kv && row_doc[r] == col_doc[j];
            } else {
                keep = true;
            }
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
    __shared__ int32_t counts[2];

    const int qb = blockIdx.x, b = blockIdx.y;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int q0 = qb * kBlock;

    if constexpr (KIND == FLEX_MASK_DOCUMENT) {
        for (int r = threadIdx.x; r < kBlock; r += kBmThreads) row_doc[r] = m.doc_ids[(int64_t)b * m.doc_len + q0 + r];
        __syncthreads();
    }
    for (int kvb = warp; kvb < nkvb; kvb += kBmWarps) {
        const uint8_t st = classify_tile<KIND>(m, b, q0, kvb * kBlock, lane, row_doc);
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
    const int nqb = q_len / kBlock, nkvb = kv_len / kBlock;
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
