// Internal declarations shared by the CUDA translation units of the library:
// the device-side mask description, the mask_mod predicate, the kernel
// launchers called by the C-ABI layer, and the per-device workspace.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda.h>

#include "../../include/flexattn.h"

namespace flex {

constexpr int kBlock = 128;         // compute tile (128 x 128); BlockMask blocks of other sizes map onto it
constexpr int kMaxKvBlocks = 1024;  // kv tiles (of 128) per row the kernels stage on chip
constexpr int kMinListBlock = 16, kMaxListBlock = 1024;  // BlockMask block sizes: powers of two in this range

__host__ __device__ constexpr bool valid_block_size(int b) {
    return b >= kMinListBlock && b <= kMaxListBlock && (b & (b - 1)) == 0;
}
// Blocks of size bs along a length (the last one may reach past it).
__host__ __device__ constexpr int ceil_div(int64_t len, int bs) { return (int)((len + bs - 1) / bs); }

// mask_mod as the kernels see it.
struct MaskDesc {
    int32_t kind;
    int32_t window;
    int32_t prefix;
    int32_t doc_len;            // row length of doc_ids (== q_len == kv_len)
    const int32_t *doc_ids;     // [B, doc_len]
    int32_t q_len, kv_len;      // positions at or past these are padding: masked
};

// Tiles along a length: the last one may reach past it (padding, masked).
__host__ __device__ constexpr int ceil_blocks(int64_t len) { return (int)((len + kBlock - 1) / kBlock); }

// mask_mod(b, h, q, kv) for the enumerated kinds.  No kind depends on h.
__host__ __device__ __forceinline__ bool mask_mod(const MaskDesc &m, int b, int q, int kv) {
    switch (m.kind) {
        case FLEX_MASK_CAUSAL:
            return q >= kv;
        case FLEX_MASK_SLIDING_WINDOW:
            return q >= kv && q - kv < m.window;
        case FLEX_MASK_CAUSAL_PREFIX:
            return (q <= m.prefix && kv <= m.prefix) || q >= kv;
        case FLEX_MASK_DOCUMENT:
            return q >= kv && m.doc_ids[(int64_t)b * m.doc_len + q] == m.doc_ids[(int64_t)b * m.doc_len + kv];
        default:
            return true;
    }
}

// The interval kinds keep, for a fixed row q, exactly the kv in [lo, hi].
// Returns false for kinds whose kept set is not an interval (document).
__host__ __device__ __forceinline__ bool mask_row_interval(const MaskDesc &m, int q, int &lo, int &hi) {
    switch (m.kind) {
        case FLEX_MASK_CAUSAL:
            lo = 0;
            hi = q;
            return true;
        case FLEX_MASK_SLIDING_WINDOW:
            lo = q - m.window + 1;
            hi = q;
            return true;
        case FLEX_MASK_CAUSAL_PREFIX:
            lo = 0;
            hi = q <= m.prefix ? m.prefix : q;
            return true;
        case FLEX_MASK_ALL:
            lo = 0;
            hi = 0x7fffffff;
            return true;
        default:
            return false;
    }
}

// Problem description handed from the C-ABI layer to the attention launchers.
struct AttnProblem {
    int B, H, q_len, kv_len, D;
    int q_block, kv_block, nqb, nkvb;                // BlockMask granularity: block sizes, blocks per row/column
    int nqt, nkvt;                                   // 128-tiles along q and kv
    int bh_begin, bh_count;                          // the (b, h) pairs b * H + h in [bh_begin, +bh_count) are computed
    int64_t q_stride[4], k_stride[4], v_stride[4];  // elements
    const void *q, *k, *v;
    void *out;                                       // contiguous [B,H,q_len,D]
    float *lse;                                      // contiguous [B,H,q_len]
    const int32_t *kv_num, *kv_idx, *full_num, *full_idx;
    MaskDesc mask;
    int score_kind;
    float score_param;
    float scale;
    int prescale;                                    // PRESCALE_QK: Q is scaled (rounded to its dtype) before QK^T
    float *row_max;                                  // OUTPUT_MAX: contiguous [B,H,q_len] or null
    int *status;                                     // device status word
};

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_block_mask(const MaskDesc &mask, int B, int H, int q_len, int kv_len, int q_block, int kv_block,
                              int32_t *kv_num, int32_t *kv_idx, int32_t *full_num, int32_t *full_idx,
                              cudaStream_t stream);
cudaError_t launch_attn_fp32(const AttnProblem &p, cudaStream_t stream);
cudaError_t launch_attn_bf16(const AttnProblem &p, cudaStream_t stream);

// TMA tensor map of a bf16 [B, H, S, D] tensor with element strides st
// (st[3] == 1): 64 x 128 boxes (head dims x rows), 128-byte swizzle.
bool make_bf16_tile_map(CUtensorMap *map, const void *base, int B, int H, int S, int D, const int64_t st[4]);

cudaError_t launch_wait_timeout_selftest(int *status, uint64_t limit_ns, cudaStream_t stream);

// The per-device workspace holding the status word (allocated once per device).
int *device_status_word(int *err);

// Status codes a kernel writes into the status word.
constexpr int kDeviceTimeout = 1;

}  // namespace flex
