// Host side of the bf16 tensor-core attention: TMA tensor maps for Q, K, V
// (4-D [B, H, S, D] views with 64 x 128 boxes and 128-byte swizzle) and
// dispatch on head dim and score kind.
#include <algorithm>
#include <mutex>

#include "attn_bf16_launch.cuh"

namespace flex {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

}  // namespace

// [B, H, S, D] bf16 with element strides st (st[3] == 1) as a 4-D tensor map
// whose box is 64 (D) x 128 (S) x 1 x 1.
bool make_bf16_tile_map(CUtensorMap *map, const void *base, int B, int H, int S, int D, const int64_t st[4]) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)H, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)st[2] * 2, (cuuint64_t)st[1] * 2, (cuuint64_t)st[0] * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)kBlock, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_attn_bf16(const AttnProblem &p, cudaStream_t stream) {
    CUtensorMap tq, tk, tv;
    if (!make_bf16_tile_map(&tq, p.q, p.B, p.H, p.q_len, p.D, p.q_stride) ||
        !make_bf16_tile_map(&tk, p.k, p.B, p.H, p.kv_len, p.D, p.k_stride) ||
        !make_bf16_tile_map(&tv, p.v, p.B, p.H, p.kv_len, p.D, p.v_stride))
        return cudaErrorInvalidValue;
    Bf16Params kp;
    kp.B = p.B;
    kp.H = p.H;
    kp.q_len = p.q_len;
    kp.kv_len = p.kv_len;
    kp.nqt = p.nqt;
    kp.nkvt = p.nkvt;
    kp.npairs = (p.nqt + 1) / 2;
    kp.bh_begin = p.bh_begin;
    kp.nbh = p.bh_count;
    // (b, h) pairs scheduled together: as many as keep their K and V within
    // 64 MB of L2 (at least kHeadGroup), so that with small heads the longest
    // items of more heads run first and fewer short ones are left at the end
    // of the grid (measured: causal + prefix B4 H16 S4096 D64 -7%, document +
    // softcap B8 H16 S8192 D128 -8%; 8 heads of S16384 D128 as fast as 4)
    {
        const int64_t kv_bytes = 4 * (int64_t)p.kv_len * p.D;  // K and V of one (b, h), bf16
        const int64_t fit = (int64_t(64) << 20) / kv_bytes;
        kp.head_group = (int)std::max<int64_t>(kHeadGroup, std::min<int64_t>(fit, p.bh_count));
    }
    kp.lists = TileLists{p.kv_num, p.kv_idx, p.full_num, p.full_idx, p.nqb, p.nkvb, p.q_block, p.kv_block, p.nkvt};
    kp.mask = p.mask;
    // PRESCALE_QK moves the scale onto Q (in shared memory); the scores then take 1
    kp.scale = p.prescale ? 1.f : p.scale;
    kp.prescale = p.prescale ? p.scale : 0.f;
    kp.score_param = p.score_param;
    kp.out = static_cast<uint16_t *>(p.out);
    kp.lse = p.lse;
    kp.row_max = p.row_max;
    kp.status = p.status;
    return p.D == 64 ? launch_bf16_d64(tq, tk, tv, kp, p.score_kind, stream)
                     : launch_bf16_d128(tq, tk, tv, kp, p.score_kind, stream);
}

}  // namespace flex
