// Launch of the tensor-core backward kernel for one walking direction;
// included by one translation unit per direction so the instantiations
// compile in parallel.
#pragma once

#include "attn_bwd_tc.cuh"

namespace flex {

template <int D, int SCORE, bool DOC, bool KV_MAJOR>
cudaError_t launch_bwd_tc_kernel(const CUtensorMap (&maps)[4], const BwdTcParams &kp, cudaStream_t stream) {
    using C = BwdTcCfg<D, KV_MAJOR>;
    auto kernel = attn_bwd_tc_kernel<D, SCORE, DOC, KV_MAJOR>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    // one CTA per (batch, head, owned block); the grid is split so it stays
    // within the launch limit
    const int per = (int)std::min<int64_t>(kp.nbh, (int64_t)INT32_MAX / kp.nblocks);
    for (int begin = 0; begin < kp.nbh; begin += per) {
        BwdTcParams part = kp;
        part.bh_begin = kp.bh_begin + begin;
        part.nbh = std::min(per, kp.nbh - begin);
        kernel<<<(unsigned)((int64_t)part.nbh * part.nblocks), kBwdThreads, C::kSmemBytes, stream>>>(
            maps[0], maps[1], maps[2], maps[3], part);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int D, bool DOC, bool KV_MAJOR>
cudaError_t launch_bwd_tc_score(const CUtensorMap (&maps)[4], const BwdTcParams &kp, int score_kind,
                                cudaStream_t stream) {
    switch (score_kind) {
        case FLEX_SCORE_SOFTCAP:
            return launch_bwd_tc_kernel<D, FLEX_SCORE_SOFTCAP, DOC, KV_MAJOR>(maps, kp, stream);
        case FLEX_SCORE_ALIBI:
            return launch_bwd_tc_kernel<D, FLEX_SCORE_ALIBI, DOC, KV_MAJOR>(maps, kp, stream);
        default:
            return launch_bwd_tc_kernel<D, FLEX_SCORE_IDENTITY, DOC, KV_MAJOR>(maps, kp, stream);
    }
}

template <bool KV_MAJOR>
cudaError_t launch_bwd_tc_dir(const CUtensorMap (&maps)[4], const BwdTcParams &kp, int D, int score_kind,
                              cudaStream_t stream) {
    const bool doc = kp.mask.kind == FLEX_MASK_DOCUMENT;
    if (D == 64)
        return doc ? launch_bwd_tc_score<64, true, KV_MAJOR>(maps, kp, score_kind, stream)
                   : launch_bwd_tc_score<64, false, KV_MAJOR>(maps, kp, score_kind, stream);
    return doc ? launch_bwd_tc_score<128, true, KV_MAJOR>(maps, kp, score_kind, stream)
               : launch_bwd_tc_score<128, false, KV_MAJOR>(maps, kp, score_kind, stream);
}

}  // namespace flex
