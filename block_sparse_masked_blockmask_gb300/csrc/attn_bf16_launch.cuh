// Launch of the bf16 tensor-core attention kernel for one head dim; included
// by one translation unit per head dim so the instantiations compile in parallel.
#pragma once

#include "attn_bf16_kernel.cuh"

namespace flex {

template <int D, int SCORE, bool DOC, bool BLOCKS128>
cudaError_t launch_bf16_kernel(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                               const Bf16Params &kp, cudaStream_t stream) {
    using C = Bf16Cfg<D>;
    auto kernel = attn_bf16_kernel<D, SCORE, DOC, BLOCKS128>;
    // The in-kernel register split assumes exactly kRegsAtLaunch registers per
    // thread at launch; any other count could stall the increase, so refuse.
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, kernel);
    if (e != cudaSuccess) return e;
    if (attr.numRegs != (int)kRegsAtLaunch) return cudaErrorInvalidDeviceFunction;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((int64_t)kp.nbh * kp.npairs);
    kernel<<<grid, kAttnThreads, C::kSmemBytes, stream>>>(tq, tk, tv, kp);
    return cudaGetLastError();
}

template <int D, bool DOC, bool BLOCKS128>
cudaError_t launch_bf16_score(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                              const Bf16Params &kp, int score_kind, cudaStream_t stream) {
    switch (score_kind) {
        case FLEX_SCORE_SOFTCAP:
            return launch_bf16_kernel<D, FLEX_SCORE_SOFTCAP, DOC, BLOCKS128>(tq, tk, tv, kp, stream);
        case FLEX_SCORE_ALIBI:
            return launch_bf16_kernel<D, FLEX_SCORE_ALIBI, DOC, BLOCKS128>(tq, tk, tv, kp, stream);
        default:
            return launch_bf16_kernel<D, FLEX_SCORE_IDENTITY, DOC, BLOCKS128>(tq, tk, tv, kp, stream);
    }
}

template <int D, bool DOC>
cudaError_t launch_bf16_blocks(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                               const Bf16Params &kp, int score_kind, cudaStream_t stream) {
    return kp.lists.own_bs == kBlock && kp.lists.walk_bs == kBlock
               ? launch_bf16_score<D, DOC, true>(tq, tk, tv, kp, score_kind, stream)
               : launch_bf16_score<D, DOC, false>(tq, tk, tv, kp, score_kind, stream);
}

template <int D>
cudaError_t launch_bf16_dim(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const Bf16Params &kp, int score_kind, cudaStream_t stream) {
    return kp.mask.kind == FLEX_MASK_DOCUMENT ? launch_bf16_blocks<D, true>(tq, tk, tv, kp, score_kind, stream)
                                              : launch_bf16_blocks<D, false>(tq, tk, tv, kp, score_kind, stream);
}

cudaError_t launch_bf16_d64(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const Bf16Params &kp, int score_kind, cudaStream_t stream);
cudaError_t launch_bf16_d128(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                             const Bf16Params &kp, int score_kind, cudaStream_t stream);

}  // namespace flex
