// Launchers of the backward pass (attn_bwd.cu), called by the C-ABI layer.
#pragma once

#include "flex_internal.h"

namespace flex {

// delta, dK/dV and dQ kernels; out and lse of p are the forward's outputs,
// read here.
cudaError_t launch_attn_bwd(const AttnProblem &p, int dtype, const void *dout, const int32_t *q_num,
                            const int32_t *q_idx, const int32_t *fq_num, const int32_t *fq_idx, void *dq, void *dk,
                            void *dv, float *delta, cudaStream_t stream);
struct BwdTcParams;
// Tensor-core backward kernels (bf16): dK and dV per kv block, dQ per q block.
// maps: the two resident tensors, then the two walked ones (TMA tensor maps).
cudaError_t launch_bwd_tc_dkdv(const CUtensorMap (&maps)[4], const BwdTcParams &kp, int D, int score_kind,
                               cudaStream_t stream);
cudaError_t launch_bwd_tc_dq(const CUtensorMap (&maps)[4], const BwdTcParams &kp, int D, int score_kind,
                             cudaStream_t stream);
// q blocks per kv block the tensor-core backward walks on chip (NQB limit for bf16)
constexpr int kBwdTcMaxQBlocks = 2048;

// q side of the BlockMask from its kv side.
cudaError_t launch_block_mask_transpose(const int32_t *kv_num, const int32_t *kv_idx, const int32_t *full_num,
                                        const int32_t *full_idx, int B, int H, int nqb, int nkvb, int32_t *q_num,
                                        int32_t *q_idx, int32_t *fq_num, int32_t *fq_idx, cudaStream_t stream);

}  // namespace flex
