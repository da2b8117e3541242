// bf16 tensor-core attention, head dim 64.
#include "attn_bf16_launch.cuh"

namespace flex {
cudaError_t launch_bf16_d64(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const Bf16Params &kp, int score_kind, cudaStream_t stream) {
    return launch_bf16_dim<64>(tq, tk, tv, kp, score_kind, stream);
}
}  // namespace flex
