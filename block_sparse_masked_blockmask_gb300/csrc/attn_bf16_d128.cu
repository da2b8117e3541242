// bf16 tensor-core attention, head dim 128.
#include "attn_bf16_launch.cuh"

namespace flex {
cudaError_t launch_bf16_d128(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                             const Bf16Params &kp, int score_kind, cudaStream_t stream) {
    return launch_bf16_dim<128>(tq, tk, tv, kp, score_kind, stream);
}
}  // namespace flex
