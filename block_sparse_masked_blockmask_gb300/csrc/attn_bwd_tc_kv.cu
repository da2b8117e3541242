// Tensor-core backward, dK and dV (one CTA per kv block, walking the q side of the BlockMask).
#include <algorithm>

#include "attn_bwd_tc_launch.cuh"
#include "bwd_internal.h"

namespace flex {
cudaError_t launch_bwd_tc_dkdv(const CUtensorMap (&maps)[4], const BwdTcParams &kp, int D, int score_kind,
                               cudaStream_t stream) {
    return launch_bwd_tc_dir<true>(maps, kp, D, score_kind, stream);
}
}  // namespace flex
