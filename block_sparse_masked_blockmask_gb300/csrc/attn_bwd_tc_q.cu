// Tensor-core backward, dQ (one CTA per q block, walking the kv side of the BlockMask).
#include <algorithm>

#include "attn_bwd_tc_launch.cuh"
#include "bwd_internal.h"

namespace flex {
cudaError_t launch_bwd_tc_dq(const CUtensorMap (&maps)[4], const BwdTcParams &kp, int D, int score_kind,
                             cudaStream_t stream) {
    return launch_bwd_tc_dir<false>(maps, kp, D, score_kind, stream);
}
}  // namespace flex
