"""Float64 CPU oracle for the block-sparse FlexAttention forward.

Test infrastructure only: the tests, the package smoke check and the bench's
CPU-baseline leg use it; the product path never does.
"""
from .oracle import (Oracle, attention, attention_bwd, attention_bwd_dq_rows, attention_opts,  # noqa: F401
                     block_mask, block_mask_q,
                     build, compile_oracle, default,
                     mask_value, num_threads, workload_attention, workload_block_mask)
