"""Failure detection without a GPU fault: a device wait that runs out (an
mbarrier nobody arrives at, limit 50 ms) is reported through the status word,
the word is cleared by reading it, and the context stays usable."""
import time

import pytest

import oracle
from block_sparse_masked_blockmask_gb300 import flexattn as fa
from block_sparse_masked_blockmask_gb300 import workloads as W
from gpu_harness import compare, run_attention

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    assert fa.flex_device_status() == fa.FLEX_OK
    t0 = time.perf_counter()
    fa.flex_selftest_wait_timeout(50)
    assert fa.flex_device_status() == fa.FLEX_ERR_DEVICE_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 0.04 <= elapsed < 5.0, elapsed
    assert fa.flex_device_status() == fa.FLEX_OK  # cleared by the read
    # the context still runs the real kernels correctly
    w = W.scaled(W.BF16_CAUSAL_ALIBI_S16384, B=1, H=2, S=512)
    q, k, v, _ = W.workload_inputs(w)
    out, lse, _ = run_attention(q, k, v, w.mask, w.score, w.scale, w.dtype)
    ref_out, ref_lse = oracle.workload_attention(w, q, k, v)
    compare(out, lse, ref_out, ref_lse, w.dtype, "after timeout")


def test_selftest_rejects_bad_limits():
    for bad in (0, 60001):
        with pytest.raises(fa.FlexError) as e:
            fa.flex_selftest_wait_timeout(bad)
        assert e.value.code == fa.FLEX_ERR_INVALID_ARG
