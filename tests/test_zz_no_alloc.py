"""flex_attention_fwd_noalloc: the attention entry point for callers that
cannot let the library allocate device memory (stream capture, host
frameworks that own all device allocations, fixed-footprint processes).

It must give the same results as flex_attention_fwd on the same inputs, call
after call: each case here makes two calls in a row through the C-ABI and
compares both with flex_attention_fwd within the parity tolerances.  This file
is collected last on purpose and depends on no state left by other tests.
"""
import numpy as np
import pytest
import torch

from block_sparse_masked_blockmask_gb300 import flexattn as fa
from block_sparse_masked_blockmask_gb300 import workloads as W
from gpu_harness import TOL, device_tensor

pytestmark = pytest.mark.gpu

CASES = [
    W.scaled(W.BF16_CAUSAL_ALIBI_S16384, B=1, H=4, S=2048),
    W.scaled(W.BF16_DOC_SOFTCAP_S8192, B=2, H=2, S=2048),
    W.scaled(W.BF16_PREFIX1024_S4096, B=1, H=3, S=1536),
    W.FP32_CAUSAL_S256,
]


class _DeviceWord:
    """The library's 4-byte status word as a device array torch can read.

    The word lives in the library's static device scratch; exposing its
    address through __cuda_array_interface__ lets torch copy it to the host
    with no other CUDA runtime in the test."""

    def __init__(self, address: int):
        self.__cuda_array_interface__ = {"shape": (1,), "typestr": "<i4", "data": (address, False),
                                         "version": 3}


def _read_word(address: int) -> int:
    return int(torch.as_tensor(_DeviceWord(address), device="cuda").cpu()[0])


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name if w.B * w.H * w.S > 2048 else w.name)
def test_noalloc_matches_flex_attention_fwd_twice(w):
    q, k, v, docs = W.workload_inputs(w)
    dq, dk, dv = (device_tensor(x, w.dtype) for x in (q, k, v))
    dd = torch.from_numpy(docs).cuda() if docs is not None else None
    bm = fa.flex_block_mask_create(w.mask, w.B, w.H, w.S, w.S, 128, window=w.window, prefix=w.prefix, doc_ids=dd)
    ref_out, ref_lse = fa.flex_attention_fwd(dq, dk, dv, bm, w.score, w.score_param, w.scale)
    torch.cuda.synchronize()
    ref_out = ref_out.float().cpu().numpy()
    ref_lse = ref_lse.cpu().numpy()
    tol_out, tol_lse = TOL[w.dtype]
    for call in range(2):
        out = torch.full_like(dq, float("nan"))
        lse = torch.full((w.B, w.H, w.S), float("nan"), dtype=torch.float32, device="cuda")
        word = fa.flex_attention_fwd_noalloc(dq, dk, dv, bm, out, lse, w.score, w.score_param, w.scale)
        torch.cuda.synchronize()
        assert word is not None and word % 256 == 0
        o = out.float().cpu().numpy()
        l_ = lse.cpu().numpy()
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(l_)), f"call {call}: unwritten output"
        assert np.max(np.abs(o - ref_out)) <= tol_out, f"call {call}: out differs"
        assert np.max(np.abs(l_ - ref_lse)) <= tol_lse, f"call {call}: lse differs"
        assert _read_word(word) == 0, f"call {call}: status word set"
