"""flex_attention_fwd_noalloc: the attention entry point for callers that
cannot let the library allocate device memory (stream capture, host
frameworks that own all device allocations, fixed-footprint processes).

It must give the same results as flex_attention_fwd on the same inputs, call
after call: each case here makes two calls in a row through the C-ABI and
compares both with flex_attention_fwd within the parity tolerances.  This file
is collected last on purpose and depends on no state left by other tests.
"""
import ctypes
import ctypes.util
import glob
import os

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


def _cudart():
    """The CUDA runtime, to read the status word back (None if not found)."""
    names = [ctypes.util.find_library("cudart")]
    tdir = os.path.dirname(torch.__file__)
    names += glob.glob(os.path.join(tdir, "lib", "libcudart*.so*"))
    names += glob.glob(os.path.join(os.path.dirname(tdir), "nvidia", "cuda_runtime", "lib", "libcudart.so*"))
    names += glob.glob("/usr/local/cuda/lib64/libcudart.so*")
    for n in names:
        if not n:
            continue
        try:
            lib = ctypes.CDLL(n)
            lib.cudaMemcpy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int]
            lib.cudaMemcpy.restype = ctypes.c_int
            return lib
        except OSError:
            continue
    return None


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
    cudart = _cudart()
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
        if cudart is not None:
            host = ctypes.c_int(-1)
            assert cudart.cudaMemcpy(ctypes.byref(host), ctypes.c_void_p(word), 4, 2) == 0
            assert host.value == 0, f"call {call}: status word {host.value}"
