"""flex_attention_fwd_host: host inputs and outputs, copies overlapped with the
work in chunks of (b, h) pairs.  It runs the same kernels on the same values as
flex_block_mask_create + flex_attention_fwd, so its outputs must equal theirs
bit for bit (each (b, h, q-block pair) is computed by one CTA on its own), and
one case is also checked against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_masked_blockmask_gb300 import flexattn as fa
from block_sparse_masked_blockmask_gb300 import workloads as W
from gpu_harness import compare, run_attention

pytestmark = pytest.mark.gpu


def _host(x: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "bf16":
        t = torch.from_numpy(W.bf16_bits(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.contiguous().pin_memory()


def _run_host(q, k, v, mask, score, scale, dtype, chunks, window=0, prefix=0, doc_ids=None, score_param=0.0):
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    hq, hk, hv = (_host(x, dtype) for x in (q, k, v))
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    hout = torch.empty((B, H, Sq, D), dtype=tdt).pin_memory()
    hlse = torch.empty((B, H, Sq), dtype=torch.float32).pin_memory()
    hdoc = None if doc_ids is None else torch.from_numpy(np.ascontiguousarray(doc_ids, np.int32)).pin_memory()
    bufs = fa.DeviceBuffers(B, H, Sq, Skv, D, tdt, document=doc_ids is not None)
    fa.flex_attention_fwd_host(hq, hk, hv, bufs, mask, hout, hlse, window=window, prefix=prefix, doc_ids=hdoc,
                               score_kind=score, score_param=score_param, scale=scale, chunks=chunks)
    torch.cuda.synchronize()
    assert fa.flex_device_status() == fa.FLEX_OK
    return hout.float().numpy().astype(np.float64), hlse.numpy().astype(np.float64)


CASES = [
    ("bf16", 2, 3, 384, 64, W.MASK_CAUSAL, W.SCORE_ALIBI, 0.0, {}),
    ("bf16", 2, 2, 512, 128, W.MASK_DOCUMENT, W.SCORE_SOFTCAP, 50.0, {}),
    ("bf16", 1, 4, 640, 128, W.MASK_SLIDING_WINDOW, W.SCORE_IDENTITY, 0.0, {"window": 200}),
    ("fp32", 1, 3, 256, 64, W.MASK_CAUSAL_PREFIX, W.SCORE_IDENTITY, 0.0, {"prefix": 130}),
]


@pytest.mark.parametrize("chunks", [1, 3, 64])
@pytest.mark.parametrize("dtype,B,H,S,D,mask,score,param,mkw", CASES, ids=lambda x: str(x))
def test_host_api_equals_device_api(dtype, B, H, S, D, mask, score, param, mkw, chunks):
    q, k, v = W.draw_qkv(B, H, S, D, seed=21, dtype=dtype)
    docs = None
    if mask == W.MASK_DOCUMENT:
        docs = np.zeros((B, S), np.int32)
        for b in range(B):
            docs[b, 100 + 37 * b:] += 1
            docs[b, 300:] += 1
    scale = 1.0 / np.sqrt(D)
    out_h, lse_h = _run_host(q, k, v, mask, score, scale, dtype, chunks, doc_ids=docs, score_param=param, **mkw)
    out_d, lse_d, _ = run_attention(q, k, v, mask, score, scale, dtype, doc_ids=docs, score_param=param, **mkw)
    assert np.array_equal(out_h, out_d) and np.array_equal(lse_h, lse_d)


def test_host_api_against_oracle():
    B, H, S, D = 2, 2, 512, 128
    q, k, v = W.draw_qkv(B, H, S, D, seed=22)
    out, lse = _run_host(q, k, v, W.MASK_CAUSAL, W.SCORE_ALIBI, 1 / np.sqrt(D), "bf16", chunks=4)
    ref_out, ref_lse = oracle.attention(q, k, v, W.MASK_CAUSAL, W.SCORE_ALIBI, 1 / np.sqrt(D))
    compare(out, lse, ref_out, ref_lse, "bf16", "host api")
