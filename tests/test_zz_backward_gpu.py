"""Backward pass (flex_attention_bwd) and the q side of the BlockMask vs the oracle.

The q-side lists are compared bit for bit.  dq, dk, dv are compared per
tensor: max-abs error <= 1e-2 * max|ref| for bf16 and <= 1e-4 *
max(1, max|ref|) for fp32, plus 1e-4 absolute: with one key per row the
exact dq and dk are 0 and the fp32 difference dP - delta leaves ~1e-6
there.  The bf16 path runs on the tensor cores: P and dS enter the MMAs
rounded to bf16 (2^-9 relative each, errors that average out over the
summed keys), each gradient is rounded to bf16 (2^-9), and delta = dout . out
is taken from the forward's bf16-rounded out (2^-9 on the row term of dS),
so 1e-2 = 5 x 2^-9 of the largest gradient bounds their sum.  The fp32 path
runs on the tensor cores with every operand split into three bf16 parts
(six part products, float32 accumulation: about 2^-22 relative per
product), well inside 1e-4.  The forward's out and lse come from the
library's own forward, as a caller would pass them; the oracle
differentiates the exact attention.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_masked_blockmask_gb300 import flexattn as fa
from block_sparse_masked_blockmask_gb300 import workloads as W
from gpu_harness import device_tensor, gpu_block_mask, sample_rows

pytestmark = pytest.mark.gpu

REL = {"bf16": 1e-2, "fp32": 1e-4}


def _docs(B, S, seed):
    rng = np.random.default_rng(seed)
    d = np.zeros((B, S), np.int32)
    for b in range(B):
        for c in np.sort(rng.choice(np.arange(1, S), size=min(3, S - 1), replace=False)):
            d[b, c:] += 1
    return d


MASKS = [
    (W.MASK_CAUSAL, {}),
    (W.MASK_SLIDING_WINDOW, {"window": 100}),
    (W.MASK_CAUSAL_PREFIX, {"prefix": 150}),
    (W.MASK_DOCUMENT, {}),
    (W.MASK_ALL, {}),
]
SCORES = [(W.SCORE_IDENTITY, 0.0), (W.SCORE_SOFTCAP, 2.0), (W.SCORE_ALIBI, 0.0)]


@pytest.mark.parametrize("mask,mkw", MASKS, ids=lambda x: str(x))
@pytest.mark.parametrize("q_len,kv_len", [(1, 1), (300, 300), (1000, 1000), (4096, 4096), (200, 333), (333, 200)])
def test_block_mask_transpose(mask, mkw, q_len, kv_len):
    if mask == W.MASK_DOCUMENT and (q_len != kv_len or q_len % 4):
        pytest.skip("document masks: Q_LEN == KV_LEN, a multiple of 4")
    B, H = 2, 3
    docs = _docs(B, q_len, 1) if mask == W.MASK_DOCUMENT else None
    bm = gpu_block_mask(mask, B, H, q_len, kv_len, doc_ids=docs, **mkw)
    bq = fa.flex_block_mask_transpose(bm)
    torch.cuda.synchronize()
    got = bq.as_numpy()
    ref = oracle.block_mask_q(mask, B, H, q_len, kv_len, 128, doc_ids=docs, **mkw)
    for key in fa.BlockMaskQ.KEYS:
        assert got[key].dtype == np.int32
        assert np.array_equal(got[key], ref[key]), f"{key} m{mask} {q_len}x{kv_len}"


def _backward(q, k, v, g, mask, score, scale, dtype, window=0, prefix=0, doc_ids=None, score_param=0.0):
    dq_, dk_, dv_, dg = (device_tensor(x, dtype) for x in (q, k, v, g))
    B, H, Sq, _ = dq_.shape
    bm = gpu_block_mask(mask, B, H, Sq, dk_.shape[2], window, prefix, doc_ids)
    bq = fa.flex_block_mask_transpose(bm)
    out, lse = fa.flex_attention_fwd(dq_, dk_, dv_, bm, score, score_param, scale)
    grads = fa.flex_attention_bwd(dq_, dk_, dv_, out, lse, dg, bm, bq, score, score_param, scale)
    assert fa.flex_device_status() == fa.FLEX_OK
    return [x.float().cpu().numpy().astype(np.float64) for x in grads]


def _compare(got, ref, dtype, what):
    for name, a, b in zip(("dq", "dk", "dv"), got, ref):
        assert a.shape == b.shape and np.all(np.isfinite(a)), f"{what} {name}"
        scale = max(1.0, float(np.max(np.abs(b)))) if dtype == "fp32" else float(np.max(np.abs(b)))
        err = float(np.max(np.abs(a - b)))
        assert err <= REL[dtype] * scale + 1e-4, f"{what} {name}: max-abs {err:.3e} > {REL[dtype]:.0e} x {scale:.3e}"


def _draw(B, H, Sq, Skv, D, seed, dtype):
    q, k, v = W.draw_qkv(B, H, Sq, D, seed=seed, dtype=dtype, S_kv=Skv)
    g = W.draw_qkv(B, H, Sq, D, seed=seed + 1000, dtype=dtype)[0]
    return q, k, v, g


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mask,mkw", MASKS, ids=lambda x: str(x))
@pytest.mark.parametrize("score,param", SCORES, ids=lambda x: str(x))
def test_backward_small(dtype, D, mask, mkw, score, param):
    # S = 384: three q blocks and three kv blocks
    B, H, S = 2, 2, 384
    q, k, v, g = _draw(B, H, S, S, D, 31, dtype)
    docs = _docs(B, S, 2) if mask == W.MASK_DOCUMENT else None
    scale = 1.0 / np.sqrt(D)
    got = _backward(q, k, v, g, mask, score, scale, dtype, doc_ids=docs, score_param=param, **mkw)
    ref = oracle.attention_bwd(q, k, v, g, mask, score, scale, doc_ids=docs, score_param=param, **mkw)
    _compare(got, ref, dtype, f"{dtype} D{D} m{mask} s{score}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("q_len,kv_len", [(300, 300), (1, 1), (200, 333), (333, 200), (129, 1)])
@pytest.mark.parametrize("mask,mkw", [(W.MASK_CAUSAL, {}), (W.MASK_CAUSAL_PREFIX, {"prefix": 150}),
                                      (W.MASK_ALL, {})], ids=lambda x: str(x))
def test_backward_ragged(dtype, q_len, kv_len, mask, mkw):
    B, H, D = 1, 2, 128
    q, k, v, g = _draw(B, H, q_len, kv_len, D, 32, dtype)
    got = _backward(q, k, v, g, mask, W.SCORE_ALIBI, 0.1, dtype, **mkw)
    ref = oracle.attention_bwd(q, k, v, g, mask, W.SCORE_ALIBI, 0.1, **mkw)
    _compare(got, ref, dtype, f"{dtype} {q_len}x{kv_len} m{mask}")


def test_backward_empty_rows_give_zero():
    B, H, S, D = 1, 2, 256, 64
    q, k, v, g = _draw(B, H, S, S, D, 33, "bf16")
    got = _backward(q, k, v, g, W.MASK_SLIDING_WINDOW, W.SCORE_IDENTITY, 0.125, "bf16", window=0)
    assert all(np.all(x == 0.0) for x in got)


def test_backward_medium():
    # causal + ALiBi, bf16, D = 128, S = 2048: every gradient against the oracle
    B, H, S, D = 1, 2, 2048, 128
    q, k, v, g = _draw(B, H, S, S, D, 34, "bf16")
    scale = 1.0 / np.sqrt(D)
    got = _backward(q, k, v, g, W.MASK_CAUSAL, W.SCORE_ALIBI, scale, "bf16")
    ref = oracle.attention_bwd(q, k, v, g, W.MASK_CAUSAL, W.SCORE_ALIBI, scale)
    _compare(got, ref, "bf16", "medium")


@pytest.mark.parametrize("D", [64, 128])
def test_backward_medium_fp32(D):
    # causal + softcap, fp32, S = 2048: sixteen q tiles per head, so the
    # two-stage chunk rings of the tensor-core kernels wrap many times
    B, H, S = 1, 2, 2048
    q, k, v, g = _draw(B, H, S, S, D, 36, "fp32")
    scale = 1.0 / np.sqrt(D)
    got = _backward(q, k, v, g, W.MASK_CAUSAL, W.SCORE_SOFTCAP, scale, "fp32", score_param=20.0)
    ref = oracle.attention_bwd(q, k, v, g, W.MASK_CAUSAL, W.SCORE_SOFTCAP, scale, score_param=20.0)
    _compare(got, ref, "fp32", f"medium fp32 D{D}")


@pytest.mark.parametrize("D", [64, 128])
def test_backward_fp32_long_q_side(D):
    # more than 2048 q tiles (Q_LEN 262400, KV_LEN 1024): dK/dV take the
    # CUDA-core kernels, dQ the tensor cores.  Sliding window 256: q row i
    # sees keys i - 255 .. i, so rows from 1279 on see none, and the exact
    # gradients are those of the first 1280 q rows alone (the oracle's)
    # with dq = 0 past them
    B, H, Sq, Skv, Sc, W_ = 1, 1, 262400, 1024, 1280, 256
    q, k, v = W.draw_qkv(B, H, Sc, D, seed=37, dtype="fp32", S_kv=Skv)
    g = W.draw_qkv(B, H, Sc, D, seed=38, dtype="fp32")[0]
    rng = np.random.default_rng(39)
    pad = lambda x: np.concatenate([x, rng.standard_normal((B, H, Sq - Sc, D), dtype=np.float32)], axis=2)
    got = _backward(pad(q), k, v, pad(g), W.MASK_SLIDING_WINDOW, W.SCORE_IDENTITY, 1.0 / np.sqrt(D), "fp32",
                    window=W_)
    ref = oracle.attention_bwd(q, k, v, g, W.MASK_SLIDING_WINDOW, W.SCORE_IDENTITY, 1.0 / np.sqrt(D), window=W_)
    assert np.all(got[0][:, :, Sc:] == 0.0), "dq past the last row with keys"
    _compare([got[0][:, :, :Sc], got[1], got[2]], ref, "fp32", f"long q side D{D}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_backward_under_graph_capture(dtype):
    # flex_attention_bwd recorded into a CUDA graph (dq on the library's side
    # stream, forked from and joined into the captured stream) and replayed
    # gives the eager call's gradients bit for bit
    B, H, S, D = 1, 2, 512, 64
    q, k, v, g = _draw(B, H, S, S, D, 40, dtype)
    dq_, dk_, dv_, dg = (device_tensor(x, dtype) for x in (q, k, v, g))
    bm = gpu_block_mask(W.MASK_CAUSAL, B, H, S, S, 0, 0, None)
    bq = fa.flex_block_mask_transpose(bm)
    out, lse = fa.flex_attention_fwd(dq_, dk_, dv_, bm, W.SCORE_ALIBI, 0.0, 0.125)
    eager = [x.clone() for x in fa.flex_attention_bwd(dq_, dk_, dv_, out, lse, dg, bm, bq, W.SCORE_ALIBI, 0.0, 0.125)]
    torch.cuda.synchronize()
    grads = [torch.full_like(x, float("nan")) for x in eager]
    delta = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fa.flex_attention_bwd(dq_, dk_, dv_, out, lse, dg, bm, bq, W.SCORE_ALIBI, 0.0, 0.125,
                              dq=grads[0], dk=grads[1], dv=grads[2], delta=delta)
    graph.replay()
    torch.cuda.synchronize()
    assert fa.flex_device_status() == fa.FLEX_OK
    for name, a, e in zip(("dq", "dk", "dv"), grads, eager):
        assert torch.equal(a, e), f"{dtype} {name}: replay differs from the eager call"


def test_backward_at_scale():
    # the headline shape's sequence length (causal + ALiBi, S = 16384, two
    # heads): dq on sampled rows against the oracle (a row's dq needs only
    # that row), and over every row the sums that the softmax fixes: each row
    # of dS sums to 0, so sum_j dK_j = 0, and sum_j dV_j = sum_i dO_i
    B, H, S, D = 1, 2, 16384, 128
    q, k, v, g = _draw(B, H, S, S, D, 35, "bf16")
    scale = 1.0 / np.sqrt(D)
    dq, dk, dv = _backward(q, k, v, g, W.MASK_CAUSAL, W.SCORE_ALIBI, scale, "bf16")
    rows = sample_rows(B, H, S, 256, seed=5)
    ref = oracle.attention_bwd_dq_rows(q, k, v, g, rows, W.MASK_CAUSAL, W.SCORE_ALIBI, scale)
    err = float(np.max(np.abs(dq.reshape(-1, D)[rows] - ref)))
    assert err <= REL["bf16"] * float(np.max(np.abs(ref))) + 1e-4, f"sampled dq rows: max-abs {err:.3e}"
    assert np.all(np.isfinite(dq)) and np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))
    gsum = g.astype(np.float64).sum(axis=2)
    assert np.max(np.abs(dv.sum(axis=2) - gsum)) <= 1e-2 * np.sqrt(S) * np.max(np.abs(dv)) + 1e-2 * np.max(np.abs(gsum))
    assert np.max(np.abs(dk.sum(axis=2))) <= 1e-2 * np.sqrt(S) * np.max(np.abs(dk))
