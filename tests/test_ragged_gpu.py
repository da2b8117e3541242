"""Lengths that are not multiples of the 128 block (tail tiles) vs the oracle.

The BlockMask is compared bit for bit (positions past a length count as
masked, so tail tiles are never full); attention out/lse/row max within the
usual tolerances (bf16 1e-2 / 5e-3, fp32 1e-4).  Buffers are followed by a
guard region that must come back untouched: no row past Q_LEN is written.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_masked_blockmask_gb300 import flexattn as fa
from block_sparse_masked_blockmask_gb300 import workloads as W
from gpu_harness import TOL, block_masks_equal, compare, device_tensor, gpu_block_mask, sample_rows

pytestmark = pytest.mark.gpu


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
@pytest.mark.parametrize("q_len,kv_len", [(1, 1), (127, 127), (129, 129), (300, 300), (1000, 1000), (4100, 4100),
                                          (200, 333), (333, 200), (5, 1000)])
def test_block_mask_ragged(mask, mkw, q_len, kv_len):
    if mask == W.MASK_DOCUMENT and (q_len != kv_len or q_len % 4):
        pytest.skip("document masks: Q_LEN == KV_LEN, a multiple of 4")
    B, H = 2, 3
    docs = _docs(B, q_len, 1) if mask == W.MASK_DOCUMENT else None
    bm = gpu_block_mask(mask, B, H, q_len, kv_len, doc_ids=docs, **mkw)
    ref = oracle.block_mask(mask, B, H, q_len, kv_len, 128, doc_ids=docs, **mkw)
    block_masks_equal(bm, ref, f"m{mask} {q_len}x{kv_len}")


def _guarded(shape, dtype):
    """A contiguous tensor of `shape` followed by a 4096-element guard of NaN bits."""
    n = int(np.prod(shape))
    flat = torch.empty(n + 4096, dtype=dtype, device="cuda")
    flat.fill_(float("nan"))
    return flat[:n].view(shape), flat[n:]


def _run(q, k, v, mask, score, scale, dtype, window=0, prefix=0, doc_ids=None, score_param=0.0):
    dq, dk, dv = (device_tensor(x, dtype) for x in (q, k, v))
    B, H, Sq, D = dq.shape
    bm = gpu_block_mask(mask, B, H, Sq, dk.shape[2], window, prefix, doc_ids)
    out, g_out = _guarded((B, H, Sq, D), dq.dtype)
    lse, g_lse = _guarded((B, H, Sq), torch.float32)
    mx, g_mx = _guarded((B, H, Sq), torch.float32)
    fa.flex_attention_fwd_opts(dq, dk, dv, bm, score, score_param, scale, out=out, lse=lse, max_scores=mx)
    assert fa.flex_device_status() == fa.FLEX_OK
    for g in (g_out, g_lse, g_mx):
        assert bool(torch.isnan(g.float()).all()), "a write past Q_LEN"
    f64 = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    return f64(out), f64(lse), f64(mx)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mask,mkw", MASKS, ids=lambda x: str(x))
@pytest.mark.parametrize("score,param", SCORES, ids=lambda x: str(x))
@pytest.mark.parametrize("S", [300, 1000])
def test_attention_ragged(dtype, D, mask, mkw, score, param, S):
    B, H = 2, 3
    q, k, v = W.draw_qkv(B, H, S, D, seed=21, dtype=dtype)
    docs = _docs(B, S, 2) if mask == W.MASK_DOCUMENT else None
    scale = 1.0 / np.sqrt(D)
    out, lse, mx = _run(q, k, v, mask, score, scale, dtype, doc_ids=docs, score_param=param, **mkw)
    ro, rl, rx = oracle.attention_opts(q, k, v, mask, score, scale, doc_ids=docs, score_param=param, **mkw)
    what = f"{dtype} D{D} m{mask} s{score} S{S}"
    compare(out, lse, ro, rl, dtype, what)
    fin = np.isfinite(rx)
    assert np.array_equal(np.isfinite(mx), fin), what
    assert np.max(np.abs(mx[fin] - rx[fin])) <= TOL[dtype][1], what


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("q_len,kv_len", [(1, 1), (1, 300), (129, 129), (200, 333), (333, 200), (130, 1)])
@pytest.mark.parametrize("mask,mkw", [(W.MASK_CAUSAL, {}), (W.MASK_CAUSAL_PREFIX, {"prefix": 150}),
                                      (W.MASK_ALL, {})], ids=lambda x: str(x))
def test_attention_ragged_rectangular(dtype, q_len, kv_len, mask, mkw):
    B, H, D = 1, 2, 128
    q, k, v = W.draw_qkv(B, H, q_len, D, seed=22, dtype=dtype, S_kv=kv_len)
    out, lse, mx = _run(q, k, v, mask, W.SCORE_ALIBI, 0.1, dtype, **mkw)
    ro, rl, rx = oracle.attention_opts(q, k, v, mask, W.SCORE_ALIBI, 0.1, **mkw)
    compare(out, lse, ro, rl, dtype, f"{dtype} {q_len}x{kv_len} m{mask}")


def test_attention_ragged_long():
    # causal + ALiBi, bf16, D = 128 at S = 5000 (39 tiles, a 8-row tail):
    # sampled rows against the oracle, properties over every row
    B, H, S, D = 1, 4, 5000, 128
    q, k, v = W.draw_qkv(B, H, S, D, seed=23, dtype="bf16")
    scale = 1.0 / np.sqrt(D)
    out, lse, mx = _run(q, k, v, W.MASK_CAUSAL, W.SCORE_ALIBI, scale, "bf16")
    tail = np.concatenate([h * S + np.arange(S - 8, S) for h in range(H)]).astype(np.int64)  # the 8 tail rows
    rows = np.unique(np.concatenate([sample_rows(B, H, S, 256, seed=4), tail]))
    ro, rl, rx = oracle.attention_opts(q, k, v, W.MASK_CAUSAL, W.SCORE_ALIBI, scale, rows=rows)
    compare(out.reshape(-1, D)[rows], lse.reshape(-1)[rows], ro, rl, "bf16", "ragged long")
    assert np.max(np.abs(mx.reshape(-1)[rows] - rx)) <= TOL["bf16"][1]
    n = np.arange(S, dtype=np.float64)[None, None, :] + 1.0
    assert np.all(np.isfinite(out)) and np.all(mx <= lse + 5e-3) and np.all(lse <= mx + np.log(n) + 5e-3)


@pytest.mark.parametrize("mask,mkw", [(W.MASK_CAUSAL, {}), (W.MASK_DOCUMENT, {})], ids=lambda x: str(x))
def test_host_api_ragged(mask, mkw):
    # flex_attention_fwd_host on ragged lengths: the same bits as the device path
    B, H, S, D = 2, 3, 1000, 128
    q, k, v = W.draw_qkv(B, H, S, D, seed=24, dtype="bf16")
    docs = _docs(B, S, 3) if mask == W.MASK_DOCUMENT else None
    dq, dk, dv = (device_tensor(x, "bf16") for x in (q, k, v))
    bm = gpu_block_mask(mask, B, H, S, S, doc_ids=docs)
    out, lse = fa.flex_attention_fwd(dq, dk, dv, bm, W.SCORE_ALIBI, 0.0, 0.09)
    torch.cuda.synchronize()
    hq, hk, hv = (x.cpu().pin_memory() for x in (dq, dk, dv))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    hlse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    hdoc = torch.from_numpy(docs).pin_memory() if docs is not None else None
    bufs = fa.DeviceBuffers(B, H, S, S, D, dq.dtype, document=docs is not None)
    fa.flex_attention_fwd_host(hq, hk, hv, bufs, mask, hout, hlse, doc_ids=hdoc, score_kind=W.SCORE_ALIBI,
                               score_param=0.0, scale=0.09, chunks=3)
    torch.cuda.synchronize()
    assert fa.flex_device_status() == fa.FLEX_OK
    assert torch.equal(hout, out.cpu()) and torch.equal(hlse, lse.cpu())
