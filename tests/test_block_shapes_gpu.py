"""BlockMasks whose blocks are not 128 x 128, and Q_BLOCK != KV_BLOCK.

The BlockMask tuple of the flex_attention op carries a Q block size and a KV
block size.  The build kernel writes the BlockMask at those sizes (bit-exact
against the oracle, kv side and q side); the attention and backward kernels
compute on 128 x 128 tiles and read a BlockMask of any of these sizes as such
tiles, so out, lse and the gradients must match the oracle within the same
tolerances as at 128 (the block sizes change which tiles are computed, never
the result).
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_masked_blockmask_gb300 import flexattn as fa
from block_sparse_masked_blockmask_gb300 import workloads as W
from gpu_harness import TOL, compare, device_tensor

pytestmark = pytest.mark.gpu

SHAPES = [(64, 64), (256, 256), (64, 128), (128, 256), (256, 64), (16, 1024), (1024, 32)]
MASKS = [
    (W.MASK_CAUSAL, {}),
    (W.MASK_SLIDING_WINDOW, {"window": 100}),
    (W.MASK_CAUSAL_PREFIX, {"prefix": 300}),
    (W.MASK_DOCUMENT, {}),
    (W.MASK_ALL, {}),
]


def _docs(B, S, seed):
    rng = np.random.default_rng(seed)
    d = np.zeros((B, S), np.int32)
    for b in range(B):
        for c in np.sort(rng.choice(np.arange(1, S), size=4, replace=False)):
            d[b, c:] += 1
    return d


def _bm(mask, B, H, q_len, kv_len, qbs, kbs, mkw, docs):
    dd = None if docs is None else torch.from_numpy(docs).cuda()
    bm = fa.flex_block_mask_create(mask, B, H, q_len, kv_len, qbs, kv_block=kbs, doc_ids=dd, **mkw)
    torch.cuda.synchronize()
    return bm


@pytest.mark.parametrize("qbs,kbs", SHAPES, ids=lambda x: str(x))
@pytest.mark.parametrize("mask,mkw", MASKS, ids=lambda x: str(x))
@pytest.mark.parametrize("q_len,kv_len", [(1000, 1000), (512, 512), (300, 700)])
def test_block_mask_bit_exact(qbs, kbs, mask, mkw, q_len, kv_len):
    if mask == W.MASK_DOCUMENT and q_len != kv_len:
        pytest.skip("document masks: Q_LEN == KV_LEN")
    B, H = 2, 2
    docs = _docs(B, q_len, 5) if mask == W.MASK_DOCUMENT else None
    bm = _bm(mask, B, H, q_len, kv_len, qbs, kbs, mkw, docs)
    ref = oracle.block_mask(mask, B, H, q_len, kv_len, qbs, kv_block=kbs, doc_ids=docs, **mkw)
    got = bm.as_numpy()
    for key, val in ref.items():
        assert np.array_equal(got[key], val), f"{key} {qbs}x{kbs} m{mask} {q_len}x{kv_len}"
    bq = fa.flex_block_mask_transpose(bm)
    torch.cuda.synchronize()
    refq = oracle.block_mask_q(mask, B, H, q_len, kv_len, qbs, kv_block=kbs, doc_ids=docs, **mkw)
    gotq = bq.as_numpy()
    for key, val in refq.items():
        assert np.array_equal(gotq[key], val), f"{key} {qbs}x{kbs} m{mask} {q_len}x{kv_len}"


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("qbs,kbs", SHAPES, ids=lambda x: str(x))
@pytest.mark.parametrize("mask,mkw", MASKS, ids=lambda x: str(x))
@pytest.mark.parametrize("score,param", [(W.SCORE_IDENTITY, 0.0), (W.SCORE_SOFTCAP, 20.0), (W.SCORE_ALIBI, 0.0)],
                         ids=lambda x: str(x))
def test_attention(dtype, qbs, kbs, mask, mkw, score, param):
    # S = 1000: ragged tail tiles at every block size
    B, H, S, D = 1, 2, 1000, 64
    q, k, v = W.draw_qkv(B, H, S, D, seed=41, dtype=dtype)
    docs = _docs(B, S, 6) if mask == W.MASK_DOCUMENT else None
    dq, dk, dv = (device_tensor(x, dtype) for x in (q, k, v))
    bm = _bm(mask, B, H, S, S, qbs, kbs, mkw, docs)
    scale = 1.0 / np.sqrt(D)
    out, lse = fa.flex_attention_fwd(dq, dk, dv, bm, score, param, scale)
    assert fa.flex_device_status() == fa.FLEX_OK
    ref_out, ref_lse = oracle.attention(q, k, v, mask, score, scale, doc_ids=docs, score_param=param, **mkw)
    compare(out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ref_out, ref_lse,
            dtype, f"{dtype} {qbs}x{kbs} m{mask} s{score}")


def test_attention_matches_block_128():
    # the headline kind at D = 128 with coarse and fine blocks: bit-identical
    # to the 128 x 128 BlockMask wherever both compute the same tiles with the
    # same full / partial classes (causal: 256 x 256 blocks make the diagonal
    # 128-tiles' neighbours partial, which changes nothing in the result)
    B, H, S, D = 1, 4, 2048, 128
    q, k, v = W.draw_qkv(B, H, S, D, seed=42)
    dq, dk, dv = (device_tensor(x, "bf16") for x in (q, k, v))
    outs = []
    for qbs, kbs in [(128, 128), (64, 64), (256, 256), (64, 256)]:
        bm = _bm(W.MASK_CAUSAL, B, H, S, S, qbs, kbs, {}, None)
        o, l = fa.flex_attention_fwd(dq, dk, dv, bm, W.SCORE_ALIBI, 0.0, 1 / np.sqrt(D))
        outs.append((o.float().cpu().numpy(), l.cpu().numpy()))
    # 64 x 64 blocks fold into exactly the 128-tiles and classes of 128 x 128
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    ref_out, ref_lse = oracle.attention(q, k, v, W.MASK_CAUSAL, W.SCORE_ALIBI, 1 / np.sqrt(D))
    for o, l in outs:
        compare(o.astype(np.float64), l.astype(np.float64), ref_out, ref_lse, "bf16", "causal alibi")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("qbs,kbs", [(64, 64), (256, 256), (64, 256), (256, 32)], ids=lambda x: str(x))
@pytest.mark.parametrize("mask,mkw", [(W.MASK_CAUSAL, {}), (W.MASK_DOCUMENT, {}),
                                      (W.MASK_CAUSAL_PREFIX, {"prefix": 300})], ids=lambda x: str(x))
def test_backward(dtype, qbs, kbs, mask, mkw):
    B, H, S, D = 1, 2, 700, 128
    q, k, v = W.draw_qkv(B, H, S, D, seed=43, dtype=dtype)
    g = W.draw_qkv(B, H, S, D, seed=44, dtype=dtype)[0]
    docs = _docs(B, S, 7) if mask == W.MASK_DOCUMENT else None
    dq_, dk_, dv_, dg = (device_tensor(x, dtype) for x in (q, k, v, g))
    bm = _bm(mask, B, H, S, S, qbs, kbs, mkw, docs)
    bq = fa.flex_block_mask_transpose(bm)
    scale = 1.0 / np.sqrt(D)
    out, lse = fa.flex_attention_fwd(dq_, dk_, dv_, bm, W.SCORE_ALIBI, 0.0, scale)
    grads = fa.flex_attention_bwd(dq_, dk_, dv_, out, lse, dg, bm, bq, W.SCORE_ALIBI, 0.0, scale)
    assert fa.flex_device_status() == fa.FLEX_OK
    ref = oracle.attention_bwd(q, k, v, g, mask, W.SCORE_ALIBI, scale, doc_ids=docs, **mkw)
    rel = {"bf16": 1e-2, "fp32": 1e-4}[dtype]
    for name, a, r in zip(("dq", "dk", "dv"), grads, ref):
        a = a.float().cpu().numpy().astype(np.float64)
        sc = max(1.0, float(np.max(np.abs(r)))) if dtype == "fp32" else float(np.max(np.abs(r)))
        err = float(np.max(np.abs(a - r)))
        assert err <= rel * sc + 1e-4, f"{dtype} {qbs}x{kbs} m{mask} {name}: {err:.3e}"
