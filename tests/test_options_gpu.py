"""Kernel options of the attention forward (flex_attention_fwd_opts) vs the oracle.

OUTPUT_MAX: the row max of the masked, modified scores, checked like lse
(bf16 5e-3, fp32 1e-4 max-abs; -inf rows exactly).  PRESCALE_QK: q rounded
to its dtype after scaling; the bf16 inputs here are drawn so that this
rounding moves lse by far more than the tolerance, so only a kernel that
rounds q~ as the oracle does passes.  ROWS_GUARANTEED_SAFE: results equal
the default call bit for bit.

Those bf16 inputs (|q| x 8, |k| x 4) make the scores spread by tens, so a
row's softmax sits on one or two keys.  The tensor-core path rounds P to
bf16 before P V (relative error <= 2^-9) and out to bf16 (another 2^-9), so
there out may be off by up to 2^-8 max|v| (0.016 for these v), not the 1e-2
that holds for N(0, 1) inputs where the weights spread over many keys; lse
keeps its 5e-3.  A CPU emulation of the kernel's arithmetic (q~ rounded as
the oracle does, fp32 scores, the thresholded running max, P in bf16) gives
1.5e-2 on the causal case, the GPU's figure; rounding q~ any other way moves
out by ~0.2 and lse by ~0.2.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_masked_blockmask_gb300 import flexattn as fa
from block_sparse_masked_blockmask_gb300 import workloads as W
from gpu_harness import TOL, compare, device_tensor, gpu_block_mask, sample_rows

pytestmark = pytest.mark.gpu


def _run(q, k, v, mask, score, scale, dtype, prescale=False, safe=False, output_max=True, window=0, prefix=0,
         doc_ids=None, score_param=0.0):
    dq, dk, dv = (device_tensor(x, dtype) for x in (q, k, v))
    bm = gpu_block_mask(mask, dq.shape[0], dq.shape[1], dq.shape[2], dk.shape[2], window, prefix, doc_ids)
    out, lse, mx = fa.flex_attention_fwd_opts(dq, dk, dv, bm, score, score_param, scale, prescale_qk=prescale,
                                              rows_guaranteed_safe=safe, output_max=output_max)
    assert fa.flex_device_status() == fa.FLEX_OK
    f64 = lambda t: None if t is None else t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    return f64(out), f64(lse), f64(mx)


def _compare_max(mx, ref_mx, dtype, what):
    empty = np.isneginf(ref_mx)
    assert np.array_equal(np.isneginf(mx), empty), f"{what}: empty rows differ"
    assert np.all(np.isfinite(mx[~empty])), f"{what}: non-finite row max"
    err = float(np.max(np.abs(mx[~empty] - ref_mx[~empty]))) if (~empty).any() else 0.0
    assert err <= TOL[dtype][1], f"{what}: row max max-abs {err:.3e} > {TOL[dtype][1]:.0e}"


def _docs(B, S, seed):
    rng = np.random.default_rng(seed)
    d = np.zeros((B, S), np.int32)
    for b in range(B):
        for c in np.sort(rng.choice(np.arange(1, S), size=3, replace=False)):
            d[b, c:] += 1
    return d


MASKS = [
    (W.MASK_CAUSAL, {}),
    (W.MASK_SLIDING_WINDOW, {"window": 100}),
    (W.MASK_CAUSAL_PREFIX, {"prefix": 200}),
    (W.MASK_DOCUMENT, {}),
    (W.MASK_ALL, {}),
]
SCORES = [(W.SCORE_IDENTITY, 0.0), (W.SCORE_SOFTCAP, 2.0), (W.SCORE_ALIBI, 0.0)]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mask,mkw", MASKS, ids=lambda x: str(x))
@pytest.mark.parametrize("score,param", SCORES, ids=lambda x: str(x))
def test_output_max(dtype, D, mask, mkw, score, param):
    # S = 384: three q blocks, one work item with a single Q tile
    B, H, S = 2, 3, 384
    q, k, v = W.draw_qkv(B, H, S, D, seed=11, dtype=dtype)
    docs = _docs(B, S, 4) if mask == W.MASK_DOCUMENT else None
    scale = 1.0 / np.sqrt(D)
    out, lse, mx = _run(q, k, v, mask, score, scale, dtype, doc_ids=docs, score_param=param, **mkw)
    ref_out, ref_lse, ref_mx = oracle.attention_opts(q, k, v, mask, score, scale, doc_ids=docs,
                                                     score_param=param, **mkw)
    what = f"{dtype} D{D} m{mask} s{score}"
    compare(out, lse, ref_out, ref_lse, dtype, what)
    _compare_max(mx, ref_mx, dtype, what)
    assert np.all(mx <= lse + TOL[dtype][1])


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_output_max_empty_rows(dtype):
    B, H, S, D = 1, 2, 256, 64
    q, k, v = W.draw_qkv(B, H, S, D, seed=12, dtype=dtype)
    out, lse, mx = _run(q, k, v, W.MASK_SLIDING_WINDOW, W.SCORE_ALIBI, 0.125, dtype, window=0)
    assert np.all(out == 0.0) and np.all(np.isneginf(lse)) and np.all(np.isneginf(mx))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("mask,mkw", MASKS, ids=lambda x: str(x))
def test_output_max_leaves_out_and_lse_alone(dtype, mask, mkw):
    B, H, S, D = 1, 4, 512, 128
    q, k, v = W.draw_qkv(B, H, S, D, seed=13, dtype=dtype)
    docs = _docs(B, S, 5) if mask == W.MASK_DOCUMENT else None
    dq, dk, dv = (device_tensor(x, dtype) for x in (q, k, v))
    bm = gpu_block_mask(mask, B, H, S, S, doc_ids=docs, **mkw)
    o0, l0 = fa.flex_attention_fwd(dq, dk, dv, bm, W.SCORE_ALIBI, 0.0, 0.09)
    o1, l1, m1 = fa.flex_attention_fwd_opts(dq, dk, dv, bm, W.SCORE_ALIBI, 0.0, 0.09, output_max=True)
    o2, l2, m2 = fa.flex_attention_fwd_opts(dq, dk, dv, bm, W.SCORE_ALIBI, 0.0, 0.09)
    torch.cuda.synchronize()
    assert m2 is None
    assert torch.equal(o0, o1) and torch.equal(l0, l1) and torch.equal(o0, o2) and torch.equal(l0, l2)


def _prescale_inputs(B, H, S, D, seed):
    # large |q| and |k|: bf16(scale q) differs from scale q by up to 2^-9
    # relative, which moves the scores (and lse) by ~1e-1, far above 5e-3
    q, k, v = W.draw_qkv(B, H, S, D, seed=seed, dtype="bf16")
    return W.round_to_bf16(q * 8.0), W.round_to_bf16(k * 4.0), v


@pytest.mark.parametrize("mask,mkw", MASKS, ids=lambda x: str(x))
@pytest.mark.parametrize("score,param", SCORES, ids=lambda x: str(x))
def test_prescale_bf16(mask, mkw, score, param):
    B, H, S, D = 1, 3, 384, 128
    q, k, v = _prescale_inputs(B, H, S, D, 14)
    docs = _docs(B, S, 6) if mask == W.MASK_DOCUMENT else None
    scale = 1.0 / np.sqrt(D)
    out, lse, mx = _run(q, k, v, mask, score, scale, "bf16", prescale=True, doc_ids=docs, score_param=param, **mkw)
    ref_out, ref_lse, ref_mx = oracle.attention_opts(q, k, v, mask, score, scale, doc_ids=docs, score_param=param,
                                                     prescale="bf16", **mkw)
    what = f"prescale bf16 m{mask} s{score}"
    compare(out, lse, ref_out, ref_lse, "bf16", what, tol=(max(TOL["bf16"][0], 2.0**-8 * np.max(np.abs(v))),
                                                         TOL["bf16"][1]))
    _compare_max(mx, ref_mx, "bf16", what)
    # the inputs do tell the rounding apart (softcap 2 squeezes the scores, so
    # there the rounding moves lse by less)
    _, plain_lse, _ = oracle.attention_opts(q, k, v, mask, score, scale, doc_ids=docs, score_param=param, **mkw)
    if score != W.SCORE_SOFTCAP:
        assert np.max(np.abs(plain_lse - ref_lse)) > 10 * TOL["bf16"][1], "inputs do not exercise the rounding"


@pytest.mark.parametrize("mask,mkw", MASKS, ids=lambda x: str(x))
@pytest.mark.parametrize("score,param", SCORES, ids=lambda x: str(x))
def test_prescale_fp32(mask, mkw, score, param):
    B, H, S, D = 1, 3, 384, 64
    q, k, v = W.draw_qkv(B, H, S, D, seed=15, dtype="fp32")
    docs = _docs(B, S, 7) if mask == W.MASK_DOCUMENT else None
    scale = 0.3
    out, lse, mx = _run(q, k, v, mask, score, scale, "fp32", prescale=True, doc_ids=docs, score_param=param, **mkw)
    ref_out, ref_lse, ref_mx = oracle.attention_opts(q, k, v, mask, score, scale, doc_ids=docs, score_param=param,
                                                     prescale="f32", **mkw)
    compare(out, lse, ref_out, ref_lse, "fp32", f"prescale fp32 m{mask} s{score}")
    _compare_max(mx, ref_mx, "fp32", f"prescale fp32 m{mask} s{score}")


def test_prescale_power_of_two_fp32_is_exact():
    # q * 2^-3 is exact, and so is every partial sum of the dot product
    B, H, S, D = 1, 2, 384, 128
    q, k, v = W.draw_qkv(B, H, S, D, seed=16, dtype="fp32")
    o0, l0, m0 = _run(q, k, v, W.MASK_CAUSAL, W.SCORE_ALIBI, 0.125, "fp32")
    o1, l1, m1 = _run(q, k, v, W.MASK_CAUSAL, W.SCORE_ALIBI, 0.125, "fp32", prescale=True)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1) and np.array_equal(m0, m1)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("mask,mkw", MASKS + [(W.MASK_SLIDING_WINDOW, {"window": 0})], ids=lambda x: str(x))
def test_rows_guaranteed_safe_changes_nothing(dtype, mask, mkw):
    # the promise holds for every mask here but W = 0, whose empty rows still
    # come out as out = 0, lse = -inf
    B, H, S, D = 1, 2, 512, 128
    q, k, v = W.draw_qkv(B, H, S, D, seed=17, dtype=dtype)
    docs = _docs(B, S, 8) if mask == W.MASK_DOCUMENT else None
    a = _run(q, k, v, mask, W.SCORE_SOFTCAP, 0.1, dtype, doc_ids=docs, score_param=20.0, **mkw)
    b = _run(q, k, v, mask, W.SCORE_SOFTCAP, 0.1, dtype, safe=True, doc_ids=docs, score_param=20.0, **mkw)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("prescale", [False, True])
def test_options_at_scale(prescale):
    # causal + ALiBi, bf16, D = 128 at S = 16384 (the long-sequence shape the
    # bench times, one batch and four heads): all options on, sampled rows
    B, H, S, D = 1, 4, 16384, 128
    q, k, v = W.draw_qkv(B, H, S, D, seed=18, dtype="bf16")
    scale = 1.0 / np.sqrt(D)
    out, lse, mx = _run(q, k, v, W.MASK_CAUSAL, W.SCORE_ALIBI, scale, "bf16", prescale=prescale, safe=True)
    rows = sample_rows(B, H, S, 256, seed=3)
    ref_out, ref_lse, ref_mx = oracle.attention_opts(q, k, v, W.MASK_CAUSAL, W.SCORE_ALIBI, scale, rows=rows,
                                                     prescale="bf16" if prescale else None)
    compare(out.reshape(-1, D)[rows], lse.reshape(-1)[rows], ref_out, ref_lse, "bf16", "options at scale")
    _compare_max(mx.reshape(-1)[rows], ref_mx, "bf16", "options at scale")
    # properties over every row: causal rows are never empty, max <= lse <= max + ln(q + 1)
    n = np.arange(S, dtype=np.float64)[None, None, :] + 1.0
    assert np.all(np.isfinite(mx)) and np.all(mx <= lse + 5e-3) and np.all(lse <= mx + np.log(n) + 5e-3)
