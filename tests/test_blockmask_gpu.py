"""BlockMask build kernel vs the oracle: bit-exact on every int32 tensor."""
import numpy as np
import pytest

import oracle
from block_sparse_masked_blockmask_gb300 import workloads as W
from gpu_harness import block_masks_equal, gpu_block_mask

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", W.CONFIGS, ids=lambda w: w.name)
def test_configs_bit_exact(w):
    docs = W.document_ids(w.B, w.S, w.seed) if w.mask == W.MASK_DOCUMENT else None
    ref = oracle.workload_block_mask(w, docs)
    bm = gpu_block_mask(w.mask, w.B, w.H, w.S, w.S, w.window, w.prefix, docs)
    block_masks_equal(bm, ref, w.name)


@pytest.mark.parametrize("S", [128, 256, 384, 1024])
@pytest.mark.parametrize("window", [0, 1, 127, 128, 129, 256])
def test_sliding_window_sweep(S, window):
    ref = oracle.block_mask(W.MASK_SLIDING_WINDOW, 1, 2, S, S, 128, window=window)
    block_masks_equal(gpu_block_mask(W.MASK_SLIDING_WINDOW, 1, 2, S, S, window=window), ref, f"W{window}")


@pytest.mark.parametrize("S", [128, 256, 384, 1024])
@pytest.mark.parametrize("prefix", [0, 127, 128, 1024])
def test_causal_prefix_sweep(S, prefix):
    ref = oracle.block_mask(W.MASK_CAUSAL_PREFIX, 2, 1, S, S, 128, prefix=prefix)
    block_masks_equal(gpu_block_mask(W.MASK_CAUSAL_PREFIX, 2, 1, S, S, prefix=prefix), ref, f"P{prefix}")


@pytest.mark.parametrize("q_len,kv_len", [(128, 384), (384, 128), (256, 1024), (1024, 256)])
@pytest.mark.parametrize("mask", [W.MASK_CAUSAL, W.MASK_ALL, W.MASK_CAUSAL_PREFIX])
def test_rectangular(q_len, kv_len, mask):
    ref = oracle.block_mask(mask, 1, 3, q_len, kv_len, 128, prefix=200)
    block_masks_equal(gpu_block_mask(mask, 1, 3, q_len, kv_len, prefix=200), ref, "rect")


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_document_random_layouts(seed):
    S, B = 2048, 3
    rng = np.random.default_rng(seed)
    contiguous = W.document_ids(B, S, seed=seed, lo=60, hi=500)
    scattered = rng.integers(0, 3, size=(B, S)).astype(np.int32)  # ids need not be contiguous
    for docs in (contiguous, scattered):
        ref = oracle.block_mask(W.MASK_DOCUMENT, B, 2, S, S, 128, doc_ids=docs)
        block_masks_equal(gpu_block_mask(W.MASK_DOCUMENT, B, 2, S, S, doc_ids=docs), ref, "doc")


def test_max_kv_blocks():
    S = 128 * 1024
    ref = oracle.block_mask(W.MASK_SLIDING_WINDOW, 1, 1, S, S, 128, window=300)
    block_masks_equal(gpu_block_mask(W.MASK_SLIDING_WINDOW, 1, 1, S, S, window=300), ref, "max")
