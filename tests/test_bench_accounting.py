"""The bench's FLOP accounting and its recorded-traffic lookup (CPU only).

Unmasked-block FLOPs are 4 * 128 * 128 * D per computed tile (full or
partial).  The per-(b, h) tile counts are pinned twice: by the numbers a
brute-force count gives for these masks (causal S256: 1 full + 2 partial;
causal with a 256-wide window at S2048: 15 + 30; causal or both below 1024
at S4096: 532 + 32), and by a numpy count of the dense mask in the test.
"""
import numpy as np
import pytest

import bench
import oracle
from block_sparse_masked_blockmask_gb300 import workloads as W


def dense_tile_counts(w):
    """(full, partial) 128 x 128 tiles of the workload's mask, from the dense boolean matrix."""
    i = np.arange(w.S)[:, None]
    j = np.arange(w.S)[None, :]
    if w.mask == W.MASK_CAUSAL:
        m = i >= j
    elif w.mask == W.MASK_SLIDING_WINDOW:
        m = (i >= j) & (i - j < w.window)
    elif w.mask == W.MASK_CAUSAL_PREFIX:
        m = (i >= j) | ((i <= w.prefix) & (j <= w.prefix))
    else:
        raise ValueError(w.mask)
    n = w.S // 128
    t = m.reshape(n, 128, n, 128).sum(axis=(1, 3))
    return int((t == 128 * 128).sum()), int(((t > 0) & (t < 128 * 128)).sum())


@pytest.mark.parametrize("w,full,partial", [(W.FP32_CAUSAL_S256, 1, 2), (W.BF16_WINDOW256_S2048, 15, 30),
                                            (W.BF16_PREFIX1024_S4096, 532, 32)], ids=lambda x: getattr(x, "name", x))
def test_unmasked_block_flops(w, full, partial):
    assert dense_tile_counts(w) == (full, partial)
    bm = oracle.workload_block_mask(w)
    assert set(bm["full_kv_num_blocks"].reshape(w.B * w.H, -1).sum(axis=1).tolist()) == {full}
    assert set(bm["kv_num_blocks"].reshape(w.B * w.H, -1).sum(axis=1).tolist()) == {partial}
    assert bench.unmasked_block_flops(w, bm) == w.B * w.H * (full + partial) * 4.0 * 128 * 128 * w.D


def test_headline_flops_closed_form():
    # causal S16384: 128 * 129 / 2 tiles per (b, h), B2 H32, D128
    w = W.BF16_CAUSAL_ALIBI_S16384
    assert w.B * w.H * (128 * 129 // 2) * 4.0 * 128 * 128 * w.D == pytest.approx(4.432e12, rel=1e-3)


def test_recorded_traffic_is_tied_to_its_workload():
    assert bench.recorded_traffic("no_such_workload") is None
    value = bench.recorded_traffic(W.BF16_CAUSAL_ALIBI_S16384.name)
    # present while the kernel sources match the digest it was captured with, else None
    assert value is None or value > 0.0
