"""Helpers for the GPU parity tests: move the seeded inputs to the device,
run the C-ABI path, and compare with the oracle."""
from __future__ import annotations

import numpy as np
import torch

from block_sparse_masked_blockmask_gb300 import flexattn as fa
from block_sparse_masked_blockmask_gb300 import workloads as W

# Tolerances of the path: bf16 inputs with fp32 accumulation, and fp32 inputs.
TOL = {"bf16": (1e-2, 5e-3), "fp32": (1e-4, 1e-4)}


def device_tensor(x: np.ndarray, dtype: str) -> torch.Tensor:
    """The exact values of x (already bf16-representable for bf16) on the GPU."""
    if dtype == "bf16":
        bits = W.bf16_bits(x).view(np.int16)
        return torch.from_numpy(bits).to("cuda").view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to("cuda")


def gpu_block_mask(mask, B, H, q_len, kv_len, window=0, prefix=0, doc_ids=None):
    dd = None if doc_ids is None else torch.from_numpy(np.ascontiguousarray(doc_ids, np.int32)).to("cuda")
    bm = fa.flex_block_mask_create(mask, B, H, q_len, kv_len, 128, window=window, prefix=prefix, doc_ids=dd)
    torch.cuda.synchronize()
    return bm


def run_attention(q, k, v, mask, score, scale, dtype, window=0, prefix=0, doc_ids=None, score_param=0.0,
                  device_inputs=None):
    """(out float64, lse float64, block mask) from the CUDA path."""
    if device_inputs is None:
        dq, dk, dv = (device_tensor(x, dtype) for x in (q, k, v))
    else:
        dq, dk, dv = device_inputs
    B, H, Sq, _ = dq.shape
    Skv = dk.shape[2]
    bm = gpu_block_mask(mask, B, H, Sq, Skv, window, prefix, doc_ids)
    out, lse = fa.flex_attention_fwd(dq, dk, dv, bm, score, score_param, scale)
    assert fa.flex_device_status() == fa.FLEX_OK
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), bm


def compare(out, lse, ref_out, ref_lse, dtype, what="", tol=None):
    """Element-wise max-abs check; -inf LSE (empty rows) must match exactly.

    tol: (out, lse) tolerances in place of the dtype's, for inputs outside
    the N(0, 1) draws those were set for (a scalar, or an array of
    per-element out bounds).
    """
    tol_out, tol_lse = TOL[dtype] if tol is None else tol
    assert out.shape == ref_out.shape and lse.shape == ref_lse.shape
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    empty = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: empty rows differ"
    assert np.all(np.isfinite(lse[~empty])), f"{what}: non-finite lse"
    if empty.any():
        assert np.all(out[empty] == 0.0), f"{what}: empty rows must be 0"
    err_l = float(np.max(np.abs(lse[~empty] - ref_lse[~empty]))) if (~empty).any() else 0.0
    if np.ndim(tol_out):
        over = np.abs(out - ref_out) - tol_out
        worst = float(np.max(over)) if out.size else -1.0
        assert worst <= 0.0, f"{what}: out exceeds its per-element bound by {worst:.3e}"
        err_o = float(np.max(np.abs(out - ref_out))) if out.size else 0.0
    else:
        err_o = float(np.max(np.abs(out - ref_out))) if out.size else 0.0
        assert err_o <= tol_out, f"{what}: out max-abs {err_o:.3e} > {tol_out:.0e}"
    assert err_l <= tol_lse, f"{what}: lse max-abs {err_l:.3e} > {tol_lse:.0e}"
    return err_o, err_l


def sample_rows(B: int, H: int, S: int, n: int, seed: int = 1) -> np.ndarray:
    """Flat row ids: every q-block's first and last row of a few heads, plus random rows."""
    rng = np.random.default_rng(seed)
    bh = rng.integers(0, B * H, size=4)
    edges = []
    for x in bh:
        for qb in range(0, S // 128, max(1, S // 128 // 8)):
            edges += [x * S + qb * 128, x * S + qb * 128 + 127]
    edges += [0, S - 1, (B * H - 1) * S, B * H * S - 1]
    rand = rng.integers(0, B * H * S, size=n)
    return np.unique(np.concatenate([np.asarray(edges, np.int64), rand.astype(np.int64)]))


def block_masks_equal(gpu_bm, ref: dict, what=""):
    got = gpu_bm.as_numpy()
    for key in ("kv_num_blocks", "kv_indices", "full_kv_num_blocks", "full_kv_indices"):
        assert got[key].dtype == np.int32
        assert np.array_equal(got[key], ref[key]), f"{what}: {key} differs"
