"""Pins that tie the float64 oracle to something other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with:
  * a library routine (PyTorch's CPU scaled-dot-product attention, which also
    returns the log-sum-exp) on cases that reduce to it: the all-true mask,
    the causal mask, the causal + bidirectional prefix mask (prefix rows are
    plain attention over keys 0..P, the rest causal), the document mask
    (causal attention inside each document slice), the sliding window (each
    row is plain attention over its window slice);
  * closed forms (ALiBi with zero scores is a truncated geometric series;
    softcap scores built through atanh; block counts of causal, sliding
    window and prefix masks; document tiles from the document intervals);
  * special cases (constant V, W = 1, W = 0, first causal row, a huge cap);
  * a pure-Python brute force on tiny shapes (math.exp, plain loops);
  * for the kernel options: PyTorch's float32 -> bfloat16 conversion and a
    nearest-neighbour check of the oracle's bfloat16 rounding, exact
    power-of-two prescaling, brute force on a prescaled q computed outside
    the oracle, and the bounds max S <= lse <= max S + ln n of the row max.

The mutation test compiles deliberately broken copies of oracle.c and checks
that at least one pin fails for each.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

from block_sparse_masked_blockmask_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _sdpa(q, k, v, scale, causal=False):
    """(out, lse) from PyTorch's CPU flash attention in float64."""
    tq, tk, tv = (torch.from_numpy(np.asarray(x, np.float64)) for x in (q, k, v))
    out, lse = torch.ops.aten._scaled_dot_product_flash_attention_for_cpu(
        tq, tk, tv, 0.0, causal, scale=scale)
    return out.numpy(), lse.numpy()


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


def _close(a, b, tol, what):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), f"{what}: finiteness differs"
    assert np.array_equal(a[~fin], b[~fin]), f"{what}: infinities differ"
    err = float(np.max(np.abs(a[fin] - b[fin]))) if fin.any() else 0.0
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


# --------------------------------------------------------------- library pins
def pin_all_true_mask_is_textbook_attention(orc):
    for (B, H, sq, skv, D, scale, seed) in [(2, 3, 40, 56, 8, 0.37, 1), (1, 2, 33, 33, 16, 0.25, 2)]:
        q, k, v = _rand((B, H, sq, D), seed), _rand((B, H, skv, D), seed + 1), _rand((B, H, skv, D), seed + 2)
        out, lse = orc.attention(q, k, v, W.MASK_ALL, W.SCORE_IDENTITY, scale)
        ro, rl = _sdpa(q, k, v, scale)
        _close(out, ro, 1e-12, "all-true out")
        _close(lse, rl, 1e-12, "all-true lse")


def pin_causal_mask_is_library_causal(orc):
    B, H, S, D, scale = 2, 2, 48, 8, 0.5
    q, k, v = _rand((B, H, S, D), 3), _rand((B, H, S, D), 4), _rand((B, H, S, D), 5)
    out, lse = orc.attention(q, k, v, W.MASK_CAUSAL, W.SCORE_IDENTITY, scale)
    ro, rl = _sdpa(q, k, v, scale, causal=True)
    _close(out, ro, 1e-12, "causal out")
    _close(lse, rl, 1e-12, "causal lse")


def pin_causal_prefix_splits_into_library_calls(orc):
    # rows q <= P attend to keys 0..P (both bounds inclusive); rows q > P are causal.
    B, H, S, D, P, scale = 1, 2, 40, 4, 13, 0.5
    q, k, v = _rand((B, H, S, D), 6), _rand((B, H, S, D), 7), _rand((B, H, S, D), 8)
    out, lse = orc.attention(q, k, v, W.MASK_CAUSAL_PREFIX, W.SCORE_IDENTITY, scale, prefix=P)
    po, pl = _sdpa(q[:, :, :P + 1], k[:, :, :P + 1], v[:, :, :P + 1], scale)
    co, cl = _sdpa(q, k, v, scale, causal=True)
    _close(out[:, :, :P + 1], po, 1e-12, "prefix rows out")
    _close(lse[:, :, :P + 1], pl, 1e-12, "prefix rows lse")
    _close(out[:, :, P + 1:], co[:, :, P + 1:], 1e-12, "causal rows out")
    _close(lse[:, :, P + 1:], cl[:, :, P + 1:], 1e-12, "causal rows lse")


def pin_document_mask_is_per_document_causal(orc):
    lengths = [5, 11, 3, 9]
    S, B, H, D, scale = sum(lengths), 1, 2, 4, 0.6
    doc = np.repeat(np.arange(len(lengths), dtype=np.int32), lengths)[None, :]
    q, k, v = _rand((B, H, S, D), 9), _rand((B, H, S, D), 10), _rand((B, H, S, D), 11)
    out, lse = orc.attention(q, k, v, W.MASK_DOCUMENT, W.SCORE_IDENTITY, scale, doc_ids=doc)
    s0 = 0
    for L in lengths:
        sl = slice(s0, s0 + L)
        ro, rl = _sdpa(q[:, :, sl], k[:, :, sl], v[:, :, sl], scale, causal=True)
        _close(out[:, :, sl], ro, 1e-12, "document out")
        _close(lse[:, :, sl], rl, 1e-12, "document lse")
        s0 += L


def pin_sliding_window_rows_are_window_slices(orc):
    B, H, S, D, Wd, scale = 1, 2, 24, 4, 5, 0.5
    q, k, v = _rand((B, H, S, D), 12), _rand((B, H, S, D), 13), _rand((B, H, S, D), 14)
    out, lse = orc.attention(q, k, v, W.MASK_SLIDING_WINDOW, W.SCORE_IDENTITY, scale, window=Wd)
    for i in range(S):
        lo = max(0, i - Wd + 1)
        ro, rl = _sdpa(q[:, :, i:i + 1], k[:, :, lo:i + 1], v[:, :, lo:i + 1], scale)
        _close(out[:, :, i:i + 1], ro, 1e-12, f"window row {i} out")
        _close(lse[:, :, i:i + 1], rl, 1e-12, f"window row {i} lse")


def pin_huge_softcap_is_identity(orc):
    B, H, S, D, scale = 1, 2, 20, 8, 0.35
    q, k, v = _rand((B, H, S, D), 15), _rand((B, H, S, D), 16), _rand((B, H, S, D), 17)
    out, lse = orc.attention(q, k, v, W.MASK_CAUSAL, W.SCORE_SOFTCAP, scale, score_param=1e30)
    ro, rl = _sdpa(q, k, v, scale, causal=True)
    _close(out, ro, 1e-12, "softcap 1e30 out")
    _close(lse, rl, 1e-12, "softcap 1e30 lse")


# ------------------------------------------------------------- closed forms
def pin_softcap_through_atanh(orc):
    # q = [1, 0], k_j = [c_j, 0], scale = 1: the scaled score of key j is c_j.  With
    # c_j = cap * atanh(x_j), cap * tanh(c_j / cap) = cap * x_j (up to the
    # float32 rounding of c_j), so the softcapped scores are known.
    cap = 50.0
    x = np.linspace(-0.06, 0.05, 17)
    kj = (cap * np.arctanh(x)).astype(np.float32)
    q = np.array([1.0, 0.0], np.float32).reshape(1, 1, 1, 2)
    k = np.stack([kj, np.zeros_like(kj)], -1)[None, None]
    v = np.stack([np.arange(x.size, dtype=np.float32), np.ones(x.size, np.float32)], -1)[None, None]
    out, lse = orc.attention(q, k, v, W.MASK_ALL, W.SCORE_SOFTCAP, 1.0, score_param=cap)
    s = cap * x
    p = np.exp(s - s.max())
    ref_lse = s.max() + math.log(p.sum())
    ref_out = (p / p.sum()) @ np.asarray(v[0, 0], np.float64)
    # float32 rounding of k_j moves each score by < 1e-5
    _close(lse[0, 0], [ref_lse], 1e-5, "softcap lse")
    _close(out[0, 0, 0], ref_out, 1e-4, "softcap out")


def pin_alibi_zero_scores_geometric(orc):
    # q = k = 0: scores are the bias -slope_h (i - j), slope_h = 2^(-8(h+1)/H).
    # Causal row i: weights r^d over d = i - j in 0..i with r = exp(-slope_h):
    #   lse_i = ln((1 - r^(i+1)) / (1 - r)),  E[d] = sum d r^d / sum r^d,
    #   out_i = [i - E[d], 1] for v_j = [j, 1].
    B, H, S = 1, 4, 20
    q = np.zeros((B, H, S, 2), np.float32)
    k = np.zeros((B, H, S, 2), np.float32)
    v = np.zeros((B, H, S, 2), np.float32)
    v[..., 0] = np.arange(S, dtype=np.float32)
    v[..., 1] = 1.0
    out, lse = orc.attention(q, k, v, W.MASK_CAUSAL, W.SCORE_ALIBI, 0.125)
    for h in range(H):
        r = math.exp(-(2.0 ** (-8.0 * (h + 1) / H)))
        for i in range(S):
            n = i
            zsum = (1 - r ** (n + 1)) / (1 - r)
            dsum = r * (1 - (n + 1) * r ** n + n * r ** (n + 1)) / (1 - r) ** 2
            _close([lse[0, h, i]], [math.log(zsum)], 1e-12, f"alibi lse h{h} i{i}")
            # the closed form cancels in (1 - r)^2 for small slopes: 1e-9
            _close(out[0, h, i], [i - dsum / zsum, 1.0], 1e-9, f"alibi out h{h} i{i}")


# ----------------------------------------------------------- special cases
def pin_constant_v_gives_constant_out(orc):
    B, H, S, D = 2, 2, 32, 4
    q, k = _rand((B, H, S, D), 18), _rand((B, H, S, D), 19)
    v = np.full((B, H, S, D), 0.75, np.float32)
    doc = np.repeat(np.arange(4, dtype=np.int32), 8)[None, :].repeat(B, 0)
    for mask, kw in [(W.MASK_CAUSAL, {}), (W.MASK_SLIDING_WINDOW, {"window": 3}),
                     (W.MASK_CAUSAL_PREFIX, {"prefix": 9}), (W.MASK_DOCUMENT, {"doc_ids": doc}),
                     (W.MASK_ALL, {})]:
        for score, sp in [(W.SCORE_IDENTITY, 0.0), (W.SCORE_SOFTCAP, 2.0), (W.SCORE_ALIBI, 0.0)]:
            out, lse = orc.attention(q, k, v, mask, score, 0.5, score_param=sp, **kw)
            assert np.all(np.isfinite(lse))
            # the weights sum to 1 up to a few double roundings per key
            assert np.max(np.abs(out - 0.75)) <= 1e-13, (mask, score)


def pin_window_one_and_zero(orc):
    B, H, S, D, scale = 1, 2, 16, 4, 0.5
    q, k, v = _rand((B, H, S, D), 20), _rand((B, H, S, D), 21), _rand((B, H, S, D), 22)
    out, lse = orc.attention(q, k, v, W.MASK_SLIDING_WINDOW, W.SCORE_IDENTITY, scale, window=1)
    _close(out, v, 1e-15, "W=1 out = v")
    diag = scale * np.einsum("bhsd,bhsd->bhs", q.astype(np.float64), k.astype(np.float64))
    _close(lse, diag, 1e-12, "W=1 lse = diagonal score")
    out0, lse0 = orc.attention(q, k, v, W.MASK_SLIDING_WINDOW, W.SCORE_IDENTITY, scale, window=0)
    assert np.all(out0 == 0.0) and np.all(np.isneginf(lse0)), "W=0 rows must be empty"


def pin_first_causal_row_is_v0(orc):
    B, H, S, D = 2, 2, 12, 4
    q, k, v = _rand((B, H, S, D), 23), _rand((B, H, S, D), 24), _rand((B, H, S, D), 25)
    for score, sp in [(W.SCORE_IDENTITY, 0.0), (W.SCORE_SOFTCAP, 3.0), (W.SCORE_ALIBI, 0.0)]:
        out, _ = orc.attention(q, k, v, W.MASK_CAUSAL, score, 0.5, score_param=sp)
        _close(out[:, :, 0], v[:, :, 0], 1e-15, "causal row 0")


def pin_alibi_diagonal_has_no_bias(orc):
    # Sliding window W=1 keeps only the diagonal, where the ALiBi bias is 0.
    B, H, S, D = 1, 4, 10, 4
    q, k, v = _rand((B, H, S, D), 26), _rand((B, H, S, D), 27), _rand((B, H, S, D), 28)
    _, la = orc.attention(q, k, v, W.MASK_SLIDING_WINDOW, W.SCORE_ALIBI, 0.5, window=1)
    _, li = orc.attention(q, k, v, W.MASK_SLIDING_WINDOW, W.SCORE_IDENTITY, 0.5, window=1)
    _close(la, li, 0.0, "alibi diagonal")


# -------------------------------------------------------- block-mask forms
def _rows_are_permutations(bm):
    for key in ("kv_indices", "full_kv_indices"):
        idx = bm[key]
        n = idx.shape[-1]
        assert np.array_equal(np.sort(idx, axis=-1), np.broadcast_to(np.arange(n), idx.shape)), key


def _expected_lists(status_rows):
    """status_rows [NQB, NKVB] in {0 empty, 1 partial, 2 full} -> the four tensors (one (b,h))."""
    nq, nk = status_rows.shape
    out = {k: [] for k in ("kv_num_blocks", "kv_indices", "full_kv_num_blocks", "full_kv_indices")}
    for r in range(nq):
        part = [j for j in range(nk) if status_rows[r, j] == 1]
        full = [j for j in range(nk) if status_rows[r, j] == 2]
        out["kv_num_blocks"].append(len(part))
        out["kv_indices"].append(part + [j for j in range(nk) if j not in part])
        out["full_kv_num_blocks"].append(len(full))
        out["full_kv_indices"].append(full + [j for j in range(nk) if j not in full])
    return {k: np.asarray(v, np.int32) for k, v in out.items()}


def _check_lists(bm, status, what):
    """status: [B, H, NQB, NKVB] expected tile classes."""
    _rows_are_permutations(bm)
    B, H = status.shape[:2]
    for b in range(B):
        for h in range(H):
            exp = _expected_lists(status[b, h])
            for key, val in exp.items():
                assert np.array_equal(bm[key][b, h], val), f"{what}: {key} (b={b}, h={h})"


def pin_causal_block_counts_closed_form(orc):
    for nb in (1, 2, 5, 16):
        S = nb * 128
        bm = orc.block_mask(W.MASK_CAUSAL, 1, 2, S, S, 128)
        assert bm["full_kv_num_blocks"].sum() == 2 * nb * (nb - 1) // 2
        assert bm["kv_num_blocks"].sum() == 2 * nb
        qb = np.arange(nb)[:, None]
        kb = np.arange(nb)[None, :]
        status = np.where(kb < qb, 2, np.where(kb == qb, 1, 0))
        _check_lists(bm, np.broadcast_to(status, (1, 2, nb, nb)), f"causal nb={nb}")


def pin_ragged_causal_block_counts_closed_form(orc):
    # S not a multiple of 128: the mask is padded with false to whole tiles, so
    # in the last q block (rows past S are padding) every tile 0..qb holds
    # some true pairs but none is full; the other rows are as for whole tiles
    # (kv tile NB-1 sits above their diagonal, empty)
    for S in (1, 127, 129, 300, 1000):
        nb = -(-S // 128)
        bm = orc.block_mask(W.MASK_CAUSAL, 1, 2, S, S, 128)
        qb = np.arange(nb)[:, None]
        kb = np.arange(nb)[None, :]
        status = np.where(kb < qb, 2, np.where(kb == qb, 1, 0))
        status[nb - 1, :] = 1
        _check_lists(bm, np.broadcast_to(status, (1, 2, nb, nb)), f"ragged causal S={S}")
    # rectangular: Q_LEN 200, KV_LEN 333 with the all-true mask: only the tile
    # of whole rows and whole columns (q block 0, kv blocks 0 and 1) is full
    bm = orc.block_mask(W.MASK_ALL, 1, 1, 200, 333, 128)
    status = np.array([[2, 2, 1], [1, 1, 1]])
    _check_lists(bm, status[None, None], "ragged all-true 200x333")


def pin_sliding_window_block_counts_closed_form(orc):
    # W = 256 = 2 blocks: row qb has kv block qb-1 full, qb-2 and qb partial.
    nb, S = 16, 2048
    bm = orc.block_mask(W.MASK_SLIDING_WINDOW, 2, 1, S, S, 128, window=256)
    assert np.all(bm["kv_num_blocks"].sum(-1) == nb + (nb - 2))
    assert np.all(bm["full_kv_num_blocks"].sum(-1) == nb - 1)
    qb = np.arange(nb)[:, None]
    kb = np.arange(nb)[None, :]
    status = np.where(kb == qb - 1, 2, np.where((kb == qb) | (kb == qb - 2), 1, 0))
    _check_lists(bm, np.broadcast_to(status, (2, 1, nb, nb)), "window 256")


def pin_causal_prefix_block_counts_closed_form(orc):
    # P = 1024 (inclusive): q blocks 0..8 see kv blocks 0..7 in full and kv
    # block 8 (which holds only kv = 1024 for rows < 1024, and is the diagonal
    # for q block 8) as partial; q blocks >= 9 are causal.
    nb, S, P = 32, 4096, 1024
    bm = orc.block_mask(W.MASK_CAUSAL_PREFIX, 1, 2, S, S, 128, prefix=P)
    assert np.all(bm["full_kv_num_blocks"].sum(-1) == 532)
    assert np.all(bm["kv_num_blocks"].sum(-1) == 32)
    status = np.zeros((nb, nb), np.int64)
    for r in range(nb):
        if r <= 8:
            status[r, :8] = 2
            status[r, 8] = 1
        else:
            status[r, :r] = 2
            status[r, r] = 1
    _check_lists(bm, np.broadcast_to(status, (1, 2, nb, nb)), "prefix 1024")


def pin_document_blocks_from_intervals(orc):
    # Contiguous documents: a tile below the diagonal is full when its rows and
    # columns lie in one document, partial when the last column's document is
    # the first row's document, empty otherwise; the diagonal tile is partial.
    B, S, blk = 2, 2048, 128
    doc = W.document_ids(B, S, seed=3, lo=100, hi=700)
    bm = orc.block_mask(W.MASK_DOCUMENT, B, 1, S, S, blk, doc_ids=doc)
    nb = S // blk
    status = np.zeros((B, 1, nb, nb), np.int64)
    for b in range(B):
        d = doc[b]
        for qb in range(nb):
            r0, r1 = d[qb * blk], d[qb * blk + blk - 1]
            for kb in range(qb + 1):
                c0, c1 = d[kb * blk], d[kb * blk + blk - 1]
                if kb == qb:
                    status[b, 0, qb, kb] = 1
                elif r0 == r1 == c0 == c1:
                    status[b, 0, qb, kb] = 2
                elif c1 == r0:
                    status[b, 0, qb, kb] = 1
    _check_lists(bm, status, "document")


def pin_golden_causal_prefix_predicate(orc):
    path = os.path.join(GOLDEN, "causal_prefix_predicate.txt")
    n = 0
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            P, qi, kv, expect = (int(x) for x in line.split())
            got = orc.mask_value(W.MASK_CAUSAL_PREFIX, qi, kv, prefix=P)
            assert got == bool(expect), (P, qi, kv, expect)
            n += 1
    assert n >= 8


# ------------------------------------------------------------ brute force
def _bf_mask(kind, b, h, i, j, window, prefix, doc):
    if kind == W.MASK_CAUSAL:
        return i >= j
    if kind == W.MASK_SLIDING_WINDOW:
        return i >= j and i - j < window
    if kind == W.MASK_CAUSAL_PREFIX:
        return (i <= prefix and j <= prefix) or i >= j
    if kind == W.MASK_DOCUMENT:
        return doc[b][i] == doc[b][j] and i >= j
    return True


def _bf_score(kind, param, t, h, H, i, j):
    if kind == W.SCORE_SOFTCAP:
        return param * math.tanh(t / param)
    if kind == W.SCORE_ALIBI:
        return t - 2.0 ** (-8.0 * (h + 1) / H) * (i - j)
    return t


def brute_force(q, k, v, mask, score, scale, window=0, prefix=0, doc=None, param=0.0, block=2, kv_block=None):
    """Plain Python loops: (out, lse, block status, row max) for tiny shapes.

    Tiles are block (Q_BLOCK) rows by kv_block (KV_BLOCK, default: block) columns."""
    kv_block = block if kv_block is None else kv_block
    B, H, S, D = q.shape
    out = [[[[0.0] * D for _ in range(S)] for _ in range(H)] for _ in range(B)]
    lse = [[[0.0] * S for _ in range(H)] for _ in range(B)]
    rmax = [[[0.0] * S for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            for i in range(S):
                row = []
                for j in range(S):
                    if _bf_mask(mask, b, h, i, j, window, prefix, doc):
                        t = scale * math.fsum(float(q[b, h, i, d]) * float(k[b, h, j, d]) for d in range(D))
                        row.append((j, _bf_score(score, param, t, h, H, i, j)))
                if not row:
                    lse[b][h][i] = -math.inf
                    rmax[b][h][i] = -math.inf
                    continue
                mx = max(s for _, s in row)
                rmax[b][h][i] = mx
                L = mx + math.log(math.fsum(math.exp(s - mx) for _, s in row))
                lse[b][h][i] = L
                for d in range(D):
                    out[b][h][i][d] = math.fsum(math.exp(s - L) * float(v[b, h, j, d]) for j, s in row)
    nqb, nkb = -(-S // block), -(-S // kv_block)  # tiles past S are padded with false
    status = np.zeros((B, H, nqb, nkb), np.int64)
    for b in range(B):
        for h in range(H):
            for qb in range(nqb):
                for kb in range(nkb):
                    c = sum(_bf_mask(mask, b, h, i, j, window, prefix, doc)
                            for i in range(qb * block, min(S, qb * block + block))
                            for j in range(kb * kv_block, min(S, kb * kv_block + kv_block)))
                    status[b, h, qb, kb] = 2 if c == block * kv_block else (1 if c else 0)
    return np.asarray(out), np.asarray(lse), status, np.asarray(rmax)


def pin_brute_force_block_shapes(orc):
    # BlockMasks whose Q block and KV block differ (the tuple carries both
    # sizes), against the brute-force tile classes of the same dense mask
    B, H = 2, 1
    for S, qbs, kbs in [(12, 2, 4), (12, 4, 2), (13, 4, 2), (10, 2, 4), (16, 8, 2), (9, 1, 4)]:
        q = k = v = _rand((B, H, S, 2), S)
        doc = np.zeros((B, S), np.int32)
        doc[0, S // 3:] = 1
        doc[1, S // 2:] = 1
        for mask, kw in [(W.MASK_CAUSAL, {}), (W.MASK_SLIDING_WINDOW, {"window": 3}),
                         (W.MASK_CAUSAL_PREFIX, {"prefix": 5}), (W.MASK_DOCUMENT, {"doc": doc}),
                         (W.MASK_ALL, {})]:
            _, _, bs, _ = brute_force(q, k, v, mask, W.SCORE_IDENTITY, 0.5, block=qbs, kv_block=kbs,
                                      window=kw.get("window", 0), prefix=kw.get("prefix", 0), doc=kw.get("doc"))
            okw = {"window": kw.get("window", 0), "prefix": kw.get("prefix", 0), "doc_ids": kw.get("doc")}
            bm = orc.block_mask(mask, B, H, S, S, qbs, kv_block=kbs, **okw)
            _check_lists(bm, bs, f"brute block mask S{S} {qbs}x{kbs} m{mask}")
            bq = orc.block_mask_q(mask, B, H, S, S, qbs, kv_block=kbs, **okw)
            for b in range(B):
                for h in range(H):
                    exp = _expected_lists(bs[b, h].T)
                    for key, qkey in (("kv_num_blocks", "q_num_blocks"), ("kv_indices", "q_indices"),
                                      ("full_kv_num_blocks", "full_q_num_blocks"),
                                      ("full_kv_indices", "full_q_indices")):
                        assert np.array_equal(bq[qkey][b, h], exp[key]), f"{qkey} S{S} {qbs}x{kbs} m{mask}"


def pin_causal_block_shapes_closed_form(orc):
    # causal, Q_BLOCK a and KV_BLOCK c: tile (i, j) holds rows a i .. a i + a - 1
    # and columns c j .. c j + c - 1; it is full when its first row reaches
    # its last column (a i >= c j + c - 1) and empty when its last row is
    # before its first column (a i + a - 1 < c j)
    for S, a, c in [(1024, 64, 128), (1024, 128, 64), (1024, 256, 128), (1000, 64, 256), (768, 256, 64)]:
        bm = orc.block_mask(W.MASK_CAUSAL, 1, 1, S, S, a, kv_block=c)
        nqb, nkb = -(-S // a), -(-S // c)
        for i in range(nqb):
            full = [j for j in range(nkb) if a * i >= c * j + c - 1 and c * j + c <= S and a * i + a <= S]
            part = [j for j in range(nkb) if not (a * i + a - 1 < c * j) and j not in full]
            assert list(bm["full_kv_indices"][0, 0, i, :len(full)]) == full, (S, a, c, i)
            assert list(bm["kv_indices"][0, 0, i, :len(part)]) == part, (S, a, c, i)
            assert bm["full_kv_num_blocks"][0, 0, i] == len(full) and bm["kv_num_blocks"][0, 0, i] == len(part)


def pin_brute_force_tiny(orc):
    B, H, D = 2, 2, 3
    for S, block in [(8, 2), (12, 4), (16, 4), (7, 2), (10, 4), (13, 4)]:
        q, k, v = _rand((B, H, S, D), S), _rand((B, H, S, D), S + 1), _rand((B, H, S, D), S + 2)
        doc = np.zeros((B, S), np.int32)
        doc[0, S // 3:] = 1
        doc[1, S // 2:] = 1
        doc[1, S - 2:] = 2
        for mask, kw in [(W.MASK_CAUSAL, {}), (W.MASK_SLIDING_WINDOW, {"window": 3}),
                         (W.MASK_CAUSAL_PREFIX, {"prefix": 5}), (W.MASK_DOCUMENT, {"doc": doc}),
                         (W.MASK_ALL, {})]:
            for score, sp in [(W.SCORE_IDENTITY, 0.0), (W.SCORE_SOFTCAP, 0.9), (W.SCORE_ALIBI, 0.0)]:
                bo, bl, bs, bx = brute_force(q, k, v, mask, score, 0.7, param=sp, block=block,
                                             window=kw.get("window", 0), prefix=kw.get("prefix", 0),
                                             doc=kw.get("doc"))
                okw = {"window": kw.get("window", 0), "prefix": kw.get("prefix", 0),
                       "doc_ids": kw.get("doc")}
                oo, ol = orc.attention(q, k, v, mask, score, 0.7, score_param=sp, **okw)
                _close(oo, bo, 1e-12, f"brute out S{S} m{mask} s{score}")
                _close(ol, bl, 1e-12, f"brute lse S{S} m{mask} s{score}")
                _, _, ox = orc.attention_opts(q, k, v, mask, score, 0.7, score_param=sp, **okw)
                _close(ox, bx, 1e-12, f"brute row max S{S} m{mask} s{score}")
                bm = orc.block_mask(mask, B, H, S, S, block, **okw)
                _check_lists(bm, bs, f"brute block mask S{S} m{mask}")


# ------------------------------------------------------------ kernel options
def _bf16(x):
    """float32 values -> bfloat16 values by PyTorch's conversion (one rounding, ties to even)."""
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16).float().numpy()


def pin_round_bf16_is_library_conversion(orc):
    # float32 inputs: PyTorch's float32 -> bfloat16 conversion is the reference
    rng = np.random.default_rng(40)
    bits = rng.integers(0, 2**31 - 1, 4000, dtype=np.int64).astype(np.uint32)
    bits = bits[(bits & 0x7F800000) != 0x7F800000]                       # no inf / nan
    ties = (rng.integers(0, 0x7F7F, 2000, dtype=np.int64).astype(np.uint32) << 16) | 0x8000
    edge = np.array([0x7F7F0000, 0x7F7F7FFF, 0x7F7F8000, 0x7F7F8001, 0x7F7FFFFF, 0x7F000000,
                     0x00800000, 0x00807FFF, 0x00808000, 0x00018000, 0x00008000, 0x00007FFF,
                     0x00000001, 0x3F808000, 0x3F818000], np.uint32)
    x = np.concatenate([bits, ties, edge]).view(np.float32)
    x = np.concatenate([x, -x])
    ref = _bf16(x).astype(np.float64)
    got = np.array([orc.round_bf16(float(t)) for t in x])
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, f"bf16 rounding differs at {x[bad[:4]]}: {got[bad[:4]]} vs {ref[bad[:4]]}"


def pin_round_bf16_nearest_on_exact_products(orc):
    # scale * q (q bfloat16, scale float32) has up to 32 significant bits: the
    # result must be a bfloat16 no farther from x than either bfloat16
    # neighbour, and the even one on a tie
    rng = np.random.default_rng(41)
    q = _bf16(rng.standard_normal(3000).astype(np.float32))
    for scale in (1 / math.sqrt(128), 1 / math.sqrt(96), 0.3):
        x = q.astype(np.float64) * float(np.float32(scale))
        r = np.array([orc.round_bf16(t) for t in x])
        rb = torch.from_numpy(r.astype(np.float32)).to(torch.bfloat16)
        assert np.array_equal(rb.float().numpy().astype(np.float64), r), "not a bfloat16 value"
        b = rb.view(torch.int16).numpy().astype(np.int32)
        d0 = np.abs(x - r)
        for off in (-1, 1):
            nb = torch.from_numpy((b + off).astype(np.int16)).view(torch.bfloat16).float().numpy()
            d1 = np.abs(x - nb.astype(np.float64))
            assert np.all(d0 <= d1), f"a neighbour is nearer (scale {scale})"
            assert np.all((b[d0 == d1] & 1) == 0), f"tie not to even (scale {scale})"


def pin_prescale_power_of_two_scale_changes_nothing(orc):
    # scale = 2^-3 multiplies exactly in both storage types
    B, H, S, D = 1, 2, 24, 8
    q, k, v = _bf16(_rand((B, H, S, D), 42)), _bf16(_rand((B, H, S, D), 43)), _rand((B, H, S, D), 44)
    for mask, kw in [(W.MASK_CAUSAL, {}), (W.MASK_SLIDING_WINDOW, {"window": 5})]:
        for score, sp in [(W.SCORE_IDENTITY, 0.0), (W.SCORE_SOFTCAP, 1.5), (W.SCORE_ALIBI, 0.0)]:
            o0, l0, m0 = orc.attention_opts(q, k, v, mask, score, 0.125, score_param=sp, **kw)
            for ps in ("bf16", "f32"):
                o1, l1, m1 = orc.attention_opts(q, k, v, mask, score, 0.125, score_param=sp,
                                                prescale=ps, **kw)
                _close(o1, o0, 0.0, f"prescale {ps} out")
                _close(l1, l0, 0.0, f"prescale {ps} lse")
                _close(m1, m0, 0.0, f"prescale {ps} row max")


def pin_prescale_is_attention_on_rounded_q(orc):
    # bfloat16: a scale with 8 significant bits keeps scale * q exact in
    # float32, so PyTorch's conversion gives q~ with one rounding; float32:
    # numpy rounds the exact double product once.  Brute force on q~, scale 1.
    B, H, S, D = 1, 2, 12, 4
    k, v = _rand((B, H, S, D), 46), _rand((B, H, S, D), 47)
    qb = _bf16(_rand((B, H, S, D), 45) * 3.0)
    qf = _rand((B, H, S, D), 48)
    cases = [("bf16", qb, 179 / 256, _bf16((qb.astype(np.float64) * (179 / 256)).astype(np.float32))),
             ("f32", qf, float(np.float32(0.3)), (qf.astype(np.float64) * float(np.float32(0.3))).astype(np.float32))]
    for ps, q, scale, qt in cases:
        assert not np.array_equal(qt.astype(np.float64), q.astype(np.float64) * scale), "no rounding exercised"
        for mask, kw in [(W.MASK_CAUSAL, {}), (W.MASK_ALL, {})]:
            for score, sp in [(W.SCORE_IDENTITY, 0.0), (W.SCORE_SOFTCAP, 0.9), (W.SCORE_ALIBI, 0.0)]:
                bo, bl, _, bx = brute_force(qt, k, v, mask, score, 1.0, param=sp, block=4, **kw)
                oo, ol, ox = orc.attention_opts(q, k, v, mask, score, scale, score_param=sp,
                                                prescale=ps, **kw)
                _close(oo, bo, 1e-12, f"prescale {ps} out m{mask} s{score}")
                _close(ol, bl, 1e-12, f"prescale {ps} lse m{mask} s{score}")
                _close(ox, bx, 1e-12, f"prescale {ps} row max m{mask} s{score}")


def pin_row_max_bounds_lse(orc):
    # max_j S_j <= ln sum_j exp(S_j) <= max_j S_j + ln n over the n unmasked
    # keys of a row; equality on the left when n = 1; empty rows give -inf
    B, H, S, D = 2, 2, 40, 8
    q, k, v = _rand((B, H, S, D), 49), _rand((B, H, S, D), 50), _rand((B, H, S, D), 51)
    doc = np.repeat(np.arange(5, dtype=np.int32), 8)[None, :].repeat(B, 0)
    for mask, kw, bkw in [(W.MASK_CAUSAL, {}, {}), (W.MASK_SLIDING_WINDOW, {"window": 7}, {"window": 7}),
                          (W.MASK_CAUSAL_PREFIX, {"prefix": 11}, {"prefix": 11}),
                          (W.MASK_DOCUMENT, {"doc_ids": doc}, {"doc": doc}), (W.MASK_ALL, {}, {})]:
        n = np.array([[[sum(_bf_mask(mask, b, h, i, j, bkw.get("window", 0), bkw.get("prefix", 0),
                                     bkw.get("doc")) for j in range(S))
                        for i in range(S)] for h in range(H)] for b in range(B)], np.float64)
        for score, sp in [(W.SCORE_IDENTITY, 0.0), (W.SCORE_SOFTCAP, 2.0), (W.SCORE_ALIBI, 0.0)]:
            _, lse, mx = orc.attention_opts(q, k, v, mask, score, 0.6, score_param=sp, **kw)
            assert np.all(mx <= lse + 1e-12), (mask, score)
            assert np.all(lse <= mx + np.log(n) + 1e-12), (mask, score)
    _, lse, mx = orc.attention_opts(q, k, v, W.MASK_SLIDING_WINDOW, W.SCORE_ALIBI, 0.6, window=1)
    _close(mx, lse, 1e-12, "W=1 row max = lse")
    o0, l0, m0 = orc.attention_opts(q, k, v, W.MASK_SLIDING_WINDOW, W.SCORE_IDENTITY, 0.6, window=0)
    assert np.all(np.isneginf(m0)) and np.all(np.isneginf(l0)) and np.all(o0 == 0.0), "W=0 rows"


# ------------------------------------------------------------------ backward
def _dense_mask(kind, B, S, window=0, prefix=0, doc=None):
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    if kind == W.MASK_CAUSAL:
        m = i >= j
    elif kind == W.MASK_SLIDING_WINDOW:
        m = (i >= j) & (i - j < window)
    elif kind == W.MASK_CAUSAL_PREFIX:
        m = ((i <= prefix) & (j <= prefix)) | (i >= j)
    elif kind == W.MASK_DOCUMENT:
        return np.stack([(doc[b][:, None] == doc[b][None, :]) & (i >= j) for b in range(B)])[:, None]
    else:
        m = np.ones((S, S), bool)
    return np.broadcast_to(m, (B, 1, S, S))


def _sdpa_grads(q, k, v, dout, scale, attn_mask):
    """(dq, dk, dv) of sum(dout * out) through PyTorch's float64 CPU attention (autograd)."""
    tq, tk, tv = (torch.tensor(np.asarray(x, np.float64), requires_grad=True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=attn_mask, scale=scale)
    out.backward(torch.tensor(np.asarray(dout, np.float64)))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


def pin_backward_is_library_autograd(orc):
    # identity score: a boolean mask; ALiBi: the bias as an additive float mask
    B, H, S, D, scale = 2, 3, 40, 8, 0.45
    q, k, v, g = (_rand((B, H, S, D), 60 + t) for t in range(4))
    doc = np.repeat(np.arange(5, dtype=np.int32), 8)[None, :].repeat(B, 0)
    for mask, kw in [(W.MASK_CAUSAL, {}), (W.MASK_SLIDING_WINDOW, {"window": 6}),
                     (W.MASK_CAUSAL_PREFIX, {"prefix": 13}), (W.MASK_DOCUMENT, {"doc": doc}), (W.MASK_ALL, {})]:
        dm = _dense_mask(mask, B, S, kw.get("window", 0), kw.get("prefix", 0), kw.get("doc"))
        okw = {"window": kw.get("window", 0), "prefix": kw.get("prefix", 0), "doc_ids": kw.get("doc")}
        ref = _sdpa_grads(q, k, v, g, scale, torch.from_numpy(np.ascontiguousarray(dm)))
        got = orc.attention_bwd(q, k, v, g, mask, W.SCORE_IDENTITY, scale, **okw)
        for name, a, b in zip("qkv", got, ref):
            _close(a, b, 1e-10, f"backward d{name} m{mask} identity")
        slopes = 2.0 ** (-8.0 * (np.arange(H) + 1) / H)
        i = np.arange(S)[:, None]
        j = np.arange(S)[None, :]
        bias = -slopes[None, :, None, None] * (i - j)[None, None]
        fm = np.where(dm, bias, -np.inf)
        ref = _sdpa_grads(q, k, v, g, scale, torch.from_numpy(np.ascontiguousarray(fm)))
        got = orc.attention_bwd(q, k, v, g, mask, W.SCORE_ALIBI, scale, **okw)
        for name, a, b in zip("qkv", got, ref):
            _close(a, b, 1e-10, f"backward d{name} m{mask} alibi")


def pin_backward_softcap_finite_differences(orc):
    # central differences of L = sum(dout * out) through the (pinned) forward;
    # inputs on a 2^-8 grid so q +- 2^-12 is exact in float32
    B, H, S, D, scale, cap = 1, 2, 7, 3, 0.8, 0.9
    q, k, v, g = (np.round(_rand((B, H, S, D), 70 + t) * 256) / 256 for t in range(4))
    q, k, v, g = (x.astype(np.float32) for x in (q, k, v, g))
    h = 2.0 ** -12
    for mask, kw in [(W.MASK_CAUSAL, {}), (W.MASK_SLIDING_WINDOW, {"window": 3})]:
        dq, dk, dv = orc.attention_bwd(q, k, v, g, mask, W.SCORE_SOFTCAP, scale, score_param=cap, **kw)

        def loss(qq, kk, vv):
            out, _ = orc.attention(qq, kk, vv, mask, W.SCORE_SOFTCAP, scale, score_param=cap, **kw)
            return float(np.sum(out * g.astype(np.float64)))

        for which, grad in ((0, dq), (1, dk), (2, dv)):
            base = [q, k, v]
            fd = np.zeros_like(grad)
            for idx in np.ndindex(*base[which].shape):
                hi, lo = [x.copy() for x in base], [x.copy() for x in base]
                hi[which][idx] += np.float32(h)
                lo[which][idx] -= np.float32(h)
                fd[idx] = (loss(*hi) - loss(*lo)) / (2 * h)
            _close(grad, fd, 2e-6, f"softcap d{'qkv'[which]} m{mask} vs finite differences")


def pin_backward_invariants(orc):
    # identity and ALiBi: every softmax row of dS sums to 0, so sum_j dK_j = 0;
    # the weights of a row sum to 1, so sum_j dV_j = sum of dout over rows
    # with a key; V equal on every key: out does not depend on q or k
    B, H, S, D = 2, 2, 48, 8
    q, k, v, g = (_rand((B, H, S, D), 80 + t) for t in range(4))
    doc = np.repeat(np.arange(6, dtype=np.int32), 8)[None, :].repeat(B, 0)
    for mask, kw in [(W.MASK_CAUSAL, {}), (W.MASK_SLIDING_WINDOW, {"window": 5}),
                     (W.MASK_CAUSAL_PREFIX, {"prefix": 20}), (W.MASK_DOCUMENT, {"doc_ids": doc}),
                     (W.MASK_ALL, {})]:
        for score in (W.SCORE_IDENTITY, W.SCORE_ALIBI):
            dq, dk, dv = orc.attention_bwd(q, k, v, g, mask, score, 0.6, **kw)
            _close(dk.sum(axis=2), np.zeros((B, H, D)), 1e-11, f"sum dK m{mask} s{score}")
            _close(dv.sum(axis=2), g.astype(np.float64).sum(axis=2), 1e-11, f"sum dV m{mask} s{score}")
        vc = np.broadcast_to(_rand((B, H, 1, D), 90), (B, H, S, D)).copy()
        for score, sp in [(W.SCORE_IDENTITY, 0.0), (W.SCORE_SOFTCAP, 1.5), (W.SCORE_ALIBI, 0.0)]:
            dq, dk, _ = orc.attention_bwd(q, k, vc, g, mask, score, 0.6, score_param=sp, **kw)
            assert np.max(np.abs(dq)) < 1e-12 and np.max(np.abs(dk)) < 1e-12, f"constant V m{mask} s{score}"
    # an empty row (W = 0) contributes nothing
    dq, dk, dv = orc.attention_bwd(q, k, v, g, W.MASK_SLIDING_WINDOW, W.SCORE_IDENTITY, 0.6, window=0)
    assert not dq.any() and not dk.any() and not dv.any()


def pin_backward_dq_rows_match_the_full_backward(orc):
    # the row-sampled dq is the full backward's dq, row for row and bit for bit
    B, H, S, D = 2, 2, 40, 8
    q, k, v, g = (_rand((B, H, S, D), 95 + t) for t in range(4))
    rows = np.array([0, 1, 39, 40, 77, 120, 159], np.int64)
    for mask, kw in [(W.MASK_CAUSAL, {}), (W.MASK_SLIDING_WINDOW, {"window": 0})]:
        for score, sp in [(W.SCORE_SOFTCAP, 1.5), (W.SCORE_ALIBI, 0.0)]:
            dq, _, _ = orc.attention_bwd(q, k, v, g, mask, score, 0.6, score_param=sp, **kw)
            got = orc.attention_bwd_dq_rows(q, k, v, g, rows, mask, score, 0.6, score_param=sp, **kw)
            _close(got, dq.reshape(-1, D)[rows], 0.0, f"dq rows m{mask} s{score}")


def pin_block_mask_q_is_the_transpose(orc):
    # brute-force tile classes, transposed: for kv block j, the q blocks of its
    # partial / full tiles ascending, then the rest ascending
    B, H = 2, 2
    for S, block in [(8, 2), (12, 4), (13, 4), (10, 4)]:
        q = k = v = _rand((B, H, S, 2), S)
        doc = np.zeros((B, S), np.int32)
        doc[0, S // 3:] = 1
        doc[1, S // 2:] = 1
        for mask, kw in [(W.MASK_CAUSAL, {}), (W.MASK_SLIDING_WINDOW, {"window": 3}),
                         (W.MASK_CAUSAL_PREFIX, {"prefix": 5}), (W.MASK_DOCUMENT, {"doc": doc}),
                         (W.MASK_ALL, {})]:
            _, _, status, _ = brute_force(q, k, v, mask, W.SCORE_IDENTITY, 0.5, block=block,
                                          window=kw.get("window", 0), prefix=kw.get("prefix", 0), doc=kw.get("doc"))
            bq = orc.block_mask_q(mask, B, H, S, S, block, window=kw.get("window", 0), prefix=kw.get("prefix", 0),
                                  doc_ids=kw.get("doc"))
            for b in range(B):
                for h in range(H):
                    exp = _expected_lists(status[b, h].T)
                    for key, qkey in (("kv_num_blocks", "q_num_blocks"), ("kv_indices", "q_indices"),
                                      ("full_kv_num_blocks", "full_q_num_blocks"),
                                      ("full_kv_indices", "full_q_indices")):
                        assert np.array_equal(bq[qkey][b, h], exp[key]), f"{qkey} S{S} m{mask} b{b} h{h}"
    # rectangular and ragged: the all-true mask at Q_LEN 200, KV_LEN 333 has
    # full tiles only where both the rows and the columns are whole
    bq = orc.block_mask_q(W.MASK_ALL, 1, 1, 200, 333, 128)
    exp = _expected_lists(np.array([[2, 2, 1], [1, 1, 1]]).T)
    for key, qkey in (("kv_num_blocks", "q_num_blocks"), ("kv_indices", "q_indices"),
                      ("full_kv_num_blocks", "full_q_num_blocks"), ("full_kv_indices", "full_q_indices")):
        assert np.array_equal(bq[qkey][0, 0], exp[key]), f"{qkey} 200x333"


ALL_PINS = [
    pin_all_true_mask_is_textbook_attention,
    pin_causal_mask_is_library_causal,
    pin_causal_prefix_splits_into_library_calls,
    pin_document_mask_is_per_document_causal,
    pin_sliding_window_rows_are_window_slices,
    pin_huge_softcap_is_identity,
    pin_softcap_through_atanh,
    pin_alibi_zero_scores_geometric,
    pin_constant_v_gives_constant_out,
    pin_window_one_and_zero,
    pin_first_causal_row_is_v0,
    pin_alibi_diagonal_has_no_bias,
    pin_causal_block_counts_closed_form,
    pin_ragged_causal_block_counts_closed_form,
    pin_sliding_window_block_counts_closed_form,
    pin_causal_prefix_block_counts_closed_form,
    pin_document_blocks_from_intervals,
    pin_golden_causal_prefix_predicate,
    pin_brute_force_tiny,
    pin_brute_force_block_shapes,
    pin_causal_block_shapes_closed_form,
    pin_round_bf16_is_library_conversion,
    pin_round_bf16_nearest_on_exact_products,
    pin_prescale_power_of_two_scale_changes_nothing,
    pin_prescale_is_attention_on_rounded_q,
    pin_row_max_bounds_lse,
    pin_backward_is_library_autograd,
    pin_backward_softcap_finite_differences,
    pin_backward_invariants,
    pin_block_mask_q_is_the_transpose,
    pin_backward_dq_rows_match_the_full_backward,
]
