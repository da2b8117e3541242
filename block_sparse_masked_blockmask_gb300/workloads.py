"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no part of the attention or BlockMask arithmetic: it only
draws the random tensors, rounds them to the storage dtype and lays out the
document ids.  Both the CUDA path and the CPU oracle receive exactly the
numbers produced here.

Workloads follow the five synthetic configurations of the FlexAttention
forward study ("[Inductor][Flex Attention] Add Subtiling Option for Alpha
Scaling", PyTorch PR #167356, and "Performance for templated attention
strangely bad for a combination of causal + upper square mask", PyTorch issue
#124369): Q, K, V ~ N(0, 1), seed 0, 128x128 blocks.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# Mask and score kinds; the integer values are the C-ABI enums of flexattn.h.
MASK_CAUSAL = 0
MASK_SLIDING_WINDOW = 1
MASK_CAUSAL_PREFIX = 2
MASK_DOCUMENT = 3
MASK_ALL = 4

SCORE_IDENTITY = 0
SCORE_SOFTCAP = 1
SCORE_ALIBI = 2

MASK_NAMES = {MASK_CAUSAL: "causal", MASK_SLIDING_WINDOW: "sliding_window",
              MASK_CAUSAL_PREFIX: "causal_prefix", MASK_DOCUMENT: "document",
              MASK_ALL: "all"}
SCORE_NAMES = {SCORE_IDENTITY: "identity", SCORE_SOFTCAP: "softcap", SCORE_ALIBI: "alibi"}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic attention problem: shapes, dtype, mask_mod and score_mod."""
    name: str
    dtype: str            # "fp32" or "bf16"
    B: int
    H: int
    S: int                # Q_LEN == KV_LEN
    D: int
    mask: int
    score: int
    window: int = 0       # sliding-window width W (mask keeps 0 <= q-kv < W)
    prefix: int = 0       # bidirectional prefix bound P (inclusive)
    softcap: float = 0.0  # cap of cap*tanh(s/cap)
    seed: int = 0
    block: int = 128

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def score_param(self) -> float:
        return self.softcap if self.score == SCORE_SOFTCAP else 0.0


# The five configurations, named by what they are.
FP32_CAUSAL_S256 = Workload("fp32_causal_b1h2s256d64", "fp32", 1, 2, 256, 64,
                            MASK_CAUSAL, SCORE_IDENTITY)
BF16_WINDOW256_S2048 = Workload("bf16_window256_b2h8s2048d64", "bf16", 2, 8, 2048, 64,
                                MASK_SLIDING_WINDOW, SCORE_IDENTITY, window=256)
BF16_PREFIX1024_S4096 = Workload("bf16_causal_prefix1024_b4h16s4096d64", "bf16", 4, 16, 4096, 64,
                                 MASK_CAUSAL_PREFIX, SCORE_IDENTITY, prefix=1024)
BF16_DOC_SOFTCAP_S8192 = Workload("bf16_document_softcap50_b8h16s8192d128", "bf16", 8, 16, 8192, 128,
                                  MASK_DOCUMENT, SCORE_SOFTCAP, softcap=50.0)
BF16_CAUSAL_ALIBI_S16384 = Workload("bf16_causal_alibi_b2h32s16384d128", "bf16", 2, 32, 16384, 128,
                                    MASK_CAUSAL, SCORE_ALIBI)

CONFIGS = [FP32_CAUSAL_S256, BF16_WINDOW256_S2048, BF16_PREFIX1024_S4096,
           BF16_DOC_SOFTCAP_S8192, BF16_CAUSAL_ALIBI_S16384]


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even).

    Returns float32 values that are exactly representable in bfloat16.
    Inputs are finite normal draws, so NaN handling is not needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    r = (u + bias) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def bf16_bits(x_rounded: np.ndarray) -> np.ndarray:
    """The bfloat16 bit patterns (uint16) of values already rounded by round_to_bf16."""
    u = np.ascontiguousarray(x_rounded, dtype=np.float32).view(np.uint32)
    return (u >> np.uint32(16)).astype(np.uint16)


def draw_qkv(B: int, H: int, S: int, D: int, seed: int = 0, dtype: str = "bf16",
             S_kv: int | None = None):
    """Q, K, V ~ N(0,1) drawn in the order q, k, v from default_rng(seed).

    Returned as float32 arrays holding exactly the values the device sees
    (rounded to bfloat16 when dtype == "bf16").
    """
    S_kv = S if S_kv is None else S_kv
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, S, D), dtype=np.float32)
    k = rng.standard_normal((B, H, S_kv, D), dtype=np.float32)
    v = rng.standard_normal((B, H, S_kv, D), dtype=np.float32)
    if dtype == "bf16":
        q, k, v = round_to_bf16(q), round_to_bf16(k), round_to_bf16(v)
    elif dtype != "fp32":
        raise ValueError(f"unknown dtype {dtype}")
    return q, k, v


def document_lengths(S: int, rng: np.random.Generator, lo: int = 256, hi: int = 2048) -> list[int]:
    """Split S tokens into documents with lengths in [lo, hi] that sum to S.

    Lengths are drawn uniformly from [lo, min(hi, R - lo)] while the remainder
    R exceeds hi; the remainder then forms the last document.
    """
    if S < lo:
        return [S]
    out = []
    R = S
    while R > hi:
        L = int(rng.integers(lo, min(hi, R - lo) + 1))
        out.append(L)
        R -= L
    out.append(R)
    return out


def document_ids(B: int, S: int, seed: int = 0, lo: int = 256, hi: int = 2048) -> np.ndarray:
    """Per batch row b (in order), the running document index of each token, int32 [B, S]."""
    rng = np.random.default_rng(seed + 1000)
    ids = np.empty((B, S), dtype=np.int32)
    for b in range(B):
        pos = 0
        for d, L in enumerate(document_lengths(S, rng, lo, hi)):
            ids[b, pos:pos + L] = d
            pos += L
    return ids


def workload_inputs(w: Workload):
    """(q, k, v, doc_ids) for a workload; doc_ids is None unless the mask is a document mask."""
    q, k, v = draw_qkv(w.B, w.H, w.S, w.D, w.seed, w.dtype)
    docs = document_ids(w.B, w.S, w.seed) if w.mask == MASK_DOCUMENT else None
    return q, k, v, docs


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(w, **changes)
