"""Python entry to the float64 CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package smoke check
and by the bench's CPU-baseline leg, never by the product path.  It builds
``liboracle.so`` from ``oracle.c`` with gcc on first use and calls it through
ctypes; it imports nothing from the CUDA package.

The arithmetic lives in oracle.c; this file only marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
LIBRARY = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None


def compile_oracle(src: str, dst: str) -> str:
    """gcc -O2 -fopenmp build of an oracle source file into a shared library."""
    tmp = dst + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, dst)
    return dst


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so when missing or stale."""
    stale = (not os.path.exists(LIBRARY)) or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE)
    if force or stale:
        compile_oracle(SOURCE, LIBRARY)
    return LIBRARY


def _ptr(a, ctype):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctype))


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i32p = ctypes.POINTER(ctypes.c_int32)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        I, L, D = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_block_mask.argtypes = [I, I, I, i32p, I, I, I, I, I, I, i32p, i32p, i32p, i32p]
        lib.oracle_block_mask.restype = I
        lib.oracle_attention.argtypes = [f32p, f32p, f32p, I, I, I, I, I, I, I, I, i32p,
                                         I, D, D, i64p, L, f64p, f64p]
        lib.oracle_attention.restype = I
        lib.oracle_attention_opts.argtypes = [f32p, f32p, f32p, I, I, I, I, I, I, I, I, i32p,
                                              I, D, D, I, i64p, L, f64p, f64p, f64p]
        lib.oracle_attention_opts.restype = I
        lib.oracle_block_mask_q.argtypes = [I, I, I, i32p, I, I, I, I, I, I, i32p, i32p, i32p, i32p]
        lib.oracle_block_mask_q.restype = I
        lib.oracle_attention_bwd.argtypes = [f32p, f32p, f32p, f32p, I, I, I, I, I, I, I, I, i32p,
                                             I, D, D, f64p, f64p, f64p]
        lib.oracle_attention_bwd.restype = I
        lib.oracle_attention_bwd_dq_rows.argtypes = [f32p, f32p, f32p, f32p, I, I, I, I, I, I, I, I, i32p,
                                                     I, D, D, i64p, L, f64p]
        lib.oracle_attention_bwd_dq_rows.restype = I
        lib.oracle_round_bf16.argtypes = [D]
        lib.oracle_round_bf16.restype = D
        lib.oracle_mask_value.argtypes = [I, I, I, i32p, L, L, L, L, L]
        lib.oracle_mask_value.restype = I
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = I
        self.lib = lib
        self.path = path

    def block_mask(self, kind: int, B: int, H: int, q_len: int, kv_len: int, block: int = 128,
                   window: int = 0, prefix: int = 0, doc_ids=None, kv_block: int | None = None) -> dict:
        """kv_num_blocks, kv_indices, full_kv_num_blocks, full_kv_indices (int32).

        Tiles are block (Q_BLOCK) rows by kv_block (KV_BLOCK, default: block) columns.
        """
        kv_block = block if kv_block is None else kv_block
        nqb, nkvb = -(-q_len // block), -(-kv_len // kv_block)  # ceil: tail tiles padded with false
        out = {
            "kv_num_blocks": np.zeros((B, H, nqb), np.int32),
            "kv_indices": np.zeros((B, H, nqb, nkvb), np.int32),
            "full_kv_num_blocks": np.zeros((B, H, nqb), np.int32),
            "full_kv_indices": np.zeros((B, H, nqb, nkvb), np.int32),
        }
        doc = None if doc_ids is None else np.ascontiguousarray(doc_ids, dtype=np.int32)
        rc = self.lib.oracle_block_mask(kind, window, prefix, _ptr(doc, ctypes.c_int32), B, H,
                                        q_len, kv_len, block, kv_block,
                                        _ptr(out["kv_num_blocks"], ctypes.c_int32),
                                        _ptr(out["kv_indices"], ctypes.c_int32),
                                        _ptr(out["full_kv_num_blocks"], ctypes.c_int32),
                                        _ptr(out["full_kv_indices"], ctypes.c_int32))
        if rc != 0:
            raise ValueError(f"oracle_block_mask failed with {rc}")
        return out

    def attention(self, q, k, v, mask_kind: int, score_kind: int, scale: float, window: int = 0,
                  prefix: int = 0, doc_ids=None, score_param: float = 0.0, rows=None):
        """(out float64, lse float64) of the plain definition.

        q: [B,H,Sq,D], k, v: [B,H,Skv,D] float32 (the exact device values).
        rows: optional flat row ids ((b*H+h)*Sq + i); then out is [len(rows), D].
        """
        q = np.ascontiguousarray(q, dtype=np.float32)
        k = np.ascontiguousarray(k, dtype=np.float32)
        v = np.ascontiguousarray(v, dtype=np.float32)
        B, H, s_q, D = q.shape
        s_kv = k.shape[2]
        doc = None if doc_ids is None else np.ascontiguousarray(doc_ids, dtype=np.int32)
        if rows is None:
            out = np.zeros((B, H, s_q, D), np.float64)
            lse = np.zeros((B, H, s_q), np.float64)
            rp, nrows = None, 0
        else:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            out = np.zeros((rows.size, D), np.float64)
            lse = np.zeros((rows.size,), np.float64)
            rp, nrows = _ptr(rows, ctypes.c_int64), rows.size
        rc = self.lib.oracle_attention(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float),
                                       _ptr(v, ctypes.c_float), B, H, s_q, s_kv, D, mask_kind,
                                       window, prefix, _ptr(doc, ctypes.c_int32), score_kind,
                                       float(score_param), float(scale), rp, nrows,
                                       _ptr(out, ctypes.c_double), _ptr(lse, ctypes.c_double))
        if rc != 0:
            raise ValueError(f"oracle_attention failed with {rc}")
        return out, lse

    PRESCALE = {None: 0, "bf16": 1, "f32": 2}

    def attention_opts(self, q, k, v, mask_kind: int, score_kind: int, scale: float,
                       window: int = 0, prefix: int = 0, doc_ids=None, score_param: float = 0.0,
                       rows=None, prescale: str | None = None):
        """(out, lse, row_max) float64 under the kernel options.

        OUTPUT_MAX is always on here (row_max); prescale None, "bf16" or "f32"
        selects PRESCALE_QK with that storage type.  Other arguments as attention().
        """
        q = np.ascontiguousarray(q, dtype=np.float32)
        k = np.ascontiguousarray(k, dtype=np.float32)
        v = np.ascontiguousarray(v, dtype=np.float32)
        B, H, s_q, D = q.shape
        s_kv = k.shape[2]
        doc = None if doc_ids is None else np.ascontiguousarray(doc_ids, dtype=np.int32)
        if rows is None:
            out = np.zeros((B, H, s_q, D), np.float64)
            lse = np.zeros((B, H, s_q), np.float64)
            rp, nrows = None, 0
        else:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            out = np.zeros((rows.size, D), np.float64)
            lse = np.zeros((rows.size,), np.float64)
            rp, nrows = _ptr(rows, ctypes.c_int64), rows.size
        row_max = np.zeros_like(lse)
        rc = self.lib.oracle_attention_opts(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float),
                                            _ptr(v, ctypes.c_float), B, H, s_q, s_kv, D, mask_kind,
                                            window, prefix, _ptr(doc, ctypes.c_int32), score_kind,
                                            float(score_param), float(scale), self.PRESCALE[prescale],
                                            rp, nrows, _ptr(out, ctypes.c_double),
                                            _ptr(lse, ctypes.c_double), _ptr(row_max, ctypes.c_double))
        if rc != 0:
            raise ValueError(f"oracle_attention_opts failed with {rc}")
        return out, lse, row_max

    def block_mask_q(self, kind: int, B: int, H: int, q_len: int, kv_len: int, block: int = 128,
                     window: int = 0, prefix: int = 0, doc_ids=None, kv_block: int | None = None) -> dict:
        """q_num_blocks, q_indices, full_q_num_blocks, full_q_indices (int32): the transposed lists."""
        kv_block = block if kv_block is None else kv_block
        nqb, nkvb = -(-q_len // block), -(-kv_len // kv_block)
        out = {
            "q_num_blocks": np.zeros((B, H, nkvb), np.int32),
            "q_indices": np.zeros((B, H, nkvb, nqb), np.int32),
            "full_q_num_blocks": np.zeros((B, H, nkvb), np.int32),
            "full_q_indices": np.zeros((B, H, nkvb, nqb), np.int32),
        }
        doc = None if doc_ids is None else np.ascontiguousarray(doc_ids, dtype=np.int32)
        rc = self.lib.oracle_block_mask_q(kind, window, prefix, _ptr(doc, ctypes.c_int32), B, H, q_len, kv_len,
                                          block, kv_block, _ptr(out["q_num_blocks"], ctypes.c_int32),
                                          _ptr(out["q_indices"], ctypes.c_int32),
                                          _ptr(out["full_q_num_blocks"], ctypes.c_int32),
                                          _ptr(out["full_q_indices"], ctypes.c_int32))
        if rc != 0:
            raise ValueError(f"oracle_block_mask_q failed with {rc}")
        return out

    def attention_bwd(self, q, k, v, dout, mask_kind: int, score_kind: int, scale: float, window: int = 0,
                      prefix: int = 0, doc_ids=None, score_param: float = 0.0):
        """(dq, dk, dv) float64: the gradients of sum(dout * out) for out = attention(q, k, v)."""
        q, k, v, dout = (np.ascontiguousarray(x, dtype=np.float32) for x in (q, k, v, dout))
        B, H, s_q, D = q.shape
        s_kv = k.shape[2]
        doc = None if doc_ids is None else np.ascontiguousarray(doc_ids, dtype=np.int32)
        dq = np.zeros((B, H, s_q, D), np.float64)
        dk = np.zeros((B, H, s_kv, D), np.float64)
        dv = np.zeros((B, H, s_kv, D), np.float64)
        rc = self.lib.oracle_attention_bwd(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float),
                                           _ptr(v, ctypes.c_float), _ptr(dout, ctypes.c_float), B, H, s_q, s_kv,
                                           D, mask_kind, window, prefix, _ptr(doc, ctypes.c_int32), score_kind,
                                           float(score_param), float(scale), _ptr(dq, ctypes.c_double),
                                           _ptr(dk, ctypes.c_double), _ptr(dv, ctypes.c_double))
        if rc != 0:
            raise ValueError(f"oracle_attention_bwd failed with {rc}")
        return dq, dk, dv

    def attention_bwd_dq_rows(self, q, k, v, dout, rows, mask_kind: int, score_kind: int, scale: float,
                              window: int = 0, prefix: int = 0, doc_ids=None, score_param: float = 0.0):
        """dq of the flat rows ((b*H + h)*Sq + i) in `rows`: float64 [len(rows), D]."""
        q, k, v, dout = (np.ascontiguousarray(x, dtype=np.float32) for x in (q, k, v, dout))
        B, H, s_q, D = q.shape
        s_kv = k.shape[2]
        doc = None if doc_ids is None else np.ascontiguousarray(doc_ids, dtype=np.int32)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        dq = np.zeros((rows.size, D), np.float64)
        rc = self.lib.oracle_attention_bwd_dq_rows(_ptr(q, ctypes.c_float), _ptr(k, ctypes.c_float),
                                                   _ptr(v, ctypes.c_float), _ptr(dout, ctypes.c_float), B, H, s_q,
                                                   s_kv, D, mask_kind, window, prefix, _ptr(doc, ctypes.c_int32),
                                                   score_kind, float(score_param), float(scale),
                                                   _ptr(rows, ctypes.c_int64), rows.size, _ptr(dq, ctypes.c_double))
        if rc != 0:
            raise ValueError(f"oracle_attention_bwd_dq_rows failed with {rc}")
        return dq

    def round_bf16(self, x: float) -> float:
        return float(self.lib.oracle_round_bf16(float(x)))

    def mask_value(self, kind: int, q: int, kv: int, b: int = 0, h: int = 0, window: int = 0,
                   prefix: int = 0, doc_ids=None) -> bool:
        doc = None if doc_ids is None else np.ascontiguousarray(doc_ids, dtype=np.int32)
        doc_len = 0 if doc is None else doc.shape[-1]
        r = self.lib.oracle_mask_value(kind, window, prefix, _ptr(doc, ctypes.c_int32), doc_len,
                                       b, h, q, kv)
        if r < 0:
            raise ValueError("bad mask kind")
        return bool(r)

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    # workload helpers (see block_sparse_masked_blockmask_gb300.workloads.Workload)
    def workload_attention(self, w, q, k, v, doc_ids=None, rows=None):
        return self.attention(q, k, v, w.mask, w.score, w.scale, window=w.window,
                              prefix=w.prefix, doc_ids=doc_ids, score_param=w.score_param,
                              rows=rows)

    def workload_block_mask(self, w, doc_ids=None, block: int | None = None):
        return self.block_mask(w.mask, w.B, w.H, w.S, w.S, block or w.block, window=w.window,
                               prefix=w.prefix, doc_ids=doc_ids)


def default() -> Oracle:
    """The oracle built from oracle.c (built on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def attention(*a, **kw):
    return default().attention(*a, **kw)


def block_mask(*a, **kw):
    return default().block_mask(*a, **kw)


def mask_value(*a, **kw):
    return default().mask_value(*a, **kw)


def attention_opts(*a, **kw):
    return default().attention_opts(*a, **kw)


def attention_bwd(*a, **kw):
    return default().attention_bwd(*a, **kw)


def block_mask_q(*a, **kw):
    return default().block_mask_q(*a, **kw)


def attention_bwd_dq_rows(*a, **kw):
    return default().attention_bwd_dq_rows(*a, **kw)


def num_threads() -> int:
    return default().num_threads()


def workload_attention(*a, **kw):
    return default().workload_attention(*a, **kw)


def workload_block_mask(*a, **kw):
    return default().workload_block_mask(*a, **kw)
