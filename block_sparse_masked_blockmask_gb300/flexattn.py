"""Thin Python binding of the C-ABI in include/flexattn.h.

Argument marshalling only: torch tensors supply device memory and
torch.cuda streams supply the cudaStream_t; every step of the path runs in
the CUDA kernels of libflexattn.so.  There is no fallback: if the library is
missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from . import _build

FLEX_OK = 0
FLEX_ERR_INVALID_ARG = -1
FLEX_ERR_UNSUPPORTED = -2
FLEX_ERR_SHAPE = -3
FLEX_ERR_ALIGNMENT = -4
FLEX_ERR_CUDA = -5
FLEX_ERR_DEVICE_TIMEOUT = -6

FLEX_MASK_CAUSAL = 0
FLEX_MASK_SLIDING_WINDOW = 1
FLEX_MASK_CAUSAL_PREFIX = 2
FLEX_MASK_DOCUMENT = 3
FLEX_MASK_ALL = 4

FLEX_SCORE_IDENTITY = 0
FLEX_SCORE_SOFTCAP = 1
FLEX_SCORE_ALIBI = 2

FLEX_DTYPE_BF16 = 0
FLEX_DTYPE_FP32 = 1

EXPORTED = ("flex_block_mask_sizes", "flex_block_mask_sizes_qkv", "flex_block_mask_create", "flex_block_mask_create_qkv",
            "flex_block_mask_transpose", "flex_attention_fwd",
            "flex_attention_fwd_opts", "flex_attention_bwd", "flex_attention_fwd_noalloc", "flex_attention_fwd_host", "flex_device_status",
            "flex_selftest_wait_timeout", "flex_status_string")


class FlexError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {flex_status_string(code)} ({code})")


class flex_mask_params(ctypes.Structure):
    _fields_ = [("window", ctypes.c_int32), ("prefix", ctypes.c_int32), ("doc_ids", ctypes.c_void_p)]


class flex_block_mask(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("kv_len", ctypes.c_int32), ("q_block", ctypes.c_int32), ("kv_block", ctypes.c_int32),
                ("nqb", ctypes.c_int32), ("nkvb", ctypes.c_int32), ("mask_kind", ctypes.c_int32),
                ("params", flex_mask_params),
                ("kv_num_blocks", ctypes.c_void_p), ("kv_indices", ctypes.c_void_p),
                ("full_kv_num_blocks", ctypes.c_void_p), ("full_kv_indices", ctypes.c_void_p)]


class flex_tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


class flex_block_mask_q(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("q_len", ctypes.c_int32),
                ("kv_len", ctypes.c_int32), ("q_block", ctypes.c_int32), ("kv_block", ctypes.c_int32),
                ("nqb", ctypes.c_int32), ("nkvb", ctypes.c_int32),
                ("q_num_blocks", ctypes.c_void_p), ("q_indices", ctypes.c_void_p),
                ("full_q_num_blocks", ctypes.c_void_p), ("full_q_indices", ctypes.c_void_p)]


class flex_kernel_options(ctypes.Structure):
    _fields_ = [("prescale_qk", ctypes.c_int32), ("rows_guaranteed_safe", ctypes.c_int32),
                ("max_scores", ctypes.c_void_p)]


class flex_device_buffers(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("lse", ctypes.c_void_p), ("doc_ids", ctypes.c_void_p), ("kv_num_blocks", ctypes.c_void_p),
                ("kv_indices", ctypes.c_void_p), ("full_kv_num_blocks", ctypes.c_void_p),
                ("full_kv_indices", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIBRARY


def load_library():
    """Load libflexattn.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; "
                                   "g.build()')")
            lib = ctypes.CDLL(path)
            i32, i64p, vp = ctypes.c_int32, ctypes.POINTER(ctypes.c_int64), ctypes.c_void_p
            lib.flex_block_mask_sizes.argtypes = [i32, i32, i32, i32, i32, i64p, i64p]
            lib.flex_block_mask_sizes.restype = ctypes.c_int
            lib.flex_block_mask_sizes_qkv.argtypes = [i32, i32, i32, i32, i32, i32, i64p, i64p]
            lib.flex_block_mask_sizes_qkv.restype = ctypes.c_int
            lib.flex_block_mask_create.argtypes = [i32, ctypes.POINTER(flex_mask_params), i32, i32, i32, i32, i32,
                                                   ctypes.POINTER(flex_block_mask), vp]
            lib.flex_block_mask_create.restype = ctypes.c_int
            lib.flex_block_mask_create_qkv.argtypes = [i32, ctypes.POINTER(flex_mask_params), i32, i32, i32, i32,
                                                       i32, i32, ctypes.POINTER(flex_block_mask), vp]
            lib.flex_block_mask_create_qkv.restype = ctypes.c_int
            tp = ctypes.POINTER(flex_tensor)
            lib.flex_attention_fwd.argtypes = [tp, tp, tp, ctypes.POINTER(flex_block_mask), i32, ctypes.c_float,
                                               ctypes.c_float, vp, vp, vp]
            lib.flex_attention_fwd.restype = ctypes.c_int
            lib.flex_attention_fwd_opts.argtypes = [tp, tp, tp, ctypes.POINTER(flex_block_mask), i32,
                                                    ctypes.c_float, ctypes.c_float, vp, vp,
                                                    ctypes.POINTER(flex_kernel_options), vp]
            lib.flex_attention_fwd_opts.restype = ctypes.c_int
            lib.flex_block_mask_transpose.argtypes = [ctypes.POINTER(flex_block_mask),
                                                      ctypes.POINTER(flex_block_mask_q), vp]
            lib.flex_block_mask_transpose.restype = ctypes.c_int
            lib.flex_attention_bwd.argtypes = [tp, tp, tp, vp, vp, vp, ctypes.POINTER(flex_block_mask),
                                               ctypes.POINTER(flex_block_mask_q), i32, ctypes.c_float,
                                               ctypes.c_float, vp, vp, vp, vp, vp]
            lib.flex_attention_bwd.restype = ctypes.c_int
            lib.flex_attention_fwd_noalloc.argtypes = [tp, tp, tp, ctypes.POINTER(flex_block_mask), i32,
                                                       ctypes.c_float, ctypes.c_float, vp, vp, vp,
                                                       ctypes.POINTER(ctypes.POINTER(ctypes.c_int))]
            lib.flex_attention_fwd_noalloc.restype = ctypes.c_int
            lib.flex_attention_fwd_host.argtypes = [tp, tp, tp, i32, ctypes.POINTER(flex_mask_params), i32,
                                                    ctypes.c_float, ctypes.c_float, vp, vp,
                                                    ctypes.POINTER(flex_device_buffers), i32, vp]
            lib.flex_attention_fwd_host.restype = ctypes.c_int
            lib.flex_device_status.argtypes = [vp]
            lib.flex_device_status.restype = ctypes.c_int
            lib.flex_selftest_wait_timeout.argtypes = [ctypes.c_uint32, vp]
            lib.flex_selftest_wait_timeout.restype = ctypes.c_int
            lib.flex_status_string.argtypes = [ctypes.c_int]
            lib.flex_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def _stream_handle(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def flex_status_string(code: int) -> str:
    return load_library().flex_status_string(int(code)).decode()


def flex_block_mask_sizes(B: int, H: int, q_len: int, kv_len: int, block: int = 128,
                          kv_block: int | None = None) -> tuple[int, int]:
    """Element counts of the count and index tensors (Q_BLOCK = block, KV_BLOCK = kv_block or block)."""
    n_num, n_idx = ctypes.c_int64(), ctypes.c_int64()
    if kv_block is None:
        rc = load_library().flex_block_mask_sizes(B, H, q_len, kv_len, block, ctypes.byref(n_num),
                                                  ctypes.byref(n_idx))
    else:
        rc = load_library().flex_block_mask_sizes_qkv(B, H, q_len, kv_len, block, kv_block, ctypes.byref(n_num),
                                                      ctypes.byref(n_idx))
    if rc != FLEX_OK:
        raise FlexError(rc, "flex_block_mask_sizes")
    return n_num.value, n_idx.value


class BlockMask:
    """Device BlockMask: the C struct plus the torch tensors that own its buffers."""

    def __init__(self, struct: flex_block_mask, tensors: dict, doc_ids):
        self.struct = struct
        self.kv_num_blocks = tensors["kv_num_blocks"]
        self.kv_indices = tensors["kv_indices"]
        self.full_kv_num_blocks = tensors["full_kv_num_blocks"]
        self.full_kv_indices = tensors["full_kv_indices"]
        self.doc_ids = doc_ids  # keeps the document ids alive while the mask is in use

    def as_numpy(self) -> dict:
        return {k: getattr(self, k).cpu().numpy() for k in
                ("kv_num_blocks", "kv_indices", "full_kv_num_blocks", "full_kv_indices")}


class BlockMaskQ:
    """Device q side of a BlockMask: the C struct plus the torch tensors that own its buffers."""

    KEYS = ("q_num_blocks", "q_indices", "full_q_num_blocks", "full_q_indices")

    def __init__(self, struct: flex_block_mask_q, tensors: dict):
        self.struct = struct
        for key in self.KEYS:
            setattr(self, key, tensors[key])

    def as_numpy(self) -> dict:
        return {k: getattr(self, k).cpu().numpy() for k in self.KEYS}


def flex_block_mask_transpose(block_mask: BlockMask, stream=None) -> BlockMaskQ:
    """The q side of a BlockMask (asynchronous on `stream`)."""
    s = block_mask.struct
    device = block_mask.kv_num_blocks.device
    t = {
        "q_num_blocks": torch.empty((s.B, s.H, s.nkvb), dtype=torch.int32, device=device),
        "q_indices": torch.empty((s.B, s.H, s.nkvb, s.nqb), dtype=torch.int32, device=device),
        "full_q_num_blocks": torch.empty((s.B, s.H, s.nkvb), dtype=torch.int32, device=device),
        "full_q_indices": torch.empty((s.B, s.H, s.nkvb, s.nqb), dtype=torch.int32, device=device),
    }
    bq = flex_block_mask_q()
    for key in BlockMaskQ.KEYS:
        setattr(bq, key, t[key].data_ptr())
    with torch.cuda.device(device):
        rc = load_library().flex_block_mask_transpose(ctypes.byref(s), ctypes.byref(bq),
                                                      _stream_handle(stream, device))
    if rc != FLEX_OK:
        raise FlexError(rc, "flex_block_mask_transpose")
    return BlockMaskQ(bq, t)


def flex_block_mask_create(mask_kind: int, B: int, H: int, q_len: int, kv_len: int, block: int = 128,
                           window: int = 0, prefix: int = 0, doc_ids: torch.Tensor | None = None,
                           device=None, stream=None, kv_block: int | None = None) -> BlockMask:
    """Build a BlockMask on the device (asynchronous on `stream`).

    Tiles are block (Q_BLOCK) rows by kv_block (KV_BLOCK; default: block)
    columns; flex_block_mask_create_qkv is called when kv_block is given.
    """
    device = torch.device(device) if device is not None else (
        doc_ids.device if doc_ids is not None else torch.device("cuda", torch.cuda.current_device()))
    n_num, n_idx = flex_block_mask_sizes(B, H, q_len, kv_len, block, kv_block)
    kvb = block if kv_block is None else kv_block
    nqb, nkvb = -(-q_len // block), -(-kv_len // kvb)  # a tail tile may reach past a length
    t = {
        "kv_num_blocks": torch.empty((B, H, nqb), dtype=torch.int32, device=device),
        "kv_indices": torch.empty((B, H, nqb, nkvb), dtype=torch.int32, device=device),
        "full_kv_num_blocks": torch.empty((B, H, nqb), dtype=torch.int32, device=device),
        "full_kv_indices": torch.empty((B, H, nqb, nkvb), dtype=torch.int32, device=device),
    }
    assert t["kv_num_blocks"].numel() == n_num and t["kv_indices"].numel() == n_idx
    if doc_ids is not None:
        doc_ids = doc_ids.to(device=device, dtype=torch.int32).contiguous()
    params = flex_mask_params(window, prefix, doc_ids.data_ptr() if doc_ids is not None else None)
    bm = flex_block_mask()
    bm.kv_num_blocks = t["kv_num_blocks"].data_ptr()
    bm.kv_indices = t["kv_indices"].data_ptr()
    bm.full_kv_num_blocks = t["full_kv_num_blocks"].data_ptr()
    bm.full_kv_indices = t["full_kv_indices"].data_ptr()
    with torch.cuda.device(device):
        if kv_block is None:
            rc = load_library().flex_block_mask_create(mask_kind, ctypes.byref(params), B, H, q_len, kv_len, block,
                                                       ctypes.byref(bm), _stream_handle(stream, device))
        else:
            rc = load_library().flex_block_mask_create_qkv(mask_kind, ctypes.byref(params), B, H, q_len, kv_len,
                                                           block, kv_block, ctypes.byref(bm),
                                                           _stream_handle(stream, device))
    if rc != FLEX_OK:
        raise FlexError(rc, "flex_block_mask_create")
    return BlockMask(bm, t, doc_ids)


_DTYPES = {torch.bfloat16: FLEX_DTYPE_BF16, torch.float32: FLEX_DTYPE_FP32}


def _tensor(x: torch.Tensor) -> flex_tensor:
    if x.dim() != 4:
        raise ValueError("expected a [B, H, S, D] tensor")
    if x.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {x.dtype}")
    t = flex_tensor()
    t.data = x.data_ptr()
    t.dtype = _DTYPES[x.dtype]
    for i in range(4):
        t.shape[i] = x.shape[i]
        t.stride[i] = x.stride(i)
    return t


def flex_attention_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, block_mask: BlockMask,
                       score_kind: int = FLEX_SCORE_IDENTITY, score_param: float = 0.0,
                       scale: float | None = None, out: torch.Tensor | None = None,
                       lse: torch.Tensor | None = None, stream=None):
    """Block-sparse attention forward; returns (out, lse).  Asynchronous on `stream`."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    B, H, Sq, D = q.shape
    if out is None:
        out = torch.empty((B, H, Sq, D), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if not out.is_contiguous() or not lse.is_contiguous() or lse.dtype != torch.float32:
        raise ValueError("out and lse must be contiguous; lse float32")
    tq, tk, tv = _tensor(q), _tensor(k), _tensor(v)
    with torch.cuda.device(q.device):
        rc = load_library().flex_attention_fwd(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                               ctypes.byref(block_mask.struct), score_kind, float(score_param),
                                               float(scale), ctypes.c_void_p(out.data_ptr()),
                                               ctypes.c_void_p(lse.data_ptr()), _stream_handle(stream, q.device))
    if rc != FLEX_OK:
        raise FlexError(rc, "flex_attention_fwd")
    return out, lse


def flex_attention_fwd_opts(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, block_mask: BlockMask,
                            score_kind: int = FLEX_SCORE_IDENTITY, score_param: float = 0.0,
                            scale: float | None = None, out: torch.Tensor | None = None,
                            lse: torch.Tensor | None = None, prescale_qk: bool = False,
                            rows_guaranteed_safe: bool = False, output_max: bool = False,
                            max_scores: torch.Tensor | None = None, stream=None):
    """flex_attention_fwd with the op's kernel options; returns (out, lse, max_scores).

    max_scores (float32 [B, H, Sq]) is allocated when output_max is set and
    none is given; it is None when OUTPUT_MAX is off.
    """
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    B, H, Sq, D = q.shape
    if out is None:
        out = torch.empty((B, H, Sq, D), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if max_scores is None and output_max:
        max_scores = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if not out.is_contiguous() or not lse.is_contiguous() or lse.dtype != torch.float32:
        raise ValueError("out and lse must be contiguous; lse float32")
    if max_scores is not None and (not max_scores.is_contiguous() or max_scores.dtype != torch.float32
                                   or max_scores.shape != (B, H, Sq)):
        raise ValueError("max_scores must be a contiguous float32 [B, H, q_len] tensor")
    opts = flex_kernel_options(int(bool(prescale_qk)), int(bool(rows_guaranteed_safe)),
                               None if max_scores is None else max_scores.data_ptr())
    tq, tk, tv = _tensor(q), _tensor(k), _tensor(v)
    with torch.cuda.device(q.device):
        rc = load_library().flex_attention_fwd_opts(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                                    ctypes.byref(block_mask.struct), score_kind,
                                                    float(score_param), float(scale),
                                                    ctypes.c_void_p(out.data_ptr()),
                                                    ctypes.c_void_p(lse.data_ptr()), ctypes.byref(opts),
                                                    _stream_handle(stream, q.device))
    if rc != FLEX_OK:
        raise FlexError(rc, "flex_attention_fwd_opts")
    return out, lse, max_scores


def flex_attention_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
                       dout: torch.Tensor, block_mask: BlockMask, block_mask_q: BlockMaskQ,
                       score_kind: int = FLEX_SCORE_IDENTITY, score_param: float = 0.0,
                       scale: float | None = None, dq: torch.Tensor | None = None, dk: torch.Tensor | None = None,
                       dv: torch.Tensor | None = None, delta: torch.Tensor | None = None, stream=None):
    """Gradients (dq, dk, dv) of sum(dout * out); asynchronous on `stream`."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    B, H, Sq, D = q.shape
    Skv = k.shape[2]
    dq = torch.empty((B, H, Sq, D), dtype=q.dtype, device=q.device) if dq is None else dq
    dk = torch.empty((B, H, Skv, D), dtype=q.dtype, device=q.device) if dk is None else dk
    dv = torch.empty((B, H, Skv, D), dtype=q.dtype, device=q.device) if dv is None else dv
    delta = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device) if delta is None else delta
    for name, t in (("out", out), ("dout", dout), ("dq", dq), ("dk", dk), ("dv", dv)):
        if not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError(f"{name} must be contiguous in q's dtype")
    if not lse.is_contiguous() or lse.dtype != torch.float32 or not delta.is_contiguous():
        raise ValueError("lse and delta must be contiguous float32")
    tq, tk, tv = _tensor(q), _tensor(k), _tensor(v)
    with torch.cuda.device(q.device):
        rc = load_library().flex_attention_bwd(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                               ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
                                               ctypes.c_void_p(dout.data_ptr()), ctypes.byref(block_mask.struct),
                                               ctypes.byref(block_mask_q.struct), score_kind, float(score_param),
                                               float(scale), ctypes.c_void_p(dq.data_ptr()),
                                               ctypes.c_void_p(dk.data_ptr()), ctypes.c_void_p(dv.data_ptr()),
                                               ctypes.c_void_p(delta.data_ptr()), _stream_handle(stream, q.device))
    if rc != FLEX_OK:
        raise FlexError(rc, "flex_attention_bwd")
    return dq, dk, dv


def flex_attention_fwd_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, block_mask: BlockMask,
                               out: torch.Tensor, lse: torch.Tensor, score_kind: int = FLEX_SCORE_IDENTITY,
                               score_param: float = 0.0, scale: float | None = None, stream=None):
    """flex_attention_fwd into caller-provided out/lse without any device allocation by the library.

    Returns the device address (int) of the status word the call uses; after the
    stream finishes, a nonzero word means a kernel gave up on a wait.
    """
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    tq, tk, tv = _tensor(q), _tensor(k), _tensor(v)
    status = ctypes.POINTER(ctypes.c_int)()
    with torch.cuda.device(q.device):
        rc = load_library().flex_attention_fwd_noalloc(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                                       ctypes.byref(block_mask.struct), score_kind,
                                                       float(score_param), float(scale),
                                                       ctypes.c_void_p(out.data_ptr()),
                                                       ctypes.c_void_p(lse.data_ptr()),
                                                       _stream_handle(stream, q.device), ctypes.byref(status))
    if rc != FLEX_OK:
        raise FlexError(rc, "flex_attention_fwd_noalloc")
    return ctypes.cast(status, ctypes.c_void_p).value


class DeviceBuffers:
    """Device working memory of flex_attention_fwd_host, allocated (and owned) through torch."""

    def __init__(self, B: int, H: int, q_len: int, kv_len: int, D: int, dtype: torch.dtype,
                 document: bool = False, device=None):
        device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.q = torch.empty((B, H, q_len, D), dtype=dtype, device=device)
        self.k = torch.empty((B, H, kv_len, D), dtype=dtype, device=device)
        self.v = torch.empty((B, H, kv_len, D), dtype=dtype, device=device)
        self.out = torch.empty((B, H, q_len, D), dtype=dtype, device=device)
        self.lse = torch.empty((B, H, q_len), dtype=torch.float32, device=device)
        self.doc_ids = torch.empty((B, q_len), dtype=torch.int32, device=device) if document else None
        nqb, nkvb = -(-q_len // 128), -(-kv_len // 128)
        self.kv_num_blocks = torch.empty((B, H, nqb), dtype=torch.int32, device=device)
        self.kv_indices = torch.empty((B, H, nqb, nkvb), dtype=torch.int32, device=device)
        self.full_kv_num_blocks = torch.empty((B, H, nqb), dtype=torch.int32, device=device)
        self.full_kv_indices = torch.empty((B, H, nqb, nkvb), dtype=torch.int32, device=device)
        self.device = device

    def struct(self) -> flex_device_buffers:
        d = flex_device_buffers()
        for name in ("q", "k", "v", "out", "lse", "kv_num_blocks", "kv_indices", "full_kv_num_blocks",
                     "full_kv_indices"):
            setattr(d, name, getattr(self, name).data_ptr())
        d.doc_ids = self.doc_ids.data_ptr() if self.doc_ids is not None else None
        return d


def flex_attention_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, buffers: DeviceBuffers,
                            mask_kind: int, out: torch.Tensor, lse: torch.Tensor, window: int = 0, prefix: int = 0,
                            doc_ids: torch.Tensor | None = None, score_kind: int = FLEX_SCORE_IDENTITY,
                            score_param: float = 0.0, scale: float | None = None, chunks: int = 8,
                            stream=None) -> None:
    """BlockMask build + attention from host q, k, v into host out, lse (see include/flexattn.h).

    q, k, v, out, lse (and doc_ids) are contiguous CPU tensors, pinned for the
    copies to overlap; `buffers` is the device working memory.  Asynchronous on
    `stream`: the host outputs are valid once the stream has passed the call.
    """
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    for t in (q, k, v, out, lse) + ((doc_ids,) if doc_ids is not None else ()):
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError("host tensors must be contiguous CPU tensors")
    if lse.dtype != torch.float32 or out.dtype != q.dtype:
        raise ValueError("out has the inputs' dtype, lse is float32")
    if doc_ids is not None and doc_ids.dtype != torch.int32:
        raise ValueError("doc_ids must be int32")
    tq, tk, tv = _tensor(q), _tensor(k), _tensor(v)
    params = flex_mask_params(window, prefix, doc_ids.data_ptr() if doc_ids is not None else None)
    dev = buffers.struct()
    with torch.cuda.device(buffers.device):
        rc = load_library().flex_attention_fwd_host(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv), mask_kind,
                                                    ctypes.byref(params), score_kind, float(score_param),
                                                    float(scale), ctypes.c_void_p(out.data_ptr()),
                                                    ctypes.c_void_p(lse.data_ptr()), ctypes.byref(dev), int(chunks),
                                                    _stream_handle(stream, buffers.device))
    if rc != FLEX_OK:
        raise FlexError(rc, "flex_attention_fwd_host")


def flex_selftest_wait_timeout(limit_ms: int = 50, stream=None, device=None) -> None:
    """Enqueue the bounded-wait failure check (see include/flexattn.h)."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        rc = load_library().flex_selftest_wait_timeout(int(limit_ms), _stream_handle(stream, device))
    if rc != FLEX_OK:
        raise FlexError(rc, "flex_selftest_wait_timeout")


def flex_device_status(stream=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        return int(load_library().flex_device_status(_stream_handle(stream, device)))
