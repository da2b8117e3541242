"""The C-ABI library builds for sm_103a, loads, exports every symbol the
header declares, and rejects bad arguments on the host (no GPU needed: every
call here fails validation before any CUDA call)."""
import ctypes
import os
import re

import pytest

from block_sparse_masked_blockmask_gb300 import _build, flexattn as fa

HEADER = os.path.join(_build.INCLUDE, "flexattn.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return fa.load_library()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"FLEX_API\s+[\w\s\*]+?\b(flex_\w+)\s*\(", text)


def test_header_declares_the_calls():
    names = declared_functions()
    assert sorted(names) == sorted(fa.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in (fa.FLEX_OK, fa.FLEX_ERR_INVALID_ARG, fa.FLEX_ERR_UNSUPPORTED, fa.FLEX_ERR_SHAPE,
                 fa.FLEX_ERR_ALIGNMENT, fa.FLEX_ERR_CUDA, fa.FLEX_ERR_DEVICE_TIMEOUT):
        s = fa.flex_status_string(code)
        assert s and s != "unknown status"
    assert fa.flex_status_string(12345) == "unknown status"


def test_block_mask_sizes_other_blocks(lib):
    # Q_BLOCK and KV_BLOCK: powers of two from 16 to 1024, possibly different
    assert fa.flex_block_mask_sizes(2, 3, 1024, 1024, 64) == (2 * 3 * 16, 2 * 3 * 16 * 16)
    assert fa.flex_block_mask_sizes(1, 1, 1000, 300, 256, kv_block=64) == (4, 4 * 5)
    assert fa.flex_block_mask_sizes(1, 1, 100, 100, 16, kv_block=1024) == (7, 7)
    with pytest.raises(fa.FlexError) as e:
        fa.flex_block_mask_sizes(1, 1, 128, 128, 128, kv_block=100)
    assert e.value.code == fa.FLEX_ERR_UNSUPPORTED


def test_block_mask_sizes(lib):
    assert fa.flex_block_mask_sizes(2, 32, 16384, 16384) == (2 * 32 * 128, 2 * 32 * 128 * 128)
    assert fa.flex_block_mask_sizes(1, 1, 128, 384) == (1, 3)
    # lengths need not be multiples of the block: the tail tile is counted
    assert fa.flex_block_mask_sizes(1, 1, 100, 128) == (1, 1)
    assert fa.flex_block_mask_sizes(2, 3, 129, 300) == (2 * 3 * 2, 2 * 3 * 2 * 3)
    assert fa.flex_block_mask_sizes(1, 1, 1, 128 * 1024) == (1, 1024)
    for args, code in [((0, 1, 128, 128), fa.FLEX_ERR_INVALID_ARG),
                       ((1, 1, 0, 128), fa.FLEX_ERR_INVALID_ARG),
                       ((1, 1, 128, 128, 96), fa.FLEX_ERR_UNSUPPORTED),  # not a power of two
                       ((1, 1, 128, 128, 8), fa.FLEX_ERR_UNSUPPORTED),
                       ((1, 1, 128, 128, 2048), fa.FLEX_ERR_UNSUPPORTED),
                       ((1, 1, 128, 128 * 1024 + 1), fa.FLEX_ERR_UNSUPPORTED),
                       ((1, 1, 128, 128 * 1025), fa.FLEX_ERR_UNSUPPORTED)]:
        with pytest.raises(fa.FlexError) as e:
            fa.flex_block_mask_sizes(*args)
        assert e.value.code == code, args


def _call_create(lib, kind, params, B=1, H=1, q=256, kv=256, block=128, buffers=True):
    bm = fa.flex_block_mask()
    if buffers:  # non-null dummies: validation must fail before they are touched
        bm.kv_num_blocks = bm.kv_indices = bm.full_kv_num_blocks = bm.full_kv_indices = 0x1000
    p = None if params is None else ctypes.byref(params)
    return lib.flex_block_mask_create(kind, p, B, H, q, kv, block, ctypes.byref(bm), None)


def test_block_mask_create_rejects_bad_arguments(lib):
    assert _call_create(lib, 7, None) == fa.FLEX_ERR_INVALID_ARG
    assert _call_create(lib, fa.FLEX_MASK_CAUSAL, None, buffers=False) == fa.FLEX_ERR_INVALID_ARG
    assert _call_create(lib, fa.FLEX_MASK_CAUSAL, None, q=-200) == fa.FLEX_ERR_INVALID_ARG
    assert _call_create(lib, fa.FLEX_MASK_CAUSAL, None, block=96) == fa.FLEX_ERR_UNSUPPORTED
    assert _call_create(lib, fa.FLEX_MASK_CAUSAL, None, block=2048) == fa.FLEX_ERR_UNSUPPORTED
    assert _call_create(lib, fa.FLEX_MASK_SLIDING_WINDOW, None) == fa.FLEX_ERR_INVALID_ARG
    assert _call_create(lib, fa.FLEX_MASK_SLIDING_WINDOW, fa.flex_mask_params(-1, 0, None)) == \
        fa.FLEX_ERR_INVALID_ARG
    assert _call_create(lib, fa.FLEX_MASK_DOCUMENT, fa.flex_mask_params(0, 0, None)) == fa.FLEX_ERR_INVALID_ARG
    assert _call_create(lib, fa.FLEX_MASK_DOCUMENT, fa.flex_mask_params(0, 0, 0x1000), kv=384) == \
        fa.FLEX_ERR_SHAPE
    assert _call_create(lib, fa.FLEX_MASK_DOCUMENT, fa.flex_mask_params(0, 0, 0x1004)) == fa.FLEX_ERR_ALIGNMENT


def _tensor(dtype, shape, stride=None, data=0x10000):
    t = fa.flex_tensor()
    t.data = data
    t.dtype = dtype
    if stride is None:
        stride = [shape[1] * shape[2] * shape[3], shape[2] * shape[3], shape[3], 1]
    for i in range(4):
        t.shape[i] = shape[i]
        t.stride[i] = stride[i]
    return t


def _mask_struct(B=1, H=2, q=256, kv=256, kind=fa.FLEX_MASK_CAUSAL):
    bm = fa.flex_block_mask()
    bm.B, bm.H, bm.q_len, bm.kv_len, bm.q_block, bm.kv_block = B, H, q, kv, 128, 128
    bm.nqb, bm.nkvb, bm.mask_kind = -(-q // 128), -(-kv // 128), kind
    bm.kv_num_blocks = bm.kv_indices = bm.full_kv_num_blocks = bm.full_kv_indices = 0x1000
    return bm


def _doc_mask_struct(S):
    bm = _mask_struct(q=S, kv=S, kind=fa.FLEX_MASK_DOCUMENT)
    bm.params.doc_ids = 0x4000
    return bm


def _doc_kv_mask_struct(q, kv):
    bm = _mask_struct(q=q, kv=kv, kind=fa.FLEX_MASK_DOCUMENT)
    bm.params.doc_ids = 0x4000
    return bm


def _fwd(lib, q, k, v, bm, score=fa.FLEX_SCORE_IDENTITY, param=0.0, scale=0.125, out=0x20000, lse=0x30000):
    return lib.flex_attention_fwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(bm), score,
                                  param, scale, ctypes.c_void_p(out), ctypes.c_void_p(lse), None)


def test_attention_rejects_bad_arguments(lib):
    bf = fa.FLEX_DTYPE_BF16
    q = _tensor(bf, [1, 2, 256, 64])
    bm = _mask_struct()
    cases = [
        (dict(q=_tensor(bf, [1, 2, 256, 96]), k=_tensor(bf, [1, 2, 256, 96]), v=_tensor(bf, [1, 2, 256, 96])),
         fa.FLEX_ERR_UNSUPPORTED),
        (dict(k=_tensor(fa.FLEX_DTYPE_FP32, [1, 2, 256, 64])), fa.FLEX_ERR_INVALID_ARG),
        (dict(k=_tensor(bf, [1, 3, 256, 64])), fa.FLEX_ERR_SHAPE),
        (dict(v=_tensor(bf, [1, 2, 256, 64], stride=[32768, 16384, 64, 2])), fa.FLEX_ERR_ALIGNMENT),
        (dict(v=_tensor(bf, [1, 2, 256, 64], stride=[32768, 16384, 68, 1])), fa.FLEX_ERR_ALIGNMENT),
        (dict(k=_tensor(bf, [1, 2, 256, 64], data=0x10002)), fa.FLEX_ERR_ALIGNMENT),
        (dict(out=0x20008), fa.FLEX_ERR_ALIGNMENT),
        (dict(lse=0), fa.FLEX_ERR_INVALID_ARG),
        (dict(score=3), fa.FLEX_ERR_INVALID_ARG),
        (dict(score=fa.FLEX_SCORE_SOFTCAP, param=0.0), fa.FLEX_ERR_INVALID_ARG),
        (dict(scale=float("nan")), fa.FLEX_ERR_INVALID_ARG),
        (dict(bm=_mask_struct(H=3)), fa.FLEX_ERR_SHAPE),
        (dict(bm=_mask_struct(q=384, kv=384)), fa.FLEX_ERR_SHAPE),
        (dict(bm=_mask_struct(kind=9)), fa.FLEX_ERR_INVALID_ARG),
        (dict(q=_tensor(bf, [1, 2, 200, 64])), fa.FLEX_ERR_SHAPE),  # the BlockMask is for 256 rows
        (dict(bm=_mask_struct(q=256, kv=200)), fa.FLEX_ERR_SHAPE),  # ... or for 200 kv rows
        # document masks need Q_LEN a multiple of 4
        (dict(q=_tensor(bf, [1, 2, 202, 64]), k=_tensor(bf, [1, 2, 202, 64]), v=_tensor(bf, [1, 2, 202, 64]),
              bm=_doc_mask_struct(202)), fa.FLEX_ERR_UNSUPPORTED),
        # ... and Q_LEN == KV_LEN: a caller-filled document BlockMask with more
        # kv rows than ids per row is refused before anything is launched
        (dict(k=_tensor(bf, [1, 2, 384, 64]), v=_tensor(bf, [1, 2, 384, 64]),
              bm=_doc_kv_mask_struct(256, 384)), fa.FLEX_ERR_SHAPE),
    ]
    for change, code in cases:
        args = dict(q=q, k=_tensor(bf, [1, 2, 256, 64]), v=_tensor(bf, [1, 2, 256, 64]), bm=bm)
        args.update(change)
        rc = _fwd(lib, args.pop("q"), args.pop("k"), args.pop("v"), args.pop("bm"), **args)
        assert rc == code, (change, rc)


def test_product_path_has_no_oracle_dependency():
    pkg = os.path.dirname(_build.__file__)
    for root, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(root, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "liboracle" not in text, f


def test_host_entry_point_rejects_bad_arguments(lib):
    # every case fails its checks before any CUDA call
    bf = fa.FLEX_DTYPE_BF16
    dev = fa.flex_device_buffers()
    for name, addr in (("q", 0x10000), ("k", 0x20000), ("v", 0x30000), ("out", 0x40000), ("lse", 0x50000),
                       ("kv_num_blocks", 0x60000), ("kv_indices", 0x70000), ("full_kv_num_blocks", 0x80000),
                       ("full_kv_indices", 0x90000)):
        setattr(dev, name, addr)

    def call(q=None, k=None, v=None, kind=fa.FLEX_MASK_CAUSAL, params=None, score=fa.FLEX_SCORE_IDENTITY,
             out=0x100000, lse=0x200000, devbuf=dev, chunks=4):
        q = q or _tensor(bf, [1, 2, 256, 64])
        k = k or _tensor(bf, [1, 2, 256, 64])
        v = v or _tensor(bf, [1, 2, 256, 64])
        return lib.flex_attention_fwd_host(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), kind,
                                           ctypes.byref(params) if params is not None else None, score, 0.0, 0.125,
                                           ctypes.c_void_p(out), ctypes.c_void_p(lse),
                                           ctypes.byref(devbuf) if devbuf is not None else None, chunks, None)

    assert call(chunks=0) == fa.FLEX_ERR_INVALID_ARG
    assert call(chunks=65) == fa.FLEX_ERR_INVALID_ARG
    assert call(devbuf=None) == fa.FLEX_ERR_INVALID_ARG
    assert call(out=0) == fa.FLEX_ERR_INVALID_ARG
    # host tensors must be contiguous
    assert call(v=_tensor(bf, [1, 2, 256, 64], stride=[65536, 32768, 64, 1])) == fa.FLEX_ERR_INVALID_ARG
    assert call(kind=9) == fa.FLEX_ERR_INVALID_ARG
    assert call(kind=fa.FLEX_MASK_SLIDING_WINDOW) == fa.FLEX_ERR_INVALID_ARG  # needs params
    assert call(kind=fa.FLEX_MASK_DOCUMENT, params=fa.flex_mask_params(0, 0, 0x1000)) == fa.FLEX_ERR_INVALID_ARG
    assert call(q=_tensor(bf, [1, 2, 200, 64], stride=[1, 1, 1, 1])) == fa.FLEX_ERR_INVALID_ARG  # not contiguous
    assert call(k=_tensor(bf, [1, 3, 256, 64])) == fa.FLEX_ERR_SHAPE
    assert call(score=7) == fa.FLEX_ERR_INVALID_ARG
    unaligned = fa.flex_device_buffers.from_buffer_copy(dev)
    unaligned.out = 0x40008
    assert call(devbuf=unaligned) == fa.FLEX_ERR_ALIGNMENT


def test_options_entry_point_rejects_bad_arguments(lib):
    # flex_attention_fwd_opts: the checks of flex_attention_fwd plus the options',
    # all before any CUDA call
    bf = fa.FLEX_DTYPE_BF16
    q, k, v = (_tensor(bf, [1, 2, 256, 64]) for _ in range(3))
    bm = _mask_struct()

    def call(opts, q=q, score=fa.FLEX_SCORE_IDENTITY):
        return lib.flex_attention_fwd_opts(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.byref(bm),
                                           score, 0.0, 0.125, ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000),
                                           ctypes.byref(opts) if opts is not None else None, None)

    assert call(fa.flex_kernel_options(2, 0, None)) == fa.FLEX_ERR_INVALID_ARG
    assert call(fa.flex_kernel_options(0, -1, None)) == fa.FLEX_ERR_INVALID_ARG
    assert call(fa.flex_kernel_options(1, 1, 0x40002)) == fa.FLEX_ERR_ALIGNMENT
    # the shared checks come first and still apply
    assert call(fa.flex_kernel_options(1, 0, 0x40000), score=3) == fa.FLEX_ERR_INVALID_ARG
    assert call(None, q=_tensor(bf, [1, 2, 384, 64])) == fa.FLEX_ERR_SHAPE


def test_backward_entry_points_reject_bad_arguments(lib):
    # flex_block_mask_transpose and flex_attention_bwd: every case fails its
    # checks before any CUDA call
    bf = fa.FLEX_DTYPE_BF16
    bm = _mask_struct()
    bq = fa.flex_block_mask_q()
    bq.B, bq.H, bq.q_len, bq.kv_len, bq.q_block, bq.kv_block, bq.nqb, bq.nkvb = 1, 2, 256, 256, 128, 128, 2, 2
    bq.q_num_blocks = bq.q_indices = bq.full_q_num_blocks = bq.full_q_indices = 0x2000
    assert lib.flex_block_mask_transpose(None, ctypes.byref(bq), None) == fa.FLEX_ERR_INVALID_ARG
    empty = fa.flex_block_mask_q()
    assert lib.flex_block_mask_transpose(ctypes.byref(bm), ctypes.byref(empty), None) == fa.FLEX_ERR_INVALID_ARG
    q, k, v = (_tensor(bf, [1, 2, 256, 64]) for _ in range(3))

    def call(bq=bq, dq=0x40000, delta=0x50000, dout=0x60000, score=fa.FLEX_SCORE_IDENTITY):
        return lib.flex_attention_bwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), ctypes.c_void_p(0x20000),
                                      ctypes.c_void_p(0x30000), ctypes.c_void_p(dout), ctypes.byref(bm),
                                      ctypes.byref(bq) if bq is not None else None, score, 0.0, 0.125,
                                      ctypes.c_void_p(dq), ctypes.c_void_p(0x70000), ctypes.c_void_p(0x80000),
                                      ctypes.c_void_p(delta), None)

    assert call(bq=None) == fa.FLEX_ERR_INVALID_ARG
    assert call(dq=0x40008) == fa.FLEX_ERR_ALIGNMENT
    assert call(delta=0x50002) == fa.FLEX_ERR_ALIGNMENT
    assert call(dout=0) == fa.FLEX_ERR_INVALID_ARG
    assert call(score=5) == fa.FLEX_ERR_INVALID_ARG
    other = fa.flex_block_mask_q.from_buffer_copy(bq)
    other.nkvb = 3
    assert call(bq=other) == fa.FLEX_ERR_SHAPE
