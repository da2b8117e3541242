// C-ABI layer (include/flexattn.h): argument validation on the host, the
// per-device status word, and dispatch to the kernels.  Nothing here computes
// attention or block classes; every step of the path runs in the kernels.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "bwd_internal.h"

namespace flex {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_ws_mutex;
int *g_status[kMaxDevices] = {nullptr};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_mask_kind(int k) { return k >= FLEX_MASK_CAUSAL && k <= FLEX_MASK_ALL; }

int check_sizes(int32_t B, int32_t H, int32_t q_len, int32_t kv_len, int32_t q_block, int32_t kv_block) {
    if (B <= 0 || H <= 0 || q_len <= 0 || kv_len <= 0 || q_block <= 0 || kv_block <= 0) return FLEX_ERR_INVALID_ARG;
    if (!valid_block_size(q_block) || !valid_block_size(kv_block)) return FLEX_ERR_UNSUPPORTED;
    if (ceil_blocks(kv_len) > kMaxKvBlocks) return FLEX_ERR_UNSUPPORTED;
    if (B > 65535 || H > 65535) return FLEX_ERR_UNSUPPORTED;
    return FLEX_OK;
}

int check_tensor(const flex_tensor *t, int dtype, int64_t B, int64_t H, int64_t S, int64_t D) {
    if (!t || !t->data) return FLEX_ERR_INVALID_ARG;
    if (t->dtype != dtype) return FLEX_ERR_INVALID_ARG;
    if (t->shape[0] != B || t->shape[1] != H || t->shape[2] != S || t->shape[3] != D) return FLEX_ERR_SHAPE;
    if (t->stride[3] != 1) return FLEX_ERR_ALIGNMENT;
    const int64_t elem = dtype == FLEX_DTYPE_BF16 ? 2 : 4;
    for (int i = 0; i < 3; ++i)
        if (t->stride[i] <= 0 || (t->stride[i] * elem) % 16 != 0 || t->stride[i] * elem >= (int64_t(1) << 40))
            return FLEX_ERR_ALIGNMENT;
    if (!aligned16(t->data)) return FLEX_ERR_ALIGNMENT;
    return FLEX_OK;
}

// The argument checks of flex_attention_fwd (shared by every attention entry
// point); on success p describes the whole problem, all (b, h) pairs, and
// everything but the status word.
int prepare_attention(const flex_tensor *q, const flex_tensor *k, const flex_tensor *v, const flex_block_mask *bm,
                      int32_t score_kind, float score_param, float scale, void *out, float *lse, AttnProblem &p) {
    if (!q || !k || !v || !bm || !out || !lse) return FLEX_ERR_INVALID_ARG;
    const int dtype = q->dtype;
    if (dtype != FLEX_DTYPE_BF16 && dtype != FLEX_DTYPE_FP32) return FLEX_ERR_INVALID_ARG;
    if (score_kind < FLEX_SCORE_IDENTITY || score_kind > FLEX_SCORE_ALIBI) return FLEX_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return FLEX_ERR_INVALID_ARG;
    if (score_kind == FLEX_SCORE_SOFTCAP && !(score_param > 0.f && std::isfinite(score_param)))
        return FLEX_ERR_INVALID_ARG;
    const int64_t B = q->shape[0], H = q->shape[1], Sq = q->shape[2], D = q->shape[3], Skv = k->shape[2];
    if (B <= 0 || H <= 0 || Sq <= 0 || Skv <= 0 || D <= 0) return FLEX_ERR_SHAPE;
    if (D != 64 && D != 128) return FLEX_ERR_UNSUPPORTED;
    if (Sq > INT32_MAX || Skv > INT32_MAX) return FLEX_ERR_UNSUPPORTED;
    int rc = check_tensor(q, dtype, B, H, Sq, D);
    if (rc == FLEX_OK) rc = check_tensor(k, dtype, B, H, Skv, D);
    if (rc == FLEX_OK) rc = check_tensor(v, dtype, B, H, Skv, D);
    if (rc != FLEX_OK) return rc;
    if (!aligned16(out) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return FLEX_ERR_ALIGNMENT;
    // BlockMask consistency
    if (!valid_mask_kind(bm->mask_kind)) return FLEX_ERR_INVALID_ARG;
    rc = check_sizes(bm->B, bm->H, bm->q_len, bm->kv_len, bm->q_block, bm->kv_block);
    if (rc != FLEX_OK) return rc;
    if (bm->B != B || bm->H != H || bm->q_len != Sq || bm->kv_len != Skv) return FLEX_ERR_SHAPE;
    if (bm->nqb != ceil_div(bm->q_len, bm->q_block) || bm->nkvb != ceil_div(bm->kv_len, bm->kv_block))
        return FLEX_ERR_SHAPE;
    if (!bm->kv_num_blocks || !bm->kv_indices || !bm->full_kv_num_blocks || !bm->full_kv_indices)
        return FLEX_ERR_INVALID_ARG;
    if (bm->mask_kind == FLEX_MASK_DOCUMENT && (!bm->params.doc_ids || !aligned16(bm->params.doc_ids)))
        return FLEX_ERR_INVALID_ARG;
    // document ids are one row per batch entry, indexed by q and by kv alike
    if (bm->mask_kind == FLEX_MASK_DOCUMENT && Sq != Skv) return FLEX_ERR_SHAPE;
    // each kv tile's document ids are bulk-copied as whole 16-byte words
    if (bm->mask_kind == FLEX_MASK_DOCUMENT && Sq % 4 != 0) return FLEX_ERR_UNSUPPORTED;
    if (bm->mask_kind == FLEX_MASK_SLIDING_WINDOW && bm->params.window < 0) return FLEX_ERR_INVALID_ARG;
    if (B * H * ((ceil_blocks(Sq) + 1) / 2) > INT32_MAX) return FLEX_ERR_UNSUPPORTED;

    p.B = (int)B;
    p.H = (int)H;
    p.bh_begin = 0;
    p.bh_count = (int)(B * H);
    p.q_len = (int)Sq;
    p.kv_len = (int)Skv;
    p.D = (int)D;
    p.q_block = bm->q_block;
    p.kv_block = bm->kv_block;
    p.nqb = bm->nqb;
    p.nkvb = bm->nkvb;
    p.nqt = ceil_blocks(Sq);
    p.nkvt = ceil_blocks(Skv);
    for (int i = 0; i < 4; ++i) {
        p.q_stride[i] = q->stride[i];
        p.k_stride[i] = k->stride[i];
        p.v_stride[i] = v->stride[i];
    }
    p.q = q->data;
    p.k = k->data;
    p.v = v->data;
    p.out = out;
    p.lse = lse;
    p.kv_num = bm->kv_num_blocks;
    p.kv_idx = bm->kv_indices;
    p.full_num = bm->full_kv_num_blocks;
    p.full_idx = bm->full_kv_indices;
    p.mask = MaskDesc{bm->mask_kind, bm->params.window, bm->params.prefix, bm->q_len, bm->params.doc_ids,
                      bm->q_len, bm->kv_len};
    p.score_kind = score_kind;
    p.score_param = score_param;
    p.scale = scale;
    p.prescale = 0;
    p.row_max = nullptr;
    p.status = nullptr;
    return FLEX_OK;
}

cudaError_t launch_attention(const AttnProblem &p, int dtype, cudaStream_t s) {
    return dtype == FLEX_DTYPE_BF16 ? launch_attn_bf16(p, s) : launch_attn_fp32(p, s);
}

}  // namespace

int *device_status_word(int *err) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = FLEX_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    if (!g_status[dev]) {
        int *p = nullptr;
        if (cudaMalloc(&p, 256) != cudaSuccess || cudaMemset(p, 0, 256) != cudaSuccess) {
            *err = FLEX_ERR_CUDA;
            return nullptr;
        }
        g_status[dev] = p;
    }
    *err = FLEX_OK;
    return g_status[dev];
}

// ----------------------------------------------------------------------------
// Scratch for flex_attention_fwd_noalloc.  Some callers cannot let a library
// call cudaMalloc: code that enqueues work while a stream is being captured,
// plug-ins whose host framework owns every device allocation, and processes
// that must not grow device memory after start-up.  For them the status word
// that the attention kernel writes on a timed-out wait lives in this
// file-scope device array instead of the cudaMalloc'd per-device workspace.
// Every GPU that loads the library holds these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_noalloc_mutex;
int *g_noalloc_word[kMaxDevices] = {nullptr};

// Device address of the static scratch on the current device.  Looked up once
// per device (cudaGetSymbolAddress, checked) with that device current; the
// host-side name of the array is not a device address.
int *noalloc_scratch_address(int *err) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = FLEX_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_word[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
            *err = FLEX_ERR_CUDA;
            return nullptr;
        }
        g_noalloc_word[dev] = static_cast<int *>(ptr);
    }
    *err = FLEX_OK;
    return g_noalloc_word[dev];
}

// ----------------------------------------------------------------------------
// Streams and events of flex_attention_fwd_host, created once per device: the
// host-to-device copies run on `in`, the device-to-host copies on `out`, the
// BlockMask build and the attention launches on the caller's stream.
constexpr int kMaxHostChunks = 64;
struct HostPipe {
    std::mutex enqueue;  // one call enqueues at a time (the events are shared)
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, out_done = nullptr;
    cudaEvent_t in_done[kMaxHostChunks] = {}, attn_done[kMaxHostChunks] = {};
};
std::mutex g_pipe_mutex;
HostPipe *g_pipe[kMaxDevices] = {nullptr};

HostPipe *host_pipe(int *err) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *err = FLEX_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_pipe_mutex);
    if (!g_pipe[dev]) {
        HostPipe *hp = new HostPipe();
        bool ok = cudaStreamCreateWithFlags(&hp->in, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&hp->out, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaEventCreateWithFlags(&hp->start, cudaEventDisableTiming) == cudaSuccess &&
                  cudaEventCreateWithFlags(&hp->out_done, cudaEventDisableTiming) == cudaSuccess;
        for (int c = 0; ok && c < kMaxHostChunks; ++c)
            ok = cudaEventCreateWithFlags(&hp->in_done[c], cudaEventDisableTiming) == cudaSuccess &&
                 cudaEventCreateWithFlags(&hp->attn_done[c], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {  // the handles created so far stay with the process
            *err = FLEX_ERR_CUDA;
            return nullptr;
        }
        g_pipe[dev] = hp;
    }
    *err = FLEX_OK;
    return g_pipe[dev];
}

bool is_contiguous(const flex_tensor *t) {
    return t->stride[3] == 1 && t->stride[2] == t->shape[3] && t->stride[1] == t->shape[2] * t->shape[3] &&
           t->stride[0] == t->shape[1] * t->shape[2] * t->shape[3];
}

}  // namespace

}  // namespace flex

using namespace flex;

extern "C" {

int flex_block_mask_sizes_qkv(int32_t B, int32_t H, int32_t q_len, int32_t kv_len, int32_t q_block,
                              int32_t kv_block, int64_t *num_elems, int64_t *idx_elems) {
    if (!num_elems || !idx_elems) return FLEX_ERR_INVALID_ARG;
    const int rc = check_sizes(B, H, q_len, kv_len, q_block, kv_block);
    if (rc != FLEX_OK) return rc;
    const int64_t nqb = ceil_div(q_len, q_block), nkvb = ceil_div(kv_len, kv_block);
    *num_elems = (int64_t)B * H * nqb;
    *idx_elems = (int64_t)B * H * nqb * nkvb;
    return FLEX_OK;
}

int flex_block_mask_sizes(int32_t B, int32_t H, int32_t q_len, int32_t kv_len, int32_t block, int64_t *num_elems,
                          int64_t *idx_elems) {
    return flex_block_mask_sizes_qkv(B, H, q_len, kv_len, block, block, num_elems, idx_elems);
}

int flex_block_mask_create(int32_t mask_kind, const flex_mask_params *params, int32_t B, int32_t H, int32_t q_len,
                           int32_t kv_len, int32_t block, flex_block_mask *bm, void *stream) {
    return flex_block_mask_create_qkv(mask_kind, params, B, H, q_len, kv_len, block, block, bm, stream);
}

int flex_block_mask_create_qkv(int32_t mask_kind, const flex_mask_params *params, int32_t B, int32_t H,
                               int32_t q_len, int32_t kv_len, int32_t q_block, int32_t kv_block, flex_block_mask *bm,
                               void *stream) {
    if (!bm || !valid_mask_kind(mask_kind)) return FLEX_ERR_INVALID_ARG;
    const int rc = check_sizes(B, H, q_len, kv_len, q_block, kv_block);
    if (rc != FLEX_OK) return rc;
    if (!bm->kv_num_blocks || !bm->kv_indices || !bm->full_kv_num_blocks || !bm->full_kv_indices)
        return FLEX_ERR_INVALID_ARG;
    flex_mask_params prm = {0, 0, nullptr};
    if (params) prm = *params;
    if (mask_kind == FLEX_MASK_SLIDING_WINDOW && (!params || prm.window < 0)) return FLEX_ERR_INVALID_ARG;
    if (mask_kind == FLEX_MASK_CAUSAL_PREFIX && !params) return FLEX_ERR_INVALID_ARG;
    if (mask_kind == FLEX_MASK_DOCUMENT) {
        if (!params || !prm.doc_ids) return FLEX_ERR_INVALID_ARG;
        if (q_len != kv_len) return FLEX_ERR_SHAPE;
        if (!aligned16(prm.doc_ids)) return FLEX_ERR_ALIGNMENT;
    }
    bm->B = B;
    bm->H = H;
    bm->q_len = q_len;
    bm->kv_len = kv_len;
    bm->q_block = q_block;
    bm->kv_block = kv_block;
    bm->nqb = ceil_div(q_len, q_block);
    bm->nkvb = ceil_div(kv_len, kv_block);
    bm->mask_kind = mask_kind;
    bm->params = prm;
    MaskDesc md{mask_kind, prm.window, prm.prefix, q_len, prm.doc_ids, q_len, kv_len};
    const cudaError_t e = launch_block_mask(md, B, H, q_len, kv_len, q_block, kv_block, bm->kv_num_blocks,
                                            bm->kv_indices, bm->full_kv_num_blocks, bm->full_kv_indices,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FLEX_OK : FLEX_ERR_CUDA;
}

int flex_attention_fwd(const flex_tensor *q, const flex_tensor *k, const flex_tensor *v, const flex_block_mask *bm,
                       int32_t score_kind, float score_param, float scale, void *out, float *lse, void *stream) {
    AttnProblem p;
    const int rc = prepare_attention(q, k, v, bm, score_kind, score_param, scale, out, lse, p);
    if (rc != FLEX_OK) return rc;
    int err = FLEX_OK;
    p.status = device_status_word(&err);
    if (!p.status) return err;
    return launch_attention(p, q->dtype, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FLEX_OK : FLEX_ERR_CUDA;
}

int flex_attention_fwd_opts(const flex_tensor *q, const flex_tensor *k, const flex_tensor *v,
                            const flex_block_mask *bm, int32_t score_kind, float score_param, float scale,
                            void *out, float *lse, const flex_kernel_options *opts, void *stream) {
    AttnProblem p;
    int rc = prepare_attention(q, k, v, bm, score_kind, score_param, scale, out, lse, p);
    if (rc != FLEX_OK) return rc;
    if (opts) {
        if ((opts->prescale_qk != 0 && opts->prescale_qk != 1) ||
            (opts->rows_guaranteed_safe != 0 && opts->rows_guaranteed_safe != 1))
            return FLEX_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(opts->max_scores) & 3u) return FLEX_ERR_ALIGNMENT;
        // scale 0 makes q~ = 0: the same scores as scaling after QK^T
        p.prescale = opts->prescale_qk && scale != 0.f;
        p.row_max = opts->max_scores;
        // rows_guaranteed_safe needs nothing: the kernels carry no per-tile
        // guard for rows without an unmasked score (see the header)
    }
    int err = FLEX_OK;
    p.status = device_status_word(&err);
    if (!p.status) return err;
    return launch_attention(p, q->dtype, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FLEX_OK : FLEX_ERR_CUDA;
}

int flex_block_mask_transpose(const flex_block_mask *bm, flex_block_mask_q *bq, void *stream) {
    if (!bm || !bq) return FLEX_ERR_INVALID_ARG;
    int rc = check_sizes(bm->B, bm->H, bm->q_len, bm->kv_len, bm->q_block, bm->kv_block);
    if (rc != FLEX_OK) return rc;
    if (bm->nqb != ceil_div(bm->q_len, bm->q_block) || bm->nkvb != ceil_div(bm->kv_len, bm->kv_block))
        return FLEX_ERR_SHAPE;
    if (!bm->kv_num_blocks || !bm->kv_indices || !bm->full_kv_num_blocks || !bm->full_kv_indices)
        return FLEX_ERR_INVALID_ARG;
    if (!bq->q_num_blocks || !bq->q_indices || !bq->full_q_num_blocks || !bq->full_q_indices)
        return FLEX_ERR_INVALID_ARG;
    bq->B = bm->B;
    bq->H = bm->H;
    bq->q_len = bm->q_len;
    bq->kv_len = bm->kv_len;
    bq->q_block = bm->q_block;
    bq->kv_block = bm->kv_block;
    bq->nqb = bm->nqb;
    bq->nkvb = bm->nkvb;
    return launch_block_mask_transpose(bm->kv_num_blocks, bm->kv_indices, bm->full_kv_num_blocks,
                                       bm->full_kv_indices, bm->B, bm->H, bm->nqb, bm->nkvb, bq->q_num_blocks,
                                       bq->q_indices, bq->full_q_num_blocks, bq->full_q_indices,
                                       static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? FLEX_OK
               : FLEX_ERR_CUDA;
}

int flex_attention_bwd(const flex_tensor *q, const flex_tensor *k, const flex_tensor *v, const void *out,
                       const float *lse, const void *dout, const flex_block_mask *bm, const flex_block_mask_q *bq,
                       int32_t score_kind, float score_param, float scale, void *dq, void *dk, void *dv,
                       float *delta, void *stream) {
    AttnProblem p;
    int rc = prepare_attention(q, k, v, bm, score_kind, score_param, scale, const_cast<void *>(out),
                               const_cast<float *>(lse), p);
    if (rc != FLEX_OK) return rc;
    if (!dout || !bq || !dq || !dk || !dv || !delta) return FLEX_ERR_INVALID_ARG;
    if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
        (reinterpret_cast<uintptr_t>(delta) & 3u))
        return FLEX_ERR_ALIGNMENT;
    if (bq->B != bm->B || bq->H != bm->H || bq->q_len != bm->q_len || bq->kv_len != bm->kv_len ||
        bq->q_block != bm->q_block || bq->kv_block != bm->kv_block || bq->nqb != bm->nqb || bq->nkvb != bm->nkvb)
        return FLEX_ERR_SHAPE;
    if (!bq->q_num_blocks || !bq->q_indices || !bq->full_q_num_blocks || !bq->full_q_indices)
        return FLEX_ERR_INVALID_ARG;
    // the tensor-core backward holds a kv tile's list of q tiles on chip
    if (q->dtype == FLEX_DTYPE_BF16 && p.nqt > kBwdTcMaxQBlocks) return FLEX_ERR_UNSUPPORTED;
    return launch_attn_bwd(p, q->dtype, dout, bq->q_num_blocks, bq->q_indices, bq->full_q_num_blocks,
                           bq->full_q_indices, dq, dk, dv, delta, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? FLEX_OK
               : FLEX_ERR_CUDA;
}

int flex_device_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FLEX_ERR_CUDA;
    int err = FLEX_OK;
    int *status = device_status_word(&err);
    if (!status) return err;
    int host = 0;
    if (cudaMemcpy(&host, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FLEX_ERR_CUDA;
    if (host != 0 && cudaMemset(status, 0, sizeof(int)) != cudaSuccess) return FLEX_ERR_CUDA;
    return host == 0 ? FLEX_OK : FLEX_ERR_DEVICE_TIMEOUT;
}

int flex_selftest_wait_timeout(uint32_t limit_ms, void *stream) {
    if (limit_ms == 0 || limit_ms > 60000) return FLEX_ERR_INVALID_ARG;
    int err = FLEX_OK;
    int *status = device_status_word(&err);
    if (!status) return err;
    const cudaError_t e =
        launch_wait_timeout_selftest(status, (uint64_t)limit_ms * 1000000ull, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FLEX_OK : FLEX_ERR_CUDA;
}

const char *flex_status_string(int status) {
    switch (status) {
        case FLEX_OK:
            return "ok";
        case FLEX_ERR_INVALID_ARG:
            return "invalid argument";
        case FLEX_ERR_UNSUPPORTED:
            return "unsupported configuration";
        case FLEX_ERR_SHAPE:
            return "shapes, lengths or BlockMask sizes disagree";
        case FLEX_ERR_ALIGNMENT:
            return "pointer or stride not 16-byte aligned, or inner stride is not 1";
        case FLEX_ERR_CUDA:
            return "CUDA error";
        case FLEX_ERR_DEVICE_TIMEOUT:
            return "a kernel gave up on a device-side wait";
        default:
            return "unknown status";
    }
}

int flex_attention_fwd_noalloc(const flex_tensor *q, const flex_tensor *k, const flex_tensor *v,
                               const flex_block_mask *bm, int32_t score_kind, float score_param, float scale,
                               void *out, float *lse, void *stream, const int **device_status) {
    if (device_status) *device_status = nullptr;
    // the same argument checks as flex_attention_fwd
    AttnProblem p;
    const int rc = prepare_attention(q, k, v, bm, score_kind, score_param, scale, out, lse, p);
    if (rc != FLEX_OK) return rc;

    // The kernel's scratch is one int status word whatever the problem size;
    // anything larger than the static array is refused.
    constexpr size_t kScratchNeeded = sizeof(int);
    if (kScratchNeeded > kNoAllocScratchBytes) return FLEX_ERR_UNSUPPORTED;
    int err = FLEX_OK;
    int *status = noalloc_scratch_address(&err);
    if (!status) return err;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the kernel only ever sets the word, so every call starts it at zero
    if (cudaMemsetAsync(status, 0, kScratchNeeded, s) != cudaSuccess) return FLEX_ERR_CUDA;
    p.status = status;
    if (launch_attention(p, q->dtype, s) != cudaSuccess) return FLEX_ERR_CUDA;
    if (device_status) *device_status = status;
    return FLEX_OK;
}

int flex_attention_fwd_host(const flex_tensor *q, const flex_tensor *k, const flex_tensor *v, int32_t mask_kind,
                            const flex_mask_params *params, int32_t score_kind, float score_param, float scale,
                            void *out, float *lse, const flex_device_buffers *dev, int32_t chunks, void *stream) {
    if (!q || !k || !v || !out || !lse || !dev) return FLEX_ERR_INVALID_ARG;
    if (chunks < 1 || chunks > kMaxHostChunks) return FLEX_ERR_INVALID_ARG;
    if (!q->data || !k->data || !v->data) return FLEX_ERR_INVALID_ARG;
    if (!is_contiguous(q) || !is_contiguous(k) || !is_contiguous(v)) return FLEX_ERR_INVALID_ARG;
    if (!valid_mask_kind(mask_kind)) return FLEX_ERR_INVALID_ARG;
    const bool doc = mask_kind == FLEX_MASK_DOCUMENT;
    if ((mask_kind == FLEX_MASK_SLIDING_WINDOW || mask_kind == FLEX_MASK_CAUSAL_PREFIX || doc) && !params)
        return FLEX_ERR_INVALID_ARG;
    if (mask_kind == FLEX_MASK_SLIDING_WINDOW && params->window < 0) return FLEX_ERR_INVALID_ARG;
    if (doc && (!params->doc_ids || !dev->doc_ids)) return FLEX_ERR_INVALID_ARG;
    if (doc && !aligned16(dev->doc_ids)) return FLEX_ERR_ALIGNMENT;
    const int64_t B64 = q->shape[0], H64 = q->shape[1], Sq64 = q->shape[2], Skv64 = k->shape[2];
    if (B64 <= 0 || H64 <= 0 || Sq64 <= 0 || Skv64 <= 0) return FLEX_ERR_SHAPE;
    if (B64 > INT32_MAX || H64 > INT32_MAX || Sq64 > INT32_MAX || Skv64 > INT32_MAX) return FLEX_ERR_UNSUPPORTED;
    const int B = (int)B64, H = (int)H64, Sq = (int)Sq64, Skv = (int)Skv64;
    int rc = check_sizes(B, H, Sq, Skv, kBlock, kBlock);
    if (rc != FLEX_OK) return rc;
    if (doc && Sq != Skv) return FLEX_ERR_SHAPE;

    // The same problem on the caller's device buffers, checked in full before
    // anything is enqueued.
    flex_tensor dq = *q, dk = *k, dv = *v;
    dq.data = dev->q;
    dk.data = dev->k;
    dv.data = dev->v;
    flex_block_mask bm = {};
    bm.B = B;
    bm.H = H;
    bm.q_len = Sq;
    bm.kv_len = Skv;
    bm.q_block = kBlock;
    bm.kv_block = kBlock;
    bm.nqb = ceil_blocks(Sq);
    bm.nkvb = ceil_blocks(Skv);
    bm.mask_kind = mask_kind;
    bm.params = params ? *params : flex_mask_params{0, 0, nullptr};
    bm.params.doc_ids = doc ? dev->doc_ids : nullptr;
    bm.kv_num_blocks = dev->kv_num_blocks;
    bm.kv_indices = dev->kv_indices;
    bm.full_kv_num_blocks = dev->full_kv_num_blocks;
    bm.full_kv_indices = dev->full_kv_indices;
    AttnProblem p;
    rc = prepare_attention(&dq, &dk, &dv, &bm, score_kind, score_param, scale, dev->out, dev->lse, p);
    if (rc != FLEX_OK) return rc;
    int err = FLEX_OK;
    p.status = device_status_word(&err);
    if (!p.status) return err;
    HostPipe *hp = host_pipe(&err);
    if (!hp) return err;

    std::lock_guard<std::mutex> lock(hp->enqueue);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t elem = q->dtype == FLEX_DTYPE_BF16 ? 2 : 4;
    const int64_t D = q->shape[3];
    const int64_t q_row = Sq64 * D * elem, kv_row = Skv64 * D * elem;  // bytes per (b, h) pair
    const int nbh = B * H;
    const int per = (nbh + chunks - 1) / chunks;
    const int nch = (nbh + per - 1) / per;
    auto ok = [](cudaError_t e) { return e == cudaSuccess; };
    bool good = ok(cudaEventRecord(hp->start, s)) && ok(cudaStreamWaitEvent(hp->in, hp->start, 0)) &&
                ok(cudaStreamWaitEvent(hp->out, hp->start, 0));
    // document ids and the BlockMask (all heads; cheap) on the caller's stream
    if (good && doc)
        good = ok(cudaMemcpyAsync(dev->doc_ids, params->doc_ids, (size_t)B64 * Sq64 * sizeof(int32_t),
                                  cudaMemcpyHostToDevice, s));
    if (good)
        good = ok(launch_block_mask(p.mask, B, H, Sq, Skv, kBlock, kBlock, bm.kv_num_blocks, bm.kv_indices,
                                    bm.full_kv_num_blocks, bm.full_kv_indices, s));
    // inputs of every chunk, back to back on the copy-in stream
    for (int c = 0; good && c < nch; ++c) {
        const int64_t b0 = (int64_t)c * per, n = std::min<int64_t>(per, nbh - b0);
        good = ok(cudaMemcpyAsync(static_cast<char *>(dev->q) + b0 * q_row,
                                  static_cast<const char *>(q->data) + b0 * q_row, n * q_row,
                                  cudaMemcpyHostToDevice, hp->in)) &&
               ok(cudaMemcpyAsync(static_cast<char *>(dev->k) + b0 * kv_row,
                                  static_cast<const char *>(k->data) + b0 * kv_row, n * kv_row,
                                  cudaMemcpyHostToDevice, hp->in)) &&
               ok(cudaMemcpyAsync(static_cast<char *>(dev->v) + b0 * kv_row,
                                  static_cast<const char *>(v->data) + b0 * kv_row, n * kv_row,
                                  cudaMemcpyHostToDevice, hp->in)) &&
               ok(cudaEventRecord(hp->in_done[c], hp->in));
    }
    // attention of each chunk once its inputs are in, results back as they finish
    for (int c = 0; good && c < nch; ++c) {
        const int64_t b0 = (int64_t)c * per, n = std::min<int64_t>(per, nbh - b0);
        p.bh_begin = (int)b0;
        p.bh_count = (int)n;
        good = ok(cudaStreamWaitEvent(s, hp->in_done[c], 0)) && ok(launch_attention(p, q->dtype, s)) &&
               ok(cudaEventRecord(hp->attn_done[c], s)) && ok(cudaStreamWaitEvent(hp->out, hp->attn_done[c], 0)) &&
               ok(cudaMemcpyAsync(static_cast<char *>(out) + b0 * q_row, static_cast<const char *>(dev->out) + b0 * q_row,
                                  n * q_row, cudaMemcpyDeviceToHost, hp->out)) &&
               ok(cudaMemcpyAsync(lse + b0 * Sq64, dev->lse + b0 * Sq64, n * Sq64 * sizeof(float),
                                  cudaMemcpyDeviceToHost, hp->out));
    }
    if (good) good = ok(cudaEventRecord(hp->out_done, hp->out)) && ok(cudaStreamWaitEvent(s, hp->out_done, 0));
    return good ? FLEX_OK : FLEX_ERR_CUDA;
}

}  // extern "C"
