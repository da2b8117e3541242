/*
 * flexattn.h -- C-ABI of the GB300 (sm_103a) block-sparse FlexAttention forward.
 *
 * Two calls do the work:
 *   flex_block_mask_create  builds a BlockMask from an enumerated mask_mod;
 *   flex_attention_fwd      runs softmax(mask(score_mod(Q K^T * scale))) V
 *                           block-sparsely from that BlockMask and returns the
 *                           output and the per-row log-sum-exp
 *                           (flex_attention_fwd_opts: the same with the op's
 *                           kernel options, e.g. the row max as a third output).
 *   flex_attention_bwd      the gradients dq, dk, dv of the same attention,
 *                           walking the q side of the BlockMask
 *                           (flex_block_mask_transpose) for dk and dv.
 * Helpers size the BlockMask buffers, name status codes and read the device
 * status word.
 *
 * Sources of the semantics (web pages on PyTorch FlexAttention):
 *  - "[Inductor][Flex Attention] Add Subtiling Option for Alpha Scaling"
 *    (PyTorch PR #167356): the flex_attention higher-order op signature
 *    flex_attention(q, k, v, score_mod, block_mask, scale, kernel_options),
 *    the BlockMask tuple (kv_num_blocks, kv_indices, full_kv_num_blocks,
 *    full_kv_indices, ..., Q_BLOCK = KV_BLOCK = 128, mask_mod), the
 *    OUTPUT_LOGSUMEXP option, and the online-softmax step forward_block_mn
 *    (l_i = l_i * alpha + sum(p); acc = acc * alpha; acc += p @ v).
 *  - "Performance for templated attention strangely bad for a combination of
 *    causal + upper square mask" (PyTorch issue #124369): masked scores become
 *    -inf (torch.where); the causal + upper-square predicate
 *    (q <= 1024 and kv <= 1024) or (q >= kv).
 *
 * Conventions shared by every call:
 *  - Every pointer named "device" is CUDA device memory owned by the caller;
 *    the library never frees caller memory and keeps no per-call state.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Work is enqueued asynchronously on it; the calls do not
 *    synchronise the host except where stated.
 *  - Return value: FLEX_OK (0) or a negative flex_status.  Argument errors
 *    are detected on the host before anything is enqueued.  A CUDA launch
 *    error returns FLEX_ERR_CUDA.  A device-side wait that exceeds its time
 *    limit does not hang: the kernel records FLEX_ERR_DEVICE_TIMEOUT in the
 *    device status word and returns; read it with flex_device_status().
 *  - The library allocates one small per-device workspace (the status word)
 *    with cudaMalloc the first time a device is used; call any entry point
 *    once before capturing a stream into a CUDA graph.
 *  - Indices and counts are int32.  Lengths are any positive int32 (KV_LEN
 *    up to 131072): the last tile along a length may reach past it, and the
 *    positions past a length count as masked.
 *  - Block sizes (Q_BLOCK, KV_BLOCK) are powers of two from 16 to 1024 and
 *    may differ.  The kernels compute on 128 x 128 tiles and read a
 *    BlockMask of any of these sizes as such tiles: a 128-tile is computed
 *    when some block overlapping it is listed, and skips mask_mod when every
 *    block overlapping it is full.
 */
#ifndef FLEXATTN_H
#define FLEXATTN_H

#include <stdint.h>

#if defined(__GNUC__)
#define FLEX_API __attribute__((visibility("default")))
#else
#define FLEX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FLEX_OK = 0,
    FLEX_ERR_INVALID_ARG = -1,     /* null pointer, bad enum, bad scale/parameter            */
    FLEX_ERR_UNSUPPORTED = -2,     /* head dim, dtype or size outside what the kernels cover  */
    FLEX_ERR_SHAPE = -3,           /* shapes or BlockMask sizes disagree                      */
    FLEX_ERR_ALIGNMENT = -4,       /* pointer or stride not 16-byte aligned / inner stride!=1 */
    FLEX_ERR_CUDA = -5,            /* a CUDA runtime/driver call failed                       */
    FLEX_ERR_DEVICE_TIMEOUT = -6   /* a kernel gave up on a wait (reported by status word)    */
} flex_status;

/* The enumerated mask_mods (b = batch, h = head, q = query row, kv = key row). */
typedef enum {
    FLEX_MASK_CAUSAL = 0,          /* q >= kv                                               */
    FLEX_MASK_SLIDING_WINDOW = 1,  /* q >= kv and q - kv < window                           */
    FLEX_MASK_CAUSAL_PREFIX = 2,   /* (q <= prefix and kv <= prefix) or q >= kv (inclusive) */
    FLEX_MASK_DOCUMENT = 3,        /* doc_ids[b][q] == doc_ids[b][kv] and q >= kv           */
    FLEX_MASK_ALL = 4              /* every pair (dense attention; for checks and timing)   */
} flex_mask_kind;

/* The enumerated score_mods, applied to the scaled score s = scale * q.k. */
typedef enum {
    FLEX_SCORE_IDENTITY = 0,       /* s                                                     */
    FLEX_SCORE_SOFTCAP = 1,        /* cap * tanh(s / cap), cap = score_param > 0            */
    FLEX_SCORE_ALIBI = 2           /* s - slope_h * (q - kv), slope_h = 2^(-8 (h+1) / H)    */
} flex_score_kind;

typedef enum {
    FLEX_DTYPE_BF16 = 0,           /* bfloat16 storage; tensor-core path, fp32 accumulation */
    FLEX_DTYPE_FP32 = 1            /* float32 storage; float32-accurate tensor-core forward */
} flex_dtype;

/* Parameters of a mask_mod.  Unused fields are ignored for kinds that do not need them. */
typedef struct {
    int32_t window;                /* FLEX_MASK_SLIDING_WINDOW: W >= 0 (W = 0 masks everything) */
    int32_t prefix;                /* FLEX_MASK_CAUSAL_PREFIX: P, inclusive bound                */
    const int32_t *doc_ids;        /* FLEX_MASK_DOCUMENT: device, [B, Q_LEN] int32, contiguous   */
} flex_mask_params;

/*
 * A BlockMask at Q_BLOCK x KV_BLOCK granularity (the BlockMask tuple of the
 * flex_attention op, kv side).  For every (b, h, q-block qb) and kv block:
 *   full     the mask_mod is true on the whole tile  -> listed in full_kv_*
 *   partial  true on some of the tile                -> listed in kv_*
 *   empty    true nowhere                            -> listed in neither
 * NQB = ceil(Q_LEN / Q_BLOCK), NKVB = ceil(KV_LEN / KV_BLOCK).  Positions
 * past Q_LEN or KV_LEN count as masked (the mask padded with false to whole
 * tiles), so a tile reaching past either length is never full; the
 * attention kernels rely on that to bound the tail tiles.
 * kv_num_blocks[b,h,qb] counts the partial tiles; kv_indices[b,h,qb,:] holds
 * their kv-block indices in ascending order followed by all other kv-block
 * indices in ascending order, so each row is a permutation of 0..NKVB-1.
 * full_kv_num_blocks / full_kv_indices follow the same layout for full tiles.
 * The mask kind and parameters are kept because the attention kernel
 * evaluates the mask_mod on partial tiles only.
 */
typedef struct {
    int32_t B, H, q_len, kv_len;
    int32_t q_block, kv_block;     /* tile rows and columns (Q_BLOCK, KV_BLOCK)   */
    int32_t nqb, nkvb;             /* ceil(q_len / q_block), ceil(kv_len / kv_block) */
    int32_t mask_kind;             /* flex_mask_kind the mask was built from      */
    flex_mask_params params;       /* its parameters (doc_ids stays caller-owned) */
    int32_t *kv_num_blocks;        /* device, [B, H, NQB]        int32            */
    int32_t *kv_indices;           /* device, [B, H, NQB, NKVB]  int32            */
    int32_t *full_kv_num_blocks;   /* device, [B, H, NQB]        int32            */
    int32_t *full_kv_indices;      /* device, [B, H, NQB, NKVB]  int32            */
} flex_block_mask;

/* A strided 4-D tensor [B, H, S, D] (strides in elements; stride[3] must be 1). */
typedef struct {
    const void *data;              /* device */
    int32_t dtype;                 /* flex_dtype */
    int32_t reserved;
    int64_t shape[4];
    int64_t stride[4];
} flex_tensor;

/*
 * Element counts of the BlockMask buffers for the given sizes, with
 * Q_BLOCK = KV_BLOCK = block:
 * *num_elems = B*H*NQB (each of kv_num_blocks, full_kv_num_blocks),
 * *idx_elems = B*H*NQB*NKVB (each of kv_indices, full_kv_indices).
 * Errors: FLEX_ERR_INVALID_ARG (null outputs, non-positive sizes),
 * FLEX_ERR_UNSUPPORTED (block not a power of two in 16..1024, KV_LEN >
 * 131072, B or H > 65535).
 */
FLEX_API int flex_block_mask_sizes(int32_t B, int32_t H, int32_t q_len, int32_t kv_len, int32_t block,
                          int64_t *num_elems, int64_t *idx_elems);

/* flex_block_mask_sizes with separate Q_BLOCK and KV_BLOCK (same errors). */
FLEX_API int flex_block_mask_sizes_qkv(int32_t B, int32_t H, int32_t q_len, int32_t kv_len, int32_t q_block,
                                       int32_t kv_block, int64_t *num_elems, int64_t *idx_elems);

/*
 * Build the BlockMask of an enumerated mask_mod on the device (the block
 * mask that create_block_mask produces for the flex_attention op, see the
 * BlockMask tuple in PyTorch PR #167356; predicate of the causal + prefix
 * kind from PyTorch issue #124369).
 *   in : bm->kv_num_blocks, kv_indices, full_kv_num_blocks, full_kv_indices
 *        point to caller-allocated device buffers sized by flex_block_mask_sizes.
 *   out: every other field of *bm is filled (sizes, mask kind, parameters), and
 *        the four buffers are written by a kernel enqueued on `stream`.
 * params may be NULL for kinds without parameters.  doc_ids must stay valid
 * while the BlockMask is used by flex_attention_fwd.  Tiles are block x block
 * (Q_BLOCK = KV_BLOCK = block).
 * Errors: FLEX_ERR_INVALID_ARG, FLEX_ERR_SHAPE, FLEX_ERR_UNSUPPORTED (as
 * flex_block_mask_sizes), FLEX_ERR_CUDA.
 */
FLEX_API int flex_block_mask_create(int32_t mask_kind, const flex_mask_params *params, int32_t B, int32_t H,
                           int32_t q_len, int32_t kv_len, int32_t block, flex_block_mask *bm,
                           void *stream);

/*
 * flex_block_mask_create with tiles of q_block rows by kv_block columns (the
 * BlockMask tuple's Q_BLOCK and KV_BLOCK fields); buffers sized by
 * flex_block_mask_sizes_qkv.  Same arguments otherwise, same errors.
 */
FLEX_API int flex_block_mask_create_qkv(int32_t mask_kind, const flex_mask_params *params, int32_t B, int32_t H,
                                        int32_t q_len, int32_t kv_len, int32_t q_block, int32_t kv_block,
                                        flex_block_mask *bm, void *stream);

/*
 * Block-sparse attention forward (the flex_attention op of PyTorch PR
 * #167356 with OUTPUT_LOGSUMEXP): for every (b, h, q)
 *   s[kv]   = score_mod(scale * q.k[kv])   on every tile listed in bm
 *   s[kv]   = -inf where mask_mod is false (evaluated on partial tiles only;
 *             tiles in neither list are skipped entirely)
 *   out[q]  = sum_kv exp(s[kv] - lse[q]) v[kv],  lse[q] = ln sum_kv exp(s[kv])
 * and a row with no unmasked score gets out = 0, lse = -inf.
 *   q    : [B, H, q_len, D];  k, v : [B, H, kv_len, D]; same dtype, B, H, D.
 *          D in {64, 128}.  bf16 needs 16-byte-aligned base and strides.
 *          Document masks need Q_LEN (== KV_LEN) a multiple of 4 (each
 *          tile's ids are copied in whole 16-byte words).
 *   bm   : a BlockMask for (B, H, q_len, kv_len) from flex_block_mask_create.
 *   score_kind, score_param : flex_score_kind and the softcap value.
 *   scale: multiplies q.k before score_mod (finite).
 *   out  : device, contiguous [B, H, q_len, D] in q's dtype, 16-byte aligned.
 *   lse  : device, contiguous [B, H, q_len] float32, natural logarithm.
 * Errors: FLEX_ERR_INVALID_ARG, FLEX_ERR_SHAPE, FLEX_ERR_ALIGNMENT,
 * FLEX_ERR_UNSUPPORTED, FLEX_ERR_CUDA.  Asynchronous on `stream`.
 */
FLEX_API int flex_attention_fwd(const flex_tensor *q, const flex_tensor *k, const flex_tensor *v,
                       const flex_block_mask *bm, int32_t score_kind, float score_param,
                       float scale, void *out, float *lse, void *stream);

/*
 * flex_attention_fwd for callers that cannot allocate device memory.  (No
 * counterpart in the pages: it exists for how the library is called, not for
 * what it computes.)
 *
 * flex_attention_fwd keeps the status word its kernels write on a timed-out
 * wait in a small workspace that it cudaMalloc's the first time a device is
 * used.  Some callers cannot allow that: code that enqueues work while a
 * stream is being captured, plug-ins whose host framework owns every device
 * allocation, processes that must not grow device memory after start-up.
 * This entry point computes exactly what flex_attention_fwd computes, with the
 * same arguments, checks and errors, and allocates nothing: the status word
 * lives in a static 256-byte device array inside the library, which every GPU
 * that loads the library holds until the process exits.  The status word is
 * 4 bytes whatever the problem size; a request for more scratch than the
 * array holds is refused with FLEX_ERR_UNSUPPORTED.
 *   - The first call on a device looks up that array's device address (once
 *     per device, with the device current); make that first call before any
 *     stream capture.
 *   - Each call clears the status word on `stream` (cudaMemsetAsync) before
 *     launching.  All calls share the one array and it keeps the last call's
 *     contents, so calls whose work overlaps on the GPU (other streams, other
 *     threads) race on it.
 *   - device_status (may be NULL): set to the device address of the status
 *     word.  After `stream` has finished, 0 means every wait completed and a
 *     nonzero value means a kernel gave up on a wait (outputs unspecified).
 *     Read it with a device-to-host copy; flex_device_status() does not see it.
 * Errors: as flex_attention_fwd.
 */
FLEX_API int flex_attention_fwd_noalloc(const flex_tensor *q, const flex_tensor *k, const flex_tensor *v,
                                        const flex_block_mask *bm, int32_t score_kind, float score_param,
                                        float scale, void *out, float *lse, void *stream,
                                        const int **device_status);

/*
 * Device buffers that flex_attention_fwd_host works in.  The caller allocates
 * and owns them (16-byte aligned, contiguous) and must not touch them until
 * `stream` has passed the call:
 *   q, k, v     [B, H, S, D] in the inputs' dtype (S = q_len for q, kv_len for k, v)
 *   out         [B, H, q_len, D] in the inputs' dtype;  lse [B, H, q_len] float32
 *   doc_ids     [B, q_len] int32 (document masks; may be NULL otherwise)
 *   kv_num_blocks ... full_kv_indices: the BlockMask index buffers, sized as
 *               flex_block_mask_sizes gives.
 */
typedef struct {
    void *q, *k, *v, *out;
    float *lse;
    int32_t *doc_ids;
    int32_t *kv_num_blocks, *kv_indices, *full_kv_num_blocks, *full_kv_indices;
} flex_device_buffers;

/*
 * flex_block_mask_create followed by flex_attention_fwd for inputs and outputs
 * in host memory, with the copies overlapped with the work.  (No counterpart
 * in the pages: it exists for callers whose tensors live on the host.)
 *   q, k, v   host tensors, contiguous [B, H, S, D], dtype and shapes as for
 *             flex_attention_fwd; page-locked (pinned) memory lets the copies
 *             run asynchronously and overlap.
 *   mask_kind, params  as for flex_block_mask_create, except that
 *             params->doc_ids (document masks) is a host array [B, q_len].
 *   score_kind, score_param, scale  as for flex_attention_fwd.
 *   out, lse  host, contiguous [B, H, q_len, D] (inputs' dtype) and
 *             [B, H, q_len] float32; written by the time `stream` has passed
 *             the call.
 *   dev       the device buffers described above.
 *   chunks    1..64: the (b, h) pairs are split into this many contiguous
 *             ranges.  The inputs of all ranges are copied in back to back on
 *             a library stream; the attention of a range starts on `stream`
 *             as soon as its inputs are in, and its out and lse are copied back
 *             on a second library stream while the next range computes.  The
 *             BlockMask of all heads is built once, on `stream`.
 * Both library streams are created once per device, wait for `stream` at the
 * start of the call, and `stream` waits for them at its end, so the call is
 * ordered on `stream` like any other.  Calls from several host threads on one
 * device enqueue one at a time.  Results are those of flex_attention_fwd.
 * Errors: FLEX_ERR_INVALID_ARG (a NULL or non-contiguous tensor, chunks out of
 * range, a missing parameter or buffer), and those of flex_block_mask_create
 * and flex_attention_fwd, all detected before anything is enqueued;
 * FLEX_ERR_CUDA if enqueueing fails.
 */
FLEX_API int flex_attention_fwd_host(const flex_tensor *q, const flex_tensor *k, const flex_tensor *v,
                                     int32_t mask_kind, const flex_mask_params *params, int32_t score_kind,
                                     float score_param, float scale, void *out, float *lse,
                                     const flex_device_buffers *dev, int32_t chunks, void *stream);

/*
 * Kernel options of the flex_attention op (its kernel_options dictionary in
 * PyTorch PR #167356, which names OUTPUT_MAX, PRESCALE_QK and
 * ROWS_GUARANTEED_SAFE and defaults each to False).  A zeroed struct is the
 * default and gives exactly what flex_attention_fwd gives.
 *   prescale_qk   0 or 1.  PRESCALE_QK: q is multiplied by scale before
 *                 Q K^T, the product rounded once to q's dtype (bfloat16 or
 *                 float32, to nearest, ties to even), and the scores are
 *                 score_mod(q~ . k[kv]) with no further scale.  The result
 *                 differs from the default by that rounding only (none when
 *                 scale is a power of two).
 *   rows_guaranteed_safe  0 or 1.  ROWS_GUARANTEED_SAFE: the caller promises
 *                 that every row keeps at least one unmasked score.  The
 *                 option exists so a kernel may drop its guard for rows with
 *                 none; these kernels carry no such guard in their inner
 *                 loops (a finite floor on the running max makes all-masked
 *                 tiles contribute exp(-inf) = 0), so the option changes
 *                 neither results nor speed, and rows that break the promise
 *                 still get out = 0, lse = -inf.
 *   max_scores    OUTPUT_MAX: NULL, or device, contiguous [B, H, q_len]
 *                 float32, 4-byte aligned: the row maximum of the masked,
 *                 modified scores s[kv] (natural units, like lse), -inf for a
 *                 row with no unmasked score.
 */
typedef struct {
    int32_t prescale_qk;
    int32_t rows_guaranteed_safe;
    float *max_scores;
} flex_kernel_options;

/*
 * flex_attention_fwd with kernel options; opts may be NULL (all default).
 * Arguments, results and errors as flex_attention_fwd, plus
 * FLEX_ERR_INVALID_ARG for an option flag other than 0 or 1 and
 * FLEX_ERR_ALIGNMENT for a misaligned max_scores.
 */
FLEX_API int flex_attention_fwd_opts(const flex_tensor *q, const flex_tensor *k, const flex_tensor *v,
                                     const flex_block_mask *bm, int32_t score_kind, float score_param,
                                     float scale, void *out, float *lse, const flex_kernel_options *opts,
                                     void *stream);

/*
 * The q side of a BlockMask (the q_num_blocks, q_indices, full_q_num_blocks,
 * full_q_indices fields of the flex_attention op's BlockMask tuple, which
 * its backward pass reads): for every (b, h, kv block j), the q blocks whose
 * tile with j is partial (full), ascending, followed by all other q blocks
 * ascending, so each row is a permutation of 0..NQB-1.
 */
typedef struct {
    int32_t B, H, q_len, kv_len, q_block, kv_block, nqb, nkvb;
    int32_t *q_num_blocks;         /* device, [B, H, NKVB]       int32 */
    int32_t *q_indices;            /* device, [B, H, NKVB, NQB]  int32 */
    int32_t *full_q_num_blocks;    /* device, [B, H, NKVB]       int32 */
    int32_t *full_q_indices;       /* device, [B, H, NKVB, NQB]  int32 */
} flex_block_mask_q;

/*
 * Fill the q side of a BlockMask from its kv side on the device.
 *   in : bm from flex_block_mask_create (its selected kv-block lists are
 *        ascending, as that call writes them); bq's four buffers,
 *        caller-allocated device memory of the sizes above.
 *   out: bq's size fields, and its buffers written by a kernel on `stream`.
 * Errors: FLEX_ERR_INVALID_ARG (null struct or buffer), FLEX_ERR_SHAPE,
 * FLEX_ERR_UNSUPPORTED (as flex_block_mask_sizes), FLEX_ERR_CUDA.
 */
FLEX_API int flex_block_mask_transpose(const flex_block_mask *bm, flex_block_mask_q *bq, void *stream);

/*
 * Backward pass of flex_attention_fwd (the flex_attention_backward op of
 * PyTorch PR #167356's tests): the gradients of sum(dout * out) with respect
 * to q, k and v, for every (b, h), with t = scale q.k, s = score_mod(t) on the
 * BlockMask's tiles (mask_mod on partial tiles), P = exp(s - lse):
 *   dv[j] = sum_i P[i,j] dout[i]
 *   dS[i,j] = P[i,j] (dout[i].v[j] - dout[i].out[i]) score_mod'(t[i,j])
 *   dq[i] = scale sum_j dS[i,j] k[j],   dk[j] = scale sum_i dS[i,j] q[i]
 * (score_mod' is 1 for identity and ALiBi, 1 - tanh^2(t / cap) for softcap).
 *   q, k, v, bm, score_kind, score_param, scale: as given to the forward.
 *   out, lse: device, the forward's outputs (contiguous, q's dtype; float32).
 *   dout: device, contiguous [B, H, q_len, D] in q's dtype, 16-byte aligned.
 *   bq:   the q side of bm, from flex_block_mask_transpose.
 *   dq:   device, contiguous [B, H, q_len, D]; dk, dv: [B, H, kv_len, D];
 *         q's dtype, 16-byte aligned.
 *   delta: device workspace, [B, H, q_len] float32 (dout[i].out[i]).
 * Rows whose lse is -inf (no unmasked score) contribute nothing.  bf16
 * inputs run on the tensor cores (S, dP and the gradient products as tcgen05
 * MMAs with fp32 accumulation; P and dS rounded to bf16 as MMA operands) and
 * need Q_LEN <= 262144 (2048 tiles of 128 rows); fp32 inputs keep float32
 * accuracy on the tensor cores (each operand split into three bf16 parts,
 * six MMAs per product), except dk and dv of q sides longer than 2048
 * tiles, computed in fp32 on the CUDA cores.  Errors: those of
 * flex_attention_fwd, FLEX_ERR_SHAPE when
 * bq does not match bm, and FLEX_ERR_UNSUPPORTED for bf16 with Q_LEN >
 * 262144.  Asynchronous on `stream`: dq is computed on a library stream
 * (created by the first call on a device that is not made during a stream
 * capture) that forks from `stream` after the work already queued there and
 * joins it again, so that its kernel fills the SMs the dk/dv kernel leaves
 * idle; without that stream dq follows dk and dv on `stream`.  Either way
 * the call stays ordered on `stream` like any other, also under stream
 * capture.  Calls from several host threads on one device enqueue one at a
 * time.
 */
FLEX_API int flex_attention_bwd(const flex_tensor *q, const flex_tensor *k, const flex_tensor *v, const void *out,
                                const float *lse, const void *dout, const flex_block_mask *bm,
                                const flex_block_mask_q *bq, int32_t score_kind, float score_param, float scale,
                                void *dq, void *dk, void *dv, float *delta, void *stream);

/*
 * Synchronises `stream`, then returns and clears the device status word of
 * the current device: FLEX_OK, or FLEX_ERR_DEVICE_TIMEOUT if a kernel gave up
 * on a wait since the last call.  FLEX_ERR_CUDA if the synchronisation failed.
 */
FLEX_API int flex_device_status(void *stream);

/*
 * Diagnostic of the failure path: enqueues on `stream` a one-warp kernel that
 * waits on an mbarrier no thread arrives at, using the same bounded wait as the
 * attention kernel but with a limit of `limit_ms` milliseconds (1..60000).
 * The wait gives up, the kernel records FLEX_ERR_DEVICE_TIMEOUT in the device
 * status word and returns; flex_device_status() then reports it and clears
 * it.  The GPU context stays usable.  Errors: FLEX_ERR_INVALID_ARG,
 * FLEX_ERR_CUDA.
 */
FLEX_API int flex_selftest_wait_timeout(uint32_t limit_ms, void *stream);

/* A static, human-readable name for a flex_status value. */
FLEX_API const char *flex_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FLEXATTN_H */
