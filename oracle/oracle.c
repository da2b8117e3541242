/*
 * Plain float64 CPU oracle for the block-sparse FlexAttention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header or constant table with the
 * CUDA library; the mask and score kinds are numbered like the C-ABI enums so
 * that the same integers can be passed to both.
 *
 * What it computes, written out as the plain definition (no tiling, no
 * online softmax, no reordering):
 *
 *   mask_mod (b,h,q,kv)  -> bool        "Performance for templated attention
 *       strangely bad for a combination of causal + upper square mask"
 *       (PyTorch issue #124369), the mask written with torch.where: a masked
 *       score becomes -inf; the causal + upper-square predicate is
 *       (q <= P and kv <= P) or (q >= kv) with inclusive bounds.
 *   score_mod(t,b,h,q,kv) -> t'         "[Inductor][Flex Attention] Add
 *       Subtiling Option for Alpha Scaling" (PyTorch PR #167356), the
 *       flex_attention higher-order op: scale is its own argument and the
 *       score_mod graph acts on the scaled score QK^T*scale.
 *   attention            -> out, lse    softmax over kv of the masked,
 *       modified scores, times V, plus the per-row log-sum-exp
 *       (OUTPUT_LOGSUMEXP in the same op's options); a row with no
 *       unmasked score gives out = 0 and lse = -inf (the guard that the
 *       ROWS_GUARANTEED_SAFE option lets a caller skip).
 *   kernel options       the same op's kernel_options, read plainly:
 *       OUTPUT_MAX   a third output, the row maximum of the masked,
 *                    modified scores (natural units like lse; -inf for a
 *                    row with no unmasked score);
 *       PRESCALE_QK  Q is multiplied by scale before QK^T: the product
 *                    scale * q is rounded once to the inputs' storage type
 *                    (bfloat16 or float32, ties to even) and the scores are
 *                    score_mod(q~ . k) with no further scale.
 *   backward             -> dq, dk, dv      the gradients of sum(dO * out)
 *       (the flex_attention_backward op of the same PR's tests, which takes
 *       the forward's out, lse and the output gradient and returns the
 *       three gradients), written out as the softmax-attention chain rule;
 *       the q side of the BlockMask (q_num_blocks, q_indices, ...), which
 *       the same tuple carries for that pass, as the transpose of the kv
 *       side.
 *   block mask           -> kv_num_blocks, kv_indices, full_kv_num_blocks,
 *       full_kv_indices   (the BlockMask tuple passed to the same op, which
 *       carries a Q block size and a KV block size): each Q_BLOCK x KV_BLOCK
 *       tile of the dense mask is full (all true), partial (some true) or
 *       empty; each row of an index tensor lists the selected kv blocks in
 *       ascending order followed by the unselected ones, also ascending (a
 *       stable descending sort of the 0/1 tile row).
 *
 * Inputs are float32 arrays holding the exact values the device reads
 * (bf16 values are exact in float32); every product and sum is taken in
 * double.
 *
 * Parity pins: see the tests (textbook attention through a library routine,
 * closed-form block counts, ALiBi and softcap closed forms, brute force on
 * tiny shapes).  No function here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_MASK_CAUSAL 0
#define OR_MASK_SLIDING_WINDOW 1
#define OR_MASK_CAUSAL_PREFIX 2
#define OR_MASK_DOCUMENT 3
#define OR_MASK_ALL 4

#define OR_SCORE_IDENTITY 0
#define OR_SCORE_SOFTCAP 1
#define OR_SCORE_ALIBI 2

#define OR_OK 0
#define OR_ERR_ARG -1
#define OR_ERR_NOMEM -2

typedef struct {
    int kind;
    int window;            /* sliding window W: keep 0 <= q - kv < W      */
    int prefix;            /* prefix P: (q <= P and kv <= P) or q >= kv    */
    const int32_t *doc;    /* [B, len] document id of every position      */
    int64_t doc_len;
} or_mask;

/* mask_mod(b, h, q, kv): the enumerated predicates. */
static int or_mask_mod(const or_mask *m, int64_t b, int64_t h, int64_t q, int64_t kv)
{
    (void)h;
    switch (m->kind) {
    case OR_MASK_CAUSAL:
        return q >= kv;
    case OR_MASK_SLIDING_WINDOW:
        return q >= kv && (q - kv) < (int64_t)m->window;
    case OR_MASK_CAUSAL_PREFIX:
        return (q <= (int64_t)m->prefix && kv <= (int64_t)m->prefix) || q >= kv;
    case OR_MASK_DOCUMENT:
        return m->doc[b * m->doc_len + q] == m->doc[b * m->doc_len + kv] && q >= kv;
    case OR_MASK_ALL:
        return 1;
    default:
        return 0;
    }
}

/* score_mod(t, b, h, q, kv) applied to the scaled score t = scale * q.k */
static double or_score_mod(int kind, double param, double t, int64_t h, int64_t H,
                           int64_t q, int64_t kv)
{
    switch (kind) {
    case OR_SCORE_SOFTCAP:
        return param * tanh(t / param);
    case OR_SCORE_ALIBI: {
        /* slope_h = 2^(-8 (h+1) / H), h counted from 0 */
        double slope = pow(2.0, -8.0 * (double)(h + 1) / (double)H);
        return t - slope * (double)(q - kv);
    }
    default:
        return t;
    }
}

static int or_mask_ok(int kind)
{
    return kind >= OR_MASK_CAUSAL && kind <= OR_MASK_ALL;
}

#define OR_PRESCALE_NONE 0
#define OR_PRESCALE_BF16 1
#define OR_PRESCALE_F32 2

/*
 * x rounded to bfloat16 (8 significant bits, float32's exponent range,
 * subnormal quantum 2^-133), ties to even, overflow to +-inf.  One rounding
 * from the exact double value.
 */
static double or_round_bf16(double x)
{
    if (x == 0.0 || !isfinite(x)) return x;
    int e;
    (void)frexp(x, &e);              /* 2^(e-1) <= |x| < 2^e */
    int quantum = e - 8;
    if (quantum < -133) quantum = -133;
    const double r = ldexp(nearbyint(ldexp(x, -quantum)), quantum);  /* default mode: ties to even */
    const double bf16_max = ldexp(255.0, 120);                       /* (2 - 2^-7) 2^127 */
    return fabs(r) > bf16_max ? copysign(INFINITY, x) : r;
}

/* q~ = scale * q rounded to the storage type (PRESCALE_QK) */
static double or_prescale(int prescale, double scale, float q)
{
    const double x = scale * (double)q;  /* exact: 24 x 24 bits fit a double */
    if (prescale == OR_PRESCALE_BF16) return or_round_bf16(x);
    return (double)(float)x;
}

/*
 * Dense mask evaluated tile by tile; one Q_BLOCK-row band of the mask is
 * materialised at a time to bound memory.  Lengths need not be multiples of
 * the block sizes: the dense mask is padded with false to whole tiles
 * (NQB = ceil(Q_LEN / Q_BLOCK), NKVB = ceil(KV_LEN / KV_BLOCK)), so a tile
 * that reaches past either length is never full.  Output layouts:
 *   kv_num, full_num : [B, H, NQB]
 *   kv_idx, full_idx : [B, H, NQB, NKVB]
 */
int oracle_block_mask(int kind, int window, int prefix, const int32_t *doc,
                      int B, int H, int q_len, int kv_len, int q_block, int kv_block,
                      int32_t *kv_num, int32_t *kv_idx,
                      int32_t *full_num, int32_t *full_idx)
{
    if (!or_mask_ok(kind) || B <= 0 || H <= 0 || q_len <= 0 || kv_len <= 0 || q_block <= 0 || kv_block <= 0)
        return OR_ERR_ARG;
    if (kind == OR_MASK_DOCUMENT && (doc == NULL || q_len != kv_len))
        return OR_ERR_ARG;
    const int64_t nqb = ((int64_t)q_len + q_block - 1) / q_block;
    const int64_t nkvb = ((int64_t)kv_len + kv_block - 1) / kv_block;
    or_mask m = {kind, window, prefix, doc, (int64_t)q_len};
    int err = OR_OK;

#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
        for (int64_t qb = 0; qb < nqb; ++qb) {
            int64_t b = bh / H, h = bh % H;
            /* the dense mask of rows [qb*q_block, (qb+1)*q_block) */
            unsigned char *band = (unsigned char *)malloc((size_t)q_block * (size_t)kv_len);
            int64_t *count = (int64_t *)calloc((size_t)nkvb, sizeof(int64_t));
            if (!band || !count) {
                free(band);
                free(count);
#pragma omp atomic write
                err = OR_ERR_NOMEM;
                continue;
            }
            for (int64_t r = 0; r < q_block; ++r)
                for (int64_t kv = 0; kv < kv_len; ++kv)  /* columns past KV_LEN: padding, false */
                    band[r * kv_len + kv] = qb * q_block + r < q_len  /* rows past Q_LEN: padding, false */
                                                ? (unsigned char)or_mask_mod(&m, b, h, qb * q_block + r, kv)
                                                : 0;
            for (int64_t r = 0; r < q_block; ++r)
                for (int64_t kv = 0; kv < kv_len; ++kv)
                    count[kv / kv_block] += band[r * kv_len + kv];

            const int64_t all = (int64_t)q_block * kv_block;
            const int64_t row = bh * nqb + qb;
            int32_t *pi = kv_idx + row * nkvb, *fi = full_idx + row * nkvb;
            int32_t np = 0, nf = 0;
            /* selected blocks first, ascending */
            for (int64_t j = 0; j < nkvb; ++j) {
                if (count[j] > 0 && count[j] < all) pi[np++] = (int32_t)j;
                if (count[j] == all) fi[nf++] = (int32_t)j;
            }
            kv_num[row] = np;
            full_num[row] = nf;
            /* then the unselected ones, ascending */
            int32_t tp = np, tf = nf;
            for (int64_t j = 0; j < nkvb; ++j) {
                if (!(count[j] > 0 && count[j] < all)) pi[tp++] = (int32_t)j;
                if (count[j] != all) fi[tf++] = (int32_t)j;
            }
            free(band);
            free(count);
        }
    }
    return err;
}

/*
 * The q side of the BlockMask tuple (q_num_blocks, q_indices,
 * full_q_num_blocks, full_q_indices), read by the backward pass: for every
 * kv block j, the q blocks whose kv-side partial (full) list holds j, in
 * ascending order, followed by the other q blocks ascending.  Output layouts:
 *   q_num, full_q_num : [B, H, NKVB]
 *   q_idx, full_q_idx : [B, H, NKVB, NQB]
 */
int oracle_block_mask_q(int kind, int window, int prefix, const int32_t *doc,
                        int B, int H, int q_len, int kv_len, int q_block, int kv_block,
                        int32_t *q_num, int32_t *q_idx, int32_t *full_q_num, int32_t *full_q_idx)
{
    if (q_block <= 0 || kv_block <= 0 || q_len <= 0 || kv_len <= 0 || B <= 0 || H <= 0)
        return OR_ERR_ARG;
    const int64_t nqb = ((int64_t)q_len + q_block - 1) / q_block;
    const int64_t nkvb = ((int64_t)kv_len + kv_block - 1) / kv_block;
    const int64_t rows = (int64_t)B * H * nqb;
    int32_t *kn = (int32_t *)malloc((size_t)rows * sizeof(int32_t));
    int32_t *ki = (int32_t *)malloc((size_t)(rows * nkvb) * sizeof(int32_t));
    int32_t *fn = (int32_t *)malloc((size_t)rows * sizeof(int32_t));
    int32_t *fi = (int32_t *)malloc((size_t)(rows * nkvb) * sizeof(int32_t));
    unsigned char *st = (unsigned char *)calloc((size_t)(nqb * nkvb), 1);
    int err = (kn && ki && fn && fi && st) ? OR_OK : OR_ERR_NOMEM;
    if (err == OR_OK)
        err = oracle_block_mask(kind, window, prefix, doc, B, H, q_len, kv_len, q_block, kv_block, kn, ki, fn, fi);
    for (int64_t bh = 0; err == OR_OK && bh < (int64_t)B * H; ++bh) {
        /* tile classes of this (b, h) from its kv-side lists: 1 partial, 2 full */
        memset(st, 0, (size_t)(nqb * nkvb));
        for (int64_t i = 0; i < nqb; ++i) {
            const int64_t row = bh * nqb + i;
            for (int32_t t = 0; t < kn[row]; ++t) st[i * nkvb + ki[row * nkvb + t]] = 1;
            for (int32_t t = 0; t < fn[row]; ++t) st[i * nkvb + fi[row * nkvb + t]] = 2;
        }
        for (int64_t j = 0; j < nkvb; ++j) {
            const int64_t col = bh * nkvb + j;
            int32_t *pq = q_idx + col * nqb, *fq = full_q_idx + col * nqb;
            int32_t np = 0, nf = 0;
            for (int64_t i = 0; i < nqb; ++i) {
                if (st[i * nkvb + j] == 1) pq[np++] = (int32_t)i;
                if (st[i * nkvb + j] == 2) fq[nf++] = (int32_t)i;
            }
            q_num[col] = np;
            full_q_num[col] = nf;
            int32_t tp = np, tf = nf;
            for (int64_t i = 0; i < nqb; ++i) {
                if (st[i * nkvb + j] != 1) pq[tp++] = (int32_t)i;
                if (st[i * nkvb + j] != 2) fq[tf++] = (int32_t)i;
            }
        }
    }
    free(kn);
    free(ki);
    free(fn);
    free(fi);
    free(st);
    return err;
}

/*
 * One output row (b, h, i):
 *   S[j] = mask_mod(b,h,i,j) ? score_mod(scale * sum_d q[i,d] k[j,d]) : -inf
 *          (PRESCALE_QK: score_mod(sum_d q~[i,d] k[j,d]), q~ = round(scale q))
 *   no unmasked j          -> out = 0, lse = -inf, row max = -inf
 *   else  mx = max_j S[j], Z = sum_j exp(S[j] - mx), lse = mx + ln Z,
 *         out[d] = sum_j exp(S[j] - lse) v[j,d], row max = mx
 */
static void or_row(const float *q, const float *k, const float *v,
                   int64_t H, int64_t s_kv, int64_t D, const or_mask *m,
                   int score_kind, double score_param, double scale, int prescale,
                   int64_t b, int64_t h, int64_t i,
                   double *srow, unsigned char *mrow, double *qrow,
                   double *out, double *lse, double *row_max)
{
    const float *qi = q + i * D;
    for (int64_t d = 0; d < D; ++d)
        qrow[d] = prescale ? or_prescale(prescale, scale, qi[d]) : (double)qi[d];
    const double post = prescale ? 1.0 : scale;  /* the scale still to apply to q.k */
    int any = 0;
    for (int64_t j = 0; j < s_kv; ++j) {
        mrow[j] = (unsigned char)or_mask_mod(m, b, h, i, j);
        any |= mrow[j];
        double dot = 0.0;
        const float *kj = k + j * D;
        for (int64_t d = 0; d < D; ++d)
            dot += qrow[d] * (double)kj[d];
        double t = or_score_mod(score_kind, score_param, post * dot, h, H, i, j);
        srow[j] = mrow[j] ? t : -INFINITY;
    }
    if (!any) {
        for (int64_t d = 0; d < D; ++d)
            out[d] = 0.0;
        *lse = -INFINITY;
        if (row_max) *row_max = -INFINITY;
        return;
    }
    double mx = -INFINITY;
    for (int64_t j = 0; j < s_kv; ++j)
        if (mrow[j] && srow[j] > mx) mx = srow[j];
    if (row_max) *row_max = mx;
    double Z = 0.0;
    for (int64_t j = 0; j < s_kv; ++j)
        if (mrow[j]) Z += exp(srow[j] - mx);
    const double L = mx + log(Z);
    for (int64_t d = 0; d < D; ++d)
        out[d] = 0.0;
    for (int64_t j = 0; j < s_kv; ++j) {
        if (!mrow[j]) continue;
        const double p = exp(srow[j] - L);
        const float *vj = v + j * D;
        for (int64_t d = 0; d < D; ++d)
            out[d] += p * (double)vj[d];
    }
    *lse = L;
}

/*
 * q: [B, H, s_q, D], k, v: [B, H, s_kv, D], contiguous float32.
 * rows == NULL: every row; out [B, H, s_q, D], lse and row_max [B, H, s_q].
 * rows != NULL: nrows flat row ids ((b*H + h)*s_q + i); out [nrows, D],
 * lse and row_max [nrows].  row_max may be NULL (OUTPUT_MAX off).
 * prescale: OR_PRESCALE_NONE, or the storage type q~ is rounded to.
 */
int oracle_attention_opts(const float *q, const float *k, const float *v,
                          int B, int H, int s_q, int s_kv, int D,
                          int mask_kind, int window, int prefix, const int32_t *doc,
                          int score_kind, double score_param, double scale, int prescale,
                          const int64_t *rows, int64_t nrows,
                          double *out, double *lse, double *row_max)
{
    if (!or_mask_ok(mask_kind) || B <= 0 || H <= 0 || s_q <= 0 || s_kv <= 0 || D <= 0)
        return OR_ERR_ARG;
    if (score_kind < OR_SCORE_IDENTITY || score_kind > OR_SCORE_ALIBI)
        return OR_ERR_ARG;
    if (prescale < OR_PRESCALE_NONE || prescale > OR_PRESCALE_F32)
        return OR_ERR_ARG;
    if (mask_kind == OR_MASK_DOCUMENT && (doc == NULL || s_q != s_kv))
        return OR_ERR_ARG;
    if (score_kind == OR_SCORE_SOFTCAP && !(score_param > 0.0))
        return OR_ERR_ARG;
    or_mask m = {mask_kind, window, prefix, doc, (int64_t)s_q};
    const int64_t total = rows ? nrows : (int64_t)B * H * s_q;
    int err = OR_OK;

#pragma omp parallel
    {
        double *srow = (double *)malloc((size_t)s_kv * sizeof(double));
        double *qrow = (double *)malloc((size_t)D * sizeof(double));
        unsigned char *mrow = (unsigned char *)malloc((size_t)s_kv);
        if (!srow || !mrow || !qrow) {
#pragma omp atomic write
            err = OR_ERR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < total; ++r) {
                const int64_t flat = rows ? rows[r] : r;
                const int64_t i = flat % s_q, bh = flat / s_q;
                const int64_t b = bh / H, h = bh % H;
                if (b >= B) continue;
                or_row(q + bh * (int64_t)s_q * D, k + bh * (int64_t)s_kv * D,
                       v + bh * (int64_t)s_kv * D, H, s_kv, D, &m, score_kind,
                       score_param, scale, prescale, b, h, i, srow, mrow, qrow,
                       out + r * D, lse + r, row_max ? row_max + r : NULL);
            }
        }
        free(srow);
        free(qrow);
        free(mrow);
    }
    return err;
}

/* d score_mod / dt at the scaled score t */
static double or_score_grad(int kind, double param, double t)
{
    if (kind == OR_SCORE_SOFTCAP) {
        const double u = tanh(t / param);
        return 1.0 - u * u;
    }
    return 1.0;  /* identity; ALiBi adds a term that does not depend on t */
}

/*
 * The backward terms of one row i of one (b, h): dq_i, and, when dk and dv
 * are given, row i's contributions to every dk_j and dv_j.  qb .. gb point at
 * the (b, h) slices; t, pr (s_kv doubles), o (D doubles) and mk (s_kv bytes)
 * are scratch.
 */
static void or_bwd_row(const float *qb, const float *kb, const float *vb, const float *gb,
                       int64_t H, int64_t s_kv, int64_t D, const or_mask *m,
                       int score_kind, double score_param, double scale,
                       int64_t b, int64_t h, int64_t i,
                       double *t, double *pr, double *o, unsigned char *mk,
                       double *dqi, double *dkb, double *dvb)
{
    for (int64_t d = 0; d < D; ++d)
        dqi[d] = 0.0;
    /* scores and the softmax of row i */
    int any = 0;
    double mx = -INFINITY;
    for (int64_t j = 0; j < s_kv; ++j) {
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dot += (double)qb[i * D + d] * (double)kb[j * D + d];
        t[j] = scale * dot;
        mk[j] = (unsigned char)or_mask_mod(m, b, h, i, j);
        if (mk[j]) {
            any = 1;
            const double sij = or_score_mod(score_kind, score_param, t[j], h, H, i, j);
            pr[j] = sij;
            if (sij > mx) mx = sij;
        }
    }
    if (!any) return;  /* P = 0: the row contributes nothing */
    double Z = 0.0;
    for (int64_t j = 0; j < s_kv; ++j)
        if (mk[j]) Z += exp(pr[j] - mx);
    const double lse = mx + log(Z);
    for (int64_t j = 0; j < s_kv; ++j)
        pr[j] = mk[j] ? exp(pr[j] - lse) : 0.0;
    /* out_i and D_i */
    for (int64_t d = 0; d < D; ++d)
        o[d] = 0.0;
    for (int64_t j = 0; j < s_kv; ++j)
        if (mk[j])
            for (int64_t d = 0; d < D; ++d)
                o[d] += pr[j] * (double)vb[j * D + d];
    double Di = 0.0;
    for (int64_t d = 0; d < D; ++d)
        Di += (double)gb[i * D + d] * o[d];
    for (int64_t j = 0; j < s_kv; ++j) {
        if (!mk[j]) continue;
        double dp = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dp += (double)gb[i * D + d] * (double)vb[j * D + d];
        const double ds = pr[j] * (dp - Di);
        const double dt = ds * or_score_grad(score_kind, score_param, t[j]);
        for (int64_t d = 0; d < D; ++d) {
            if (dvb) dvb[j * D + d] += pr[j] * (double)gb[i * D + d];
            dqi[d] += scale * dt * (double)kb[j * D + d];
            if (dkb) dkb[j * D + d] += scale * dt * (double)qb[i * D + d];
        }
    }
}

static int or_bwd_args_ok(int B, int H, int s_q, int s_kv, int D, int mask_kind, const int32_t *doc,
                          int score_kind, double score_param)
{
    if (!or_mask_ok(mask_kind) || B <= 0 || H <= 0 || s_q <= 0 || s_kv <= 0 || D <= 0)
        return 0;
    if (score_kind < OR_SCORE_IDENTITY || score_kind > OR_SCORE_ALIBI)
        return 0;
    if (mask_kind == OR_MASK_DOCUMENT && (doc == NULL || s_q != s_kv))
        return 0;
    if (score_kind == OR_SCORE_SOFTCAP && !(score_param > 0.0))
        return 0;
    return 1;
}

/*
 * Backward pass: the gradients of L = sum_{i,d} dO[i,d] out[i,d] with
 * respect to q, k and v, for out as oracle_attention defines it.  Per (b, h),
 * with t_ij = scale q_i.k_j, S_ij = score_mod(t_ij) where mask_mod holds
 * (else -inf), P_ij = exp(S_ij - lse_i) (0 on a row with no unmasked score):
 *   dV_j = sum_i P_ij dO_i
 *   dP_ij = dO_i . v_j,   D_i = dO_i . out_i = sum_j P_ij dP_ij
 *   dS_ij = P_ij (dP_ij - D_i)          (softmax rows)
 *   dT_ij = dS_ij score_mod'(t_ij)
 *   dQ_i = scale sum_j dT_ij k_j,   dK_j = scale sum_i dT_ij q_i
 * q, k, v, dout: float32 [B, H, S, D]; dq [B, H, s_q, D], dk, dv
 * [B, H, s_kv, D] in double.  One (b, h) per thread; memory O(s_kv + D).
 */
int oracle_attention_bwd(const float *q, const float *k, const float *v, const float *dout,
                         int B, int H, int s_q, int s_kv, int D,
                         int mask_kind, int window, int prefix, const int32_t *doc,
                         int score_kind, double score_param, double scale,
                         double *dq, double *dk, double *dv)
{
    if (!or_bwd_args_ok(B, H, s_q, s_kv, D, mask_kind, doc, score_kind, score_param))
        return OR_ERR_ARG;
    or_mask m = {mask_kind, window, prefix, doc, (int64_t)s_q};
    int err = OR_OK;
    memset(dk, 0, sizeof(double) * (size_t)B * H * s_kv * D);
    memset(dv, 0, sizeof(double) * (size_t)B * H * s_kv * D);

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
        const int64_t b = bh / H, h = bh % H;
        double *t = (double *)malloc((size_t)s_kv * sizeof(double));
        double *pr = (double *)malloc((size_t)s_kv * sizeof(double));
        double *o = (double *)malloc((size_t)D * sizeof(double));
        unsigned char *mk = (unsigned char *)malloc((size_t)s_kv);
        if (!t || !pr || !o || !mk) {
#pragma omp atomic write
            err = OR_ERR_NOMEM;
        } else {
            for (int64_t i = 0; i < s_q; ++i)
                or_bwd_row(q + bh * s_q * D, k + bh * s_kv * D, v + bh * s_kv * D, dout + bh * s_q * D,
                           H, s_kv, D, &m, score_kind, score_param, scale, b, h, i, t, pr, o, mk,
                           dq + (bh * s_q + i) * D, dk + bh * s_kv * D, dv + bh * s_kv * D);
        }
        free(t);
        free(pr);
        free(o);
        free(mk);
    }
    return err;
}

/*
 * dq of the flat rows ((b*H + h)*s_q + i) listed in rows: dq [nrows, D].  A
 * row's dq needs only that row's scores, so this stays cheap at lengths where
 * the whole backward would not.
 */
int oracle_attention_bwd_dq_rows(const float *q, const float *k, const float *v, const float *dout,
                                 int B, int H, int s_q, int s_kv, int D,
                                 int mask_kind, int window, int prefix, const int32_t *doc,
                                 int score_kind, double score_param, double scale,
                                 const int64_t *rows, int64_t nrows, double *dq)
{
    if (!or_bwd_args_ok(B, H, s_q, s_kv, D, mask_kind, doc, score_kind, score_param) || !rows)
        return OR_ERR_ARG;
    or_mask m = {mask_kind, window, prefix, doc, (int64_t)s_q};
    int err = OR_OK;
#pragma omp parallel
    {
        double *t = (double *)malloc((size_t)s_kv * sizeof(double));
        double *pr = (double *)malloc((size_t)s_kv * sizeof(double));
        double *o = (double *)malloc((size_t)D * sizeof(double));
        unsigned char *mk = (unsigned char *)malloc((size_t)s_kv);
        if (!t || !pr || !o || !mk) {
#pragma omp atomic write
            err = OR_ERR_NOMEM;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < nrows; ++r) {
                const int64_t i = rows[r] % s_q, bh = rows[r] / s_q;
                if (bh >= (int64_t)B * H) continue;
                or_bwd_row(q + bh * s_q * D, k + bh * s_kv * D, v + bh * s_kv * D, dout + bh * s_q * D,
                           H, s_kv, D, &m, score_kind, score_param, scale, bh / H, bh % H, i, t, pr, o, mk,
                           dq + r * D, NULL, NULL);
            }
        }
        free(t);
        free(pr);
        free(o);
        free(mk);
    }
    return err;
}

/* the default kernel options: no prescale, no row max */
int oracle_attention(const float *q, const float *k, const float *v,
                     int B, int H, int s_q, int s_kv, int D,
                     int mask_kind, int window, int prefix, const int32_t *doc,
                     int score_kind, double score_param, double scale,
                     const int64_t *rows, int64_t nrows,
                     double *out, double *lse)
{
    return oracle_attention_opts(q, k, v, B, H, s_q, s_kv, D, mask_kind, window, prefix, doc,
                                 score_kind, score_param, scale, OR_PRESCALE_NONE, rows, nrows,
                                 out, lse, NULL);
}

/* bfloat16 rounding, exposed so tests can check it against a library conversion */
double oracle_round_bf16(double x)
{
    return or_round_bf16(x);
}

/* the single predicate, exposed so tests can check it against the pages' examples */
int oracle_mask_value(int kind, int window, int prefix, const int32_t *doc, int64_t doc_len,
                      int64_t b, int64_t h, int64_t q, int64_t kv)
{
    or_mask m = {kind, window, prefix, doc, doc_len};
    return or_mask_ok(kind) ? or_mask_mod(&m, b, h, q, kv) : -1;
}

int oracle_num_threads(void)
{
    int n = 1;
#ifdef _OPENMP
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
#endif
    return n;
}
