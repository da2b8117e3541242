// Backward pass of the block-sparse attention (the flex_attention_backward op
// of "[Inductor][Flex Attention] Add Subtiling Option for Alpha Scaling",
// PyTorch PR #167356, test diffs: it takes q, k, v, the forward's out and lse,
// and the output gradient, and returns dq, dk, dv).  Both dtypes take delta
// from the kernel below; bf16 inputs take dq, dk, dv from the tensor-core
// kernels of attn_bwd_tc.cuh, fp32 inputs from those of attn_bwd_fp32_tc.cuh
// (three-way bf16 split), except dk and dv of q sides longer than
// kBwdF32TcMaxQTiles tiles, which take the register-tiled CUDA-core kernels
// below.  The dq kernel runs on a side stream beside the dk/dv kernel.
//
// With t = scale q.k, s = score_mod(t) where mask_mod holds, P = exp(s - lse):
//   delta_i = dO_i . out_i
//   dV_j = sum_i P_ij dO_i
//   dS_ij = P_ij (dO_i . v_j - delta_i),   dT_ij = dS_ij score_mod'(t_ij)
//   dK_j = scale sum_i dT_ij q_i,          dQ_i = scale sum_j dT_ij k_j
// Three kernels: delta (one warp per row); dK and dV, one CTA per 64 kv rows
// walking the q blocks of its kv block from the q side of the BlockMask (the
// transposed lists); dQ, one CTA per 64 q rows walking the kv side as the
// forward does.  P is recomputed from the saved lse in both, so nothing is
// accumulated across CTAs.  A fourth kernel transposes the kv-side lists.
//
// The CUDA-core fp32 dK/dV and dQ kernels are register-tiled: a CTA
// of 256 threads holds its 64 owned rows of two tensors in shared memory
// and walks the other side in steps of 64 rows (two tiles of 64 x D).  Per
// step a thread computes a 4 x 4 patch of the two 64 x 64 products over D
// (the recomputed score and dP), applies score_mod, mask_mod, exp and the
// dS formula to it, writes it to shared memory transposed, and then
// accumulates a 4 x (D / 16) block of its output rows over the 64 walked
// rows; the FMAs are packed fp32x2 (fma.rn.f32x2, two per instruction).
// Rows are padded by 4 floats, so the 16-byte loads of a quarter warp fall
// in eight distinct bank groups.  At D = 64 two CTAs share an SM (at most
// 128 registers a thread, 109 KB of shared memory each); at D = 128 one
// (175 KB).
#include <mutex>

#include "attn_bwd_fp32_tc.cuh"
#include "attn_bwd_tc.cuh"
#include "bwd_internal.h"
#include "ptx.cuh"
#include "tilelist.cuh"

namespace flex {
namespace {

constexpr int kTRows = 64;       // owned rows per CTA, walked rows per step
constexpr int kTThreads = 256;

template <int D>
struct TiledCfg {
    static constexpr int kLd = D + 4;          // padded row stride of a 64 x D tile (floats)
    static constexpr int kZLd = kTRows + 4;    // padded row stride of a 64 x 64 tile
    static constexpr int kTile = kTRows * kLd;
    static constexpr int kZ = kTRows * kZLd;
    static constexpr int kCols = D / 16;       // output columns per thread (two float4 at D = 128)
    // four 64 x D tiles (two owned, two walked), two 64 x 64 tiles, two row vectors, one flag word per walked tile
    static constexpr size_t kSmem =
        (4ull * kTile + 2ull * kZ + 2ull * kTRows) * sizeof(float) + kMaxKvBlocks * sizeof(uint32_t);
};

__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4(const uint16_t *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}

// score_mod at the scaled score t, and its derivative d score_mod / dt
template <int SCORE>
__device__ __forceinline__ float score_fwd(float cap, float t, float slope, int q, int kv, float &grad) {
    if constexpr (SCORE == FLEX_SCORE_SOFTCAP) {
        const float u = tanhf(t / cap);
        grad = 1.f - u * u;
        return cap * u;
    }
    grad = 1.f;
    if constexpr (SCORE == FLEX_SCORE_ALIBI) return t - slope * (float)(q - kv);
    return t;
}

struct BwdArgs {
    const void *dout;                              // contiguous [B, H, q_len, D], input dtype
    const int32_t *q_num, *q_idx, *fq_num, *fq_idx; // q side of the BlockMask
    void *dq, *dk, *dv;                            // contiguous, input dtype
    float *delta;                                  // [B, H, q_len]
};

// delta_i = dO_i . out_i, one warp per row
template <int D, typename T>
__global__ void __launch_bounds__(256) attn_bwd_delta_kernel(AttnProblem p, BwdArgs a, int64_t rows) {
    const int64_t r = ((int64_t)blockIdx.x * 256 + threadIdx.x) / 32;
    const int lane = threadIdx.x % 32;
    if (r >= rows) return;
    const T *o = static_cast<const T *>(p.out) + r * D;
    const T *g = static_cast<const T *>(a.dout) + r * D;
    float acc = 0.f;
#pragma unroll
    for (int c = lane * 4; c < D; c += 128) {
        const float4 x = load4(o + c), y = load4(g + c);
        acc = fmaf(x.x, y.x, fmaf(x.y, y.y, fmaf(x.z, y.z, fmaf(x.w, y.w, acc))));
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) a.delta[r] = acc;
}

// 64 rows of a [.., S, D] float32 tensor (row stride `rs` elements) from
// row r0 into a padded shared-memory tile; rows at or past `len` are zeros.
template <int D>
__device__ __forceinline__ void load_rows(float *dst, const float *src, int64_t rs, int r0, int len) {
    constexpr int kV = D / 4;  // float4 per row
#pragma unroll
    for (int u = 0; u < kTRows * kV / kTThreads; ++u) {
        const int i = (int)threadIdx.x + kTThreads * u, r = i / kV, c = i % kV;
        const float4 v = r0 + r < len ? __ldg(reinterpret_cast<const float4 *>(src + (int64_t)(r0 + r) * rs) + c)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
        *reinterpret_cast<float4 *>(dst + r * TiledCfg<D>::kLd + 4 * c) = v;
    }
}

// x[i][j] = A[4 ta + i] . W[tw + 16 j] over the D columns of two padded
// 64 x D tiles, with packed fp32x2 FMAs (even and odd columns in the two
// halves of an accumulator, added at the end).
template <int D>
__device__ __forceinline__ void dots4x4(const float *a, const float *w, int ta, int tw, float (&x)[4][4]) {
    constexpr int kLd = TiledCfg<D>::kLd;
    uint64_t acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0ull;  // (0.f, 0.f)
#pragma unroll 2
    for (int d = 0; d < D; d += 4) {
        ulonglong2 ra[4], rw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            ra[i] = *reinterpret_cast<const ulonglong2 *>(a + (4 * ta + i) * kLd + d);
            rw[i] = *reinterpret_cast<const ulonglong2 *>(w + (tw + 16 * i) * kLd + d);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[i][j] = f2_fma(ra[i].x, rw[j].x, acc[i][j]);
                acc[i][j] = f2_fma(ra[i].y, rw[j].y, acc[i][j]);
            }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float lo, hi;
            f2_unpack(acc[i][j], lo, hi);
            x[i][j] = lo + hi;
        }
}

// z[i][j] (owned row 4 ta + i, walked row tw + 16 j) into the 64 x 64 tile
// stored walked-row-major: zs[tw + 16 j][4 ta + i].
__device__ __forceinline__ void store_patch(float *zs, int ta, int tw, const float (&z)[4][4]) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
        *reinterpret_cast<float4 *>(zs + (tw + 16 * j) * (kTRows + 4) + 4 * ta) =
            make_float4(z[0][j], z[1][j], z[2][j], z[3][j]);
}

// y[i][c] += sum over the 64 walked rows w of zs[w][4 ta + i] * W[w][col c],
// the thread's columns being 4 td .. 4 td + 3 and, at D = 128, 64 + the
// same, held as packed pairs: y[i][2 h] = columns (64 h + 4 td, + 1),
// y[i][2 h + 1] = (+ 2, + 3).
template <int D>
__device__ __forceinline__ void accumulate(const float *zs, const float *w, int ta, int td,
                                           uint64_t (&y)[4][TiledCfg<D>::kCols / 2]) {
    constexpr int kLd = TiledCfg<D>::kLd;
#pragma unroll 4
    for (int r = 0; r < kTRows; ++r) {
        const float4 z = *reinterpret_cast<const float4 *>(zs + r * (kTRows + 4) + 4 * ta);
        const uint64_t zz[4] = {f2_pack(z.x, z.x), f2_pack(z.y, z.y), f2_pack(z.z, z.z), f2_pack(z.w, z.w)};
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
            const ulonglong2 v = *reinterpret_cast<const ulonglong2 *>(w + r * kLd + 64 * h + 4 * td);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                y[i][2 * h] = f2_fma(zz[i], v.x, y[i][2 * h]);
                y[i][2 * h + 1] = f2_fma(zz[i], v.y, y[i][2 * h + 1]);
            }
        }
    }
}

template <int D>
__device__ __forceinline__ void store_rows(float *dst, int row0, int len, int ta, int td,
                                           const uint64_t (&y)[4][TiledCfg<D>::kCols / 2]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = row0 + 4 * ta + i;
        if (r >= len) continue;
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
            float4 o;
            f2_unpack(y[i][2 * h], o.x, o.y);
            f2_unpack(y[i][2 * h + 1], o.z, o.w);
            *reinterpret_cast<float4 *>(dst + (int64_t)r * D + 64 * h + 4 * td) = o;
        }
    }
}

// dK, dV (fp32): CTA = 64 kv rows of one kv block; the q blocks come from the
// transposed lists, each walked in two steps of 64 q rows.
template <int D, int SCORE>
__global__ void __launch_bounds__(kTThreads, D == 64 ? 2 : 1) attn_bwd_dkdv_kernel(AttnProblem p, BwdArgs a) {
    using C = TiledCfg<D>;
    extern __shared__ float4 smem4[];
    float *ks = reinterpret_cast<float *>(smem4), *vs = ks + C::kTile;   // owned
    float *qs = vs + C::kTile, *gs = qs + C::kTile;                        // walked
    float *ps = gs + C::kTile, *dss = ps + C::kZ;                          // P^T, dS^T patches (walked-row-major)
    float *ls = dss + C::kZ, *dl = ls + kTRows;
    uint32_t *flags = reinterpret_cast<uint32_t *>(dl + kTRows);

    const int kvb = blockIdx.x / 2;
    const int bh = p.bh_begin + (int)blockIdx.y, h = bh % p.H, b = bh / p.H;
    const int kv0 = kvb * kBlock + (blockIdx.x & 1) * kTRows;
    if (kv0 >= p.kv_len) return;  // the second half of a short tail tile
    const int ta = threadIdx.x / 16, tw = threadIdx.x % 16;
    const float slope = SCORE == FLEX_SCORE_ALIBI ? exp2f(-8.f * (float)(h + 1) / (float)p.H) : 0.f;
    const float *kbase = static_cast<const float *>(p.k) + b * p.k_stride[0] + h * p.k_stride[1];
    const float *vbase = static_cast<const float *>(p.v) + b * p.v_stride[0] + h * p.v_stride[1];
    load_rows<D>(ks, kbase, p.k_stride[2], kv0, p.kv_len);
    load_rows<D>(vs, vbase, p.v_stride[2], kv0, p.kv_len);
    uint64_t dk[4][C::kCols / 2], dv[4][C::kCols / 2];  // packed column pairs
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < C::kCols / 2; ++c) dk[i][c] = dv[i][c] = 0ull;

    // the q side of the BlockMask (any block sizes) read as 128-tiles, in
    // chunks of kMaxKvBlocks q tiles; counts clamped and malformed entries
    // dropped, so no load leaves the tensors
    const TileLists lists{a.q_num, a.q_idx, a.fq_num, a.fq_idx, p.nkvb, p.nqb, p.kv_block, p.q_block, p.nqt};
    const float *qbase = static_cast<const float *>(p.q) + b * p.q_stride[0] + h * p.q_stride[1];
    const float *gbase = static_cast<const float *>(a.dout) + (int64_t)bh * p.q_len * D;
    const float *lbase = p.lse + (int64_t)bh * p.q_len;
    const float *dbase = a.delta + (int64_t)bh * p.q_len;

    for (int tlo = 0; tlo < p.nqt; tlo += kMaxKvBlocks) {
      const int thi = min(p.nqt, tlo + kMaxKvBlocks);
      __syncthreads();  // the previous chunk's flags are consumed
      for (int i = threadIdx.x; i < thi - tlo; i += kTThreads) flags[i] = 0u;
      __syncthreads();
      if (threadIdx.x < 32) tl_mark_warp(lists, bh, kvb, 0, flags, tlo, thi, threadIdx.x);
      __syncthreads();
      for (int qb = tlo; qb < thi; ++qb) {
        const uint32_t w = flags[qb - tlo];  // uniform over the CTA
        if (!tl_listed(w, 0)) continue;
        const bool full = tl_full(tl_expect(lists), w, 0);
        for (int q0 = qb * kBlock; q0 < min(qb * kBlock + kBlock, p.q_len); q0 += kTRows) {
            __syncthreads();  // the previous step's walked tiles and patches are consumed
            load_rows<D>(qs, qbase, p.q_stride[2], q0, p.q_len);
            load_rows<D>(gs, gbase, D, q0, p.q_len);
            if (threadIdx.x < kTRows) {
                const int q = q0 + (int)threadIdx.x;
                ls[threadIdx.x] = q < p.q_len ? lbase[q] : -INFINITY;
                dl[threadIdx.x] = q < p.q_len ? dbase[q] : 0.f;
            }
            __syncthreads();
            float st[4][4], dp[4][4];
            dots4x4<D>(ks, qs, ta, tw, st);
            dots4x4<D>(vs, gs, ta, tw, dp);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int q = q0 + tw + 16 * j;
                const float lse = ls[tw + 16 * j], dlt = dl[tw + 16 * j];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int kv = kv0 + 4 * ta + i;
                    const bool keep = lse != -INFINITY && (full || (kv < p.kv_len && mask_mod(p.mask, b, q, kv)));
                    float pr = 0.f, dts = 0.f;
                    if (keep) {
                        float grad;
                        const float x = score_fwd<SCORE>(p.score_param, st[i][j] * p.scale, slope, q, kv, grad);
                        pr = expf(x - lse);
                        dts = p.scale * pr * (dp[i][j] - dlt) * grad;
                    }
                    st[i][j] = pr;
                    dp[i][j] = dts;
                }
            }
            store_patch(ps, ta, tw, st);
            store_patch(dss, ta, tw, dp);
            __syncthreads();
            accumulate<D>(ps, gs, ta, tw, dv);
            accumulate<D>(dss, qs, ta, tw, dk);
        }
      }
    }
    const int64_t orow = (int64_t)bh * p.kv_len;
    store_rows<D>(static_cast<float *>(a.dk) + orow * D, kv0, p.kv_len, ta, tw, dk);
    store_rows<D>(static_cast<float *>(a.dv) + orow * D, kv0, p.kv_len, ta, tw, dv);
}

// dQ (fp32): CTA = 64 q rows of one q block; the kv tiles come from the kv
// side of the BlockMask, as in the forward pass, each walked in two steps.
template <int D, int SCORE>
__global__ void __launch_bounds__(kTThreads, D == 64 ? 2 : 1) attn_bwd_dq_kernel(AttnProblem p, BwdArgs a) {
    using C = TiledCfg<D>;
    extern __shared__ float4 smem4[];
    float *qs = reinterpret_cast<float *>(smem4), *gs = qs + C::kTile;   // owned
    float *ks = gs + C::kTile, *vs = ks + C::kTile;                        // walked
    float *dss = vs + C::kTile;                                            // dS patches (walked-row-major)
    uint32_t *flags = reinterpret_cast<uint32_t *>(dss + 2 * C::kZ + 2 * kTRows);

    const int qb = blockIdx.x / 2;
    const int bh = p.bh_begin + (int)blockIdx.y, h = bh % p.H, b = bh / p.H;
    const int q0 = qb * kBlock + (blockIdx.x & 1) * kTRows;
    if (q0 >= p.q_len) return;  // the second half of a short tail tile
    const int ta = threadIdx.x / 16, tw = threadIdx.x % 16;
    const float slope = SCORE == FLEX_SCORE_ALIBI ? exp2f(-8.f * (float)(h + 1) / (float)p.H) : 0.f;
    const float *qbase = static_cast<const float *>(p.q) + b * p.q_stride[0] + h * p.q_stride[1];
    const float *gbase = static_cast<const float *>(a.dout) + (int64_t)bh * p.q_len * D;
    load_rows<D>(qs, qbase, p.q_stride[2], q0, p.q_len);
    load_rows<D>(gs, gbase, D, q0, p.q_len);
    float lse[4], dlt[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int q = q0 + 4 * ta + i;
        lse[i] = q < p.q_len ? p.lse[(int64_t)bh * p.q_len + q] : -INFINITY;
        dlt[i] = q < p.q_len ? a.delta[(int64_t)bh * p.q_len + q] : 0.f;
    }
    uint64_t dq[4][C::kCols / 2];  // packed column pairs
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < C::kCols / 2; ++c) dq[i][c] = 0ull;

    // the kv side of the BlockMask (any block sizes) read as 128-tiles (at
    // most kMaxKvBlocks kv tiles)
    const TileLists lists{p.kv_num, p.kv_idx, p.full_num, p.full_idx, p.nqb, p.nkvb, p.q_block, p.kv_block, p.nkvt};
    for (int i = threadIdx.x; i < p.nkvt; i += kTThreads) flags[i] = 0u;
    __syncthreads();
    if (threadIdx.x < 32) tl_mark_warp(lists, bh, qb, 0, flags, 0, p.nkvt, threadIdx.x);
    __syncthreads();
    const float *kbase = static_cast<const float *>(p.k) + b * p.k_stride[0] + h * p.k_stride[1];
    const float *vbase = static_cast<const float *>(p.v) + b * p.v_stride[0] + h * p.v_stride[1];

    for (int kvb = 0; kvb < p.nkvt; ++kvb) {
        const uint32_t w = flags[kvb];  // uniform over the CTA
        if (!tl_listed(w, 0)) continue;
        const bool full = tl_full(tl_expect(lists), w, 0);
        for (int kv0 = kvb * kBlock; kv0 < min(kvb * kBlock + kBlock, p.kv_len); kv0 += kTRows) {
            __syncthreads();  // the previous step's walked tiles and patch are consumed
            load_rows<D>(ks, kbase, p.k_stride[2], kv0, p.kv_len);
            load_rows<D>(vs, vbase, p.v_stride[2], kv0, p.kv_len);
            __syncthreads();
            float st[4][4], dp[4][4];
            dots4x4<D>(qs, ks, ta, tw, st);
            dots4x4<D>(gs, vs, ta, tw, dp);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int q = q0 + 4 * ta + i;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int kv = kv0 + tw + 16 * j;
                    const bool keep = lse[i] != -INFINITY && (full || (kv < p.kv_len && mask_mod(p.mask, b, q, kv)));
                    float dts = 0.f;
                    if (keep) {
                        float grad;
                        const float x = score_fwd<SCORE>(p.score_param, st[i][j] * p.scale, slope, q, kv, grad);
                        dts = p.scale * expf(x - lse[i]) * (dp[i][j] - dlt[i]) * grad;
                    }
                    dp[i][j] = dts;
                }
            }
            store_patch(dss, ta, tw, dp);
            __syncthreads();
            accumulate<D>(dss, ks, ta, tw, dq);
        }
    }
    store_rows<D>(static_cast<float *>(a.dq) + (int64_t)bh * p.q_len * D, q0, p.q_len, ta, tw, dq);
}

// Whether the ascending list[0, n) holds x.
__device__ __forceinline__ bool holds(const int32_t *list, int n, int x) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) / 2;
        const int v = list[mid];
        if (v == x) return true;
        if (v < x) lo = mid + 1;
        else hi = mid;
    }
    return false;
}

// q side of the BlockMask: one warp per (b, h, kv block j) writes, for the
// partial and the full lists, the q blocks whose kv-side list holds j
// (ascending) and then the other q blocks (ascending).
__global__ void __launch_bounds__(128) block_mask_transpose_kernel(const int32_t *kv_num, const int32_t *kv_idx,
                                                                   const int32_t *full_num, const int32_t *full_idx,
                                                                   int64_t nbh, int nqb, int nkvb, int32_t *q_num,
                                                                   int32_t *q_idx, int32_t *fq_num, int32_t *fq_idx) {
    const int64_t w = ((int64_t)blockIdx.x * 128 + threadIdx.x) / 32;
    const int lane = threadIdx.x % 32;
    if (w >= nbh * nkvb) return;
    const int64_t bh = w / nkvb;
    const int j = (int)(w % nkvb);
    const unsigned lt = (1u << lane) - 1u;
    for (int list = 0; list < 2; ++list) {
        const int32_t *num = list ? full_num : kv_num;
        const int32_t *idx = list ? full_idx : kv_idx;
        int32_t *onum = list ? fq_num : q_num;
        int32_t *oidx = (list ? fq_idx : q_idx) + w * nqb;
        int count = 0;
        for (int pass = 0; pass < 2; ++pass) {
            for (int base = 0; base < nqb; base += 32) {
                const int i = base + lane;
                bool sel = false;
                if (i < nqb) {
                    const int64_t row = bh * nqb + i;
                    sel = holds(idx + row * nkvb, num[row], j) == (pass == 0);
                }
                const unsigned bal = __ballot_sync(0xffffffffu, sel);
                if (sel) oidx[count + __popc(bal & lt)] = i;
                count += __popc(bal);
            }
            if (pass == 0 && lane == 0) onum[w] = count;
        }
    }
}

template <int D, int SCORE>
cudaError_t launch_bwd_fp32_score(const AttnProblem &p, const BwdArgs &a, bool dkdv, bool dq, cudaStream_t stream) {
    using C = TiledCfg<D>;
    cudaError_t e =
        cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D, SCORE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D, SCORE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)C::kSmem);
    if (e != cudaSuccess) return e;
    // grid.y holds at most 65535 (b, h) pairs per launch
    for (int begin = 0; begin < p.B * p.H; begin += 65535) {
        AttnProblem part = p;
        part.bh_begin = begin;
        const int count = p.B * p.H - begin < 65535 ? p.B * p.H - begin : 65535;
        if (dkdv) {
            attn_bwd_dkdv_kernel<D, SCORE><<<dim3(2 * p.nkvt, count), kTThreads, C::kSmem, stream>>>(part, a);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        if (dq) {
            attn_bwd_dq_kernel<D, SCORE><<<dim3(2 * p.nqt, count), kTThreads, C::kSmem, stream>>>(part, a);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

// The dQ launch of a backward runs on a second stream per device that forks
// from the caller's stream after delta and joins it after dQ, so that its
// CTAs fill the SMs the dK/dV kernel's last items leave idle (measured on
// one GB300: causal + prefix B4 H16 S4096 D64 0.646 -> 0.629 ms, document +
// softcap B8 H16 S8192 D128 1.935 -> 1.916 ms, causal + ALiBi B2 H32
// S16384 D128 10.29 -> 10.24 ms).  One enqueue at a time per device, since
// the fork and join events are shared.
struct BwdSide {
    std::mutex enqueue;
    cudaStream_t s2 = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int kSideDevices = 64;
std::mutex g_side_mutex;
BwdSide *g_side[kSideDevices] = {nullptr};

// The side stream of the current device, created on first use; while
// `stream` is being captured, only one that already exists (creating
// streams and events is not among the calls a capture may record).
BwdSide *bwd_side(cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kSideDevices) return nullptr;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return nullptr;
    std::lock_guard<std::mutex> lock(g_side_mutex);
    if (!g_side[dev] && cap == cudaStreamCaptureStatusNone) {
        BwdSide *b = new BwdSide();
        if (cudaStreamCreateWithFlags(&b->s2, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&b->fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&b->join, cudaEventDisableTiming) != cudaSuccess)
            return nullptr;  // the handles created so far stay with the process
        g_side[dev] = b;
    }
    return g_side[dev];
}

// dK/dV on `stream`, dQ on the side stream between a fork after the work
// already on `stream` (delta) and a join back into `stream`; both on
// `stream`, one after the other, when there is no side stream.
template <class DkDv, class Dq>
cudaError_t launch_dkdv_dq(cudaStream_t stream, DkDv &&dkdv, Dq &&dq) {
    BwdSide *side = bwd_side(stream);
    if (!side) {
        cudaGetLastError();  // a failed capture-status query leaves nothing to report
        const cudaError_t e = dkdv(stream);
        return e != cudaSuccess ? e : dq(stream);
    }
    std::lock_guard<std::mutex> lock(side->enqueue);
    cudaError_t e;
    if ((e = cudaEventRecord(side->fork, stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(side->s2, side->fork, 0)) != cudaSuccess)
        return e;
    if ((e = dkdv(stream)) != cudaSuccess) return e;
    if ((e = dq(side->s2)) != cudaSuccess) return e;
    if ((e = cudaEventRecord(side->join, side->s2)) != cudaSuccess) return e;
    return cudaStreamWaitEvent(stream, side->join, 0);
}

// fp32: delta, then dK/dV and dQ on the tensor cores (three-way bf16 split);
// dK/dV of a q side longer than kBwdF32TcMaxQTiles tiles falls to the
// register-tiled CUDA-core kernel.
template <int D>
cudaError_t launch_bwd_fp32(const AttnProblem &p, const BwdArgs &a, cudaStream_t stream) {
    const int64_t rows = (int64_t)p.B * p.H * p.q_len;
    attn_bwd_delta_kernel<D, float><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, stream>>>(p, a, rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const BwdF32TcArgs ta{static_cast<const float *>(a.dout), a.delta, a.q_num, a.q_idx, a.fq_num, a.fq_idx,
                          static_cast<float *>(a.dk), static_cast<float *>(a.dv), static_cast<float *>(a.dq)};
    auto dq = [&](cudaStream_t s) { return launch_bwd_fp32_tc_dq(p, ta, s); };
    if (p.nqt <= kBwdF32TcMaxQTiles)
        return launch_dkdv_dq(stream, [&](cudaStream_t s) { return launch_bwd_fp32_tc_dkdv(p, ta, s); }, dq);
    // dK/dV of a longer q side on the CUDA cores
    return launch_dkdv_dq(
        stream,
        [&](cudaStream_t s) {
            switch (p.score_kind) {
                case FLEX_SCORE_SOFTCAP:
                    return launch_bwd_fp32_score<D, FLEX_SCORE_SOFTCAP>(p, a, true, false, s);
                case FLEX_SCORE_ALIBI:
                    return launch_bwd_fp32_score<D, FLEX_SCORE_ALIBI>(p, a, true, false, s);
                default:
                    return launch_bwd_fp32_score<D, FLEX_SCORE_IDENTITY>(p, a, true, false, s);
            }
        },
        dq);
}

}  // namespace

cudaError_t launch_block_mask_transpose(const int32_t *kv_num, const int32_t *kv_idx, const int32_t *full_num,
                                        const int32_t *full_idx, int B, int H, int nqb, int nkvb, int32_t *q_num,
                                        int32_t *q_idx, int32_t *fq_num, int32_t *fq_idx, cudaStream_t stream) {
    const int64_t nbh = (int64_t)B * H, warps = nbh * nkvb;
    block_mask_transpose_kernel<<<(unsigned)((warps * 32 + 127) / 128), 128, 0, stream>>>(
        kv_num, kv_idx, full_num, full_idx, nbh, nqb, nkvb, q_num, q_idx, fq_num, fq_idx);
    return cudaGetLastError();
}

static_assert(kBwdTcMaxQBlocks == kBwdMaxList, "list capacity of the tensor-core backward");

namespace {

// bf16: delta on the CUDA cores, then the tensor-core dK/dV and dQ kernels.
cudaError_t launch_bwd_bf16_tc(const AttnProblem &p, const BwdArgs &a, cudaStream_t stream) {
    const int64_t rows = (int64_t)p.B * p.H * p.q_len;
    if (p.D == 64)
        attn_bwd_delta_kernel<64, uint16_t><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, stream>>>(p, a, rows);
    else
        attn_bwd_delta_kernel<128, uint16_t><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, stream>>>(p, a, rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t dstr[4] = {(int64_t)p.H * p.q_len * p.D, (int64_t)p.q_len * p.D, p.D, 1};
    CUtensorMap mq, mk, mv, mdo;
    if (!make_bf16_tile_map(&mq, p.q, p.B, p.H, p.q_len, p.D, p.q_stride) ||
        !make_bf16_tile_map(&mk, p.k, p.B, p.H, p.kv_len, p.D, p.k_stride) ||
        !make_bf16_tile_map(&mv, p.v, p.B, p.H, p.kv_len, p.D, p.v_stride) ||
        !make_bf16_tile_map(&mdo, a.dout, p.B, p.H, p.q_len, p.D, dstr))
        return cudaErrorInvalidValue;
    BwdTcParams kp;
    kp.B = p.B;
    kp.H = p.H;
    kp.q_len = p.q_len;
    kp.kv_len = p.kv_len;
    kp.bh_begin = p.bh_begin;
    kp.nbh = p.bh_count;
    kp.mask = p.mask;
    kp.scale = p.scale;
    kp.score_param = p.score_param;
    kp.lse = p.lse;
    kp.delta = a.delta;
    kp.status = p.status;
    // dK, dV: own the kv tiles, walk the q side of the BlockMask
    kp.nblocks = p.nkvt;
    kp.lists = TileLists{a.q_num, a.q_idx, a.fq_num, a.fq_idx, p.nkvb, p.nqb, p.kv_block, p.q_block, p.nqt};
    kp.out0 = static_cast<uint16_t *>(a.dv);
    kp.out1 = static_cast<uint16_t *>(a.dk);
    const CUtensorMap kv_maps[4] = {mk, mv, mq, mdo};
    // dQ: own the q tiles, walk the kv side
    BwdTcParams qp = kp;
    qp.nblocks = p.nqt;
    qp.lists = TileLists{p.kv_num, p.kv_idx, p.full_num, p.full_idx, p.nqb, p.nkvb, p.q_block, p.kv_block, p.nkvt};
    qp.out0 = static_cast<uint16_t *>(a.dq);
    qp.out1 = nullptr;
    const CUtensorMap q_maps[4] = {mq, mdo, mk, mv};
    return launch_dkdv_dq(
        stream, [&](cudaStream_t s) { return launch_bwd_tc_dkdv(kv_maps, kp, p.D, p.score_kind, s); },
        [&](cudaStream_t s) { return launch_bwd_tc_dq(q_maps, qp, p.D, p.score_kind, s); });
}

}  // namespace

cudaError_t launch_attn_bwd(const AttnProblem &p, int dtype, const void *dout, const int32_t *q_num,
                            const int32_t *q_idx, const int32_t *fq_num, const int32_t *fq_idx, void *dq, void *dk,
                            void *dv, float *delta, cudaStream_t stream) {
    const BwdArgs a{dout, q_num, q_idx, fq_num, fq_idx, dq, dk, dv, delta};
    if (dtype == FLEX_DTYPE_BF16) return launch_bwd_bf16_tc(p, a, stream);
    return p.D == 64 ? launch_bwd_fp32<64>(p, a, stream) : launch_bwd_fp32<128>(p, a, stream);
}

}  // namespace flex
