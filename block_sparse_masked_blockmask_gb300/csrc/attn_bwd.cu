// Backward pass of the block-sparse attention (the flex_attention_backward op
// of "[Inductor][Flex Attention] Add Subtiling Option for Alpha Scaling",
// PyTorch PR #167356, test diffs: it takes q, k, v, the forward's out and lse,
// and the output gradient, and returns dq, dk, dv).  fp32 inputs run on the
// CUDA cores with fp32 arithmetic (the kernels below); bf16 inputs take delta
// from the kernel below and dq, dk, dv from the tensor-core kernels of
// attn_bwd_tc.cuh.
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
// Each thread owns 32 of a row's D dims, as 8 groups of 4 contiguous floats
// spaced 4 * (threads per row) apart, so the row's threads read distinct
// shared-memory banks when they fetch the same staged row.
#include "attn_bwd_tc.cuh"
#include "bwd_internal.h"
#include "ptx.cuh"
#include "tilelist.cuh"

namespace flex {
namespace {

constexpr int kBwdRows = 64;    // rows per CTA (kv rows for dK/dV, q rows for dQ)
constexpr int kDimsPer = 32;    // dims per thread
constexpr int kGroups = kDimsPer / 4;

template <int D>
struct BwdCfg {
    static constexpr int kTpr = D / kDimsPer;          // threads per row: 2 (D = 64) or 4 (D = 128)
    static constexpr int kThreads = kBwdRows * kTpr;   // 128 or 256
    static constexpr int kStride = 4 * kTpr;           // distance between a thread's groups
    // two staged 128 x D fp32 tiles, then two 128-float row vectors
    // plus one flag word per walked tile of a chunk (the BlockMask read as 128-tiles)
    static constexpr size_t kSmem =
        2ull * kBlock * D * sizeof(float) + 2ull * kBlock * sizeof(float) + kMaxKvBlocks * sizeof(uint32_t);
};

__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4(const uint16_t *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}
__device__ __forceinline__ void store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void store4(uint16_t *p, float4 v) {
    *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
}

// score_mod at the scaled score t, and its derivative d score_mod / dt
__device__ __forceinline__ float score_fwd(int kind, float cap, float t, float slope, int q, int kv, float &grad) {
    if (kind == FLEX_SCORE_SOFTCAP) {
        const float u = tanhf(t / cap);
        grad = 1.f - u * u;
        return cap * u;
    }
    grad = 1.f;
    if (kind == FLEX_SCORE_ALIBI) return t - slope * (float)(q - kv);
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

// Stage 128 rows of a [.., S, D] tensor (row stride `rs` elements) starting
// at row r0 into shared memory as fp32; rows at or past `len` become zeros.
template <int D, int THREADS, typename T>
__device__ __forceinline__ void stage_tile(float *dst, const T *src, int64_t rs, int r0, int len) {
    for (int i = threadIdx.x; i < kBlock * D / 4; i += THREADS) {
        const int r = (i * 4) / D, c = (i * 4) % D;
        const float4 v = r0 + r < len ? load4(src + (int64_t)(r0 + r) * rs + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        reinterpret_cast<float4 *>(dst)[i] = v;
    }
}

// dK, dV: CTA = 64 kv rows of one kv block; the q blocks come from the
// transposed lists (full tiles first, then partial ones).
template <int D, typename T>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1) attn_bwd_dkdv_kernel(AttnProblem p, BwdArgs a) {
    using C = BwdCfg<D>;
    extern __shared__ float4 smem4[];
    float *qs = reinterpret_cast<float *>(smem4);
    float *gs = qs + kBlock * D;
    float *ls = gs + kBlock * D;
    float *dl = ls + kBlock;
    uint32_t *flags = reinterpret_cast<uint32_t *>(dl + kBlock);

    const int kvb = blockIdx.x / 2;
    const int bh = p.bh_begin + (int)blockIdx.y, h = bh % p.H, b = bh / p.H;
    const int row = threadIdx.x / C::kTpr, part = threadIdx.x % C::kTpr;
    const int kv = kvb * kBlock + (blockIdx.x & 1) * kBwdRows + row;
    const bool kv_in = kv < p.kv_len;

    const T *kp = static_cast<const T *>(p.k) + b * p.k_stride[0] + h * p.k_stride[1] + (int64_t)kv * p.k_stride[2];
    const T *vp = static_cast<const T *>(p.v) + b * p.v_stride[0] + h * p.v_stride[1] + (int64_t)kv * p.v_stride[2];
    float kr[kDimsPer], vr[kDimsPer], dk[kDimsPer], dv[kDimsPer];
#pragma unroll
    for (int gi = 0; gi < kGroups; ++gi) {
        const int d = gi * C::kStride + 4 * part;
        const float4 x = kv_in ? load4(kp + d) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 y = kv_in ? load4(vp + d) : make_float4(0.f, 0.f, 0.f, 0.f);
        kr[4 * gi] = x.x, kr[4 * gi + 1] = x.y, kr[4 * gi + 2] = x.z, kr[4 * gi + 3] = x.w;
        vr[4 * gi] = y.x, vr[4 * gi + 1] = y.y, vr[4 * gi + 2] = y.z, vr[4 * gi + 3] = y.w;
    }
#pragma unroll
    for (int e = 0; e < kDimsPer; ++e) dk[e] = dv[e] = 0.f;
    const float slope = exp2f(-8.f * (float)(h + 1) / (float)p.H);

    // the q side of the BlockMask (any block sizes) read as 128-tiles, in
    // chunks of kMaxKvBlocks q tiles; counts clamped and malformed entries
    // dropped, so no load leaves the tensors
    const TileLists lists{a.q_num, a.q_idx, a.fq_num, a.fq_idx, p.nkvb, p.nqb, p.kv_block, p.q_block, p.nqt};
    const T *qbase = static_cast<const T *>(p.q) + b * p.q_stride[0] + h * p.q_stride[1];
    const T *gbase = static_cast<const T *>(a.dout) + (int64_t)bh * p.q_len * D;
    const float *lbase = p.lse + (int64_t)bh * p.q_len;
    const float *dbase = a.delta + (int64_t)bh * p.q_len;

    for (int tlo = 0; tlo < p.nqt; tlo += kMaxKvBlocks) {
      const int thi = min(p.nqt, tlo + kMaxKvBlocks);
      __syncthreads();  // the previous chunk's flags are consumed
      for (int i = threadIdx.x; i < thi - tlo; i += C::kThreads) flags[i] = 0u;
      __syncthreads();
      if (threadIdx.x < 32) tl_mark_warp(lists, bh, kvb, 0, flags, tlo, thi, threadIdx.x);
      __syncthreads();
      for (int qb = tlo; qb < thi; ++qb) {
        const uint32_t w = flags[qb - tlo];  // uniform over the CTA
        if (!tl_listed(w, 0)) continue;
        const bool full = tl_full(tl_expect(lists), w, 0);
        const int q0 = qb * kBlock;
        __syncthreads();  // the previous q block is consumed
        stage_tile<D, C::kThreads>(qs, qbase, p.q_stride[2], q0, p.q_len);
        stage_tile<D, C::kThreads>(gs, gbase, D, q0, p.q_len);
        for (int r = threadIdx.x; r < kBlock; r += C::kThreads) {
            const bool in = q0 + r < p.q_len;
            ls[r] = in ? lbase[q0 + r] : -INFINITY;
            dl[r] = in ? dbase[q0 + r] : 0.f;
        }
        __syncthreads();
        for (int r = 0; r < kBlock; ++r) {
            const int q = q0 + r;
            float qv[kDimsPer], gv[kDimsPer];
            float t4[4] = {0.f, 0.f, 0.f, 0.f}, p4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int gi = 0; gi < kGroups; ++gi) {
                const int d = gi * C::kStride + 4 * part;
                const float4 x = reinterpret_cast<const float4 *>(qs + r * D + d)[0];
                const float4 y = reinterpret_cast<const float4 *>(gs + r * D + d)[0];
                qv[4 * gi] = x.x, qv[4 * gi + 1] = x.y, qv[4 * gi + 2] = x.z, qv[4 * gi + 3] = x.w;
                gv[4 * gi] = y.x, gv[4 * gi + 1] = y.y, gv[4 * gi + 2] = y.z, gv[4 * gi + 3] = y.w;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    t4[c] = fmaf(qv[4 * gi + c], kr[4 * gi + c], t4[c]);
                    p4[c] = fmaf(gv[4 * gi + c], vr[4 * gi + c], p4[c]);
                }
            }
            float dot = (t4[0] + t4[1]) + (t4[2] + t4[3]);
            float dp = (p4[0] + p4[1]) + (p4[2] + p4[3]);
#pragma unroll
            for (int s = 1; s < C::kTpr; s <<= 1) {
                dot += __shfl_xor_sync(0xffffffffu, dot, s);
                dp += __shfl_xor_sync(0xffffffffu, dp, s);
            }
            const float lse = ls[r];
            const bool keep = lse != -INFINITY &&
                              (full || (kv_in && q < p.q_len && mask_mod(p.mask, b, q, kv)));
            float pr = 0.f, dts = 0.f;
            if (keep) {
                float grad;
                const float x = score_fwd(p.score_kind, p.score_param, dot * p.scale, slope, q, kv, grad);
                pr = expf(x - lse);
                dts = p.scale * pr * (dp - dl[r]) * grad;
            }
#pragma unroll
            for (int e = 0; e < kDimsPer; ++e) {
                dv[e] = fmaf(pr, gv[e], dv[e]);
                dk[e] = fmaf(dts, qv[e], dk[e]);
            }
        }
      }
    }
    if (!kv_in) return;
    const int64_t orow = (int64_t)bh * p.kv_len + kv;
    T *dkp = static_cast<T *>(a.dk) + orow * D;
    T *dvp = static_cast<T *>(a.dv) + orow * D;
#pragma unroll
    for (int gi = 0; gi < kGroups; ++gi) {
        const int d = gi * C::kStride + 4 * part;
        store4(dkp + d, make_float4(dk[4 * gi], dk[4 * gi + 1], dk[4 * gi + 2], dk[4 * gi + 3]));
        store4(dvp + d, make_float4(dv[4 * gi], dv[4 * gi + 1], dv[4 * gi + 2], dv[4 * gi + 3]));
    }
}

// dQ: CTA = 64 q rows of one q block; the kv tiles come from the kv side of
// the BlockMask, as in the forward pass.
template <int D, typename T>
__global__ void __launch_bounds__(BwdCfg<D>::kThreads, 1) attn_bwd_dq_kernel(AttnProblem p, BwdArgs a) {
    using C = BwdCfg<D>;
    extern __shared__ float4 smem4[];
    float *ks = reinterpret_cast<float *>(smem4);
    float *vs = ks + kBlock * D;
    uint32_t *flags = reinterpret_cast<uint32_t *>(vs + kBlock * D + 2 * kBlock);

    const int qb = blockIdx.x / 2;
    const int bh = p.bh_begin + (int)blockIdx.y, h = bh % p.H, b = bh / p.H;
    const int row = threadIdx.x / C::kTpr, part = threadIdx.x % C::kTpr;
    const int q = qb * kBlock + (blockIdx.x & 1) * kBwdRows + row;
    const bool q_in = q < p.q_len;

    const T *qp = static_cast<const T *>(p.q) + b * p.q_stride[0] + h * p.q_stride[1] +
                  (int64_t)(q_in ? q : 0) * p.q_stride[2];
    const T *gp = static_cast<const T *>(a.dout) + ((int64_t)bh * p.q_len + (q_in ? q : 0)) * D;
    float qv[kDimsPer], gv[kDimsPer], dq[kDimsPer];
#pragma unroll
    for (int gi = 0; gi < kGroups; ++gi) {
        const int d = gi * C::kStride + 4 * part;
        const float4 x = q_in ? load4(qp + d) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 y = q_in ? load4(gp + d) : make_float4(0.f, 0.f, 0.f, 0.f);
        qv[4 * gi] = x.x, qv[4 * gi + 1] = x.y, qv[4 * gi + 2] = x.z, qv[4 * gi + 3] = x.w;
        gv[4 * gi] = y.x, gv[4 * gi + 1] = y.y, gv[4 * gi + 2] = y.z, gv[4 * gi + 3] = y.w;
    }
#pragma unroll
    for (int e = 0; e < kDimsPer; ++e) dq[e] = 0.f;
    const int64_t orow = (int64_t)bh * p.q_len + q;
    const float lse = q_in ? p.lse[orow] : -INFINITY;
    const float dlt = q_in ? a.delta[orow] : 0.f;
    const float slope = exp2f(-8.f * (float)(h + 1) / (float)p.H);

    // the kv side of the BlockMask (any block sizes) read as 128-tiles (at
    // most kMaxKvBlocks kv tiles)
    const TileLists lists{p.kv_num, p.kv_idx, p.full_num, p.full_idx, p.nqb, p.nkvb, p.q_block, p.kv_block, p.nkvt};
    for (int i = threadIdx.x; i < p.nkvt; i += C::kThreads) flags[i] = 0u;
    __syncthreads();
    if (threadIdx.x < 32) tl_mark_warp(lists, bh, qb, 0, flags, 0, p.nkvt, threadIdx.x);
    __syncthreads();
    const T *kbase = static_cast<const T *>(p.k) + b * p.k_stride[0] + h * p.k_stride[1];
    const T *vbase = static_cast<const T *>(p.v) + b * p.v_stride[0] + h * p.v_stride[1];

    for (int kvb = 0; kvb < p.nkvt; ++kvb) {
        const uint32_t w = flags[kvb];  // uniform over the CTA
        if (!tl_listed(w, 0)) continue;
        const bool full = tl_full(tl_expect(lists), w, 0);
        const int kv0 = kvb * kBlock;
        __syncthreads();
        stage_tile<D, C::kThreads>(ks, kbase, p.k_stride[2], kv0, p.kv_len);
        stage_tile<D, C::kThreads>(vs, vbase, p.v_stride[2], kv0, p.kv_len);
        __syncthreads();
        // Every thread runs the column loop, whose shuffles need all 32
        // lanes; an empty or padding row (lse = -inf) only keeps no column.
        for (int c = 0; c < kBlock; ++c) {
            const int kv = kv0 + c;
            float kc[kDimsPer];
            float t4[4] = {0.f, 0.f, 0.f, 0.f}, p4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int gi = 0; gi < kGroups; ++gi) {
                const int d = gi * C::kStride + 4 * part;
                const float4 x = reinterpret_cast<const float4 *>(ks + c * D + d)[0];
                const float4 y = reinterpret_cast<const float4 *>(vs + c * D + d)[0];
                kc[4 * gi] = x.x, kc[4 * gi + 1] = x.y, kc[4 * gi + 2] = x.z, kc[4 * gi + 3] = x.w;
                const float yv[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    t4[e] = fmaf(qv[4 * gi + e], kc[4 * gi + e], t4[e]);
                    p4[e] = fmaf(gv[4 * gi + e], yv[e], p4[e]);
                }
            }
            float dot = (t4[0] + t4[1]) + (t4[2] + t4[3]);
            float dp = (p4[0] + p4[1]) + (p4[2] + p4[3]);
#pragma unroll
            for (int s = 1; s < C::kTpr; s <<= 1) {
                dot += __shfl_xor_sync(0xffffffffu, dot, s);
                dp += __shfl_xor_sync(0xffffffffu, dp, s);
            }
            const bool keep = lse != -INFINITY && (full || (kv < p.kv_len && mask_mod(p.mask, b, q, kv)));
            float dts = 0.f;
            if (keep) {
                float grad;
                const float x = score_fwd(p.score_kind, p.score_param, dot * p.scale, slope, q, kv, grad);
                dts = p.scale * expf(x - lse) * (dp - dlt) * grad;
            }
#pragma unroll
            for (int e = 0; e < kDimsPer; ++e) dq[e] = fmaf(dts, kc[e], dq[e]);
        }
    }
    if (!q_in) return;
    T *dqp = static_cast<T *>(a.dq) + orow * D;
#pragma unroll
    for (int gi = 0; gi < kGroups; ++gi) {
        const int d = gi * C::kStride + 4 * part;
        store4(dqp + d, make_float4(dq[4 * gi], dq[4 * gi + 1], dq[4 * gi + 2], dq[4 * gi + 3]));
    }
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

template <int D, typename T>
cudaError_t launch_bwd_typed(const AttnProblem &p, const BwdArgs &a, cudaStream_t stream) {
    using C = BwdCfg<D>;
    const int64_t rows = (int64_t)p.B * p.H * p.q_len;
    attn_bwd_delta_kernel<D, T><<<(unsigned)((rows * 32 + 255) / 256), 256, 0, stream>>>(p, a, rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_bwd_dq_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
    if (e != cudaSuccess) return e;
    // grid.y holds at most 65535 (b, h) pairs per launch
    for (int begin = 0; begin < p.B * p.H; begin += 65535) {
        AttnProblem part = p;
        part.bh_begin = begin;
        const int count = p.B * p.H - begin < 65535 ? p.B * p.H - begin : 65535;
        attn_bwd_dkdv_kernel<D, T><<<dim3(2 * p.nkvt, count), C::kThreads, C::kSmem, stream>>>(part, a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        attn_bwd_dq_kernel<D, T><<<dim3(2 * p.nqt, count), C::kThreads, C::kSmem, stream>>>(part, a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
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
    e = launch_bwd_tc_dkdv(kv_maps, kp, p.D, p.score_kind, stream);
    if (e != cudaSuccess) return e;
    // dQ: own the q tiles, walk the kv side
    kp.nblocks = p.nqt;
    kp.lists = TileLists{p.kv_num, p.kv_idx, p.full_num, p.full_idx, p.nqb, p.nkvb, p.q_block, p.kv_block, p.nkvt};
    kp.out0 = static_cast<uint16_t *>(a.dq);
    kp.out1 = nullptr;
    const CUtensorMap q_maps[4] = {mq, mdo, mk, mv};
    return launch_bwd_tc_dq(q_maps, kp, p.D, p.score_kind, stream);
}

}  // namespace

cudaError_t launch_attn_bwd(const AttnProblem &p, int dtype, const void *dout, const int32_t *q_num,
                            const int32_t *q_idx, const int32_t *fq_num, const int32_t *fq_idx, void *dq, void *dk,
                            void *dv, float *delta, cudaStream_t stream) {
    const BwdArgs a{dout, q_num, q_idx, fq_num, fq_idx, dq, dk, dv, delta};
    if (dtype == FLEX_DTYPE_BF16) return launch_bwd_bf16_tc(p, a, stream);
    return p.D == 64 ? launch_bwd_typed<64, float>(p, a, stream) : launch_bwd_typed<128, float>(p, a, stream);
}

}  // namespace flex
