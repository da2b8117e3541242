// Block-sparse attention forward for float32 inputs on the CUDA cores.
//
// The same computation as the tensor-core path (the flex_attention op of
// "[Inductor][Flex Attention] Add Subtiling Option for Alpha Scaling",
// PyTorch PR #167356): for every tile listed in the BlockMask, scores
// s = score_mod(scale * q.k), masked to -inf by mask_mod on partial tiles,
// folded into an online softmax (running max m, running sum l, output rescaled
// by alpha = exp(m_old - m_new): the forward_block_mn step), then out = acc / l
// and lse = m + ln l.  All arithmetic is fp32 FFMA; no tensor cores, so the
// 1e-4 tolerance of fp32 inputs holds (a single TF32 pass would not).
//
// One CTA per (q block, head, batch); D/64 threads per query row, each owning
// 64 dims of q and of the accumulator.  K and V tiles are staged in shared
// memory and read as broadcasts.  Rows of a tail tile past the lengths are
// staged as zeros and masked (kv) or left unwritten (q).
#include "flex_internal.h"
#include "tilelist.cuh"

namespace flex {
namespace {

constexpr int kDimsPerThread = 64;
constexpr int kChunk = 16;   // columns per online-softmax update

template <int D>
struct Fp32Cfg {
    static constexpr int kTpr = D / kDimsPerThread;      // threads per row
    static constexpr int kThreads = kBlock * kTpr;
    // K and V tiles, then one flag word per kv tile (the BlockMask read as 128-tiles)
    static constexpr size_t kSmem = 2ull * kBlock * D * sizeof(float) + kMaxKvBlocks * sizeof(uint32_t);
};

__device__ __forceinline__ float score_mod_f32(int kind, float param, float s, float slope, int q, int kv) {
    if (kind == FLEX_SCORE_SOFTCAP) return param * tanhf(s / param);
    if (kind == FLEX_SCORE_ALIBI) return s - slope * (float)(q - kv);
    return s;
}

template <int D>
__global__ void __launch_bounds__(Fp32Cfg<D>::kThreads) attn_fp32_kernel(AttnProblem p) {
    using C = Fp32Cfg<D>;
    extern __shared__ float4 smem4[];
    float *ks = reinterpret_cast<float *>(smem4);
    float *vs = ks + kBlock * D;
    uint32_t *flags = reinterpret_cast<uint32_t *>(vs + kBlock * D);

    const int qb = blockIdx.x, bh = p.bh_begin + (int)blockIdx.y, h = bh % p.H, b = bh / p.H;
    const int row = threadIdx.x / C::kTpr, part = threadIdx.x % C::kTpr;
    const int q = qb * kBlock + row;

    const bool row_in = q < p.q_len;  // a tail tile's rows past Q_LEN are padding
    const float *qp = static_cast<const float *>(p.q) + b * p.q_stride[0] + h * p.q_stride[1] +
                      (int64_t)(row_in ? q : 0) * p.q_stride[2] + part * kDimsPerThread;
    // PRESCALE_QK: q~ = scale q rounded to float once, scores q~.k unscaled
    const float post = p.prescale ? 1.f : p.scale;
    float qr[kDimsPerThread], acc[kDimsPerThread];
#pragma unroll
    for (int d = 0; d < kDimsPerThread; ++d) {
        const float x = row_in ? qp[d] : 0.f;
        qr[d] = p.prescale ? __fmul_rn(x, p.scale) : x;
        acc[d] = 0.f;
    }
    const float slope = exp2f(-8.f * (float)(h + 1) / (float)p.H);
    float m = -INFINITY, l = 0.f;

    // the kv tiles of this q tile: the BlockMask's lists (any block sizes)
    // read as 128-tiles by the first warp; counts are clamped and malformed
    // entries dropped, so no load leaves the tensors
    const TileLists lists{p.kv_num, p.kv_idx, p.full_num, p.full_idx, p.nqb, p.nkvb, p.q_block, p.kv_block, p.nkvt};
    for (int i = threadIdx.x; i < p.nkvt; i += C::kThreads) flags[i] = 0u;
    __syncthreads();
    if (threadIdx.x < 32) tl_mark_warp(lists, bh, qb, 0, flags, 0, p.nkvt, threadIdx.x);
    __syncthreads();
    const float *kbase = static_cast<const float *>(p.k) + b * p.k_stride[0] + h * p.k_stride[1];
    const float *vbase = static_cast<const float *>(p.v) + b * p.v_stride[0] + h * p.v_stride[1];

    for (int kvb = 0; kvb < p.nkvt; ++kvb) {
        const uint32_t w = flags[kvb];  // the same for every thread of the CTA
        if (!tl_listed(w, 0)) continue;
        const bool full = tl_full(tl_expect(lists), w, 0);
        const int kv0 = kvb * kBlock;
        __syncthreads();  // previous tile fully consumed
        for (int i = threadIdx.x; i < kBlock * D / 4; i += C::kThreads) {
            const int r = (i * 4) / D, c = (i * 4) % D;
            const bool in = kv0 + r < p.kv_len;
            const int64_t ko = (int64_t)(kv0 + r) * p.k_stride[2] + c;
            const int64_t vo = (int64_t)(kv0 + r) * p.v_stride[2] + c;
            const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
            reinterpret_cast<float4 *>(ks)[i] = in ? *reinterpret_cast<const float4 *>(kbase + ko) : zero;
            reinterpret_cast<float4 *>(vs)[i] = in ? *reinterpret_cast<const float4 *>(vbase + vo) : zero;
        }
        __syncthreads();

        for (int c0 = 0; c0 < kBlock; c0 += kChunk) {
            float s[kChunk];
#pragma unroll
            for (int j = 0; j < kChunk; ++j) {
                const float *kr = ks + (c0 + j) * D + part * kDimsPerThread;
                float dot = 0.f;
#pragma unroll
                for (int d = 0; d < kDimsPerThread; ++d) dot = fmaf(qr[d], kr[d], dot);
                if constexpr (C::kTpr == 2) dot += __shfl_xor_sync(0xffffffffu, dot, 1);
                const int kv = kv0 + c0 + j;
                float x = score_mod_f32(p.score_kind, p.score_param, dot * post, slope, q, kv);
                // tail tiles are never full; columns past KV_LEN are
                // masked before mask_mod could read a document id there
                if (!full && (kv >= p.kv_len || !row_in || !mask_mod(p.mask, b, q, kv))) x = -INFINITY;
                s[j] = x;
            }
            float cmax = s[0];
#pragma unroll
            for (int j = 1; j < kChunk; ++j) cmax = fmaxf(cmax, s[j]);
            const float m_new = fmaxf(m, cmax);
            if (m_new == -INFINITY) continue;  // nothing unmasked in this row yet
            const float alpha = expf(m - m_new);  // 0 when m was -inf
            l *= alpha;
#pragma unroll
            for (int d = 0; d < kDimsPerThread; ++d) acc[d] *= alpha;
            m = m_new;
#pragma unroll
            for (int j = 0; j < kChunk; ++j) {
                const float pj = expf(s[j] - m);
                l += pj;
                const float *vr = vs + (c0 + j) * D + part * kDimsPerThread;
#pragma unroll
                for (int d = 0; d < kDimsPerThread; ++d) acc[d] = fmaf(pj, vr[d], acc[d]);
            }
        }
    }

    float *op = static_cast<float *>(p.out) + (((int64_t)b * p.H + h) * p.q_len + q) * D + part * kDimsPerThread;
    if (!row_in) return;
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int d = 0; d < kDimsPerThread; d += 4)
        *reinterpret_cast<float4 *>(op + d) = make_float4(acc[d] * inv, acc[d + 1] * inv, acc[d + 2] * inv,
                                                          acc[d + 3] * inv);
    const int64_t orow = ((int64_t)b * p.H + h) * p.q_len + q;
    if (part == 0) p.lse[orow] = l > 0.f ? m + logf(l) : -INFINITY;
    if (part == 0 && p.row_max) p.row_max[orow] = m;  // exact running max (OUTPUT_MAX); -inf for an empty row
}

template <int D>
cudaError_t launch_d(const AttnProblem &p, cudaStream_t stream) {
    using C = Fp32Cfg<D>;
    cudaError_t e = cudaFuncSetAttribute(attn_fp32_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::kSmem);
    if (e != cudaSuccess) return e;
    // grid.y holds at most 65535 (b, h) pairs per launch
    for (int begin = 0; begin < p.bh_count; begin += 65535) {
        AttnProblem part = p;
        part.bh_begin = p.bh_begin + begin;
        part.bh_count = p.bh_count - begin < 65535 ? p.bh_count - begin : 65535;
        attn_fp32_kernel<D><<<dim3(p.nqt, part.bh_count), C::kThreads, C::kSmem, stream>>>(part);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_attn_fp32(const AttnProblem &p, cudaStream_t stream) {
    return p.D == 64 ? launch_d<64>(p, stream) : launch_d<128>(p, stream);
}

}  // namespace flex
