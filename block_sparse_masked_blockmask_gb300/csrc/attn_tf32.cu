// Block-sparse attention forward for float32 inputs on sm_103a tensor cores,
// with the float32 accuracy of the inputs kept by split TF32 (three MMAs per
// product).
//
// What it computes is the flex_attention op of "[Inductor][Flex Attention]
// Add Subtiling Option for Alpha Scaling" (PyTorch PR #167356) with
// OUTPUT_LOGSUMEXP, as on the bf16 path: s = score_mod(scale * q.k) on every
// listed tile, -inf where mask_mod is false (partial tiles only), online
// softmax (the forward_block_mn step: running max m, running sum
// l = l * alpha + sum(p), acc = acc * alpha + p V), out = acc / l,
// lse = m + ln l; a row with no unmasked score gets out = 0, lse = -inf.
//
// Split TF32: a tcgen05 MMA of kind::tf32 reads 19 bits of each float32
// operand.  Every operand x is written as hi = x with its low 13 mantissa
// bits cleared (exactly a TF32 value) and lo = x - hi (exact in float32,
// |lo| < 2^-10 |x|), and
//   S = Qhi Khi^T + Qhi Klo^T + Qlo Khi^T,   O += Phi Vhi + Phi Vlo + Plo Vhi
// accumulate in float32 in tensor memory; the dropped lo x lo terms and the
// TF32 reading of lo are below 2^-20 relative.  The softmax runs in float32
// with expf and an exact running max.
//
// Design (one CTA per (batch, head, 128-row q tile), 288 threads):
//   warps 0-3  softmax, one thread per q row (TMEM lane = row)
//   warps 4-7  loaders: read Q once and each kv sub-tile of K and V from
//              global memory, split them into hi and lo and write them into
//              shared memory in the layout the MMAs read (128-byte swizzled
//              rows, K-major; V is transposed on the way so that every
//              operand is K-major)
//   warp 8     one thread issues every tcgen05.mma
// The kv tiles of the BlockMask (any block sizes, read as 128-tiles) are
// walked in sub-tiles of KS kv rows (64 at D = 64, 32 at D = 128, so that Q,
// its lo part and a stage of K, V fit in shared memory).  Every wait is
// bounded; on timeout the CTA records FLEX_ERR_DEVICE_TIMEOUT in the status
// word, drains its MMAs, frees TMEM and exits.
#include <cfloat>

#include "flex_internal.h"
#include "ptx.cuh"
#include "tilelist.cuh"

namespace flex {
namespace {

constexpr int kT32Threads = 288;
constexpr int kT32MmaWarp = 8;
constexpr uint32_t kT32TmemCols = 256;

template <int D>
struct T32Cfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int KS = D == 64 ? 64 : 32;                 // kv rows per sub-step
    static constexpr int NS = D == 64 ? 2 : 1;                   // stages
    static constexpr int kSub = kBlock / KS;                     // sub-steps per 128-tile
    static constexpr uint32_t kQBytes = 128 * D * 4;             // Q hi (or lo): 128 rows x D
    static constexpr uint32_t kKBytes = KS * D * 4;              // K hi (or lo): KS rows x D
    static constexpr uint32_t kVBytes = D * KS * 4;              // V^T hi (or lo): D rows x KS
    static constexpr uint32_t kQAtom = 128 * 128;                // 32 floats of K-dim, all rows
    static constexpr uint32_t kKAtom = KS * 128;
    static constexpr uint32_t kVAtom = D * 128;
    static constexpr uint32_t kQhi = 0, kQlo = kQBytes;
    static constexpr uint32_t kStage0 = 2 * kQBytes;
    static constexpr uint32_t kStageBytes = 2 * kKBytes + 2 * kVBytes;  // Khi, Klo, Vhi^T, Vlo^T
    static constexpr uint32_t kMiscOff = kStage0 + NS * kStageBytes;
    // TMEM columns: S (then Phi) | Plo | O
    static constexpr uint32_t kS = 0, kPlo = KS, kO = 2 * KS;
    static_assert(2 * KS + D <= (int)kT32TmemCols, "tensor memory");
};

struct T32Misc {
    uint64_t q_ready, stage_full[2], stage_empty[2], s_full, p_full, o_full, drain;
    uint32_t tmem_base;
    int abort;
    int n;  // 128-tiles listed for this q tile
    int pad;
    alignas(16) uint32_t flags[kMaxKvBlocks];  // listed / full count per kv tile (tilelist.cuh)
    alignas(16) uint32_t list[kMaxKvBlocks];   // kv tile | full << 16, ascending
};

template <int D>
constexpr size_t t32_smem_bytes() {
    return T32Cfg<D>::kMiscOff + sizeof(T32Misc) + 1024;
}

// Offset of float group (row r, 4-float chunk c4 along the K dimension) in a
// K-major tile with 128-byte swizzled rows: atoms of 32 floats along K, each
// atom all rows x 128 bytes; 8-row groups 1024 bytes apart; the 16-byte
// chunk index of a row XORed with the row's index within its 8-row group
// (the layout a TMA load with 128-byte swizzle writes, and the one the
// matrix descriptors below describe).
__device__ __forceinline__ uint32_t sw128_offset(int r, int c4, uint32_t atom_bytes) {
    return (uint32_t)(c4 / 8) * atom_bytes + (uint32_t)(r / 8) * 1024u + (uint32_t)(r % 8) * 128u +
           (uint32_t)(((c4 % 8) ^ (r % 8)) * 16);
}

__device__ __forceinline__ float tf32_hi(float x) { return __uint_as_float(__float_as_uint(x) & 0xFFFFE000u); }

// Instruction descriptor, kind::tf32: f32 accumulator, TF32 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(uint32_t M, uint32_t N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

template <uint32_t A_HI, uint32_t B_HI>
__device__ __forceinline__ void mma_tf32_ss(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "mov.b64 da, {%1, %5};\n\t"
        "mov.b64 db, {%2, %6};\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], da, db, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(A_HI), "n"(B_HI)
        : "memory");
}

template <uint32_t B_HI>
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "mov.b64 db, {%2, %5};\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], db, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(B_HI)
        : "memory");
}

__device__ __forceinline__ void t32_fail(T32Misc &ms, int *status) {
    *reinterpret_cast<volatile int *>(&ms.abort) = 1;
    atomicCAS(status, 0, kDeviceTimeout);
}

// A wait taken by all 32 lanes of a warp, with one outcome for the warp.
__device__ __forceinline__ bool t32_warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        const int stop = (*abort != 0) || (global_timer_ns() - t0 > kWaitLimitNs);
        if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
}

__device__ __forceinline__ void t32_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

template <int D>
__global__ void __launch_bounds__(kT32Threads, 1) attn_tf32_kernel(AttnProblem p) {
    using C = T32Cfg<D>;
    constexpr int KS = C::KS, NS = C::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    T32Misc &ms = *reinterpret_cast<T32Misc *>(smem + C::kMiscOff);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int qt = blockIdx.x, bh = p.bh_begin + (int)blockIdx.y, h = bh % p.H, b = bh / p.H;
    const int q0 = qt * kBlock;

    if (threadIdx.x == 0) {
        mbar_init(&ms.q_ready, 128);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&ms.stage_full[s], 128);
            mbar_init(&ms.stage_empty[s], 1);
        }
        mbar_init(&ms.s_full, 1);
        mbar_init(&ms.p_full, 128);
        mbar_init(&ms.o_full, 1);
        mbar_init(&ms.drain, 1);
        ms.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        // the kv tiles of this q tile: the BlockMask's lists (any block sizes)
        // read as 128-tiles; counts clamped and malformed entries dropped
        const TileLists lists{p.kv_num, p.kv_idx, p.full_num, p.full_idx, p.nqb, p.nkvb, p.q_block, p.kv_block,
                              p.nkvt};
        for (int i = lane; i < p.nkvt; i += 32) ms.flags[i] = 0u;
        __syncwarp();
        tl_mark_warp(lists, bh, qt, 0, ms.flags, 0, p.nkvt, lane);
        __syncwarp();
        const uint32_t expect = tl_expect(lists);
        const unsigned lt = (1u << lane) - 1u;
        int cnt = 0;
        for (int base = 0; base < p.nkvt; base += 32) {
            const int i = base + lane;
            const uint32_t w = i < p.nkvt ? ms.flags[i] : 0u;
            const bool on = tl_listed(w, 0);
            const unsigned bal = __ballot_sync(0xffffffffu, on);
            if (on) ms.list[cnt + __popc(bal & lt)] = (uint32_t)i | (tl_full(expect, w, 0) ? (1u << 16) : 0u);
            cnt += __popc(bal);
        }
        if (lane == 0) ms.n = cnt;
    }
    if (warp == kT32MmaWarp) {
        tmem_alloc(&ms.tmem_base, kT32TmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ms.tmem_base;
    volatile int *abort_flag = &ms.abort;
    const int nsub = ms.n * C::kSub;  // kv sub-steps

    if (warp >= 4 && warp < 8) {
        // ------------------------------------------------------------ loaders
        const int lt = threadIdx.x - 128;
        const float *qbase = static_cast<const float *>(p.q) + b * p.q_stride[0] + h * p.q_stride[1];
        const float *kbase = static_cast<const float *>(p.k) + b * p.k_stride[0] + h * p.k_stride[1];
        const float *vbase = static_cast<const float *>(p.v) + b * p.v_stride[0] + h * p.v_stride[1];
        const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
        // Q: hi and lo, 128 rows x D; PRESCALE_QK multiplies by scale first (one rounding)
        for (int i = lt; i < 128 * D / 4; i += 128) {
            const int r = i / (D / 4), c4 = i % (D / 4);
            float4 x = q0 + r < p.q_len ? *reinterpret_cast<const float4 *>(qbase + (int64_t)(q0 + r) * p.q_stride[2] +
                                                                           4 * c4)
                                        : zero;
            if (p.prescale) {
                x.x = __fmul_rn(x.x, p.scale);
                x.y = __fmul_rn(x.y, p.scale);
                x.z = __fmul_rn(x.z, p.scale);
                x.w = __fmul_rn(x.w, p.scale);
            }
            const float4 hi = make_float4(tf32_hi(x.x), tf32_hi(x.y), tf32_hi(x.z), tf32_hi(x.w));
            const float4 lo = make_float4(x.x - hi.x, x.y - hi.y, x.z - hi.z, x.w - hi.w);
            const uint32_t off = sw128_offset(r, c4, C::kQAtom);
            *reinterpret_cast<float4 *>(smem + C::kQhi + off) = hi;
            *reinterpret_cast<float4 *>(smem + C::kQlo + off) = lo;
        }
        fence_proxy_async_smem();
        mbar_arrive(&ms.q_ready);
        bool ok = true;
        for (int u = 0; u < nsub; ++u) {
            const int s = u % NS;
            const uint32_t use = (uint32_t)(u / NS);
            if (use > 0 && !t32_warp_wait(&ms.stage_empty[s], (use - 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            const int kv0 = (int)(ms.list[u / C::kSub] & 0xFFFFu) * kBlock + (u % C::kSub) * KS;
            uint8_t *st = smem + C::kStage0 + s * C::kStageBytes;
            // K: KS rows x D, hi and lo
            for (int i = lt; i < KS * D / 4; i += 128) {
                const int r = i / (D / 4), c4 = i % (D / 4);
                const float4 x = kv0 + r < p.kv_len
                                     ? *reinterpret_cast<const float4 *>(kbase + (int64_t)(kv0 + r) * p.k_stride[2] +
                                                                         4 * c4)
                                     : zero;
                const float4 hi = make_float4(tf32_hi(x.x), tf32_hi(x.y), tf32_hi(x.z), tf32_hi(x.w));
                const float4 lo = make_float4(x.x - hi.x, x.y - hi.y, x.z - hi.z, x.w - hi.w);
                const uint32_t off = sw128_offset(r, c4, C::kKAtom);
                *reinterpret_cast<float4 *>(st + off) = hi;
                *reinterpret_cast<float4 *>(st + C::kKBytes + off) = lo;
            }
            // V transposed: V^T is D rows x KS (kv contiguous), hi and lo
            for (int i = lt; i < KS * D / 4; i += 128) {
                const int r = i / (D / 4), c4 = i % (D / 4);  // kv row r, head dims 4 c4 .. 4 c4 + 3
                const float4 x = kv0 + r < p.kv_len
                                     ? *reinterpret_cast<const float4 *>(vbase + (int64_t)(kv0 + r) * p.v_stride[2] +
                                                                         4 * c4)
                                     : zero;
                const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int d = 4 * c4 + e;
                    const uint32_t off = sw128_offset(d, r / 4, C::kVAtom) + (uint32_t)(r % 4) * 4u;
                    const float hi = tf32_hi(xs[e]);
                    *reinterpret_cast<float *>(st + 2 * C::kKBytes + off) = hi;
                    *reinterpret_cast<float *>(st + 2 * C::kKBytes + C::kVBytes + off) = xs[e] - hi;
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(&ms.stage_full[s]);
        }
        if (!ok) t32_fail(ms, p.status);
    } else if (warp == kT32MmaWarp) {
        // ---------------------------------------------------------------- MMA
        if (lane == 0 && nsub > 0) {
            constexpr uint32_t idesc_s = idesc_tf32_f32(128, KS);
            constexpr uint32_t idesc_o = idesc_tf32_f32(128, D);
            constexpr uint32_t kHi = smem_desc_hi_sw128(1024);
            const uint32_t qhi = smem_desc_lo(smem_u32(smem + C::kQhi), 16);
            const uint32_t qlo = smem_desc_lo(smem_u32(smem + C::kQlo), 16);
            bool ok = mbar_wait(&ms.q_ready, 0, abort_flag);
            for (int u = 0; ok && u < nsub; ++u) {
                const int s = u % NS;
                if (!mbar_wait(&ms.stage_full[s], (uint32_t)(u / NS) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t st = smem_u32(smem + C::kStage0 + s * C::kStageBytes);
                const uint32_t khi = smem_desc_lo(st, 16), klo = smem_desc_lo(st + C::kKBytes, 16);
                const uint32_t vhi = smem_desc_lo(st + 2 * C::kKBytes, 16);
                const uint32_t vlo = smem_desc_lo(st + 2 * C::kKBytes + C::kVBytes, 16);
                // S = Qhi Khi^T + Qhi Klo^T + Qlo Khi^T (K steps of 8 floats = 32 bytes)
#pragma unroll
                for (int k = 0; k < D / 8; ++k) {
                    const uint32_t oq = ((k / 4) * C::kQAtom + (k % 4) * 32) >> 4;
                    const uint32_t ok_ = ((k / 4) * C::kKAtom + (k % 4) * 32) >> 4;
                    mma_tf32_ss<kHi, kHi>(tmem + C::kS, qhi + oq, khi + ok_, idesc_s, k > 0 ? 1u : 0u);
                    mma_tf32_ss<kHi, kHi>(tmem + C::kS, qhi + oq, klo + ok_, idesc_s, 1u);
                    mma_tf32_ss<kHi, kHi>(tmem + C::kS, qlo + oq, khi + ok_, idesc_s, 1u);
                }
                mma_commit(&ms.s_full);
                if (!mbar_wait(&ms.p_full, (uint32_t)u & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                // O += Phi Vhi + Phi Vlo + Plo Vhi (P from TMEM, 8 kv columns per step)
#pragma unroll
                for (int k = 0; k < KS / 8; ++k) {
                    const uint32_t ov = ((k / 4) * C::kVAtom + (k % 4) * 32) >> 4;
                    const uint32_t acc0 = (u > 0 || k > 0) ? 1u : 0u;
                    mma_tf32_ts<kHi>(tmem + C::kO, tmem + C::kS + 8 * k, vhi + ov, idesc_o, acc0);
                    mma_tf32_ts<kHi>(tmem + C::kO, tmem + C::kS + 8 * k, vlo + ov, idesc_o, 1u);
                    mma_tf32_ts<kHi>(tmem + C::kO, tmem + C::kPlo + 8 * k, vhi + ov, idesc_o, 1u);
                }
                mma_commit(&ms.stage_empty[s]);
            }
            if (ok) mma_commit(&ms.o_full);
            if (!ok) t32_fail(ms, p.status);
            mma_commit(&ms.drain);  // every MMA issued above completes before TMEM is freed
            int never = 0;
            (void)mbar_wait(&ms.drain, 0, &never);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ------------------------------------------------------------ softmax
        const int t = threadIdx.x;
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        const int q = q0 + t;
        const bool row_in = q < p.q_len;
        const float post = p.prescale ? 1.f : p.scale;
        const float slope = exp2f(-8.f * (float)(h + 1) / (float)p.H);
        int doc_q = 0;
        if (p.mask.kind == FLEX_MASK_DOCUMENT && row_in) doc_q = p.mask.doc_ids[(int64_t)b * p.mask.doc_len + q];
        int lo = 0, hi = -1;  // the kept kv interval of an interval mask_mod
        if (p.mask.kind != FLEX_MASK_DOCUMENT && row_in) {
            mask_row_interval(p.mask, q, lo, hi);
            hi = min(hi, p.kv_len - 1);
        }
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int u = 0; u < nsub; ++u) {
            const uint32_t e = ms.list[u / C::kSub];
            const bool full = (e >> 16) & 1u;
            const int kv0 = (int)(e & 0xFFFFu) * kBlock + (u % C::kSub) * KS;
            if (!t32_warp_wait(&ms.s_full, (uint32_t)u & 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            float x[KS];
#pragma unroll
            for (int c0 = 0; c0 < KS; c0 += 32) {
                uint32_t r[32];
                t32_ld32(trow + C::kS + c0, r);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int kv = kv0 + c0 + j;
                    float s = __uint_as_float(r[j]) * post;
                    if (p.score_kind == FLEX_SCORE_SOFTCAP) s = p.score_param * tanhf(s / p.score_param);
                    else if (p.score_kind == FLEX_SCORE_ALIBI) s -= slope * (float)(q - kv);
                    if (!full) {
                        bool keep;
                        if (p.mask.kind == FLEX_MASK_DOCUMENT)
                            keep = row_in && kv <= q && kv < p.kv_len &&
                                   p.mask.doc_ids[(int64_t)b * p.mask.doc_len + kv] == doc_q;
                        else
                            keep = kv >= lo && kv <= hi;
                        if (!keep) s = -INFINITY;
                    }
                    x[c0 + j] = s;
                }
            }
            float mt = x[0];
#pragma unroll
            for (int j = 1; j < KS; ++j) mt = fmaxf(mt, x[j]);
            const float m_new = fmaxf(m, mt);
            // the previous sub-step's O update is complete (it was issued
            // before this S), so O can be rescaled in place
            const float alpha = m_new == -INFINITY ? 1.f : expf(m - m_new);  // 0 when m was -inf
            if (u > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    t32_ld32(trow + C::kO + c0, o);
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    tmem_st32(trow + C::kO + c0, o);
                }
            }
            m = m_new;
            float sum = 0.f;
#pragma unroll
            for (int c0 = 0; c0 < KS; c0 += 32) {
                uint32_t ph[32], pl[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float pj = m == -INFINITY ? 0.f : expf(x[c0 + j] - m);
                    sum += pj;
                    const float hj = tf32_hi(pj);
                    ph[j] = __float_as_uint(hj);
                    pl[j] = __float_as_uint(pj - hj);
                }
                tmem_st32(trow + C::kS + c0, ph);  // over S columns, all read above
                tmem_st32(trow + C::kPlo + c0, pl);
            }
            l = l * alpha + sum;
            tmem_wait_st();
            tc_fence_before_sync();
            mbar_arrive(&ms.p_full);
        }
        // ------------------------------------------------------------ epilogue
        bool have = ok && nsub > 0;
        if (have && !t32_warp_wait(&ms.o_full, 0, abort_flag)) {
            have = false;
            ok = false;
        }
        if (!ok) t32_fail(ms, p.status);
        if (ok) {
            tc_fence_after_sync();
            const int64_t orow = (int64_t)bh * p.q_len + (row_in ? q : 0);
            float *op = static_cast<float *>(p.out) + orow * D;
            const bool live = have && l > 0.f;
            const float inv = live ? 1.f / l : 0.f;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {  // every lane takes the warp-collective loads
                uint32_t o[32];
                if (have) {
                    t32_ld32(trow + C::kO + c0, o);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] = 0u;
                }
                if (row_in) {
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(op + c0 + j) =
                            make_float4(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv,
                                        __uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
                }
            }
            if (row_in) {
                p.lse[orow] = live ? m + logf(l) : -INFINITY;
                if (p.row_max) p.row_max[orow] = live ? m : -INFINITY;
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kT32MmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kT32TmemCols);
    }
}

template <int D>
cudaError_t launch_tf32_d(const AttnProblem &p, cudaStream_t stream) {
    const size_t smem = t32_smem_bytes<D>();
    cudaError_t e = cudaFuncSetAttribute(attn_tf32_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // grid.y holds at most 65535 (b, h) pairs per launch
    for (int begin = 0; begin < p.bh_count; begin += 65535) {
        AttnProblem part = p;
        part.bh_begin = p.bh_begin + begin;
        part.bh_count = p.bh_count - begin < 65535 ? p.bh_count - begin : 65535;
        attn_tf32_kernel<D><<<dim3(p.nqt, part.bh_count), kT32Threads, smem, stream>>>(part);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_attn_tf32(const AttnProblem &p, cudaStream_t stream) {
    return p.D == 64 ? launch_tf32_d<64>(p, stream) : launch_tf32_d<128>(p, stream);
}

}  // namespace flex
