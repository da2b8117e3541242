// Block-sparse attention forward for float32 inputs on sm_103a tensor cores,
// with the float32 accuracy of the inputs kept by a three-way bf16 split
// (six bf16 MMAs per product).
//
// What it computes is the flex_attention op of "[Inductor][Flex Attention]
// Add Subtiling Option for Alpha Scaling" (PyTorch PR #167356) with
// OUTPUT_LOGSUMEXP, as on the bf16 path: s = score_mod(scale * q.k) on every
// listed tile, -inf where mask_mod is false (partial tiles only), online
// softmax (the forward_block_mn step: running max m, running sum
// l = l * alpha + sum(p), acc = acc * alpha + p V), out = acc / l,
// lse = m + ln l; a row with no unmasked score gets out = 0, lse = -inf.
//
// Three-way split: every float32 operand x is written as x1 + x2 + x3 with
// x1 = bf16(x), x2 = bf16(x - x1), x3 = bf16(x - x1 - x2) (round to nearest;
// both differences are exact in float32), which leaves |x - x1 - x2 - x3|
// below about 2^-27 |x|.  A product a.b is then accumulated in float32 in
// tensor memory as
//   a1 b1 + a1 b2 + a2 b1 + a1 b3 + a2 b2 + a3 b1,
// the dropped terms a2 b3, a3 b2, a3 b3 being below 2^-23 |a| |b|: float32
// accuracy on the tcgen05 kind::f16 datapath.  A bf16 MMA does twice the
// work of a TF32 MMA of the same shape, so six of them cost what three
// split-TF32 MMAs cost; the bf16 parts take half the on-chip space, which
// lets S be computed 64 kv columns at a time and double-buffered (an MMA
// issue costs ~50 cycles whatever its width up to N = 64, so narrow S MMAs
// leave the tensor cores idle).
//
// Design (one CTA per (batch, head, 128-row q tile), 512 threads at D = 64,
// 480 at D = 128; the producer warps are placed away from the MMA issuers'
// sub-partitions, see F32Cfg; roles by group):
//   warps 0-3   softmax, one thread per q row (TMEM lane = row); at the start
//               they read their Q rows, split them and write Q1, Q2, Q3
//               (bf16 pairs) into tensor memory, where the S MMAs read them
//               as the A operand
//   K group     four warps: read each chunk of 64 kv rows of K from global
//               memory, split it and write the three parts into a
//               shared-memory ring (rows of 64 bf16 per 128-byte swizzled
//               atom, as a TMA load with 128-byte swizzle writes them); the
//               loads of a chunk are issued before its slot is waited for
//   V group     four warps: the same for V, in the same row layout, which
//               the PV MMAs read as an MN-major B operand (no transpose)
//   warp 12     one thread issues the MMAs; at D = 64 the PV MMAs only, and
//   warp 13     one thread the S MMAs (the fixed ~50-cycle cost of an MMA
//               issue on one thread overlaps the other's)
// Tensor memory (512 columns): Q1 | Q2 | Q3 | O | S0 | P3_0 | S1 | P3_1
// (| S2 | P3_2 at D = 64).  S of the next chunks is computed while the
// softmax works on chunk u; P1 and P2 (bf16 pairs) overwrite their S in
// place, P3 has its own columns; S(u + NB), NB the number of S buffers, is
// issued after PV(u) (one issuer: right behind it; two: once it has
// completed).  The softmax keeps a reference
// maximum m and rescales O and l only when a chunk's maximum exceeds m by
// more than kF32RescaleNats (then waiting for PV(u - 1)); out = O / l and
// lse = m + ln l do not depend on which m was used.  The kv tiles of the
// BlockMask (any block sizes, read as 128-tiles) are walked in chunks of 64
// kv rows.  CTAs take q tiles longest first.  Every wait is bounded; on
// timeout the CTA records FLEX_ERR_DEVICE_TIMEOUT in the status word, drains
// its MMAs, frees TMEM and exits.
#include <cfloat>

#include "bf16x3.cuh"
#include "flex_internal.h"
#include "ptx.cuh"
#include "tilelist.cuh"

namespace flex {
namespace {

constexpr int kF32MmaWarp = 12;  // issues the (PV) MMAs and allocates TMEM
constexpr int kF32SWarp = 13;    // D = 64: issues the S MMAs
constexpr int kF32MaxThreads = 16 * 32;  // launch bound: at most 128 registers a thread
constexpr uint32_t kF32TmemCols = 512;
constexpr int kF32KS = 64;                // kv rows per chunk
constexpr float kF32RescaleNats = 8.0f;   // O and l are rescaled when the maximum grows by more
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct F32Cfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int KS = kF32KS;
    static constexpr int kSub = kBlock / KS;               // chunks per 128-tile
    static constexpr int kSlots = D == 128 ? 2 : 3;        // ring depth, K and V alike
    // two MMA issuers at D = 64 (S and PV MMAs, each ~50 cycles of fixed
    // issue cost at N = 64, overlap); one at D = 128, where PV's N = 128
    // MMAs keep the tensor pipe busy and S(u + 2) is better issued right
    // behind PV(u) than after a wait for its completion
    static constexpr bool kTwoIssuers = D == 64;
    // unroll of the K-step loops that issue the MMAs: rolled at D = 64, where
    // two issuers and the softmax warps share the instruction cache (measured
    // 6 % faster), unrolled at D = 128 (rolled measured 7 % slower)
    static constexpr int kUnrollK = D == 64 ? 1 : 8;
    // S/P buffers in TMEM: with two issuers S(j) must wait for PV(j - NB)
    // to complete, so each buffer is a chain S -> softmax -> PV -> S; three
    // buffers at D = 64 run three such chains at once (TMEM: 448 columns),
    // two at D = 128 (512)
    static constexpr int kSBufs = D == 64 ? 3 : 2;
    // Warp roles.  Warps are dealt to the four sub-partitions round robin
    // (warp w on sub-partition w % 4), and a thread issuing MMAs slows down
    // when its sub-partition is busy (~50 cycles an MMA alone, ~75 beside a
    // TMEM-traffic warp and a shared-memory-store warp).  D = 128: the
    // issuer (warp 12) shares its sub-partition only with softmax warp 0,
    // warps 4 and 8 stay idle, the producers run on warps 5-7, 9 (K) and
    // 10, 11, 13, 14 (V).  D = 64: PV issuer 12 and S issuer 13 each beside
    // one producer warp (V on 4, 5, 14, 15; K on 6, 7, 10, 11; 8 and 9 idle).
    static constexpr int kWarps = D == 128 ? 15 : 16;
    __device__ static int k_index(int w) {
        if (D == 64) return w == 6 || w == 7 ? w - 6 : w == 10 || w == 11 ? w - 8 : -1;
        return w >= 5 && w < 8 ? w - 5 : w == 9 ? 3 : -1;
    }
    __device__ static int v_index(int w) {
        if (D == 64) return w == 14 || w == 15 ? w - 14 : w == 4 || w == 5 ? w - 2 : -1;
        return w == 10 || w == 11 ? w - 10 : w == 13 || w == 14 ? w - 11 : -1;
    }
    static constexpr int kUnits = KS * D / 8 / 128;        // 8-float units per producer thread per chunk
    static constexpr uint32_t kAtom = KS * 128;            // 64 bf16 of a row, all KS rows
    static constexpr uint32_t kPart = KS * D * 2;          // one bf16 part of a chunk
    static constexpr uint32_t kSlot = 3 * kPart;           // parts 1 | 2 | 3
    static constexpr uint32_t kK0 = 0, kV0 = kSlots * kSlot;
    static constexpr uint32_t kMiscOff = 2 * kSlots * kSlot;
    // tensor memory columns (a column holds a bf16 pair of an A operand)
    __host__ __device__ static constexpr uint32_t q_col(int j) { return (uint32_t)(j * D / 2); }
    static constexpr uint32_t kO = 3 * D / 2;
    __host__ __device__ static constexpr uint32_t s_col(int i) { return 5 * D / 2 + (uint32_t)i * (KS + KS / 2); }
    __host__ __device__ static constexpr uint32_t p_col(int i, int j) {
        return j < 2 ? s_col(i) + (uint32_t)j * (KS / 2) : s_col(i) + KS;
    }
    static_assert(5 * D / 2 + kSBufs * (KS + KS / 2) <= (int)kF32TmemCols, "tensor memory");
    static_assert(kMiscOff % 1024 == 0, "ring alignment");
};

struct F32Misc {
    uint64_t q_ready, k_full[3], k_empty[3], v_full[3], v_empty[3];
    // per S/P buffer; pv_done[b]: the PV MMAs that read buffer b, so that
    // every parity wait on it is at most one phase behind
    uint64_t s_full[3], p_full[3], pv_done[3], o_full, drain;  // drain: one commit per issuing thread
    uint32_t tmem_base;
    int abort;
    int n;  // 128-tiles listed for this q tile
    int pad;
    alignas(16) uint32_t flags[kMaxKvBlocks];  // listed / full count per kv tile (tilelist.cuh)
    alignas(16) uint32_t list[kMaxKvBlocks];   // kv tile | full << 16, ascending
};

template <int D>
constexpr size_t f32_smem_bytes() {
    return F32Cfg<D>::kMiscOff + sizeof(F32Misc) + 1024;
}

__device__ __forceinline__ void f32_fail(F32Misc &ms, int *status) {
    *reinterpret_cast<volatile int *>(&ms.abort) = 1;
    atomicCAS(status, 0, kDeviceTimeout);
}

// One producer group (four warps, thread lt in 0..127): each chunk of KS kv
// rows of a [.., kv, D] float32 tensor is split and written, part j at
// slot + j * kPart, in 128-byte swizzled rows.  Thread lt takes units
// i = lt + 128 u (row i / (D/8), 8 floats at column 8 (i % (D/8))): a warp's
// loads are whole rows, a quarter warp's stores hit eight distinct 16-byte
// bank groups.  Not inlined: the K and V groups run one copy of the code.
template <int D>
__device__ __noinline__ bool f32_produce(F32Misc &ms, uint8_t *ring, uint64_t *full, uint64_t *empty,
                                            const float *base, int64_t row_stride, int kv_len, int nsub, int lt,
                                            int lane, volatile int *abort_flag) {
    using C = F32Cfg<D>;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int u = 0; u < nsub; ++u) {
        const int kv0 = (int)(ms.list[u / C::kSub] & 0xFFFFu) * kBlock + (u % C::kSub) * C::KS;
        float4 x[2 * C::kUnits];
#pragma unroll
        for (int j = 0; j < C::kUnits; ++j) {
            const int i = lt + 128 * j, r = i / (D / 8), c = i % (D / 8);
            const float4 *src = reinterpret_cast<const float4 *>(base + (int64_t)(kv0 + r) * row_stride) + 2 * c;
            const bool in = kv0 + r < kv_len;
            x[2 * j] = in ? __ldg(src) : zero;
            x[2 * j + 1] = in ? __ldg(src + 1) : zero;
        }
        const int s = u % C::kSlots;
        const uint32_t use = (uint32_t)(u / C::kSlots);
        if (use > 0 && !f32_warp_wait(&empty[s], (use - 1) & 1u, abort_flag)) return false;
        uint8_t *slot = ring + s * C::kSlot;
#pragma unroll
        for (int j = 0; j < C::kUnits; ++j) {
            const int i = lt + 128 * j, r = i / (D / 8), c = i % (D / 8);
            uint4 p1, p2, p3;
            split3(x[2 * j].x, x[2 * j].y, p1.x, p2.x, p3.x);
            split3(x[2 * j].z, x[2 * j].w, p1.y, p2.y, p3.y);
            split3(x[2 * j + 1].x, x[2 * j + 1].y, p1.z, p2.z, p3.z);
            split3(x[2 * j + 1].z, x[2 * j + 1].w, p1.w, p2.w, p3.w);
            const uint32_t off = sw128_chunk(r, c, C::kAtom);
            *reinterpret_cast<uint4 *>(slot + off) = p1;
            *reinterpret_cast<uint4 *>(slot + C::kPart + off) = p2;
            *reinterpret_cast<uint4 *>(slot + 2 * C::kPart + off) = p3;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
    }
    return true;
}

template <int D, int SCORE, bool DOC>
__global__ void __launch_bounds__(kF32MaxThreads, 1) attn_fp32_kernel(AttnProblem p, int bh_major) {
    using C = F32Cfg<D>;
    constexpr int KS = C::KS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    F32Misc &ms = *reinterpret_cast<F32Misc *>(smem + C::kMiscOff);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // longest first: under a causal mask the last q tiles list the most kv tiles
    const int qt = p.nqt - 1 - (int)(bh_major ? blockIdx.y : blockIdx.x);
    const int bh = p.bh_begin + (int)(bh_major ? blockIdx.x : blockIdx.y), h = bh % p.H, b = bh / p.H;
    const int q0 = qt * kBlock;

    if (threadIdx.x == 0) {
        mbar_init(&ms.q_ready, 4);
        for (int s = 0; s < C::kSlots; ++s) {
            mbar_init(&ms.k_full[s], 4);
            mbar_init(&ms.k_empty[s], 1);
            mbar_init(&ms.v_full[s], 4);
            mbar_init(&ms.v_empty[s], 1);
        }
        for (int i = 0; i < C::kSBufs; ++i) {
            mbar_init(&ms.s_full[i], 1);
            mbar_init(&ms.p_full[i], 4);
            mbar_init(&ms.pv_done[i], 1);
        }
        mbar_init(&ms.o_full, 1);
        mbar_init(&ms.drain, C::kTwoIssuers ? 2 : 1);
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
    if (warp == kF32MmaWarp) {
        tmem_alloc(&ms.tmem_base, kF32TmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ms.tmem_base;
    volatile int *abort_flag = &ms.abort;
    const int nsub = ms.n * C::kSub;  // kv chunks

    const int kidx = C::k_index(warp), vidx = C::v_index(warp);
    if (kidx >= 0) {
        // --------------------------------------------------------- K producers
        const float *kbase = static_cast<const float *>(p.k) + b * p.k_stride[0] + h * p.k_stride[1];
        if (!f32_produce<D>(ms, smem + C::kK0, ms.k_full, ms.k_empty, kbase, p.k_stride[2], p.kv_len, nsub,
                            32 * kidx + lane, lane, abort_flag))
            f32_fail(ms, p.status);
    } else if (vidx >= 0) {
        // --------------------------------------------------------- V producers
        const float *vbase = static_cast<const float *>(p.v) + b * p.v_stride[0] + h * p.v_stride[1];
        if (!f32_produce<D>(ms, smem + C::kV0, ms.v_full, ms.v_empty, vbase, p.v_stride[2], p.kv_len, nsub,
                            32 * vidx + lane, lane, abort_flag))
            f32_fail(ms, p.status);
    } else if (warp == kF32MmaWarp || (C::kTwoIssuers && warp == kF32SWarp)) {
        // ---------------------------------------------------------------- MMA
        if (lane == 0 && nsub > 0) {
            constexpr uint32_t kHi = smem_desc_hi_sw128(1024);
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, KS, 0, 0);
            constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, 0, 1);
            // the six part products t, first the largest: (A part, B part) =
            // (0,0) (0,1) (1,0) (0,2) (1,1) (2,0)
            auto pa = [](int t) { return t == 2 || t == 4 ? 1 : t == 5 ? 2 : 0; };
            auto pbp = [](int t) { return t == 1 || t == 4 ? 1 : t == 3 ? 2 : 0; };
            // S(j) = sum of the part products Q_a K_b^T into S buffer j % 2;
            // K is K-major (K steps of 16 bf16 = 32 bytes within a 64-wide atom)
            auto issue_s = [&](int j) -> bool {
                const int s = j % C::kSlots;
                if (!mbar_wait(&ms.k_full[s], (uint32_t)(j / C::kSlots) & 1u, abort_flag)) return false;
                tc_fence_after_sync();
                const uint32_t kd = smem_desc_lo(smem_u32(smem + C::kK0 + s * C::kSlot), 16);
                const uint32_t d = tmem + C::s_col(j % C::kSBufs);
#pragma unroll(C::kUnrollK)
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = ((k / 4) * C::kAtom + (k % 4) * 32) >> 4;
#pragma unroll
                    for (int t = 0; t < 6; ++t)
                        mma_ts_lo<kHi>(d, tmem + C::q_col(pa(t)) + 8 * k, kd + ((pbp(t) * C::kPart) >> 4) + off,
                                       idesc_s, (k > 0 || t > 0) ? 1u : 0u);
                }
                mma_commit(&ms.k_empty[s]);
                mma_commit(&ms.s_full[j % C::kSBufs]);
                return true;
            };
            // O += sum of the part products P_a V_b; V is MN-major (kv rows of
            // 64 head-dim elements, the 64-wide halves kAtom apart), K steps
            // of 16 kv rows = 2048 bytes
            auto issue_pv = [&](int u) -> bool {
                const int pb = u % C::kSBufs, s = u % C::kSlots;
                if (!mbar_wait(&ms.p_full[pb], (uint32_t)(u / C::kSBufs) & 1u, abort_flag) ||
                    !mbar_wait(&ms.v_full[s], (uint32_t)(u / C::kSlots) & 1u, abort_flag))
                    return false;
                tc_fence_after_sync();
                const uint32_t vd = smem_desc_lo(smem_u32(smem + C::kV0 + s * C::kSlot), C::kAtom);
#pragma unroll(C::kUnrollK)
                for (int k = 0; k < KS / 16; ++k) {
#pragma unroll
                    for (int t = 0; t < 6; ++t)
                        mma_ts_lo<kHi>(tmem + C::kO, tmem + C::p_col(pb, pa(t)) + 8 * k,
                                       vd + ((pbp(t) * C::kPart + k * 2048) >> 4), idesc_o,
                                       (u > 0 || k > 0 || t > 0) ? 1u : 0u);
                }
                mma_commit(&ms.v_empty[s]);
                mma_commit(&ms.pv_done[pb]);
                return true;
            };
            bool ok = true;
            if (!C::kTwoIssuers) {
                // one issuer: S of the first kSBufs chunks, then PV(u) and
                // S(u + kSBufs) (MMAs of one thread run in order, so
                // S(u + kSBufs) follows PV(u), which read the same buffer)
                ok = mbar_wait(&ms.q_ready, 0, abort_flag);
                if (ok) tc_fence_after_sync();
                for (int j = 0; ok && j < min(nsub, C::kSBufs); ++j) ok = issue_s(j);
                for (int u = 0; ok && u < nsub; ++u)
                    ok = issue_pv(u) && (u + C::kSBufs >= nsub || issue_s(u + C::kSBufs));
                if (ok) mma_commit(&ms.o_full);
            } else if (warp == kF32SWarp) {
                // S(j) overwrites the buffer PV(j - kSBufs) read its P from
                ok = mbar_wait(&ms.q_ready, 0, abort_flag);
                for (int j = 0; ok && j < nsub; ++j) {
                    if (j >= C::kSBufs &&
                        !mbar_wait(&ms.pv_done[j % C::kSBufs], (uint32_t)(j / C::kSBufs - 1) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    ok = issue_s(j);
                }
            } else {
                for (int u = 0; ok && u < nsub; ++u) ok = issue_pv(u);
                if (ok) mma_commit(&ms.o_full);
            }
            if (!ok) f32_fail(ms, p.status);
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
        const float slope = SCORE == FLEX_SCORE_ALIBI ? exp2f(-8.f * (float)(h + 1) / (float)p.H) : 0.f;
        int doc_q = 0;
        if (DOC && row_in) doc_q = p.mask.doc_ids[(int64_t)b * p.mask.doc_len + q];
        int lo = 0, hi = -1;  // the kept kv interval of an interval mask_mod
        if (!DOC && row_in) {
            mask_row_interval(p.mask, q, lo, hi);
            hi = min(hi, p.kv_len - 1);
        }
        bool ok = true;
        if (nsub > 0) {
            // Q row -> Q1, Q2, Q3 columns of this lane (bf16 pairs);
            // PRESCALE_QK multiplies by scale first (one rounding)
            const float *qrow = static_cast<const float *>(p.q) + b * p.q_stride[0] + h * p.q_stride[1] +
                                (int64_t)(row_in ? q : 0) * p.q_stride[2];
            const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {  // 8 loads in flight, then 16 columns of each part
                float4 x[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    x[j] = row_in ? __ldg(reinterpret_cast<const float4 *>(qrow + c0) + j) : zero;
                uint32_t w1[16], w2[16], w3[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    float a = f4_at(x[j / 2], 2 * (j % 2)), c = f4_at(x[j / 2], 2 * (j % 2) + 1);
                    if (p.prescale) {
                        a = __fmul_rn(a, p.scale);
                        c = __fmul_rn(c, p.scale);
                    }
                    split3(a, c, w1[j], w2[j], w3[j]);
                }
                const uint32_t col = (uint32_t)c0 / 2;
                tmem_st16(trow + C::q_col(0) + col, w1);
                tmem_st16(trow + C::q_col(1) + col, w2);
                tmem_st16(trow + C::q_col(2) + col, w3);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.q_ready);
        }
        float m = -INFINITY, m_true = -INFINITY, l = 0.f;
        for (int u = 0; u < nsub; ++u) {
            const int pb = u % C::kSBufs;
            const uint32_t e = ms.list[u / C::kSub];
            const bool full = (e >> 16) & 1u;
            const int kv0 = (int)(e & 0xFFFFu) * kBlock + (u % C::kSub) * KS;
            if (!f32_warp_wait(&ms.s_full[pb], (uint32_t)(u / C::kSBufs) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            float x[KS];
#pragma unroll
            for (int c0 = 0; c0 < KS; c0 += 32) {
                uint32_t r[32];
                f32_ld32(trow + C::s_col(pb) + c0, r);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int kv = kv0 + c0 + j;
                    float s = __uint_as_float(r[j]) * post;
                    if constexpr (SCORE == FLEX_SCORE_SOFTCAP) s = p.score_param * tanhf(s / p.score_param);
                    if constexpr (SCORE == FLEX_SCORE_ALIBI) s -= slope * (float)(q - kv);
                    if (!full) {
                        bool keep;
                        if constexpr (DOC)
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
            m_true = fmaxf(m_true, mt);
            // the reference maximum moves only when this chunk's exceeds it by
            // more than kF32RescaleNats (so p <= e^8); from -inf it moves to
            // the first finite maximum
            const bool grow = mt > m + kF32RescaleNats;
            if (__any_sync(0xffffffffu, grow)) {
                const float m_new = grow ? mt : m;
                const float alpha = grow ? expf(m - m_new) : 1.f;  // 0 when m was -inf
                if (u > 0) {
                    // PV(u - 1) has completed before O is rescaled in place
                    const int pv = (u - 1) % C::kSBufs;  // PV(u - 1) and, in order, every PV before it
                    if (!f32_warp_wait(&ms.pv_done[pv], (uint32_t)((u - 1) / C::kSBufs) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        f32_ld32(trow + C::kO + c0, o);
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                        tmem_st32(trow + C::kO + c0, o);
                    }
                }
                l *= alpha;
                m = m_new;
            }
            // p = e^(s - m) = 2^(s log2 e - m log2 e); a row with m = -inf has
            // every s = -inf and gets p = 2^-inf = 0
            const float mb = m == -INFINITY ? 0.f : m * kLog2e;
            float sum = 0.f;
#pragma unroll
            for (int c0 = 0; c0 < KS; c0 += 16) {  // 16 columns at a time: x is consumed as P is stored
                uint32_t w1[8], w2[8], w3[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float pa = ex2_approx(fmaf(x[c0 + 2 * j], kLog2e, -mb));
                    const float pc = ex2_approx(fmaf(x[c0 + 2 * j + 1], kLog2e, -mb));
                    sum += pa + pc;
                    split3(pa, pc, w1[j], w2[j], w3[j]);
                }
                const uint32_t col = (uint32_t)c0 / 2;
                f32_st8(trow + C::p_col(pb, 0) + col, w1);  // over S columns, all read above
                f32_st8(trow + C::p_col(pb, 1) + col, w2);
                f32_st8(trow + C::p_col(pb, 2) + col, w3);
            }
            l += sum;
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.p_full[pb]);
        }
        // ------------------------------------------------------------ epilogue
        bool have = ok && nsub > 0;
        if (have && !f32_warp_wait(&ms.o_full, 0, abort_flag)) {
            have = false;
            ok = false;
        }
        if (!ok) f32_fail(ms, p.status);
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
                    f32_ld32(trow + C::kO + c0, o);
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
                if (p.row_max) p.row_max[orow] = live ? m_true : -INFINITY;
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kF32MmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kF32TmemCols);
    }
}

template <int D, int SCORE, bool DOC>
cudaError_t launch_fp32_kernel(const AttnProblem &p, cudaStream_t stream) {
    using C = F32Cfg<D>;
    const size_t smem = f32_smem_bytes<D>();
    auto kern = attn_fp32_kernel<D, SCORE, DOC>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (p.nqt <= 65535) {
        // (b, h) pairs along x, q tiles (longest first) along y: the first
        // CTAs to run are the longest of every pair
        kern<<<dim3(p.bh_count, p.nqt), C::kWarps * 32, smem, stream>>>(p, 1);
        return cudaGetLastError();
    }
    // grid.y holds at most 65535 (b, h) pairs per launch
    for (int begin = 0; begin < p.bh_count; begin += 65535) {
        AttnProblem part = p;
        part.bh_begin = p.bh_begin + begin;
        part.bh_count = p.bh_count - begin < 65535 ? p.bh_count - begin : 65535;
        kern<<<dim3(p.nqt, part.bh_count), C::kWarps * 32, smem, stream>>>(part, 0);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int D, bool DOC>
cudaError_t launch_fp32_score(const AttnProblem &p, cudaStream_t stream) {
    switch (p.score_kind) {
        case FLEX_SCORE_SOFTCAP:
            return launch_fp32_kernel<D, FLEX_SCORE_SOFTCAP, DOC>(p, stream);
        case FLEX_SCORE_ALIBI:
            return launch_fp32_kernel<D, FLEX_SCORE_ALIBI, DOC>(p, stream);
        default:
            return launch_fp32_kernel<D, FLEX_SCORE_IDENTITY, DOC>(p, stream);
    }
}

template <int D>
cudaError_t launch_fp32_d(const AttnProblem &p, cudaStream_t stream) {
    return p.mask.kind == FLEX_MASK_DOCUMENT ? launch_fp32_score<D, true>(p, stream)
                                             : launch_fp32_score<D, false>(p, stream);
}

}  // namespace

cudaError_t launch_attn_fp32(const AttnProblem &p, cudaStream_t stream) {
    return p.D == 64 ? launch_fp32_d<64>(p, stream) : launch_fp32_d<128>(p, stream);
}

}  // namespace flex
