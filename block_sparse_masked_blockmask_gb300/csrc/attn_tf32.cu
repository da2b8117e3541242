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
// Design (one CTA per (batch, head, 128-row q tile), 416 threads):
//   warps 0-3   softmax, one thread per q row (TMEM lane = row); at the start
//               they read their Q rows, split them and write Qhi and Qlo into
//               tensor memory, where the S MMAs read them as the A operand
//   warps 4-7   K producers: read each kv chunk of KS rows of K from global
//               memory, split it into hi and lo and write both into a
//               three-slot shared-memory ring (128-byte swizzled rows,
//               K-major), the loads of chunk u + 1 issued before chunk u is
//               stored
//   warps 8-11  V producers: the same for V, transposed on the way (V^T,
//               kv contiguous) so that every operand is K-major; each thread
//               holds a 4 x 4 block (4 kv rows x 4 head dims) and writes it
//               as four 16-byte V^T pieces, the lanes of a quarter warp
//               spread over all eight 16-byte bank groups
//   warp 12     one thread issues every tcgen05.mma
// Tensor memory (512 columns): Qhi | Qlo | O | S0 | Plo0 | S1 | Plo1.  S of
// chunk u + 1 is computed while the softmax works on chunk u (two S
// buffers; P hi overwrites its S in place, P lo has its own columns), and
// the MMA thread issues PV(u) and then S(u + 2).  The softmax keeps a
// reference maximum m and rescales O and l only when a chunk's maximum
// exceeds m by more than kT32RescaleNats (then waiting for PV(u - 1));
// out = O / l and lse = m + ln l do not depend on which m was used.  The kv
// tiles of the BlockMask (any block sizes, read as 128-tiles) are walked in
// chunks of KS kv rows (32 at D = 128, 64 at D = 64).  CTAs take q tiles
// longest first.  Every wait is bounded; on timeout the CTA records
// FLEX_ERR_DEVICE_TIMEOUT in the status word, drains its MMAs, frees TMEM
// and exits.
#include <cfloat>

#include "flex_internal.h"
#include "ptx.cuh"
#include "tilelist.cuh"

namespace flex {
namespace {

constexpr int kT32KWarp = 4;      // first of the four K producer warps
constexpr int kT32VWarp = 8;      // first of the four V producer warps
constexpr int kT32MmaWarp = 12;
constexpr int kT32Threads = 13 * 32;
constexpr uint32_t kT32TmemCols = 512;
constexpr int kT32Slots = 3;                // ring depth, K and V alike
constexpr float kT32RescaleNats = 8.0f;     // O and l are rescaled when the maximum grows by more

template <int D>
struct T32Cfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int KS = D == 64 ? 64 : 32;       // kv rows per chunk
    static constexpr int kSub = kBlock / KS;            // chunks per 128-tile
    static constexpr int kPer = KS * D / 4 / 128;       // float4 per producer thread per chunk
    static constexpr uint32_t kHalf = KS * D * 4;       // the hi (or lo) part of a K or V^T chunk
    static constexpr uint32_t kSlot = 2 * kHalf;        // hi | lo
    static constexpr uint32_t kKAtom = KS * 128;        // K chunk: 32 floats of head dim, all KS rows
    static constexpr uint32_t kVAtom = D * 128;         // V^T chunk: 32 kv floats, all D rows
    static constexpr uint32_t kK0 = 0, kV0 = kT32Slots * kSlot;
    static constexpr uint32_t kMiscOff = 2 * kT32Slots * kSlot;
    // tensor memory columns
    static constexpr uint32_t kQhi = 0, kQlo = D, kO = 2 * D;
    __host__ __device__ static constexpr uint32_t s_col(int i) { return 3 * D + 2 * KS * i; }
    __host__ __device__ static constexpr uint32_t plo_col(int i) { return 3 * D + 2 * KS * i + KS; }
    static_assert(3 * D + 4 * KS <= (int)kT32TmemCols, "tensor memory");
    static_assert(kPer == 8, "producer mapping: 8 float4 per thread per chunk");
};

struct T32Misc {
    uint64_t q_ready, k_full[kT32Slots], k_empty[kT32Slots], v_full[kT32Slots], v_empty[kT32Slots];
    uint64_t s_full[2], p_full[2], pv_done, o_full, drain;
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

__device__ __forceinline__ float f4_at(const float4 &v, int e) {
    return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

// hi and lo of four floats, written to `dst` and `dst + lo_off` (16 bytes each)
__device__ __forceinline__ void t32_put_split(uint8_t *dst, uint32_t lo_off, float4 x) {
    const float4 hi = make_float4(tf32_hi(x.x), tf32_hi(x.y), tf32_hi(x.z), tf32_hi(x.w));
    *reinterpret_cast<float4 *>(dst) = hi;
    *reinterpret_cast<float4 *>(dst + lo_off) = make_float4(x.x - hi.x, x.y - hi.y, x.z - hi.z, x.w - hi.w);
}

template <int D>
__global__ void __launch_bounds__(kT32Threads, 1) attn_tf32_kernel(AttnProblem p, int bh_major) {
    using C = T32Cfg<D>;
    constexpr int KS = C::KS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    T32Misc &ms = *reinterpret_cast<T32Misc *>(smem + C::kMiscOff);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // longest first: under a causal mask the last q tiles list the most kv tiles
    const int qt = p.nqt - 1 - (int)(bh_major ? blockIdx.y : blockIdx.x);
    const int bh = p.bh_begin + (int)(bh_major ? blockIdx.x : blockIdx.y), h = bh % p.H, b = bh / p.H;
    const int q0 = qt * kBlock;

    if (threadIdx.x == 0) {
        mbar_init(&ms.q_ready, 4);
        for (int s = 0; s < kT32Slots; ++s) {
            mbar_init(&ms.k_full[s], 4);
            mbar_init(&ms.k_empty[s], 1);
            mbar_init(&ms.v_full[s], 4);
            mbar_init(&ms.v_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ms.s_full[i], 1);
            mbar_init(&ms.p_full[i], 4);
        }
        mbar_init(&ms.pv_done, 1);
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
    const int nsub = ms.n * C::kSub;  // kv chunks
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    auto chunk_kv0 = [&](int u) { return (int)(ms.list[u / C::kSub] & 0xFFFFu) * kBlock + (u % C::kSub) * KS; };

    if (warp >= kT32KWarp && warp < kT32KWarp + 4) {
        // --------------------------------------------------------- K producers
        // thread lt holds rows lt / (D/4) + 128 j / (D/4), float4 column lt % (D/4):
        // a warp's loads are whole rows, its stores one 16-byte chunk per bank group
        const int lt = threadIdx.x - 32 * kT32KWarp;
        const float *kbase = static_cast<const float *>(p.k) + b * p.k_stride[0] + h * p.k_stride[1];
        auto load = [&](int u, float4 (&x)[C::kPer]) {
            const int kv0 = chunk_kv0(u);
#pragma unroll
            for (int j = 0; j < C::kPer; ++j) {
                const int i = lt + 128 * j, r = i / (D / 4), c4 = i % (D / 4);
                x[j] = kv0 + r < p.kv_len
                           ? __ldg(reinterpret_cast<const float4 *>(kbase + (int64_t)(kv0 + r) * p.k_stride[2]) + c4)
                           : zero;
            }
        };
        float4 cur[C::kPer], nxt[C::kPer];
        if (nsub > 0) load(0, cur);
        bool ok = true;
        for (int u = 0; u < nsub; ++u) {
            if (u + 1 < nsub) load(u + 1, nxt);
            const int s = u % kT32Slots;
            const uint32_t use = (uint32_t)(u / kT32Slots);
            if (use > 0 && !t32_warp_wait(&ms.k_empty[s], (use - 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            uint8_t *slot = smem + C::kK0 + s * C::kSlot;
#pragma unroll
            for (int j = 0; j < C::kPer; ++j) {
                const int i = lt + 128 * j, r = i / (D / 4), c4 = i % (D / 4);
                t32_put_split(slot + sw128_offset(r, c4, C::kKAtom), C::kHalf, cur[j]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.k_full[s]);
#pragma unroll
            for (int j = 0; j < C::kPer; ++j) cur[j] = nxt[j];
        }
        if (!ok) t32_fail(ms, p.status);
    } else if (warp >= kT32VWarp && warp < kT32VWarp + 4) {
        // --------------------------------------------------------- V producers
        // Warp tile t (of (KS / 16) x (D / 32)): 16 kv rows x 32 head dims.
        // Lane = (row quad rq: 2 bits, float4 column: 3 bits); a thread loads
        // 4 rows of one float4 column and stores 4 V^T pieces (one head dim,
        // 4 kv each).  A quarter warp covers 4 row quads x 2 columns, whose
        // pieces land in 8 distinct 16-byte bank groups of the swizzled rows.
        const int vw = warp - kT32VWarp;
        const float *vbase = static_cast<const float *>(p.v) + b * p.v_stride[0] + h * p.v_stride[1];
        constexpr int kColTiles = D / 32;
        auto unit = [&](int jt, int &rq, int &c4) {
            const int t = vw + 4 * jt;
            rq = (t / kColTiles) * 4 + (lane & 3);
            c4 = (t % kColTiles) * 8 + (lane >> 2);
        };
        auto load = [&](int u, float4 (&x)[C::kPer]) {
            const int kv0 = chunk_kv0(u);
#pragma unroll
            for (int jt = 0; jt < 2; ++jt) {
                int rq, c4;
                unit(jt, rq, c4);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int r = 4 * rq + jj;
                    x[4 * jt + jj] =
                        kv0 + r < p.kv_len
                            ? __ldg(reinterpret_cast<const float4 *>(vbase + (int64_t)(kv0 + r) * p.v_stride[2]) + c4)
                            : zero;
                }
            }
        };
        float4 cur[C::kPer], nxt[C::kPer];
        if (nsub > 0) load(0, cur);
        bool ok = true;
        for (int u = 0; u < nsub; ++u) {
            if (u + 1 < nsub) load(u + 1, nxt);
            const int s = u % kT32Slots;
            const uint32_t use = (uint32_t)(u / kT32Slots);
            if (use > 0 && !t32_warp_wait(&ms.v_empty[s], (use - 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            uint8_t *slot = smem + C::kV0 + s * C::kSlot;
#pragma unroll
            for (int jt = 0; jt < 2; ++jt) {
                int rq, c4;
                unit(jt, rq, c4);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float4 col = make_float4(f4_at(cur[4 * jt], e), f4_at(cur[4 * jt + 1], e),
                                                   f4_at(cur[4 * jt + 2], e), f4_at(cur[4 * jt + 3], e));
                    t32_put_split(slot + sw128_offset(4 * c4 + e, rq, C::kVAtom), C::kHalf, col);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.v_full[s]);
#pragma unroll
            for (int j = 0; j < C::kPer; ++j) cur[j] = nxt[j];
        }
        if (!ok) t32_fail(ms, p.status);
    } else if (warp == kT32MmaWarp) {
        // ---------------------------------------------------------------- MMA
        if (lane == 0 && nsub > 0) {
            constexpr uint32_t idesc_s = idesc_tf32_f32(128, KS);
            constexpr uint32_t idesc_o = idesc_tf32_f32(128, D);
            constexpr uint32_t kHi = smem_desc_hi_sw128(1024);
            // S(j) = Qhi Khi^T + Qhi Klo^T + Qlo Khi^T into S buffer j % 2 (K steps of 8 floats)
            auto issue_s = [&](int j) -> bool {
                const int s = j % kT32Slots;
                if (!mbar_wait(&ms.k_full[s], (uint32_t)(j / kT32Slots) & 1u, abort_flag)) return false;
                tc_fence_after_sync();
                const uint32_t st = smem_u32(smem + C::kK0 + s * C::kSlot);
                const uint32_t khi = smem_desc_lo(st, 16), klo = smem_desc_lo(st + C::kHalf, 16);
                const uint32_t d = tmem + C::s_col(j & 1);
#pragma unroll
                for (int k = 0; k < D / 8; ++k) {
                    const uint32_t ok_ = ((k / 4) * C::kKAtom + (k % 4) * 32) >> 4;
                    mma_tf32_ts<kHi>(d, tmem + C::kQhi + 8 * k, khi + ok_, idesc_s, k > 0 ? 1u : 0u);
                    mma_tf32_ts<kHi>(d, tmem + C::kQhi + 8 * k, klo + ok_, idesc_s, 1u);
                    mma_tf32_ts<kHi>(d, tmem + C::kQlo + 8 * k, khi + ok_, idesc_s, 1u);
                }
                mma_commit(&ms.k_empty[s]);
                mma_commit(&ms.s_full[j & 1]);
                return true;
            };
            bool ok = mbar_wait(&ms.q_ready, 0, abort_flag);
            if (ok) {
                tc_fence_after_sync();
                ok = issue_s(0);
            }
            if (ok && nsub > 1) ok = issue_s(1);
            for (int u = 0; ok && u < nsub; ++u) {
                const int pb = u & 1, s = u % kT32Slots;
                if (!mbar_wait(&ms.p_full[pb], (uint32_t)(u >> 1) & 1u, abort_flag) ||
                    !mbar_wait(&ms.v_full[s], (uint32_t)(u / kT32Slots) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t st = smem_u32(smem + C::kV0 + s * C::kSlot);
                const uint32_t vhi = smem_desc_lo(st, 16), vlo = smem_desc_lo(st + C::kHalf, 16);
                // O += Phi Vhi + Phi Vlo + Plo Vhi (P from TMEM, 8 kv columns per step)
#pragma unroll
                for (int k = 0; k < KS / 8; ++k) {
                    const uint32_t ov = ((k / 4) * C::kVAtom + (k % 4) * 32) >> 4;
                    const uint32_t acc0 = (u > 0 || k > 0) ? 1u : 0u;
                    mma_tf32_ts<kHi>(tmem + C::kO, tmem + C::s_col(pb) + 8 * k, vhi + ov, idesc_o, acc0);
                    mma_tf32_ts<kHi>(tmem + C::kO, tmem + C::s_col(pb) + 8 * k, vlo + ov, idesc_o, 1u);
                    mma_tf32_ts<kHi>(tmem + C::kO, tmem + C::plo_col(pb) + 8 * k, vhi + ov, idesc_o, 1u);
                }
                mma_commit(&ms.v_empty[s]);
                mma_commit(&ms.pv_done);
                // S(u + 2) reuses the buffer PV(u) reads: MMAs of one thread run in order
                if (u + 2 < nsub && !issue_s(u + 2)) ok = false;
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
        bool ok = true;
        if (nsub > 0) {
            // Q row -> Qhi, Qlo columns of this lane; PRESCALE_QK multiplies by scale first (one rounding)
            const float *qrow = static_cast<const float *>(p.q) + b * p.q_stride[0] + h * p.q_stride[1] +
                                (int64_t)(row_in ? q : 0) * p.q_stride[2];
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 64) {  // 16 loads in flight, then four 16-column stores
                float4 x[16];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    x[j] = row_in ? __ldg(reinterpret_cast<const float4 *>(qrow + c0) + j) : zero;
#pragma unroll
                for (int part = 0; part < 4; ++part) {
                    uint32_t qh[16], ql[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        float f = f4_at(x[4 * part + j / 4], j % 4);
                        if (p.prescale) f = __fmul_rn(f, p.scale);
                        const float fh = tf32_hi(f);
                        qh[j] = __float_as_uint(fh);
                        ql[j] = __float_as_uint(f - fh);
                    }
                    tmem_st16(trow + C::kQhi + c0 + 16 * part, qh);
                    tmem_st16(trow + C::kQlo + c0 + 16 * part, ql);
                }
            }
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.q_ready);
        }
        float m = -INFINITY, m_true = -INFINITY, l = 0.f;
        for (int u = 0; u < nsub; ++u) {
            const int pb = u & 1;
            const uint32_t e = ms.list[u / C::kSub];
            const bool full = (e >> 16) & 1u;
            const int kv0 = (int)(e & 0xFFFFu) * kBlock + (u % C::kSub) * KS;
            if (!t32_warp_wait(&ms.s_full[pb], (uint32_t)(u >> 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            float x[KS];
#pragma unroll
            for (int c0 = 0; c0 < KS; c0 += 32) {
                uint32_t r[32];
                t32_ld32(trow + C::s_col(pb) + c0, r);
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
            m_true = fmaxf(m_true, mt);
            // the reference maximum moves only when this chunk's exceeds it by
            // more than kT32RescaleNats (so p <= e^8); from -inf it moves to
            // the first finite maximum
            const bool grow = mt > m + kT32RescaleNats;
            if (__any_sync(0xffffffffu, grow)) {
                const float m_new = grow ? mt : m;
                const float alpha = grow ? expf(m - m_new) : 1.f;  // 0 when m was -inf
                if (u > 0) {
                    // PV(u - 1) has completed before O is rescaled in place
                    if (!t32_warp_wait(&ms.pv_done, (uint32_t)(u - 1) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
#pragma unroll 1
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t o[32];
                        t32_ld32(trow + C::kO + c0, o);
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                        tmem_st32(trow + C::kO + c0, o);
                    }
                }
                l *= alpha;
                m = m_new;
            }
            float sum = 0.f;
#pragma unroll
            for (int c0 = 0; c0 < KS; c0 += 16) {  // 16 columns at a time: x is consumed as P is stored
                uint32_t ph[16], pl[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float pj = m == -INFINITY ? 0.f : expf(x[c0 + j] - m);
                    sum += pj;
                    const float hj = tf32_hi(pj);
                    ph[j] = __float_as_uint(hj);
                    pl[j] = __float_as_uint(pj - hj);
                }
                tmem_st16(trow + C::s_col(pb) + c0, ph);  // over S columns, all read above
                tmem_st16(trow + C::plo_col(pb) + c0, pl);
            }
            l += sum;
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.p_full[pb]);
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
                if (p.row_max) p.row_max[orow] = live ? m_true : -INFINITY;
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
    if (p.nqt <= 65535) {
        // (b, h) pairs along x, q tiles (longest first) along y: the first
        // CTAs to run are the longest of every pair
        attn_tf32_kernel<D><<<dim3(p.bh_count, p.nqt), kT32Threads, smem, stream>>>(p, 1);
        return cudaGetLastError();
    }
    // grid.y holds at most 65535 (b, h) pairs per launch
    for (int begin = 0; begin < p.bh_count; begin += 65535) {
        AttnProblem part = p;
        part.bh_begin = p.bh_begin + begin;
        part.bh_count = p.bh_count - begin < 65535 ? p.bh_count - begin : 65535;
        attn_tf32_kernel<D><<<dim3(p.nqt, part.bh_count), kT32Threads, smem, stream>>>(part, 0);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_attn_tf32(const AttnProblem &p, cudaStream_t stream) {
    return p.D == 64 ? launch_tf32_d<64>(p, stream) : launch_tf32_d<128>(p, stream);
}

}  // namespace flex
