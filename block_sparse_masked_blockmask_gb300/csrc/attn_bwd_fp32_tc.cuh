// dK, dV and dQ of the block-sparse attention for float32 inputs at head
// dims 64 and 128 on sm_103a tensor cores, with float32 accuracy kept by the three-way bf16
// split of the float32 forward (bf16x3.cuh): every operand x = x1 + x2 + x3
// and each product takes the six part products a1 b1 + a1 b2 + a2 b1 +
// a1 b3 + a2 b2 + a3 b1, accumulated in float32 in tensor memory.
//
// What it computes is the dk and dv outputs of the flex_attention_backward
// op ("[Inductor][Flex Attention] Add Subtiling Option for Alpha Scaling",
// PyTorch PR #167356, test diffs), for one 128-row kv block j, walking the q
// blocks of the q side of the BlockMask in chunks of 64 q rows i:
//   S^T  = K_j Q_i^T,  dP^T = V_j dO_i^T              (SS MMAs)
//   P^T  = exp(score_mod(scale S^T) - lse_i) where mask_mod holds, else 0
//   dS^T = scale P^T (dP^T - delta_i) score_mod'      (elementwise, float32)
//   dV_j += P^T dO_i,  dK_j += dS^T Q_i               (TS MMAs: P^T, dS^T
//                                                      read from TMEM)
// and, in a second kernel for one 128-row q block i walking the kv side in
// chunks of 64 kv rows j, S = Q_i K_j^T, dP = dO_i V_j^T, dS as above and
// dQ_i += dS K_j (its rows of P are not needed).
// Roles of the dK/dV kernel (480 threads, one CTA per kv block; the dQ
// kernel the same with Q and dO resident and K and V streamed):
//   warps 0-3   elementwise, one thread per kv row (TMEM lane = row)
//   Q group     warps 5-7, 9: split the resident K tile, then each Q chunk
//               and its lse into a two-stage ring
//   dO group    warps 10, 11, 13, 14: the resident V tile, each dO chunk and
//               its delta
//   warp 12     one thread issues every MMA (warps 4 and 8 stay idle, so
//               that the issuer shares its sub-partition with warp 0 only)
// At head dim 128 the dK/dV kernel runs two CTAs per kv block, one for dK
// and one for dV, and the dQ kernel keeps the Q parts in tensor
// memory; the comments at those kernels give their layouts.
// Tensor memory at head dim 64 (512 columns): dV | dK | two buffers of S^T (64) | dP^T (64)
// | 64 more.  P^T and dS^T are split into bf16 parts over the columns they
// were computed from, a half of the 64 q columns at a time: the parts of
// columns 32h .. 32h + 31 take S^T (dP^T) columns 32h .. 32h + 31 and 16 of
// the spare columns, so each half only overwrites columns it has already
// read.  Every wait is bounded; on timeout the CTA records
// FLEX_ERR_DEVICE_TIMEOUT, drains its MMAs, frees TMEM and exits.
#pragma once

#include <cfloat>

#include "bf16x3.cuh"
#include "flex_internal.h"
#include "ptx.cuh"
#include "tilelist.cuh"

namespace flex {

// q tiles of a kv block the kernel walks on chip (longer q sides take the
// CUDA-core kernel)
constexpr int kBwdF32TcMaxQTiles = 2048;

struct BwdF32TcArgs {
    const float *dout;                               // contiguous [B, H, q_len, 64]
    const float *delta;                              // [B, H, q_len]
    const int32_t *q_num, *q_idx, *fq_num, *fq_idx;  // q side of the BlockMask
    float *dk, *dv;                                  // contiguous [B, H, kv_len, 64]
    float *dq;                                       // contiguous [B, H, q_len, 64]
};

namespace bwdf32 {

constexpr int D = 64;
constexpr int kKvRows = 128;     // owned kv rows (MMA M)
constexpr int kQc = 64;          // q rows per chunk (MMA N of S^T and dP^T, K of dV and dK)
constexpr int kThreads = 15 * 32;
constexpr int kMmaWarp = 12;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

// shared memory: K parts | V parts | two ring stages (Q parts, dO parts, lse, delta) | misc
constexpr uint32_t kOwnPart = kKvRows * D * 2;   // 16 KB: one bf16 part of a 128 x 64 tile
constexpr uint32_t kChunkPart = kQc * D * 2;     // 8 KB: one bf16 part of a 64 x 64 chunk
constexpr uint32_t kK0 = 0, kV0 = 3 * kOwnPart;
constexpr uint32_t kStage0 = 6 * kOwnPart;
constexpr uint32_t kStQ = 0, kStDo = 3 * kChunkPart, kStLse = 6 * kChunkPart, kStDelta = kStLse + kQc * 4;
constexpr uint32_t kStageBytes = 6 * kChunkPart + 1024;  // parts, lse and delta, 1024-aligned
constexpr uint32_t kMiscOff = kStage0 + 2 * kStageBytes;

// tensor memory columns
constexpr uint32_t kDv = 0, kDk = 64;
__host__ __device__ constexpr uint32_t buf_col(int b) { return 128u + 192u * (uint32_t)b; }
// A-operand column of part `part` (0..2) of P^T (dS: + 64 and + 32 in the
// spare columns) for K step k (16 q columns: half k / 2, 8 words into it when k is odd)
__host__ __device__ constexpr uint32_t p_part_col(int b, int part, int k) {
    return part < 2 ? buf_col(b) + 32u * (uint32_t)(k / 2) + 16u * (uint32_t)part + 8u * (uint32_t)(k % 2)
                    : buf_col(b) + 128u + 16u * (uint32_t)(k / 2) + 8u * (uint32_t)(k % 2);
}
__host__ __device__ constexpr uint32_t ds_part_col(int b, int part, int k) {
    return part < 2 ? buf_col(b) + 64u + 32u * (uint32_t)(k / 2) + 16u * (uint32_t)part + 8u * (uint32_t)(k % 2)
                    : buf_col(b) + 160u + 16u * (uint32_t)(k / 2) + 8u * (uint32_t)(k % 2);
}
static_assert(buf_col(1) + 192 == kTmemCols, "tensor memory");

struct Misc {
    // ring stage s, producer group g (0: Q in the dK/dV kernel, K in the dQ
    // kernel; 1: dO, V): each half of a stage is filled and freed on its own
    uint64_t kv_ready, st_full[2][2], st_empty[2][2], s_full[2], p_full[2], acc_full, drain;
    uint32_t tmem_base;
    int abort;
    int ntiles;  // q tiles listed for this kv block
    int pad;
    alignas(16) uint32_t flags[kBwdF32TcMaxQTiles];  // listed / full count per q tile (tilelist.cuh)
    alignas(16) uint32_t list[kBwdF32TcMaxQTiles];   // q tile | full << 16, ascending
};
constexpr size_t kSmemBytes = kMiscOff + sizeof(Misc) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

// Producer group of four warps (thread lt in 0..127): the rows r0 .. r0 +
// ROWS - 1 of a [.., len, 64] float32 tensor (rows past len read as zeros)
// into registers, then split into three bf16 parts at dst + j * part_bytes
// in 128-byte swizzled rows.  Thread lt takes units i = lt + 128 u: row
// i / 8, 8 floats at column 8 (i % 8).  The loads of a chunk are issued
// before its ring slot is waited for.
template <int ROWS>
struct RowsRegs {
    float4 x[ROWS * 8 / 128 * 2];
};
template <int ROWS>
__device__ __forceinline__ void load_rows(RowsRegs<ROWS> &g, const float *src, int64_t rs, int r0, int len, int lt) {
    constexpr int kUnits = ROWS * 8 / 128;
#pragma unroll
    for (int u = 0; u < kUnits; ++u) {
        const int i = lt + 128 * u, r = i / 8, c = i % 8;
        const bool in = r0 + r < len;
        const float4 *p = reinterpret_cast<const float4 *>(src + (int64_t)(in ? r0 + r : 0) * rs) + 2 * c;
        g.x[2 * u] = in ? __ldg(p) : make_float4(0.f, 0.f, 0.f, 0.f);
        g.x[2 * u + 1] = in ? __ldg(p + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}
template <int ROWS>
__device__ __forceinline__ void store_split(uint8_t *dst, uint32_t part_bytes, const RowsRegs<ROWS> &g, int lt) {
    constexpr int kUnits = ROWS * 8 / 128;
#pragma unroll
    for (int u = 0; u < kUnits; ++u) {
        const int i = lt + 128 * u, r = i / 8, c = i % 8;
        uint4 p1, p2, p3;
        split3(g.x[2 * u].x, g.x[2 * u].y, p1.x, p2.x, p3.x);
        split3(g.x[2 * u].z, g.x[2 * u].w, p1.y, p2.y, p3.y);
        split3(g.x[2 * u + 1].x, g.x[2 * u + 1].y, p1.z, p2.z, p3.z);
        split3(g.x[2 * u + 1].z, g.x[2 * u + 1].w, p1.w, p2.w, p3.w);
        const uint32_t off = sw128_chunk(r, c, ROWS * 128);
        *reinterpret_cast<uint4 *>(dst + off) = p1;
        *reinterpret_cast<uint4 *>(dst + part_bytes + off) = p2;
        *reinterpret_cast<uint4 *>(dst + 2 * part_bytes + off) = p3;
    }
}
template <int ROWS>
__device__ __forceinline__ void load_split(uint8_t *dst, uint32_t part_bytes, const float *src, int64_t rs, int r0,
                                           int len, int lt) {
    RowsRegs<ROWS> g;
    load_rows<ROWS>(g, src, rs, r0, len, lt);
    store_split<ROWS>(dst, part_bytes, g, lt);
}

__device__ __forceinline__ void fail(Misc &ms, int *status) {
    *reinterpret_cast<volatile int *>(&ms.abort) = 1;
    atomicCAS(status, 0, kDeviceTimeout);
}

// warp -> index in the Q group (5, 6, 7, 9) or the dO group (10, 11, 13, 14), else -1
__device__ __forceinline__ int q_index(int w) { return w >= 5 && w < 8 ? w - 5 : w == 9 ? 3 : -1; }
__device__ __forceinline__ int do_index(int w) { return w == 10 || w == 11 ? w - 10 : w == 13 || w == 14 ? w - 11 : -1; }

// score_mod at the scaled score t, and its derivative d score_mod / dt
template <int SCORE>
__device__ __forceinline__ float score_t(float cap, float t, float slope, int q, int kv, float &grad) {
    if constexpr (SCORE == FLEX_SCORE_SOFTCAP) {
        const float u = tanhf(t / cap);
        grad = 1.f - u * u;
        return cap * u;
    }
    grad = 1.f;
    if constexpr (SCORE == FLEX_SCORE_ALIBI) return t - slope * (float)(q - kv);
    return t;
}

template <int SCORE>
__global__ void __launch_bounds__(16 * 32, 1) dkdv_kernel(AttnProblem p, BwdF32TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc &ms = *reinterpret_cast<Misc *>(smem + kMiscOff);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // (b, h) pairs along x, kv blocks along y (at most 1024): the first CTAs
    // to run are the kv blocks that come first in every pair (the longest q
    // sides of a causal mask)
    const int kvb = blockIdx.y;
    const int bh = p.bh_begin + (int)blockIdx.x, h = bh % p.H, b = bh / p.H;
    const int kv0 = kvb * kBlock;

    if (threadIdx.x == 0) {
        mbar_init(&ms.kv_ready, 8);
        for (int i = 0; i < 2; ++i) {
            for (int g = 0; g < 2; ++g) {
                mbar_init(&ms.st_full[i][g], 4);
                mbar_init(&ms.st_empty[i][g], 1);
            }
            mbar_init(&ms.s_full[i], 1);
            mbar_init(&ms.p_full[i], 4);
        }
        mbar_init(&ms.acc_full, 1);
        mbar_init(&ms.drain, 1);
        ms.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        // the q side of the BlockMask (any block sizes) read as 128-tiles:
        // counts clamped, malformed entries dropped
        const TileLists lists{a.q_num, a.q_idx, a.fq_num, a.fq_idx, p.nkvb, p.nqb, p.kv_block, p.q_block, p.nqt};
        for (int i = lane; i < p.nqt; i += 32) ms.flags[i] = 0u;
        __syncwarp();
        tl_mark_warp(lists, bh, kvb, 0, ms.flags, 0, p.nqt, lane);
        __syncwarp();
        const uint32_t expect = tl_expect(lists);
        const unsigned lt = (1u << lane) - 1u;
        int cnt = 0;
        for (int base = 0; base < p.nqt; base += 32) {
            const int i = base + lane;
            const uint32_t w = i < p.nqt ? ms.flags[i] : 0u;
            const bool on = tl_listed(w, 0);
            const unsigned bal = __ballot_sync(0xffffffffu, on);
            if (on) ms.list[cnt + __popc(bal & lt)] = (uint32_t)i | (tl_full(expect, w, 0) ? (1u << 16) : 0u);
            cnt += __popc(bal);
        }
        if (lane == 0) ms.ntiles = cnt;
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&ms.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ms.tmem_base;
    volatile int *abort_flag = &ms.abort;
    const int nchunk = 2 * ms.ntiles;  // two 64-row chunks per q tile
    auto chunk_q0 = [&](int j) { return (int)(ms.list[j / 2] & 0xFFFFu) * kBlock + (j % 2) * kQc; };
    const int qi = q_index(warp), di = do_index(warp);

    if (qi >= 0 || di >= 0) {
        // ----------------------------------------------------------- producers
        const int lt = 32 * (qi >= 0 ? qi : di) + lane, grp = qi >= 0 ? 0 : 1;
        if (qi >= 0) {
            const float *kbase = static_cast<const float *>(p.k) + b * p.k_stride[0] + h * p.k_stride[1];
            load_split<kKvRows>(smem + kK0, kOwnPart, kbase, p.k_stride[2], kv0, p.kv_len, lt);
        } else {
            const float *vbase = static_cast<const float *>(p.v) + b * p.v_stride[0] + h * p.v_stride[1];
            load_split<kKvRows>(smem + kV0, kOwnPart, vbase, p.v_stride[2], kv0, p.kv_len, lt);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms.kv_ready);
        const float *qbase = static_cast<const float *>(p.q) + b * p.q_stride[0] + h * p.q_stride[1];
        const float *gbase = a.dout + (int64_t)bh * p.q_len * D;
        const float *lbase = p.lse + (int64_t)bh * p.q_len;
        const float *dbase = a.delta + (int64_t)bh * p.q_len;
        bool ok = true;
        for (int j = 0; j < nchunk; ++j) {
            const int s = j & 1;
            const int q0 = chunk_q0(j);
            // this chunk's rows (and its lse or delta) into registers, then the slot
            RowsRegs<kQc> g;
            float rowv = 0.f;
            const int q = q0 + lt;
            if (qi >= 0) {
                load_rows<kQc>(g, qbase, p.q_stride[2], q0, p.q_len, lt);
                if (lt < kQc) rowv = q < p.q_len ? lbase[q] : -INFINITY;
            } else {
                load_rows<kQc>(g, gbase, D, q0, p.q_len, lt);
                if (lt < kQc) rowv = q < p.q_len ? dbase[q] : 0.f;
            }
            if (j >= 2 && !f32_warp_wait(&ms.st_empty[s][grp], (uint32_t)((j >> 1) - 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            uint8_t *st = smem + kStage0 + s * kStageBytes;
            store_split<kQc>(st + (qi >= 0 ? kStQ : kStDo), kChunkPart, g, lt);
            if (lt < kQc) reinterpret_cast<float *>(st + (qi >= 0 ? kStLse : kStDelta))[lt] = rowv;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.st_full[s][grp]);
        }
        if (!ok) fail(ms, p.status);
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0 && nchunk > 0) {
            constexpr uint32_t kHi = smem_desc_hi_sw128(1024);
            constexpr uint32_t idesc_kmaj = idesc_bf16_f32(128, kQc, 0, 0);  // S^T, dP^T: B K-major
            constexpr uint32_t idesc_mn = idesc_bf16_f32(128, D, 0, 1);      // dV, dK: B MN-major
            // the six part products t: (A part, B part) = (0,0) (0,1) (1,0) (0,2) (1,1) (2,0)
            auto pa = [](int t) { return t == 2 || t == 4 ? 1 : t == 5 ? 2 : 0; };
            auto pbp = [](int t) { return t == 1 || t == 4 ? 1 : t == 3 ? 2 : 0; };
            const uint32_t kd = smem_desc_lo(smem_u32(smem + kK0), 16), vd = smem_desc_lo(smem_u32(smem + kV0), 16);
            // S^T(j) and dP^T(j) into buffer j % 2 (K steps of 16 head dims = 32 bytes)
            // (dP^T first: the dO half of a stage is refilled while dK(j - 2) runs)
            auto issue_sdp = [&](int j) -> bool {
                const int s = j & 1;
                const uint32_t st = smem_u32(smem + kStage0 + s * kStageBytes);
                const uint32_t qd = smem_desc_lo(st + kStQ, 16), gd = smem_desc_lo(st + kStDo, 16);
                if (!mbar_wait(&ms.st_full[s][1], (uint32_t)(j >> 1) & 1u, abort_flag)) return false;
                tc_fence_after_sync();
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
#pragma unroll
                    for (int t = 0; t < 6; ++t)
                        mma_ss_lo<kHi, kHi>(tmem + buf_col(s) + 64, vd + ((pa(t) * kOwnPart + k * 32) >> 4),
                                            gd + ((pbp(t) * kChunkPart + k * 32) >> 4), idesc_kmaj,
                                            (k > 0 || t > 0) ? 1u : 0u);
                if (!mbar_wait(&ms.st_full[s][0], (uint32_t)(j >> 1) & 1u, abort_flag)) return false;
                tc_fence_after_sync();
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
#pragma unroll
                    for (int t = 0; t < 6; ++t)
                        mma_ss_lo<kHi, kHi>(tmem + buf_col(s), kd + ((pa(t) * kOwnPart + k * 32) >> 4),
                                            qd + ((pbp(t) * kChunkPart + k * 32) >> 4), idesc_kmaj,
                                            (k > 0 || t > 0) ? 1u : 0u);
                mma_commit(&ms.s_full[s]);
                return true;
            };
            // dV += P^T dO(j), dK += dS^T Q(j): A from TMEM, B MN-major (rows
            // of 64 head dims, K steps of 16 q rows = 2048 bytes)
            auto issue_acc = [&](int j) -> bool {
                const int s = j & 1;
                if (!mbar_wait(&ms.p_full[s], (uint32_t)(j >> 1) & 1u, abort_flag)) return false;
                tc_fence_after_sync();
                const uint32_t st = smem_u32(smem + kStage0 + s * kStageBytes);
                const uint32_t qm = smem_desc_lo(st + kStQ, kChunkPart), gm = smem_desc_lo(st + kStDo, kChunkPart);
                // dV, then the dO half of the stage is free; dK, then the Q half
#pragma unroll
                for (int k = 0; k < kQc / 16; ++k)
#pragma unroll
                    for (int t = 0; t < 6; ++t)
                        mma_ts_lo<kHi>(tmem + kDv, tmem + p_part_col(s, pa(t), k),
                                       gm + ((pbp(t) * kChunkPart + k * 2048) >> 4), idesc_mn,
                                       (j > 0 || k > 0 || t > 0) ? 1u : 0u);
                mma_commit(&ms.st_empty[s][1]);
#pragma unroll
                for (int k = 0; k < kQc / 16; ++k)
#pragma unroll
                    for (int t = 0; t < 6; ++t)
                        mma_ts_lo<kHi>(tmem + kDk, tmem + ds_part_col(s, pa(t), k),
                                       qm + ((pbp(t) * kChunkPart + k * 2048) >> 4), idesc_mn,
                                       (j > 0 || k > 0 || t > 0) ? 1u : 0u);
                mma_commit(&ms.st_empty[s][0]);
                return true;
            };
            bool ok = mbar_wait(&ms.kv_ready, 0, abort_flag);
            if (ok) tc_fence_after_sync();
            for (int j = 0; ok && j < min(nchunk, 2); ++j) ok = issue_sdp(j);
            // S^T(j + 2) reuses the buffer dV(j), dK(j) read: MMAs of one thread run in order
            for (int j = 0; ok && j < nchunk; ++j) ok = issue_acc(j) && (j + 2 >= nchunk || issue_sdp(j + 2));
            if (ok) mma_commit(&ms.acc_full);
            if (!ok) fail(ms, p.status);
            mma_commit(&ms.drain);  // every MMA issued above completes before TMEM is freed
            int never = 0;
            (void)mbar_wait(&ms.drain, 0, &never);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ---------------------------------------------------------- elementwise
        const int kv = kv0 + (int)threadIdx.x;
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        const float slope = SCORE == FLEX_SCORE_ALIBI ? exp2f(-8.f * (float)(h + 1) / (float)p.H) : 0.f;
        const float scale = p.scale;
        bool ok = true;
        for (int j = 0; j < nchunk; ++j) {
            const int s = j & 1;
            const bool full = (ms.list[j / 2] >> 16) & 1u;
            const int q0 = chunk_q0(j);
            // S^T and dP^T of the chunk are in TMEM; its lse and delta (written
            // by the producers) are read after their own barrier
            if (!f32_warp_wait(&ms.s_full[s], (uint32_t)(j >> 1) & 1u, abort_flag) ||
                !f32_warp_wait(&ms.st_full[s][0], (uint32_t)(j >> 1) & 1u, abort_flag) ||
                !f32_warp_wait(&ms.st_full[s][1], (uint32_t)(j >> 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const float *lse_s = reinterpret_cast<const float *>(smem + kStage0 + s * kStageBytes + kStLse);
            const float *dl_s = reinterpret_cast<const float *>(smem + kStage0 + s * kStageBytes + kStDelta);
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                uint32_t sr[32], dr[32];
                f32_ld32(trow + buf_col(s) + 32 * half, sr);
                f32_ld32(trow + buf_col(s) + 64 + 32 * half, dr);
                float pv[32], dsv[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int q = q0 + 32 * half + c;
                    const float lse = lse_s[32 * half + c];
                    const bool keep = lse != -INFINITY && (full || (kv < p.kv_len && mask_mod(p.mask, b, q, kv)));
                    float grad;
                    const float x = score_t<SCORE>(p.score_param, __uint_as_float(sr[c]) * scale, slope, q, kv, grad);
                    const float pr = keep ? ex2_approx(fmaf(x, kLog2e, -lse * kLog2e)) : 0.f;
                    pv[c] = pr;
                    dsv[c] = keep ? scale * pr * (__uint_as_float(dr[c]) - dl_s[32 * half + c]) * grad : 0.f;
                }
                uint32_t w1[16], w2[16], w3[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) split3(pv[2 * c], pv[2 * c + 1], w1[c], w2[c], w3[c]);
                // over S^T columns 32 half .. 32 half + 31, all read above
                tmem_st16(trow + buf_col(s) + 32 * half, w1);
                tmem_st16(trow + buf_col(s) + 32 * half + 16, w2);
                tmem_st16(trow + buf_col(s) + 128 + 16 * half, w3);
#pragma unroll
                for (int c = 0; c < 16; ++c) split3(dsv[2 * c], dsv[2 * c + 1], w1[c], w2[c], w3[c]);
                tmem_st16(trow + buf_col(s) + 64 + 32 * half, w1);
                tmem_st16(trow + buf_col(s) + 64 + 32 * half + 16, w2);
                tmem_st16(trow + buf_col(s) + 160 + 16 * half, w3);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.p_full[s]);
        }
        // ------------------------------------------------------------ epilogue
        const bool have = ok && nchunk > 0;
        if (have && !f32_warp_wait(&ms.acc_full, 0, abort_flag)) ok = false;
        if (!ok) fail(ms, p.status);
        if (ok) {
            tc_fence_after_sync();
            const int64_t orow = (int64_t)bh * p.kv_len + (kv < p.kv_len ? kv : 0);
#pragma unroll 1
            for (int o = 0; o < 2; ++o) {  // dV, then dK
                float *dst = (o ? a.dk : a.dv) + orow * D;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {  // every lane takes the warp-collective loads
                    uint32_t r[32];
                    if (have) {
                        f32_ld32(trow + (o ? kDk : kDv) + c0, r);
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c) r[c] = 0u;
                    }
                    if (kv < p.kv_len) {
#pragma unroll
                        for (int c = 0; c < 32; c += 4)
                            *reinterpret_cast<float4 *>(dst + c0 + c) =
                                make_float4(__uint_as_float(r[c]), __uint_as_float(r[c + 1]),
                                            __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]));
                    }
                }
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// dQ: one CTA per 128-row q block (TMEM: dQ | two buffers of S (64) and dP
// (64); the bf16 parts of dS of columns 32h .. 32h + 31 go over S columns
// 32h .. 32h + 31 and dP columns 32h .. 32h + 15).
__host__ __device__ constexpr uint32_t dq_buf_col(int b) { return 64u + 128u * (uint32_t)b; }
__host__ __device__ constexpr uint32_t dq_ds_part_col(int b, int part, int k) {
    return part < 2 ? dq_buf_col(b) + 32u * (uint32_t)(k / 2) + 16u * (uint32_t)part + 8u * (uint32_t)(k % 2)
                    : dq_buf_col(b) + 64u + 32u * (uint32_t)(k / 2) + 8u * (uint32_t)(k % 2);
}
static_assert(dq_buf_col(1) + 128 <= kTmemCols, "tensor memory");
constexpr uint32_t kQ0 = 0, kDo0 = 3 * kOwnPart;            // resident Q and dO parts
constexpr uint32_t kStK = 0, kStV = 3 * kChunkPart;          // a stage: K chunk parts, V chunk parts
constexpr uint32_t kDqStageBytes = 6 * kChunkPart;
constexpr uint32_t kDqMiscOff = kStage0 + 2 * kDqStageBytes;
constexpr size_t kDqSmemBytes = kDqMiscOff + sizeof(Misc) + 1024;
static_assert(kDqSmemBytes <= 232448, "shared memory per CTA");

template <int SCORE>
__global__ void __launch_bounds__(16 * 32, 1) dq_kernel(AttnProblem p, BwdF32TcArgs a, int bh_x) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc &ms = *reinterpret_cast<Misc *>(smem + kDqMiscOff);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // longest first: under a causal mask the last q blocks list the most kv tiles
    // (b, h) pairs along x and q tiles (longest first) along y when they fit
    // grid.y, so that the first CTAs to run are the longest of every pair
    const int qb = p.nqt - 1 - (int)(bh_x ? blockIdx.y : blockIdx.x);
    const int bh = p.bh_begin + (int)(bh_x ? blockIdx.x : blockIdx.y), h = bh % p.H, b = bh / p.H;
    const int q0 = qb * kBlock;

    if (threadIdx.x == 0) {
        mbar_init(&ms.kv_ready, 8);
        for (int i = 0; i < 2; ++i) {
            for (int g = 0; g < 2; ++g) {
                mbar_init(&ms.st_full[i][g], 4);
                mbar_init(&ms.st_empty[i][g], 1);
            }
            mbar_init(&ms.s_full[i], 1);
            mbar_init(&ms.p_full[i], 4);
        }
        mbar_init(&ms.acc_full, 1);
        mbar_init(&ms.drain, 1);
        ms.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        // the kv side of the BlockMask (any block sizes) read as 128-tiles
        const TileLists lists{p.kv_num, p.kv_idx, p.full_num, p.full_idx, p.nqb, p.nkvb, p.q_block, p.kv_block,
                              p.nkvt};
        for (int i = lane; i < p.nkvt; i += 32) ms.flags[i] = 0u;
        __syncwarp();
        tl_mark_warp(lists, bh, qb, 0, ms.flags, 0, p.nkvt, lane);
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
        if (lane == 0) ms.ntiles = cnt;
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&ms.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ms.tmem_base;
    volatile int *abort_flag = &ms.abort;
    const int nchunk = 2 * ms.ntiles;  // two 64-row chunks per kv tile
    auto chunk_kv0 = [&](int j) { return (int)(ms.list[j / 2] & 0xFFFFu) * kBlock + (j % 2) * kQc; };
    const int qi = q_index(warp), di = do_index(warp);

    if (qi >= 0 || di >= 0) {
        // ----------------------------------------------------------- producers
        const int lt = 32 * (qi >= 0 ? qi : di) + lane, grp = qi >= 0 ? 0 : 1;
        if (qi >= 0) {
            const float *qbase = static_cast<const float *>(p.q) + b * p.q_stride[0] + h * p.q_stride[1];
            load_split<kKvRows>(smem + kQ0, kOwnPart, qbase, p.q_stride[2], q0, p.q_len, lt);
        } else {
            load_split<kKvRows>(smem + kDo0, kOwnPart, a.dout + (int64_t)bh * p.q_len * D, D, q0, p.q_len, lt);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ms.kv_ready);
        const float *kbase = static_cast<const float *>(p.k) + b * p.k_stride[0] + h * p.k_stride[1];
        const float *vbase = static_cast<const float *>(p.v) + b * p.v_stride[0] + h * p.v_stride[1];
        bool ok = true;
        for (int j = 0; j < nchunk; ++j) {
            const int s = j & 1;
            const int kv0 = chunk_kv0(j);
            // this chunk's rows into registers, then the slot
            RowsRegs<kQc> g;
            if (qi >= 0)
                load_rows<kQc>(g, kbase, p.k_stride[2], kv0, p.kv_len, lt);
            else
                load_rows<kQc>(g, vbase, p.v_stride[2], kv0, p.kv_len, lt);
            if (j >= 2 && !f32_warp_wait(&ms.st_empty[s][grp], (uint32_t)((j >> 1) - 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            uint8_t *st = smem + kStage0 + s * kDqStageBytes;
            store_split<kQc>(st + (qi >= 0 ? kStK : kStV), kChunkPart, g, lt);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.st_full[s][grp]);
        }
        if (!ok) fail(ms, p.status);
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0 && nchunk > 0) {
            constexpr uint32_t kHi = smem_desc_hi_sw128(1024);
            constexpr uint32_t idesc_kmaj = idesc_bf16_f32(128, kQc, 0, 0);  // S, dP: B K-major
            constexpr uint32_t idesc_mn = idesc_bf16_f32(128, D, 0, 1);      // dQ: B MN-major
            auto pa = [](int t) { return t == 2 || t == 4 ? 1 : t == 5 ? 2 : 0; };
            auto pbp = [](int t) { return t == 1 || t == 4 ? 1 : t == 3 ? 2 : 0; };
            const uint32_t qd = smem_desc_lo(smem_u32(smem + kQ0), 16), gd = smem_desc_lo(smem_u32(smem + kDo0), 16);
            // S(j) = Q K_j^T and dP(j) = dO V_j^T into buffer j % 2
            // (dP first: V is read by nothing else, so its half of the stage
            // is free as soon as these MMAs are done)
            auto issue_sdp = [&](int j) -> bool {
                const int s = j & 1;
                const uint32_t st = smem_u32(smem + kStage0 + s * kDqStageBytes);
                const uint32_t kd = smem_desc_lo(st + kStK, 16), vd = smem_desc_lo(st + kStV, 16);
                if (!mbar_wait(&ms.st_full[s][1], (uint32_t)(j >> 1) & 1u, abort_flag)) return false;
                tc_fence_after_sync();
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
#pragma unroll
                    for (int t = 0; t < 6; ++t)
                        mma_ss_lo<kHi, kHi>(tmem + dq_buf_col(s) + 64, gd + ((pa(t) * kOwnPart + k * 32) >> 4),
                                            vd + ((pbp(t) * kChunkPart + k * 32) >> 4), idesc_kmaj,
                                            (k > 0 || t > 0) ? 1u : 0u);
                mma_commit(&ms.st_empty[s][1]);
                if (!mbar_wait(&ms.st_full[s][0], (uint32_t)(j >> 1) & 1u, abort_flag)) return false;
                tc_fence_after_sync();
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
#pragma unroll
                    for (int t = 0; t < 6; ++t)
                        mma_ss_lo<kHi, kHi>(tmem + dq_buf_col(s), qd + ((pa(t) * kOwnPart + k * 32) >> 4),
                                            kd + ((pbp(t) * kChunkPart + k * 32) >> 4), idesc_kmaj,
                                            (k > 0 || t > 0) ? 1u : 0u);
                mma_commit(&ms.s_full[s]);
                return true;
            };
            // dQ += dS K_j: A from TMEM, B MN-major (K steps of 16 kv rows = 2048 bytes)
            auto issue_acc = [&](int j) -> bool {
                const int s = j & 1;
                if (!mbar_wait(&ms.p_full[s], (uint32_t)(j >> 1) & 1u, abort_flag)) return false;
                tc_fence_after_sync();
                const uint32_t km = smem_desc_lo(smem_u32(smem + kStage0 + s * kDqStageBytes + kStK), kChunkPart);
#pragma unroll
                for (int k = 0; k < kQc / 16; ++k)
#pragma unroll
                    for (int t = 0; t < 6; ++t)
                        mma_ts_lo<kHi>(tmem + 0, tmem + dq_ds_part_col(s, pa(t), k),
                                       km + ((pbp(t) * kChunkPart + k * 2048) >> 4), idesc_mn,
                                       (j > 0 || k > 0 || t > 0) ? 1u : 0u);
                mma_commit(&ms.st_empty[s][0]);  // the K half of the stage
                return true;
            };
            bool ok = mbar_wait(&ms.kv_ready, 0, abort_flag);
            if (ok) tc_fence_after_sync();
            for (int j = 0; ok && j < min(nchunk, 2); ++j) ok = issue_sdp(j);
            // S(j + 2) reuses the buffer dQ(j) read: MMAs of one thread run in order
            for (int j = 0; ok && j < nchunk; ++j) ok = issue_acc(j) && (j + 2 >= nchunk || issue_sdp(j + 2));
            if (ok) mma_commit(&ms.acc_full);
            if (!ok) fail(ms, p.status);
            mma_commit(&ms.drain);  // every MMA issued above completes before TMEM is freed
            int never = 0;
            (void)mbar_wait(&ms.drain, 0, &never);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ---------------------------------------------------------- elementwise
        const int q = q0 + (int)threadIdx.x;
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        const float slope = SCORE == FLEX_SCORE_ALIBI ? exp2f(-8.f * (float)(h + 1) / (float)p.H) : 0.f;
        const float scale = p.scale;
        const bool q_in = q < p.q_len;
        const float lse = q_in ? p.lse[(int64_t)bh * p.q_len + q] : -INFINITY;
        const float dlt = q_in ? a.delta[(int64_t)bh * p.q_len + q] : 0.f;
        const float lb = lse * kLog2e;
        bool ok = true;
        for (int j = 0; j < nchunk; ++j) {
            const int s = j & 1;
            const bool full = (ms.list[j / 2] >> 16) & 1u;
            const int kv0 = chunk_kv0(j);
            if (!f32_warp_wait(&ms.s_full[s], (uint32_t)(j >> 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                uint32_t sr[32], dr[32];
                f32_ld32(trow + dq_buf_col(s) + 32 * half, sr);
                f32_ld32(trow + dq_buf_col(s) + 64 + 32 * half, dr);
                float dsv[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int kv = kv0 + 32 * half + c;
                    const bool keep = lse != -INFINITY && (full || (kv < p.kv_len && mask_mod(p.mask, b, q, kv)));
                    float grad;
                    const float x = score_t<SCORE>(p.score_param, __uint_as_float(sr[c]) * scale, slope, q, kv, grad);
                    const float pr = ex2_approx(fmaf(x, kLog2e, -lb));
                    dsv[c] = keep ? scale * pr * (__uint_as_float(dr[c]) - dlt) * grad : 0.f;
                }
                uint32_t w1[16], w2[16], w3[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) split3(dsv[2 * c], dsv[2 * c + 1], w1[c], w2[c], w3[c]);
                // over S columns 32 half .. + 31 and dP columns 32 half .. + 15, all read above
                tmem_st16(trow + dq_buf_col(s) + 32 * half, w1);
                tmem_st16(trow + dq_buf_col(s) + 32 * half + 16, w2);
                tmem_st16(trow + dq_buf_col(s) + 64 + 32 * half, w3);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.p_full[s]);
        }
        // ------------------------------------------------------------ epilogue
        const bool have = ok && nchunk > 0;
        if (have && !f32_warp_wait(&ms.acc_full, 0, abort_flag)) ok = false;
        if (!ok) fail(ms, p.status);
        if (ok) {
            tc_fence_after_sync();
            float *dst = a.dq + ((int64_t)bh * p.q_len + (q_in ? q : 0)) * D;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {  // every lane takes the warp-collective loads
                uint32_t r[32];
                if (have) {
                    f32_ld32(trow + c0, r);
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) r[c] = 0u;
                }
                if (q_in) {
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        *reinterpret_cast<float4 *>(dst + c0 + c) =
                            make_float4(__uint_as_float(r[c]), __uint_as_float(r[c + 1]), __uint_as_float(r[c + 2]),
                                        __uint_as_float(r[c + 3]));
                }
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// dQ at D = 128.  Q parts are the A operand of S from tensor memory (as in
// the forward), dO parts the A operand of dP from shared memory; one ring
// stage of K and V parts and one S/dP buffer (the split parts of 128 head
// dims leave no room for two), so a chunk's MMAs, its elementwise work and
// the next chunk's loads follow each other: S, dP -> dS -> dQ -> S, dP.
// TMEM: Q1 | Q2 | Q3 (64 each) | dQ (128) | S (64) | dP (64).
namespace d128 {
constexpr int D = 128;
constexpr uint32_t kQcol = 0, kDq = 192, kS = 320, kDp = 384;
__host__ __device__ constexpr uint32_t ds_part_col(int part, int k) {
    return part < 2 ? kS + 32u * (uint32_t)(k / 2) + 16u * (uint32_t)part + 8u * (uint32_t)(k % 2)
                    : kDp + 32u * (uint32_t)(k / 2) + 8u * (uint32_t)(k % 2);
}
constexpr uint32_t kDoPart = 128 * D * 2;      // 32 KB: one part of the resident dO (two 64-wide atoms)
constexpr uint32_t kDoAtom = 128 * 128;        // 128 rows x 64 bf16
constexpr uint32_t kChPart = kQc * D * 2;      // 16 KB: one part of a 64-row K or V chunk
constexpr uint32_t kChAtom = kQc * 128;        // 64 rows x 64 bf16
constexpr uint32_t kDo0 = 0, kStK = 3 * kDoPart, kStV = kStK + 3 * kChPart;
constexpr uint32_t kMiscOff = kStV + 3 * kChPart;
constexpr size_t kSmemBytes = kMiscOff + sizeof(Misc) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(kDp + 64 <= kTmemCols, "tensor memory");

// rows r0 .. r0 + 63 of a [.., len, 128] float32 tensor (zeros past len),
// split into three bf16 parts stored as tile rows row_base .. row_base + 63
// of a tile with 128-byte swizzled rows (atoms of atom_bytes) at dst + j *
// part_bytes.  Thread lt (0..127) takes units i = lt + 128 u: row i / 16, 8
// floats at column 8 (i % 16).
struct Rows64 {
    float4 x[16];
};
__device__ __forceinline__ void load64(Rows64 &g, const float *src, int64_t rs, int r0, int len, int lt) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int i = lt + 128 * u, r = i / 16, c = i % 16;
        const bool in = r0 + r < len;
        const float4 *p = reinterpret_cast<const float4 *>(src + (int64_t)(in ? r0 + r : 0) * rs) + 2 * c;
        g.x[2 * u] = in ? __ldg(p) : make_float4(0.f, 0.f, 0.f, 0.f);
        g.x[2 * u + 1] = in ? __ldg(p + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}
__device__ __forceinline__ void store64(uint8_t *dst, uint32_t part_bytes, uint32_t atom_bytes, int row_base,
                                        const Rows64 &g, int lt) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int i = lt + 128 * u, r = i / 16, c = i % 16;
        uint4 p1, p2, p3;
        split3(g.x[2 * u].x, g.x[2 * u].y, p1.x, p2.x, p3.x);
        split3(g.x[2 * u].z, g.x[2 * u].w, p1.y, p2.y, p3.y);
        split3(g.x[2 * u + 1].x, g.x[2 * u + 1].y, p1.z, p2.z, p3.z);
        split3(g.x[2 * u + 1].z, g.x[2 * u + 1].w, p1.w, p2.w, p3.w);
        const uint32_t off = sw128_chunk(row_base + r, c, atom_bytes);
        *reinterpret_cast<uint4 *>(dst + off) = p1;
        *reinterpret_cast<uint4 *>(dst + part_bytes + off) = p2;
        *reinterpret_cast<uint4 *>(dst + 2 * part_bytes + off) = p3;
    }
}
}  // namespace d128

template <int SCORE>
__global__ void __launch_bounds__(16 * 32, 1) dq128_kernel(AttnProblem p, BwdF32TcArgs a, int bh_x) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc &ms = *reinterpret_cast<Misc *>(smem + d128::kMiscOff);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // longest first: under a causal mask the last q blocks list the most kv tiles
    // (b, h) pairs along x and q tiles (longest first) along y when they fit
    // grid.y, so that the first CTAs to run are the longest of every pair
    const int qb = p.nqt - 1 - (int)(bh_x ? blockIdx.y : blockIdx.x);
    const int bh = p.bh_begin + (int)(bh_x ? blockIdx.x : blockIdx.y), h = bh % p.H, b = bh / p.H;
    const int q0 = qb * kBlock;

    // kv_ready: dO resident (4 dO-group warps) and Q in TMEM (4 elementwise
    // warps); st_full[0][g] / st_empty[0][g]: the K (g = 0) and V (g = 1)
    // halves of the single stage
    if (threadIdx.x == 0) {
        mbar_init(&ms.kv_ready, 8);
        for (int g = 0; g < 2; ++g) {
            mbar_init(&ms.st_full[0][g], 4);
            mbar_init(&ms.st_empty[0][g], 1);
        }
        mbar_init(&ms.s_full[0], 1);
        mbar_init(&ms.p_full[0], 4);
        mbar_init(&ms.acc_full, 1);
        mbar_init(&ms.drain, 1);
        ms.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        const TileLists lists{p.kv_num, p.kv_idx, p.full_num, p.full_idx, p.nqb, p.nkvb, p.q_block, p.kv_block,
                              p.nkvt};
        for (int i = lane; i < p.nkvt; i += 32) ms.flags[i] = 0u;
        __syncwarp();
        tl_mark_warp(lists, bh, qb, 0, ms.flags, 0, p.nkvt, lane);
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
        if (lane == 0) ms.ntiles = cnt;
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&ms.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ms.tmem_base;
    volatile int *abort_flag = &ms.abort;
    const int nchunk = 2 * ms.ntiles;
    auto chunk_kv0 = [&](int j) { return (int)(ms.list[j / 2] & 0xFFFFu) * kBlock + (j % 2) * kQc; };
    const int qi = q_index(warp), di = do_index(warp);

    if (qi >= 0 || di >= 0) {
        // ----------------------------------------------------------- producers
        const int lt = 32 * (qi >= 0 ? qi : di) + lane, grp = qi >= 0 ? 0 : 1;
        if (grp == 1 && nchunk > 0) {
            // the resident dO: two 64-row halves of the 128-row tile
            const float *gbase = a.dout + (int64_t)bh * p.q_len * d128::D;
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                d128::Rows64 g;
                d128::load64(g, gbase, d128::D, q0 + 64 * half, p.q_len, lt);
                d128::store64(smem + d128::kDo0, d128::kDoPart, d128::kDoAtom, 64 * half, g, lt);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.kv_ready);
        }
        const float *base = grp == 0 ? static_cast<const float *>(p.k) + b * p.k_stride[0] + h * p.k_stride[1]
                                     : static_cast<const float *>(p.v) + b * p.v_stride[0] + h * p.v_stride[1];
        const int64_t rs = grp == 0 ? p.k_stride[2] : p.v_stride[2];
        bool ok = true;
        for (int j = 0; j < nchunk; ++j) {
            d128::Rows64 g;
            d128::load64(g, base, rs, chunk_kv0(j), p.kv_len, lt);
            if (j >= 1 && !f32_warp_wait(&ms.st_empty[0][grp], (uint32_t)(j - 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            d128::store64(smem + (grp == 0 ? d128::kStK : d128::kStV), d128::kChPart, d128::kChAtom, 0, g, lt);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.st_full[0][grp]);
        }
        if (!ok) fail(ms, p.status);
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0 && nchunk > 0) {
            constexpr uint32_t kHi = smem_desc_hi_sw128(1024);
            constexpr uint32_t idesc_kmaj = idesc_bf16_f32(128, kQc, 0, 0);  // S, dP: N = 64 kv, B K-major
            constexpr uint32_t idesc_mn = idesc_bf16_f32(128, d128::D, 0, 1);      // dQ: N = 128, B MN-major
            auto pa = [](int t) { return t == 2 || t == 4 ? 1 : t == 5 ? 2 : 0; };
            auto pbp = [](int t) { return t == 1 || t == 4 ? 1 : t == 3 ? 2 : 0; };
            const uint32_t gd = smem_desc_lo(smem_u32(smem + d128::kDo0), 16);
            const uint32_t kd = smem_desc_lo(smem_u32(smem + d128::kStK), 16), vd = smem_desc_lo(smem_u32(smem + d128::kStV), 16);
            const uint32_t km = smem_desc_lo(smem_u32(smem + d128::kStK), d128::kChAtom);
            bool ok = mbar_wait(&ms.kv_ready, 0, abort_flag);
            for (int j = 0; ok && j < nchunk; ++j) {
                const uint32_t ph = (uint32_t)j & 1u;
                // dP = dO V^T (A: dO parts in shared memory), then the V half is free
                if (!mbar_wait(&ms.st_full[0][1], ph, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
#pragma unroll
                for (int k = 0; k < d128::D / 16; ++k)
#pragma unroll
                    for (int t = 0; t < 6; ++t)
                        mma_ss_lo<kHi, kHi>(tmem + d128::kDp,
                                            gd + ((pa(t) * d128::kDoPart + (k / 4) * d128::kDoAtom + (k % 4) * 32) >> 4),
                                            vd + ((pbp(t) * d128::kChPart + (k / 4) * d128::kChAtom + (k % 4) * 32) >> 4),
                                            idesc_kmaj, (k > 0 || t > 0) ? 1u : 0u);
                mma_commit(&ms.st_empty[0][1]);
                // S = Q K^T (A: Q parts in TMEM, 8 columns per K step of 16 head dims)
                if (!mbar_wait(&ms.st_full[0][0], ph, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
#pragma unroll
                for (int k = 0; k < d128::D / 16; ++k)
#pragma unroll
                    for (int t = 0; t < 6; ++t)
                        mma_ts_lo<kHi>(tmem + d128::kS, tmem + d128::kQcol + 64 * pa(t) + 8 * k,
                                       kd + ((pbp(t) * d128::kChPart + (k / 4) * d128::kChAtom + (k % 4) * 32) >> 4),
                                       idesc_kmaj, (k > 0 || t > 0) ? 1u : 0u);
                mma_commit(&ms.s_full[0]);
                // dQ += dS K (A: dS parts in TMEM; B: K MN-major, the two
                // 64-wide halves d128::kChAtom apart, K steps of 16 kv rows)
                if (!mbar_wait(&ms.p_full[0], ph, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
#pragma unroll
                for (int k = 0; k < kQc / 16; ++k)
#pragma unroll
                    for (int t = 0; t < 6; ++t)
                        mma_ts_lo<kHi>(tmem + d128::kDq, tmem + d128::ds_part_col(pa(t), k),
                                       km + ((pbp(t) * d128::kChPart + k * 2048) >> 4), idesc_mn,
                                       (j > 0 || k > 0 || t > 0) ? 1u : 0u);
                mma_commit(&ms.st_empty[0][0]);  // the K half
            }
            if (ok) mma_commit(&ms.acc_full);
            if (!ok) fail(ms, p.status);
            mma_commit(&ms.drain);
            int never = 0;
            (void)mbar_wait(&ms.drain, 0, &never);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ---------------------------------------------------------- elementwise
        const int q = q0 + (int)threadIdx.x;
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        const float slope = SCORE == FLEX_SCORE_ALIBI ? exp2f(-8.f * (float)(h + 1) / (float)p.H) : 0.f;
        const float scale = p.scale;
        const bool q_in = q < p.q_len;
        const float lse = q_in ? p.lse[(int64_t)bh * p.q_len + q] : -INFINITY;
        const float dlt = q_in ? a.delta[(int64_t)bh * p.q_len + q] : 0.f;
        const float lb = lse * kLog2e;
        bool ok = true;
        if (nchunk > 0) {
            // this row of Q -> Q1, Q2, Q3 columns of this lane (bf16 pairs)
            const float *qrow = static_cast<const float *>(p.q) + b * p.q_stride[0] + h * p.q_stride[1] +
                                (int64_t)(q_in ? q : 0) * p.q_stride[2];
#pragma unroll 1
            for (int c0 = 0; c0 < d128::D; c0 += 32) {
                float4 x[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    x[j] = q_in ? __ldg(reinterpret_cast<const float4 *>(qrow + c0) + j) : make_float4(0.f, 0.f, 0.f, 0.f);
                uint32_t w1[16], w2[16], w3[16];
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    split3(f4_at(x[j / 2], 2 * (j % 2)), f4_at(x[j / 2], 2 * (j % 2) + 1), w1[j], w2[j], w3[j]);
                tmem_st16(trow + d128::kQcol + c0 / 2, w1);
                tmem_st16(trow + d128::kQcol + 64 + c0 / 2, w2);
                tmem_st16(trow + d128::kQcol + 128 + c0 / 2, w3);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.kv_ready);
        }
        for (int j = 0; j < nchunk; ++j) {
            const bool full = (ms.list[j / 2] >> 16) & 1u;
            const int kv0 = chunk_kv0(j);
            if (!f32_warp_wait(&ms.s_full[0], (uint32_t)j & 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                uint32_t sr[32], dr[32];
                f32_ld32(trow + d128::kS + 32 * half, sr);
                f32_ld32(trow + d128::kDp + 32 * half, dr);
                float dsv[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int kv = kv0 + 32 * half + c;
                    const bool keep = lse != -INFINITY && (full || (kv < p.kv_len && mask_mod(p.mask, b, q, kv)));
                    float grad;
                    const float x = score_t<SCORE>(p.score_param, __uint_as_float(sr[c]) * scale, slope, q, kv, grad);
                    const float pr = ex2_approx(fmaf(x, kLog2e, -lb));
                    dsv[c] = keep ? scale * pr * (__uint_as_float(dr[c]) - dlt) * grad : 0.f;
                }
                uint32_t w1[16], w2[16], w3[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) split3(dsv[2 * c], dsv[2 * c + 1], w1[c], w2[c], w3[c]);
                // over S columns 32 half .. + 31 and dP columns 32 half .. + 15, all read above
                tmem_st16(trow + d128::kS + 32 * half, w1);
                tmem_st16(trow + d128::kS + 32 * half + 16, w2);
                tmem_st16(trow + d128::kDp + 32 * half, w3);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.p_full[0]);
        }
        // ------------------------------------------------------------ epilogue
        const bool have = ok && nchunk > 0;
        if (have && !f32_warp_wait(&ms.acc_full, 0, abort_flag)) ok = false;
        if (!ok) fail(ms, p.status);
        if (ok) {
            tc_fence_after_sync();
            float *dst = a.dq + ((int64_t)bh * p.q_len + (q_in ? q : 0)) * d128::D;
#pragma unroll 1
            for (int c0 = 0; c0 < d128::D; c0 += 32) {  // every lane takes the warp-collective loads
                uint32_t r[32];
                if (have) {
                    f32_ld32(trow + d128::kDq + c0, r);
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) r[c] = 0u;
                }
                if (q_in) {
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        *reinterpret_cast<float4 *>(dst + c0 + c) =
                            make_float4(__uint_as_float(r[c]), __uint_as_float(r[c + 1]), __uint_as_float(r[c + 2]),
                                        __uint_as_float(r[c + 3]));
                }
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// dK and dV at D = 128: two CTAs per 128-row kv block, so that each holds
// one accumulator of all 128 columns and only the products it needs; both
// walk the q side in chunks of 64 rows.
//   role 0 (dK): S^T = K Q^T (K parts resident in shared memory), dP^T = V
//     dO^T (V parts the A operand from tensor memory), dS^T elementwise and
//     dK += dS^T Q.  One ring stage (the resident K leaves room for no
//     second); three 64-column TMEM slots: S^T of every chunk in slot X,
//     dP^T in Y and Z by turns, so that dP^T of the next chunk is issued
//     while the elementwise warps work on this one (its dO half frees as
//     soon as this chunk's dP^T is done).  The dS^T parts go over dP^T and
//     the first half of each 32-column half of S^T.
//   role 1 (dV): S^T = K Q^T (K parts the A operand from tensor memory), P^T
//     elementwise and dV += P^T dO, through a two-stage ring; it needs
//     neither dP^T nor delta.  Two buffers of S^T (64) | P3 (32), P1 and P2
//     over S^T.
// Tensor memory (512 columns): A parts (V or K: 3 x 64) | accumulator (128) |
// 192 columns of slots or buffers.  The row values of a chunk (lse, delta)
// travel with the half of its ring stage that is freed last: the Q half in
// role 0 (read by dK), the dO half in role 1 (read by dV).
namespace d128kv {
constexpr int D = 128;
constexpr int kQr = 64;                          // q rows per chunk
constexpr uint32_t kA = 0, kAcc = 192;
constexpr uint32_t kKPart = 128 * D * 2;         // 32 KB: one part of role 0's resident K (two 64-wide atoms)
constexpr uint32_t kKAtom = 128 * 128;           // 128 rows x 64 bf16
constexpr uint32_t kCPart = kQr * D * 2;         // 16 KB: one part of a 64-row Q or dO chunk
constexpr uint32_t kCAtom = kQr * 128;           // 64 rows x 64 bf16
constexpr uint32_t kStQ = 0, kStDo = 3 * kCPart, kStRows = 6 * kCPart;  // rows: role 0 lse[64], delta[64]; role 1 lse[64]
constexpr uint32_t kStBytes = 6 * kCPart + 1024;
template <int ROLE>
struct Role;
template <>
struct Role<0> {
    static constexpr uint32_t kSt0 = 3 * kKPart;  // after the resident K
    static constexpr int kStages = 1, kRowGrp = 0, kRowVals = 128;
};
template <>
struct Role<1> {
    static constexpr uint32_t kSt0 = 0;
    static constexpr int kStages = 2, kRowGrp = 1, kRowVals = 64;
};
// role 0: slot X holds S^T, dP^T alternates between Y and Z
constexpr uint32_t kSlotX = 320;
__host__ __device__ constexpr uint32_t dp_slot(int j) { return 384u + 64u * (uint32_t)(j & 1); }
// role 1: S^T (64) | P3 (32) buffers
__host__ __device__ constexpr uint32_t s_buf(int b) { return 320u + 96u * (uint32_t)b; }
constexpr uint32_t kMiscOff = 2 * kStBytes;
static_assert(Role<0>::kSt0 + kStBytes <= kMiscOff, "role 0's shared memory");
constexpr size_t kSmemBytes = kMiscOff + sizeof(Misc) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert(dp_slot(1) + 64 == kTmemCols && s_buf(1) + 96 == kTmemCols, "tensor memory");
static_assert(Role<0>::kSt0 % 1024 == 0 && kStBytes % 1024 == 0, "ring alignment");
}  // namespace d128kv

template <int SCORE, int ROLE>
__device__ __forceinline__ void dkdv128_role(const AttnProblem &p, const BwdF32TcArgs &a, uint8_t *smem, Misc &ms,
                                             int kvb, int bh, int warp, int lane) {
    namespace c = d128kv;
    using R = c::Role<ROLE>;
    const int h = bh % p.H, b = bh / p.H;
    const int kv0 = kvb * kBlock;
    const uint32_t tmem = ms.tmem_base;
    volatile int *abort_flag = &ms.abort;
    constexpr int kPerTile = kBlock / c::kQr;
    const int nchunk = kPerTile * ms.ntiles;
    auto chunk_q0 = [&](int j) { return (int)(ms.list[j / kPerTile] & 0xFFFFu) * kBlock + (j % kPerTile) * c::kQr; };
    // ring stage of chunk j and the parity of its n-th use
    auto stage_of = [](int j) { return R::kStages == 1 ? 0 : (j & 1); };
    auto use_of = [](int j) { return R::kStages == 1 ? j : (j >> 1); };
    auto stage = [&](int s) { return smem + R::kSt0 + s * c::kStBytes; };
    const int qi = q_index(warp), di = do_index(warp);

    if (qi >= 0 || di >= 0) {
        // ----------------------------------------------------------- producers
        const int lt = 32 * (qi >= 0 ? qi : di) + lane, grp = qi >= 0 ? 0 : 1;
        if (ROLE == 0 && grp == 0 && nchunk > 0) {
            // role 0's resident K: two 64-row halves of the 128-row tile
            const float *kbase = static_cast<const float *>(p.k) + b * p.k_stride[0] + h * p.k_stride[1];
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                d128::Rows64 g;
                d128::load64(g, kbase, p.k_stride[2], kv0 + 64 * half, p.kv_len, lt);
                d128::store64(smem, c::kKPart, c::kKAtom, 64 * half, g, lt);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.kv_ready);
        }
        const float *base = grp == 0 ? static_cast<const float *>(p.q) + b * p.q_stride[0] + h * p.q_stride[1]
                                     : a.dout + (int64_t)bh * p.q_len * c::D;
        const int64_t rs = grp == 0 ? p.q_stride[2] : c::D;
        const float *lse_g = p.lse + (int64_t)bh * p.q_len, *delta_g = a.delta + (int64_t)bh * p.q_len;
        const bool rows = grp == R::kRowGrp && lt < R::kRowVals;
        bool ok = true;
        for (int j = 0; j < nchunk; ++j) {
            const int s = stage_of(j);
            const int q0 = chunk_q0(j);
            // this chunk's rows (and its row values) into registers, then the slot
            d128::Rows64 g;
            d128::load64(g, base, rs, q0, p.q_len, lt);
            // role 0: lse of rows 0-63, then their delta; role 1: lse of rows 0-63
            float rowv = 0.f;
            if (rows) {
                const bool is_lse = lt < 64;
                const int q = q0 + (is_lse ? lt : lt - 64);
                rowv = q < p.q_len ? (is_lse ? lse_g[q] : delta_g[q]) : (is_lse ? -INFINITY : 0.f);
            }
            if (j >= R::kStages &&
                !f32_warp_wait(&ms.st_empty[s][grp], (uint32_t)(use_of(j) - 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            d128::store64(stage(s) + (grp == 0 ? c::kStQ : c::kStDo), c::kCPart, c::kCAtom, 0, g, lt);
            if (rows) reinterpret_cast<float *>(stage(s) + c::kStRows)[lt] = rowv;
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.st_full[s][grp]);
        }
        if (!ok) fail(ms, p.status);
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------------------- MMA
        if (lane == 0 && nchunk > 0) {
            constexpr uint32_t kHi = smem_desc_hi_sw128(1024);
            constexpr uint32_t idesc_kmaj = idesc_bf16_f32(128, c::kQr, 0, 0);  // S^T, dP^T: N = 64 q rows
            constexpr uint32_t idesc_mn = idesc_bf16_f32(128, c::D, 0, 1);      // dK, dV: N = 128, B MN-major
            auto pa = [](int t) { return t == 2 || t == 4 ? 1 : t == 5 ? 2 : 0; };
            auto pbp = [](int t) { return t == 1 || t == 4 ? 1 : t == 3 ? 2 : 0; };
            // The K-step loops that issue MMAs stay rolled loops: unrolled,
            // the issue code no longer fits the instruction cache beside the
            // other roles' (measured: the issue rate and the elementwise warps
            // both slowed).  K-major B of a chunk (rows = q), part pt, K step
            // k of 16 head dims:
            auto kstep = [](int pt, int k) { return (pt * c::kCPart + (k / 4) * c::kCAtom + (k % 4) * 32) >> 4; };
            // S^T(j) = K Q^T into `dcol`: role 0 with K parts in shared
            // memory (SS), role 1 with K parts in TMEM (TS); frees nothing
            // (role 1 frees the Q half after it)
            auto issue_s = [&](int j, uint32_t dcol) -> bool {
                const int s = stage_of(j);
                if (!mbar_wait(&ms.st_full[s][0], (uint32_t)use_of(j) & 1u, abort_flag)) return false;
                tc_fence_after_sync();
                const uint32_t qd = smem_desc_lo(smem_u32(stage(s)) + c::kStQ, 16);
                if (ROLE == 0) {
                    const uint32_t kd = smem_desc_lo(smem_u32(smem), 16);
#pragma unroll 1
                    for (int k = 0; k < c::D / 16; ++k)
#pragma unroll
                        for (int t = 0; t < 6; ++t)
                            mma_ss_lo<kHi, kHi>(tmem + dcol,
                                                kd + ((pa(t) * c::kKPart + (k / 4) * c::kKAtom + (k % 4) * 32) >> 4),
                                                qd + kstep(pbp(t), k), idesc_kmaj, (k > 0 || t > 0) ? 1u : 0u);
                } else {
#pragma unroll 1
                    for (int k = 0; k < c::D / 16; ++k)
#pragma unroll
                        for (int t = 0; t < 6; ++t)
                            mma_ts_lo<kHi>(tmem + dcol, tmem + c::kA + 64 * pa(t) + 8 * k, qd + kstep(pbp(t), k),
                                           idesc_kmaj, (k > 0 || t > 0) ? 1u : 0u);
                    mma_commit(&ms.st_empty[s][0]);
                }
                mma_commit(&ms.s_full[ROLE == 0 ? 0 : s]);
                return true;
            };
            // role 0: dP^T(j) = V dO^T into its slot, then the dO half is free
            auto issue_dp = [&](int j) -> bool {
                if (!mbar_wait(&ms.st_full[0][1], (uint32_t)j & 1u, abort_flag)) return false;
                tc_fence_after_sync();
                const uint32_t gd = smem_desc_lo(smem_u32(stage(0)) + c::kStDo, 16);
#pragma unroll 1
                for (int k = 0; k < c::D / 16; ++k)
#pragma unroll
                    for (int t = 0; t < 6; ++t)
                        mma_ts_lo<kHi>(tmem + c::dp_slot(j), tmem + c::kA + 64 * pa(t) + 8 * k, gd + kstep(pbp(t), k),
                                       idesc_kmaj, (k > 0 || t > 0) ? 1u : 0u);
                mma_commit(&ms.st_empty[0][1]);
                return true;
            };
            // role 0: dK += dS^T Q; role 1: dV += P^T dO (B MN-major: two
            // 64-wide slabs one atom apart, K steps of 16 q rows = 2048 bytes)
            auto issue_acc = [&](int j) -> bool {
                const int s = stage_of(j);
                const int pb = ROLE == 0 ? 0 : s;
                if (!mbar_wait(&ms.p_full[pb], (uint32_t)use_of(j) & 1u, abort_flag)) return false;
                if (ROLE == 1 && !mbar_wait(&ms.st_full[s][1], (uint32_t)use_of(j) & 1u, abort_flag)) return false;
                tc_fence_after_sync();
                const uint32_t bm = smem_desc_lo(smem_u32(stage(s)) + (ROLE == 0 ? c::kStQ : c::kStDo), c::kCAtom);
#pragma unroll 1
                for (int k = 0; k < c::kQr / 16; ++k)
#pragma unroll
                    for (int t = 0; t < 6; ++t) {
                        const uint32_t ap = (uint32_t)pa(t), h32 = 32u * (uint32_t)(k / 2), o8 = 8u * (uint32_t)(k % 2);
                        // role 0: dS1, dS2 over dP^T, dS3 over the S^T slot;
                        // role 1: P1, P2 over S^T, P3 in the spare columns
                        const uint32_t col =
                            ROLE == 0 ? (ap < 2 ? c::dp_slot(j) + h32 + 16u * ap + o8 : c::kSlotX + h32 + o8)
                                      : (ap < 2 ? c::s_buf(s) + h32 + 16u * ap + o8
                                                : c::s_buf(s) + 64u + 16u * (uint32_t)(k / 2) + o8);
                        mma_ts_lo<kHi>(tmem + c::kAcc, tmem + col, bm + ((pbp(t) * c::kCPart + k * 2048) >> 4),
                                       idesc_mn, (j > 0 || k > 0 || t > 0) ? 1u : 0u);
                    }
                mma_commit(&ms.st_empty[s][ROLE == 0 ? 0 : 1]);
                return true;
            };
            bool ok = mbar_wait(&ms.kv_ready, 0, abort_flag);
            if (ok) tc_fence_after_sync();
            if (ROLE == 0) {
                // dP^T(0), S^T(0); then per chunk dP^T(j + 1) (its slot was
                // last read by dK(j - 1), issued earlier), dK(j), S^T(j + 1)
                // over the slot dK(j) read: MMAs of one thread run in order
                ok = ok && issue_dp(0) && issue_s(0, c::kSlotX);
                for (int j = 0; ok && j < nchunk; ++j)
                    ok = (j + 1 >= nchunk || issue_dp(j + 1)) && issue_acc(j) &&
                         (j + 1 >= nchunk || issue_s(j + 1, c::kSlotX));
            } else {
                for (int j = 0; ok && j < min(nchunk, 2); ++j) ok = issue_s(j, c::s_buf(j & 1));
                // S^T(j + 2) reuses the buffer dV(j) read: MMAs of one thread run in order
                for (int j = 0; ok && j < nchunk; ++j)
                    ok = issue_acc(j) && (j + 2 >= nchunk || issue_s(j + 2, c::s_buf(j & 1)));
            }
            if (ok) mma_commit(&ms.acc_full);
            if (!ok) fail(ms, p.status);
            mma_commit(&ms.drain);  // every MMA issued above completes before TMEM is freed
            int never = 0;
            (void)mbar_wait(&ms.drain, 0, &never);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ---------------------------------------------------------- elementwise
        const int kv = kv0 + (int)threadIdx.x;
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        const float slope = SCORE == FLEX_SCORE_ALIBI ? exp2f(-8.f * (float)(h + 1) / (float)p.H) : 0.f;
        const float scale = p.scale;
        bool ok = true;
        if (nchunk > 0) {
            // this kv row of V (role 0) or K (role 1) -> the three A parts (bf16 pairs)
            const bool kv_in = kv < p.kv_len;
            const float *arow =
                ROLE == 0 ? static_cast<const float *>(p.v) + b * p.v_stride[0] + h * p.v_stride[1] +
                                (int64_t)(kv_in ? kv : 0) * p.v_stride[2]
                          : static_cast<const float *>(p.k) + b * p.k_stride[0] + h * p.k_stride[1] +
                                (int64_t)(kv_in ? kv : 0) * p.k_stride[2];
#pragma unroll 1
            for (int c0 = 0; c0 < c::D; c0 += 32) {
                float4 x[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    x[i] = kv_in ? __ldg(reinterpret_cast<const float4 *>(arow + c0) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                uint32_t w1[16], w2[16], w3[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    split3(f4_at(x[i / 2], 2 * (i % 2)), f4_at(x[i / 2], 2 * (i % 2) + 1), w1[i], w2[i], w3[i]);
                tmem_st16(trow + c::kA + c0 / 2, w1);
                tmem_st16(trow + c::kA + 64 + c0 / 2, w2);
                tmem_st16(trow + c::kA + 128 + c0 / 2, w3);
            }
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.kv_ready);
        }
        for (int j = 0; j < nchunk; ++j) {
            const int s = stage_of(j);
            const bool full = (ms.list[j / kPerTile] >> 16) & 1u;
            const int q0 = chunk_q0(j);
            // S^T (and in role 0 dP^T, issued before it) are in TMEM; the row
            // values (written by the producers) are read after their own barrier
            if (!f32_warp_wait(&ms.s_full[ROLE == 0 ? 0 : s], (uint32_t)use_of(j) & 1u, abort_flag) ||
                !f32_warp_wait(&ms.st_full[s][R::kRowGrp], (uint32_t)use_of(j) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const float *rows_s = reinterpret_cast<const float *>(stage(s) + c::kStRows);
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                const uint32_t scol = ROLE == 0 ? c::kSlotX + 32u * half : c::s_buf(s) + 32u * half;
                uint32_t sr[32];
                f32_ld32(trow + scol, sr);
                if (ROLE == 0) {
                    const uint32_t dcol = c::dp_slot(j) + 32u * half;
                    uint32_t dr[32];
                    f32_ld32(trow + dcol, dr);
                    float dsv[32];
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) {
                        const int q = q0 + 32 * half + cc;
                        const float lse = rows_s[32 * half + cc];
                        const bool keep = lse != -INFINITY && (full || (kv < p.kv_len && mask_mod(p.mask, b, q, kv)));
                        float grad;
                        const float x =
                            score_t<SCORE>(p.score_param, __uint_as_float(sr[cc]) * scale, slope, q, kv, grad);
                        const float pr = keep ? ex2_approx(fmaf(x, kLog2e, -lse * kLog2e)) : 0.f;
                        dsv[cc] = keep ? scale * pr * (__uint_as_float(dr[cc]) - rows_s[64 + 32 * half + cc]) * grad
                                       : 0.f;
                    }
                    uint32_t w1[16], w2[16], w3[16];
#pragma unroll
                    for (int cc = 0; cc < 16; ++cc) split3(dsv[2 * cc], dsv[2 * cc + 1], w1[cc], w2[cc], w3[cc]);
                    // over this half's dP^T and S^T columns, all read above
                    tmem_st16(trow + dcol, w1);
                    tmem_st16(trow + dcol + 16, w2);
                    tmem_st16(trow + scol, w3);
                } else {
                    float pv[32];
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) {
                        const int q = q0 + 32 * half + cc;
                        const float lse = rows_s[32 * half + cc];
                        const bool keep = lse != -INFINITY && (full || (kv < p.kv_len && mask_mod(p.mask, b, q, kv)));
                        float grad;
                        const float x =
                            score_t<SCORE>(p.score_param, __uint_as_float(sr[cc]) * scale, slope, q, kv, grad);
                        pv[cc] = keep ? ex2_approx(fmaf(x, kLog2e, -lse * kLog2e)) : 0.f;
                    }
                    uint32_t w1[16], w2[16], w3[16];
#pragma unroll
                    for (int cc = 0; cc < 16; ++cc) split3(pv[2 * cc], pv[2 * cc + 1], w1[cc], w2[cc], w3[cc]);
                    // over S^T columns 32 half .. 32 half + 31, all read above
                    tmem_st16(trow + scol, w1);
                    tmem_st16(trow + scol + 16, w2);
                    tmem_st16(trow + c::s_buf(s) + 64 + 16 * half, w3);
                }
            }
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.p_full[ROLE == 0 ? 0 : s]);
        }
        // ------------------------------------------------------------ epilogue
        const bool have = ok && nchunk > 0;
        if (have && !f32_warp_wait(&ms.acc_full, 0, abort_flag)) ok = false;
        if (!ok) fail(ms, p.status);
        if (ok) {
            tc_fence_after_sync();
            const int64_t orow = (int64_t)bh * p.kv_len + (kv < p.kv_len ? kv : 0);
            float *dst = (ROLE == 0 ? a.dk : a.dv) + orow * c::D;
#pragma unroll 1
            for (int c0 = 0; c0 < c::D; c0 += 32) {  // every lane takes the warp-collective loads
                uint32_t r[32];
                if (have) {
                    f32_ld32(trow + c::kAcc + c0, r);
                } else {
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc) r[cc] = 0u;
                }
                if (kv < p.kv_len) {
#pragma unroll
                    for (int cc = 0; cc < 32; cc += 4)
                        *reinterpret_cast<float4 *>(dst + c0 + cc) =
                            make_float4(__uint_as_float(r[cc]), __uint_as_float(r[cc + 1]),
                                        __uint_as_float(r[cc + 2]), __uint_as_float(r[cc + 3]));
                }
            }
        }
    }
}

template <int SCORE>
__global__ void __launch_bounds__(16 * 32, 1) dkdv128_kernel(AttnProblem p, BwdF32TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Misc &ms = *reinterpret_cast<Misc *>(smem + d128kv::kMiscOff);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int kvb = (int)blockIdx.y / 2, role = (int)blockIdx.y & 1;  // role 0: dK, role 1: dV
    const int bh = p.bh_begin + (int)blockIdx.x;

    if (threadIdx.x == 0) {
        // role 0: K resident (Q group) and V in TMEM (elementwise warps); role 1: K in TMEM
        mbar_init(&ms.kv_ready, role == 0 ? 8 : 4);
        for (int i = 0; i < 2; ++i) {
            for (int g = 0; g < 2; ++g) {
                mbar_init(&ms.st_full[i][g], 4);
                mbar_init(&ms.st_empty[i][g], 1);
            }
            mbar_init(&ms.s_full[i], 1);
            mbar_init(&ms.p_full[i], 4);
        }
        mbar_init(&ms.acc_full, 1);
        mbar_init(&ms.drain, 1);
        ms.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        const TileLists lists{a.q_num, a.q_idx, a.fq_num, a.fq_idx, p.nkvb, p.nqb, p.kv_block, p.q_block, p.nqt};
        for (int i = lane; i < p.nqt; i += 32) ms.flags[i] = 0u;
        __syncwarp();
        tl_mark_warp(lists, bh, kvb, 0, ms.flags, 0, p.nqt, lane);
        __syncwarp();
        const uint32_t expect = tl_expect(lists);
        const unsigned lt = (1u << lane) - 1u;
        int cnt = 0;
        for (int base = 0; base < p.nqt; base += 32) {
            const int i = base + lane;
            const uint32_t w = i < p.nqt ? ms.flags[i] : 0u;
            const bool on = tl_listed(w, 0);
            const unsigned bal = __ballot_sync(0xffffffffu, on);
            if (on) ms.list[cnt + __popc(bal & lt)] = (uint32_t)i | (tl_full(expect, w, 0) ? (1u << 16) : 0u);
            cnt += __popc(bal);
        }
        if (lane == 0) ms.ntiles = cnt;
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&ms.tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();

    if (role == 0)
        dkdv128_role<SCORE, 0>(p, a, smem, ms, kvb, bh, warp, lane);
    else
        dkdv128_role<SCORE, 1>(p, a, smem, ms, kvb, bh, warp, lane);

    // ------------------------------------------------------------ teardown
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(ms.tmem_base, kTmemCols);
    }
}

}  // namespace bwdf32

// dK and dV of fp32 inputs on the tensor cores (p.D == 64 or 128; p.nqt <=
// kBwdF32TcMaxQTiles).
inline cudaError_t launch_bwd_fp32_tc_dkdv(const AttnProblem &p, const BwdF32TcArgs &a, cudaStream_t stream) {
    using namespace bwdf32;
    const bool d64 = p.D == 64;
    const size_t smem = d64 ? kSmemBytes : d128kv::kSmemBytes;
    // D = 128: two CTAs per kv block, one for dK and one for dV
    const unsigned gy = (unsigned)p.nkvt * (d64 ? 1u : 2u);
    static_assert(2 * kMaxKvBlocks <= 65535, "kv blocks along grid.y");
    auto pick = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        for (int begin = 0; begin < p.B * p.H; begin += 65535) {
            AttnProblem part = p;
            part.bh_begin = begin;
            const int count = p.B * p.H - begin < 65535 ? p.B * p.H - begin : 65535;
            kern<<<dim3(count, gy), kThreads, smem, stream>>>(part, a);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        return cudaSuccess;
    };
    switch (p.score_kind) {
        case FLEX_SCORE_SOFTCAP:
            return d64 ? pick(dkdv_kernel<FLEX_SCORE_SOFTCAP>) : pick(dkdv128_kernel<FLEX_SCORE_SOFTCAP>);
        case FLEX_SCORE_ALIBI:
            return d64 ? pick(dkdv_kernel<FLEX_SCORE_ALIBI>) : pick(dkdv128_kernel<FLEX_SCORE_ALIBI>);
        default:
            return d64 ? pick(dkdv_kernel<FLEX_SCORE_IDENTITY>) : pick(dkdv128_kernel<FLEX_SCORE_IDENTITY>);
    }
}

// dQ of fp32 inputs on the tensor cores (p.D == 64 or 128).
inline cudaError_t launch_bwd_fp32_tc_dq(const AttnProblem &p, const BwdF32TcArgs &a, cudaStream_t stream) {
    using namespace bwdf32;
    const size_t smem = p.D == 64 ? kDqSmemBytes : d128::kSmemBytes;
    const bool bh_x = p.nqt <= 65535;
    auto pick = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        for (int begin = 0; begin < p.B * p.H; begin += 65535) {
            AttnProblem part = p;
            part.bh_begin = begin;
            const int count = p.B * p.H - begin < 65535 ? p.B * p.H - begin : 65535;
            if (bh_x)
                kern<<<dim3(count, p.nqt), kThreads, smem, stream>>>(part, a, 1);
            else
                kern<<<dim3(p.nqt, count), kThreads, smem, stream>>>(part, a, 0);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        return cudaSuccess;
    };
    const bool d64 = p.D == 64;
    switch (p.score_kind) {
        case FLEX_SCORE_SOFTCAP:
            return d64 ? pick(dq_kernel<FLEX_SCORE_SOFTCAP>) : pick(dq128_kernel<FLEX_SCORE_SOFTCAP>);
        case FLEX_SCORE_ALIBI:
            return d64 ? pick(dq_kernel<FLEX_SCORE_ALIBI>) : pick(dq128_kernel<FLEX_SCORE_ALIBI>);
        default:
            return d64 ? pick(dq_kernel<FLEX_SCORE_IDENTITY>) : pick(dq128_kernel<FLEX_SCORE_IDENTITY>);
    }
}

}  // namespace flex
