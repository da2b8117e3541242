// Backward pass of the block-sparse attention for bf16 inputs on sm_103a
// tensor cores (the flex_attention_backward op of "[Inductor][Flex
// Attention] Add Subtiling Option for Alpha Scaling", PyTorch PR #167356,
// test diffs: q, k, v, the forward's out and lse and the output gradient in;
// dq, dk, dv out).
//
// With t = scale q.k, s = score_mod(t) where mask_mod holds (-inf elsewhere),
// P = exp(s - lse), delta_i = dO_i . out_i:
//   dV_j = sum_i P_ij dO_i
//   dS_ij = P_ij (dO_i . v_j - delta_i) score_mod'(t_ij)
//   dK_j = scale sum_i dS_ij q_i,   dQ_i = scale sum_j dS_ij k_j
//
// Two launches of one kernel template, each work item one owned 128-row block:
//   KV_MAJOR  a kv block j, walking the q blocks of the q side of the
//             BlockMask (q_num_blocks / q_indices and the full variants):
//               S^T  = K_j Q_i^T          (SS MMA, TMEM)
//               dP^T = V_j dO_i^T         (SS MMA, TMEM)
//               P^T, dS^T by the elementwise warps (bf16 back into TMEM)
//               dV_j += P^T dO_i          (TS MMA: P^T read from TMEM)
//               dK_j += dS^T Q_i          (TS MMA: dS^T read from TMEM)
//   Q-major   a q block i, walking the kv side of the BlockMask:
//               S = Q_i K_j^T, dP = dO_i V_j^T, dS, dQ_i += dS K_j.
// One CTA computes an item's output rows whole, so nothing is accumulated
// across CTAs and the result does not depend on scheduling.  P is recomputed from the saved
// lse (no running max).  Roles (320 threads, one CTA per SM):
//   warps 0-7  elementwise, two threads per owned row (TMEM lane = row):
//              warps w and w + 4 share a TMEM lane quarter, the first takes
//              the walked columns 0-63, the second 64-127 (the backward
//              needs no row reductions, so the halves never talk)
//   warp 8     scheduler and TMA: builds each work item's list, loads its
//              two resident tiles, then the two streamed tiles of each list
//              step into rings that run on across items, and takes the next
//              item from the grid (cluster launch control): the CTAs are
//              persistent, one per SM
//   warp 9     one thread issues every tcgen05.mma
// The MMA thread issues, per step n: dV(n) once P(n) is in TMEM, S(n+1)
// (into the columns P(n) was read from: MMAs execute in issue order), dK(n)
// (or dQ(n)) once dS(n) is in TMEM, then dP(n+1) (over dS(n)), so the
// elementwise work of step n+1 overlaps the accumulating MMAs of step n.
// Every wait is bounded; on timeout the CTA records FLEX_ERR_DEVICE_TIMEOUT
// in the status word, drains its copies and MMAs, frees TMEM and exits.
#pragma once

#include <cfloat>
#include <climits>
#include <cstddef>
#include <type_traits>

#include "flex_internal.h"
#include "ptx.cuh"
#include "tilelist.cuh"

namespace flex {

constexpr int kBwdThreads = 320;
constexpr int kBwdTmaWarp = 8;
constexpr int kBwdMmaWarp = 9;
constexpr int kBwdMaxList = 2048;    // list steps per CTA held on chip (q blocks of a kv block)
constexpr int kBwdHeadGroup = 4;     // (batch, head) pairs scheduled together (their tiles stay in L2)
constexpr float kBwdLog2e = 1.4426950408889634f;

struct BwdTcParams {
    int B, H, q_len, kv_len;
    int nblocks;                  // 128-tiles of the owned dimension (kv when KV_MAJOR, else q)
    int bh_begin, nbh;
    TileLists lists;              // the BlockMask side that lists the walked dimension, read as 128-tiles
    MaskDesc mask;
    float scale, score_param;
    const float *lse, *delta;     // [B, H, q_len]
    uint16_t *out0, *out1;        // KV_MAJOR: dv, dk; else dq (out1 unused); bf16, contiguous
    int *status;
};

// One work item (a 128-row block of one (batch, head)) as the scheduler
// publishes it: the walked tiles of its BlockMask list side.
struct BwdSlot {
    int n;      // list steps; -1: no more work for this CTA
    int own;    // owned block
    int bh;     // b * H + h
    int pad;
    alignas(16) uint32_t list[kBwdMaxList];  // walked tile | full << 16, ascending
};

struct BwdMisc {
    uint64_t res_full, res_empty;           // the item's two resident tiles landed / no longer read
    uint64_t a_full[4], a_empty[4];         // ring of the first streamed tile (K, or Q when KV_MAJOR)
    uint64_t b_full[4], b_empty[4];         // ring of the second (V, or dO when KV_MAJOR)
    uint64_t s_full, dp_full, p_ready, ds_ready, acc_full, drain;
    uint64_t col_ready[2];                  // the elementwise warps' per-column data of a step
    uint64_t item_ready[2], item_free[2];   // per item slot
    uint64_t clc_bar;                       // cluster-launch-control response landed
    uint32_t tmem_base;
    int abort;
    alignas(16) uint32_t clc_resp[4];
    alignas(16) float colv[2][128];         // per column of a step (see the elementwise code)
    alignas(16) float dltv[2][128];         // KV_MAJOR: -delta of each q column
    alignas(16) int32_t docv[2][128];       // document ids of the walked block's rows
    alignas(16) uint32_t words[kBwdMaxList];// per walked tile: listed bit and full-pair count (tilelist.cuh)
    BwdSlot slot[2];
};
static_assert(offsetof(BwdMisc, clc_resp) % 16 == 0, "clc_resp alignment");
static_assert(offsetof(BwdMisc, slot) % 16 == 0 && sizeof(BwdSlot) % 16 == 0, "slot alignment");
// arrivals that free an item slot: the MMA thread and the 8 elementwise warps
constexpr uint32_t kBwdItemConsumers = 9;

// The two streamed tiles of a step have rings of their own.  The first (K, or
// Q when KV_MAJOR) is read by the step's S MMA, issued a step ahead, and by
// its dQ (dK) MMA at the end of the step; the second (V, or dO) by the dP
// MMA, issued a step ahead, and when KV_MAJOR by the dV MMA in mid-step.  At
// D = 128 shared memory holds four streamed tiles: two of each when
// KV_MAJOR; otherwise three K and one V, since V is released as soon as its
// dP MMA is done and K must arrive a step before its S MMA.
template <int D, bool KV_MAJOR>
struct BwdTcCfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kAtoms = D / 64;
    static constexpr uint32_t kAtomBytes = 128 * 128;
    static constexpr uint32_t kTileBytes = 128 * D * 2;
    static constexpr int kNA = D == 128 ? (KV_MAJOR ? 2 : 3) : 4;  // ring depths
    static constexpr int kNB = D == 128 ? (KV_MAJOR ? 2 : 1) : 4;
    // rings of equal depth share the first ring's barriers (one wait and one
    // release per step for both tiles, as one stage of two tiles)
    static constexpr bool kSplit = kNA != kNB;
    static constexpr uint32_t kResOff = 0;                         // two resident tiles
    static constexpr uint32_t kAOff = 2 * kTileBytes;              // ring of the first streamed tile
    static constexpr uint32_t kBOff = kAOff + kNA * kTileBytes;    // ring of the second
    static constexpr uint32_t kMiscOff = kBOff + kNB * kTileBytes;
    static constexpr uint32_t kSmemBytes = kMiscOff + sizeof(BwdMisc) + 1024;
    // TMEM columns: S | dP | acc0 | acc1.  P (KV_MAJOR) and dS are written
    // back as bf16 over the columns they came from: the walked columns
    // 64h .. 64h + 63 of S (dP) pack into S's (dP's) columns 64h .. 64h + 31,
    // so each column half writes only where it has read.
    static constexpr uint32_t kS = 0, kDP = 128, kAcc0 = 256, kAcc1 = 256 + D;
    static constexpr uint32_t kTmemCols = 512;
};

__device__ __forceinline__ void bwd_fail(BwdMisc &ms, int *status) {
    *reinterpret_cast<volatile int *>(&ms.abort) = 1;
    atomicCAS(status, 0, kDeviceTimeout);
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ void drain_wait_bwd(uint64_t *bar, uint32_t parity) {
    int never = 0;
    (void)mbar_wait(bar, parity, &never);
}

// A wait taken by all 32 lanes of a warp, with one outcome for the warp.
__device__ __forceinline__ bool bwd_warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        const int stop = (*abort != 0) || (global_timer_ns() - t0 > kWaitLimitNs);
        if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
}

// TMEM read of 32 columns of this thread's lane, completed before returning.
__device__ __forceinline__ void bwd_tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
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

// TMEM read of 64 columns of this thread's lane (two 32-column loads, one
// wait), completed before returning.
__device__ __forceinline__ void bwd_tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]),
          "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]),
          "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]),
          "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]),
          "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(taddr), "r"(taddr + 32)
        : "memory");
}

// The q rows that keep key row kv (the enumerated interval mask_mods read
// along a column): [lo, hi], empty when lo > hi.  Rows at or past Q_LEN and
// keys at or past KV_LEN are padding.
__device__ __forceinline__ void mask_col_interval(const MaskDesc &m, int kv, int &lo, int &hi) {
    int64_t l = 0, h = (int64_t)m.q_len - 1;
    switch (m.kind) {
        case FLEX_MASK_CAUSAL:
            l = kv;
            break;
        case FLEX_MASK_SLIDING_WINDOW:  // q >= kv and q - kv < W
            l = kv;
            h = min(h, (int64_t)kv + (int64_t)m.window - 1);
            break;
        case FLEX_MASK_CAUSAL_PREFIX:   // (q <= P and kv <= P) or q >= kv
            l = kv <= m.prefix ? 0 : kv;
            break;
        default:                        // all
            break;
    }
    if (kv >= m.kv_len) h = l - 1;
    lo = (int)l;
    hi = (int)max(h, l - 1);
}

// Keep-bits of a 32-column chunk whose columns are base .. base + 31, for a
// kept interval [lo, hi] of column indices.
__device__ __forceinline__ uint32_t interval_bits(int lo, int hi, int base) {
    const int a = max(lo - base, 0), b = min(hi - base, 31);
    if (a > b) return 0u;
    return (0xFFFFFFFFu >> (31 - b)) & (0xFFFFFFFFu << a);
}

// Work item `item` of the launch (one CTA index): heads in groups of
// kBwdHeadGroup, and inside a group the heaviest blocks of causal-like masks
// first (kv block 0 has the most q blocks; the last q block the most kv
// blocks), heads innermost.
__device__ __forceinline__ void bwd_decode_item(const BwdTcParams &p, bool kv_major, int item, int &own, int &bh) {
    const int group_items = kBwdHeadGroup * p.nblocks;
    const int g0 = (item / group_items) * kBwdHeadGroup;
    const int gsize = min(kBwdHeadGroup, p.nbh - g0);
    const int r = item - (item / group_items) * group_items;
    own = kv_major ? r / gsize : p.nblocks - 1 - r / gsize;
    bh = p.bh_begin + g0 + r % gsize;
}

// The walked tiles of an item's block, with the 32 lanes of one warp: the
// BlockMask's lists (any block sizes) read as 128-tiles, in ascending order;
// counts are clamped and malformed entries dropped, so nothing is written or
// loaded out of bounds.
__device__ __forceinline__ void bwd_build_list(const BwdTcParams &p, bool kv_major, BwdMisc &ms, BwdSlot &sl, int item,
                                               int lane) {
    int own, bh;
    bwd_decode_item(p, kv_major, item, own, bh);
    const int nt = min(p.lists.walk_nt, kBwdMaxList);
    for (int i = lane; i < nt; i += 32) ms.words[i] = 0u;
    __syncwarp();
    tl_mark_warp(p.lists, bh, own, 0, ms.words, 0, nt, lane);
    __syncwarp();
    const unsigned lt = (1u << lane) - 1u;
    const uint32_t expect = tl_expect(p.lists);
    int cnt = 0;
    for (int base = 0; base < nt; base += 32) {
        const int i = base + lane;
        const uint32_t w = i < nt ? ms.words[i] : 0u;
        const bool ok = tl_listed(w, 0);
        const unsigned bal = __ballot_sync(0xffffffffu, ok);
        if (ok) sl.list[cnt + __popc(bal & lt)] = (uint32_t)i | (tl_full(expect, w, 0) ? (1u << 16) : 0u);
        cnt += __popc(bal);
    }
    if (lane == 0) {
        sl.n = cnt;
        sl.own = own;
        sl.bh = bh;
    }
}

// Persistent over work items: each CTA starts with the item of its own index
// and then takes items from CTAs of the grid that have not started yet
// (cluster launch control), so the next item's list, resident tiles and
// first streamed tiles load while the current one ends.  Every role walks the
// same sequence of published items; the ring, S/dP hand-off and column
// barriers run on across items with the CTA's global step count.
template <int D, int SCORE, bool DOC, bool KV_MAJOR>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap map_r0, const __grid_constant__ CUtensorMap map_r1,
                       const __grid_constant__ CUtensorMap map_s0, const __grid_constant__ CUtensorMap map_s1,
                       const BwdTcParams p) {
    using C = BwdTcCfg<D, KV_MAJOR>;
    constexpr int NA = C::kNA, NB = C::kNB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    BwdMisc &ms = *reinterpret_cast<BwdMisc *>(smem + C::kMiscOff);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int own_len = KV_MAJOR ? p.kv_len : p.q_len;
    const int walk_len = KV_MAJOR ? p.q_len : p.kv_len;

    if (threadIdx.x == 0) {
        mbar_init(&ms.res_full, 1);
        mbar_init(&ms.res_empty, 1);
        for (int s = 0; s < 4; ++s) {
            mbar_init(&ms.a_full[s], 1);
            mbar_init(&ms.a_empty[s], 1);
            mbar_init(&ms.b_full[s], 1);
            mbar_init(&ms.b_empty[s], 1);
        }
        mbar_init(&ms.s_full, 1);
        mbar_init(&ms.dp_full, 1);
        mbar_init(&ms.p_ready, 256);
        mbar_init(&ms.ds_ready, 256);
        mbar_init(&ms.acc_full, 1);
        mbar_init(&ms.drain, 1);
        mbar_init(&ms.col_ready[0], 128);
        mbar_init(&ms.col_ready[1], 128);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ms.item_ready[i], 1);
            mbar_init(&ms.item_free[i], kBwdItemConsumers);
        }
        mbar_init(&ms.clc_bar, 1);
        ms.abort = 0;
        fence_barrier_init();
    }
    if (warp == kBwdMmaWarp) {
        tmem_alloc(&ms.tmem_base, C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = ms.tmem_base;
    volatile int *abort_flag = &ms.abort;

    if (warp == kBwdTmaWarp) {
        // ------------------------------------------------ scheduler and TMA
        // Item n goes to slot n % 2 once every consumer has released that
        // slot's item n - 2.  The next item is taken from the grid once the
        // current one's last streamed tiles are on the way (about a ring
        // depth before its end) and its list built while the current item's
        // last steps compute.  An item's resident tiles load once the
        // previous item's MMAs are done with them (res_empty).
        if (lane == 0) {
            prefetch_tensormap(&map_r0);
            prefetch_tensormap(&map_r1);
            prefetch_tensormap(&map_s0);
            prefetch_tensormap(&map_s1);
        }
        int item = blockIdx.x;
        uint32_t g = 0;      // steps issued over all items
        uint32_t nw = 0;     // items with work (resident loads issued)
        uint32_t nclc = 0;   // launch-control responses consumed
        int na = 0, nb = 0;  // tiles issued into each ring
        bool ok = true;
        for (uint32_t it = 0;; ++it) {
            const int k = (int)(it & 1u);
            BwdSlot &sl = ms.slot[k];
            if (it >= 2 && !bwd_warp_wait(&ms.item_free[k], ((it - 2) >> 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            if (item >= 0) {
                bwd_build_list(p, KV_MAJOR, ms, sl, item, lane);
            } else if (lane == 0) {
                sl.n = -1;
            }
            __threadfence_block();  // every lane's slot writes before the release below
            __syncwarp();
            if (lane == 0) mbar_arrive(&ms.item_ready[k]);
            if (item < 0) break;
            const int N = sl.n;
            if (N > 0) {
                int lok = 1;
                if (lane == 0) {
                    const int own = sl.own, bh = sl.bh, b = bh / p.H, h = bh % p.H;
                    if (nw > 0 && !mbar_wait(&ms.res_empty, (nw - 1) & 1u, abort_flag)) lok = 0;
                    if (lok) {
                        mbar_arrive_expect_tx(&ms.res_full, 2 * C::kTileBytes);
                        for (int a = 0; a < C::kAtoms; ++a) {
                            tma_load_4d(smem + C::kResOff + a * C::kAtomBytes, &map_r0, &ms.res_full, 64 * a, own * 128,
                                        h, b);
                            tma_load_4d(smem + C::kResOff + C::kTileBytes + a * C::kAtomBytes, &map_r1, &ms.res_full,
                                        64 * a, own * 128, h, b);
                        }
                    }
                    for (int n = 0; lok && n < N; ++n) {
                        const uint32_t gn = g + (uint32_t)n;
                        const int sa = (int)(gn % NA), sb = (int)(gn % NB);
                        const uint32_t ua = gn / NA, ub = gn / NB;
                        const int blk = (int)(sl.list[n] & 0xFFFFu);
                        if (ua > 0 && !mbar_wait(&ms.a_empty[sa], (ua - 1) & 1u, abort_flag)) {
                            lok = 0;
                            break;
                        }
                        uint8_t *dst = smem + C::kAOff + sa * C::kTileBytes;
                        mbar_arrive_expect_tx(&ms.a_full[sa], (C::kSplit ? 1u : 2u) * C::kTileBytes);
                        for (int a = 0; a < C::kAtoms; ++a)
                            tma_load_4d(dst + a * C::kAtomBytes, &map_s0, &ms.a_full[sa], 64 * a, blk * 128, h, b);
                        ++na;
                        uint64_t *bbar = &ms.a_full[sa];
                        if constexpr (C::kSplit) {
                            if (ub > 0 && !mbar_wait(&ms.b_empty[sb], (ub - 1) & 1u, abort_flag)) {
                                lok = 0;
                                break;
                            }
                            bbar = &ms.b_full[sb];
                            mbar_arrive_expect_tx(bbar, C::kTileBytes);
                        }
                        dst = smem + C::kBOff + sb * C::kTileBytes;
                        for (int a = 0; a < C::kAtoms; ++a)
                            tma_load_4d(dst + a * C::kAtomBytes, &map_s1, bbar, 64 * a, blk * 128, h, b);
                        ++nb;
                    }
                }
                if (!__shfl_sync(0xffffffffu, lok, 0)) {
                    ok = false;
                    break;
                }
                g += (uint32_t)N;
                ++nw;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(&ms.clc_bar, 16u);
                clc_try_cancel(ms.clc_resp, &ms.clc_bar);
            }
            if (!bwd_warp_wait(&ms.clc_bar, nclc & 1u, abort_flag)) {
                ok = false;
                break;
            }
            ++nclc;
            int next = 0;
            if (lane == 0) next = clc_cancelled_x(ms.clc_resp);
            item = __shfl_sync(0xffffffffu, next, 0);
        }
        if (!ok && lane == 0) bwd_fail(ms, p.status);
        // every copy issued above lands before the CTA exits (lane 0 issued them)
        if (lane == 0) {
            if (nw > 0) drain_wait_bwd(&ms.res_full, (nw - 1) & 1u);
            for (int s = 0; s < NA && s < na; ++s) {
                const int last = s + ((na - 1 - s) / NA) * NA;
                drain_wait_bwd(&ms.a_full[s], (uint32_t)(last / NA) & 1u);
            }
            for (int s = 0; C::kSplit && s < NB && s < nb; ++s) {
                const int last = s + ((nb - 1 - s) / NB) * NB;
                drain_wait_bwd(&ms.b_full[s], (uint32_t)(last / NB) & 1u);
            }
        }
        __syncwarp();
    } else if (warp == kBwdMmaWarp) {
        // ------------------------------------------------------------ MMA
        if (lane == 0) {
            constexpr uint32_t idesc_ss = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t idesc_acc = idesc_bf16_f32(128, D, 0, 1);
            constexpr uint32_t kHi = smem_desc_hi_sw128(1024);
            const uint32_t r0_lo = smem_desc_lo(smem_u32(smem + C::kResOff), 16);
            const uint32_t r1_lo = smem_desc_lo(smem_u32(smem + C::kResOff + C::kTileBytes), 16);
            const uint32_t s0_lo = smem_desc_lo(smem_u32(smem + C::kAOff), 16);
            const uint32_t s1_lo = smem_desc_lo(smem_u32(smem + C::kBOff), 16);
            const uint32_t s0_mn = smem_desc_lo(smem_u32(smem + C::kAOff), C::kAtomBytes);
            const uint32_t s1_mn = smem_desc_lo(smem_u32(smem + C::kBOff), C::kAtomBytes);
            // A (M = 128 resident rows, K = D) times B^T (N = 128 walked rows, K = D), both K-major
            auto issue_ss = [&](uint32_t dcol, uint32_t a_lo, uint32_t b_lo) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = ((k / 4) * C::kAtomBytes + (k % 4) * 32) >> 4;
                    mma_ss_lo<kHi, kHi>(tmem + dcol, a_lo + off, b_lo + off, idesc_ss, k > 0 ? 1u : 0u);
                }
            };
            // acc (128 x D) += A (TMEM, 128 x 128 bf16) times B (128 walked rows x D, MN-major);
            // A's walked columns 16k .. 16k + 15 sit at TMEM column 64 (k / 4) + 8 (k % 4)
            auto issue_ts = [&](uint32_t dcol, uint32_t acol, uint32_t b_mn, bool acc) {
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_ts_lo<kHi>(tmem + dcol, tmem + acol + 64 * (k / 4) + 8 * (k % 4), b_mn + ((k * 2048) >> 4),
                                   idesc_acc, (k > 0 || acc) ? 1u : 0u);
            };
            constexpr uint32_t tile16 = C::kTileBytes >> 4;
            uint32_t g = 0, nw = 0;
            bool ok = true;
            for (uint32_t it = 0; ok; ++it) {
                const int k = (int)(it & 1u);
                const BwdSlot &sl = ms.slot[k];
                if (!mbar_wait(&ms.item_ready[k], (it >> 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const int N = sl.n;
                if (N < 0) break;
                if (N > 0) {
                    const int sa0 = (int)(g % NA), sb0 = (int)(g % NB);
                    ok = mbar_wait(&ms.res_full, nw & 1u, abort_flag) &&
                         mbar_wait(&ms.a_full[sa0], (g / NA) & 1u, abort_flag) &&
                         (!C::kSplit || mbar_wait(&ms.b_full[sb0], (g / NB) & 1u, abort_flag));
                    if (!ok) break;
                    tc_fence_after_sync();
                    issue_ss(C::kS, r0_lo, s0_lo + sa0 * tile16);
                    mma_commit(&ms.s_full);
                    issue_ss(C::kDP, r1_lo, s1_lo + sb0 * tile16);
                    mma_commit(&ms.dp_full);
                    if constexpr (C::kSplit && !KV_MAJOR) mma_commit(&ms.b_empty[sb0]);  // V is read by dP alone
                    for (int n = 0; ok && n < N; ++n) {
                        const uint32_t gn = g + (uint32_t)n;
                        const int sa = (int)(gn % NA), sb = (int)(gn % NB);
                        const bool nxt = n + 1 < N;
                        const int sa1 = (int)((gn + 1) % NA), sb1 = (int)((gn + 1) % NB);
                        if (!mbar_wait(&ms.p_ready, gn & 1u, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        if constexpr (KV_MAJOR) {
                            issue_ts(C::kAcc0, C::kS, s1_mn + sb * tile16, n > 0);  // dV += P^T dO
                            if constexpr (C::kSplit) mma_commit(&ms.b_empty[sb]);   // dO no longer read
                        }
                        if (nxt) {
                            if (!mbar_wait(&ms.a_full[sa1], ((gn + 1) / NA) & 1u, abort_flag)) {
                                ok = false;
                                break;
                            }
                            issue_ss(C::kS, r0_lo, s0_lo + sa1 * tile16);
                            mma_commit(&ms.s_full);
                        }
                        if (!mbar_wait(&ms.ds_ready, gn & 1u, abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        // dK += dS^T Q (KV_MAJOR) or dQ += dS K
                        issue_ts(KV_MAJOR ? C::kAcc1 : C::kAcc0, C::kDP, s0_mn + sa * tile16, n > 0);
                        mma_commit(&ms.a_empty[sa]);
                        if (nxt) {
                            if (C::kSplit && !mbar_wait(&ms.b_full[sb1], ((gn + 1) / NB) & 1u, abort_flag)) {
                                ok = false;
                                break;
                            }
                            issue_ss(C::kDP, r1_lo, s1_lo + sb1 * tile16);
                            mma_commit(&ms.dp_full);
                            if constexpr (C::kSplit && !KV_MAJOR) mma_commit(&ms.b_empty[sb1]);
                        }
                    }
                    if (!ok) break;
                    mma_commit(&ms.res_empty);  // the resident tiles are no longer read
                    mma_commit(&ms.acc_full);
                    g += (uint32_t)N;
                    ++nw;
                }
                mbar_arrive(&ms.item_free[k]);
            }
            if (!ok) bwd_fail(ms, p.status);
            mma_commit(&ms.drain);  // every MMA issued above completes before TMEM is freed
            drain_wait_bwd(&ms.drain, 0);
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------- elementwise
        const int t = threadIdx.x % 128;   // owned row within the block, TMEM lane
        const int half = threadIdx.x / 128;  // walked columns 64 half .. 64 half + 63
        const int cbase = 64 * half;
        const uint32_t lane_base = (uint32_t)((warp % 4) * 32) << 16;
        const uint32_t trow = tmem + lane_base;
        // base-2 score: identity/ALiBi x = k0 S + bias, softcap x = k1 tanh(k0 S)
        const float k0 = SCORE == FLEX_SCORE_SOFTCAP ? p.scale / p.score_param : p.scale * kBwdLog2e;
        const float k1 = SCORE == FLEX_SCORE_SOFTCAP ? p.score_param * kBwdLog2e : 0.f;
        const uint64_t k0_2 = f2_pack(k0, k0), k1_2 = f2_pack(k1, k1);
        const bool loader = half == 0;
        uint32_t g = 0, nw = 0;
        bool ok = true;
        for (uint32_t it = 0; ok; ++it) {
          const int k = (int)(it & 1u);
          const BwdSlot &sl = ms.slot[k];
          if (!bwd_warp_wait(&ms.item_ready[k], (it >> 1) & 1u, abort_flag)) {
              ok = false;
              break;
          }
          const int N = sl.n;
          if (N < 0) break;
          const int own = sl.own, bh = sl.bh;
          const int b = bh / p.H, h = bh % p.H;
          const int row = own * 128 + t;  // kv (KV_MAJOR) or q
          const float slope2 =
              SCORE == FLEX_SCORE_ALIBI ? kBwdLog2e * exp2f(-8.f * (float)(h + 1) / (float)p.H) : 0.f;
          const int32_t *doc_row = DOC ? p.mask.doc_ids + (int64_t)b * p.mask.doc_len : nullptr;
          int doc_own = 0;
          if constexpr (DOC) {
              if (row < own_len) doc_own = __ldg(doc_row + row);
          }
          // Q-major: the row's lse (base 2) and -delta; a row without any
          // unmasked score (lse = -inf) or past Q_LEN contributes nothing
          float lse2_row = INFINITY, ndelta_row = 0.f;
          if constexpr (!KV_MAJOR) {
              if (row < p.q_len) {
                  const float l = __ldg(p.lse + (int64_t)bh * p.q_len + row);
                  if (l != -INFINITY) lse2_row = l * kBwdLog2e;
                  ndelta_row = -__ldg(p.delta + (int64_t)bh * p.q_len + row);
              }
          }
          // Per-column data of a step, column t loaded by thread t of the first
          // half:
          //   KV_MAJOR: colv = -(lse2 + slope2 c) of q column c (-inf for a q
          //             row without unmasked scores or past Q_LEN), dltv = -delta
          //   Q-major : colv = slope2 c (ALiBi column term)
          //   DOC     : docv = document id of the walked row
          float cv = 0.f, dv_ = 0.f;
          int dc = 0;
          auto load_col = [&](int n) {
              const int blk = (int)(sl.list[n] & 0xFFFFu);
              const int r = blk * 128 + t;
              if constexpr (KV_MAJOR) {
                  float l = -INFINITY, d = 0.f;
                  if (r < p.q_len) {
                      l = __ldg(p.lse + (int64_t)bh * p.q_len + r);
                      d = __ldg(p.delta + (int64_t)bh * p.q_len + r);
                  }
                  cv = l == -INFINITY ? -INFINITY : -(l * kBwdLog2e + slope2 * (float)t);
                  dv_ = -d;
              } else {
                  cv = slope2 * (float)t;
              }
              if constexpr (DOC) dc = r < walk_len ? __ldg(doc_row + r) : 0;
          };
          auto store_col = [&](int buf) {
              ms.colv[buf][t] = cv;
              if constexpr (KV_MAJOR) ms.dltv[buf][t] = dv_;
              if constexpr (DOC) ms.docv[buf][t] = dc;
              mbar_arrive(&ms.col_ready[buf]);
          };
          if (N > 0 && loader) {
              load_col(0);
              store_col((int)(g & 1u));
          }
          for (int n = 0; n < N; ++n) {
              const uint32_t gn = g + (uint32_t)n;
              const int buf = (int)(gn & 1u);
              if (n + 1 < N && loader) load_col(n + 1);  // in flight while this step computes
              if (!bwd_warp_wait(&ms.col_ready[buf], (gn >> 1) & 1u, abort_flag)) {
                  ok = false;
                  break;
              }
              const uint32_t e = sl.list[n];
              const int blk = (int)(e & 0xFFFFu);
              const bool full = (e >> 16) & 1u;
              const int w0 = blk * 128;  // first walked row of the step
              // keep-interval of walked columns for this row (partial steps)
              int clo = 0, chi = -1;
              if (!full) {
                  int lo, hi;
                  if constexpr (KV_MAJOR) {
                      if constexpr (DOC) {  // q >= kv, q < Q_LEN (ids compared below)
                          lo = row;
                          hi = row < p.kv_len ? p.q_len - 1 : row - 1;
                      } else {
                          mask_col_interval(p.mask, row, lo, hi);
                      }
                  } else {
                      if constexpr (DOC) {  // kv <= q (Q_LEN == KV_LEN)
                          lo = 0;
                          hi = row < p.q_len ? row : -1;
                      } else {
                          if (!mask_row_interval(p.mask, row, lo, hi)) hi = lo - 1;
                          hi = min(hi, p.kv_len - 1);
                          if (row >= p.q_len) hi = lo - 1;
                      }
                  }
                  clo = lo - w0;
                  chi = hi - w0;
                  if (clo > chi) {
                      clo = 1;
                      chi = 0;
                  }
              }
              // per-row term of the exponent
              float rowc;
              if constexpr (KV_MAJOR) {
                  rowc = SCORE == FLEX_SCORE_ALIBI ? slope2 * (float)(row - w0) : 0.f;  // slope2 (kv - q) = rowc - slope2 c
              } else {
                  rowc = SCORE == FLEX_SCORE_ALIBI ? slope2 * (float)(w0 - row) - lse2_row : -lse2_row;
              }
              const uint64_t rowc2 = f2_pack(rowc, rowc);
              const float4 *colv4 = reinterpret_cast<const float4 *>(ms.colv[buf] + cbase);
              const float4 *dltv4 = reinterpret_cast<const float4 *>(ms.dltv[buf] + cbase);
              const int4 *docv4 = reinterpret_cast<const int4 *>(ms.docv[buf] + cbase);

              if (!bwd_warp_wait(&ms.s_full, gn & 1u, abort_flag)) {
                  ok = false;
                  break;
              }
              tc_fence_after_sync();
              // ---- phase 1: P (and P score_mod') from S, this half's 64 columns
              float pg[64];
              {
                  uint32_t r[64];
                  bwd_tmem_ld64(trow + C::kS + cbase, r);
                  // one column chunk; PARTIAL: apply the keep bits (full steps
                  // carry no mask work)
                  auto p_chunk = [&](auto partial, int c0, uint32_t keep) {
                      constexpr bool PARTIAL = decltype(partial)::value;
                      uint32_t pk[16];
  #pragma unroll
                      for (int j = 0; j < 16; ++j) {
                          const int c = 32 * c0 + 2 * j;  // within the half
                          uint64_t bias2;
                          if constexpr (KV_MAJOR) {
                              const float4 cc = colv4[c / 4];
                              const uint64_t cpair = (c & 2) ? f2_pack(cc.z, cc.w) : f2_pack(cc.x, cc.y);
                              bias2 = SCORE == FLEX_SCORE_ALIBI ? f2_add(rowc2, cpair) : cpair;
                          } else {
                              if constexpr (SCORE == FLEX_SCORE_ALIBI) {
                                  const float4 cc = colv4[c / 4];
                                  bias2 = f2_add(rowc2, (c & 2) ? f2_pack(cc.z, cc.w) : f2_pack(cc.x, cc.y));
                              } else {
                                  bias2 = rowc2;
                              }
                          }
                          const uint64_t s2 = f2_pack(__uint_as_float(r[c]), __uint_as_float(r[c + 1]));
                          float x0, x1, g0 = 1.f, g1 = 1.f;
                          if constexpr (SCORE == FLEX_SCORE_SOFTCAP) {
                              float t0, t1;
                              f2_unpack(f2_mul(s2, k0_2), t0, t1);
                              const float u0 = tanh_approx(t0), u1 = tanh_approx(t1);
                              f2_unpack(f2_fma(f2_pack(u0, u1), k1_2, bias2), x0, x1);
                              g0 = fmaf(-u0, u0, 1.f);
                              g1 = fmaf(-u1, u1, 1.f);
                          } else {
                              f2_unpack(f2_fma(s2, k0_2, bias2), x0, x1);
                          }
                          if constexpr (PARTIAL) {
                              if (!((keep >> (2 * j)) & 1u)) x0 = -INFINITY;
                              if (!((keep >> (2 * j + 1)) & 1u)) x1 = -INFINITY;
                          }
                          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                          if constexpr (KV_MAJOR) pk[j] = pack_bf16x2(p0, p1);
                          pg[c] = p0 * g0;
                          pg[c + 1] = p1 * g1;
                      }
                      // over this half's S columns, all read above
                      if constexpr (KV_MAJOR) tmem_st16(trow + C::kS + cbase + 16 * c0, pk);
                  };
  #pragma unroll
                  for (int c0 = 0; c0 < 2; ++c0) {
                      if (full) {
                          // (document masks keep one code path: their steps are
                          // often partial, and a second copy measured slower)
                          if constexpr (DOC) p_chunk(std::true_type{}, c0, 0xFFFFFFFFu);
                          else p_chunk(std::false_type{}, c0, 0u);
                      } else {
                          uint32_t keep = interval_bits(clo, chi, cbase + 32 * c0);
                          if constexpr (DOC) {
                              uint32_t same = 0u;
  #pragma unroll
                              for (int j = 0; j < 8; ++j) {
                                  const int4 d = docv4[8 * c0 + j];
                                  same |= ((uint32_t)(d.x == doc_own) | ((uint32_t)(d.y == doc_own) << 1) |
                                           ((uint32_t)(d.z == doc_own) << 2) | ((uint32_t)(d.w == doc_own) << 3))
                                          << (4 * j);
                              }
                              keep &= same;
                          }
                          p_chunk(std::true_type{}, c0, keep);
                      }
                  }
              }
              if constexpr (KV_MAJOR) tmem_wait_st();
              tc_fence_before_sync();
              mbar_arrive(&ms.p_ready);

              if (!bwd_warp_wait(&ms.dp_full, gn & 1u, abort_flag)) {
                  ok = false;
                  break;
              }
              tc_fence_after_sync();
              // ---- phase 2: dS = P score_mod' (dP - delta) from dP
              {
                  const uint64_t nd_row2 = f2_pack(ndelta_row, ndelta_row);
                  uint32_t r[64];
                  bwd_tmem_ld64(trow + C::kDP + cbase, r);
  #pragma unroll
                  for (int c0 = 0; c0 < 2; ++c0) {
                      uint32_t pk[16];
  #pragma unroll
                      for (int j = 0; j < 16; ++j) {
                          const int c = 32 * c0 + 2 * j;
                          uint64_t nd2;
                          if constexpr (KV_MAJOR) {
                              const float4 dd = dltv4[c / 4];
                              nd2 = (c & 2) ? f2_pack(dd.z, dd.w) : f2_pack(dd.x, dd.y);
                          } else {
                              nd2 = nd_row2;
                          }
                          const uint64_t dp2 = f2_pack(__uint_as_float(r[c]), __uint_as_float(r[c + 1]));
                          float d0, d1;
                          f2_unpack(f2_mul(f2_add(dp2, nd2), f2_pack(pg[c], pg[c + 1])), d0, d1);
                          pk[j] = pack_bf16x2(d0, d1);
                      }
                      tmem_st16(trow + C::kDP + cbase + 16 * c0, pk);  // over this half's dP columns, all read
                  }
              }
              tmem_wait_st();
              tc_fence_before_sync();
              mbar_arrive(&ms.ds_ready);
              if (n + 1 < N && loader) store_col((int)((gn + 1) & 1u));
          }
          // ----------------------------------------------------- epilogue
          bool have = ok && N > 0;
          if (have && !bwd_warp_wait(&ms.acc_full, nw & 1u, abort_flag)) {
              have = false;
              ok = false;
          }
          if (!ok) bwd_fail(ms, p.status);
          // every lane of a warp takes the (warp-collective) TMEM loads; only
          // the rows inside the length are stored
          if (ok) {
              tc_fence_after_sync();
              const bool store = row < own_len;
              const int64_t orow = (int64_t)bh * own_len + (store ? row : 0);
              // KV_MAJOR: acc0 = dV, acc1 = dK (scaled); Q-major: acc0 = dQ (scaled).
              // Each half writes D / 2 of the row's columns.
  #pragma unroll 1
              for (int which = 0; which < (KV_MAJOR ? 2 : 1); ++which) {
                  const float mul = (KV_MAJOR && which == 0) ? 1.f : p.scale;
                  uint16_t *dst = (which == 0 ? p.out0 : p.out1) + orow * D + half * (D / 2);
                  const uint32_t col = (which == 0 ? C::kAcc0 : C::kAcc1) + half * (D / 2);
  #pragma unroll 1
                  for (int c0 = 0; c0 < D / 2; c0 += 32) {
                      uint32_t o[32];
                      if (have) {
                          bwd_tmem_ld32(trow + col + c0, o);
                      } else {
  #pragma unroll
                          for (int j = 0; j < 32; ++j) o[j] = 0u;
                      }
                      uint32_t pk[16];
  #pragma unroll
                      for (int j = 0; j < 16; ++j)
                          pk[j] = pack_bf16x2(__uint_as_float(o[2 * j]) * mul, __uint_as_float(o[2 * j + 1]) * mul);
                      // whole 32-byte sectors per store
                      if (store) {
                          st_global_32B(dst + c0, &pk[0]);
                          st_global_32B(dst + c0 + 16, &pk[8]);
                      }
                  }
              }
          }
          if (N > 0) {
              g += (uint32_t)N;
              ++nw;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&ms.item_free[k]);
        }
        if (!ok) bwd_fail(ms, p.status);
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kBwdMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

}  // namespace flex

