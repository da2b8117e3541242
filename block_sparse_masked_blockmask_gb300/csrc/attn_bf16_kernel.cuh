// Block-sparse FlexAttention forward for bf16 inputs on sm_103a tensor cores.
//
// What it computes (the flex_attention op with OUTPUT_LOGSUMEXP, from
// "[Inductor][Flex Attention] Add Subtiling Option for Alpha Scaling",
// PyTorch PR #167356): for each query row, over the kv tiles its BlockMask
// lists, s = score_mod(scale * q.k) with s = -inf where mask_mod is false
// (mask_mod evaluated on partial tiles only), out = softmax(s) V and
// lse = ln sum exp(s).  The online-softmax step is the page's forward_block_mn
// (l = l * alpha + sum(p); acc = acc * alpha; acc += p V) carried out with
// the running max in base-2 units.
//
// Design for one GB300 SM (one persistent CTA per SM, 384 threads):
//   * A work item is two consecutive q blocks (two 128-row Q tiles) of one
//     (batch, head); the CTA walks the union of their kv-tile lists in
//     descending kv order, so the K/V tile staged in shared memory serves
//     both Q tiles.  After its first item (its own index) a CTA takes the
//     items of CTAs that have not started yet (cluster launch control).
//   * warp 11 (scheduler): builds each item's union list into one of two
//                         shared-memory slots, loads its Q tiles once the
//                         previous item's S MMAs are done, and fetches the
//                         next item while the current one computes.
//   * warps 8 / 10 (TMA): load the K tiles / the V tiles of each union step
//                         into a ring of shared-memory stages (128-byte
//                         swizzle, the layout tcgen05 descriptors read) that
//                         runs on across items.  At D = 64 warp 8 loads both.
//   * warp 9  (MMA)     : one thread issues tcgen05.mma: S_i = Q_i K^T into
//                         tensor memory (TMEM) and O_i += P_i V with P_i read
//                         from TMEM; order per step PV0, S0(next), PV1,
//                         S1(next), so each softmax group has two MMAs of
//                         slack while the tensor core works for the other.
//                         P_i overwrites the first 64 columns of S_i.
//     D = 64 (TMEM has room for P apart from S): warps 9 and 10 each issue
//                         one Q tile's MMAs, S two steps ahead of PV (the
//                         next S only waits for the softmax to have read the
//                         S it replaces), so the softmax never waits for an
//                         S MMA and neither tile waits behind the other's.
//   * warps 0-3 / 4-7   : softmax of Q tile 0 / 1, one thread per row (TMEM
//                         lane = row).  Score_mod on every listed tile,
//                         mask_mod only on partial tiles (the row's kept
//                         interval or document id is hoisted out of the
//                         column loop).  P goes back to TMEM as bf16.
//   * O rescale: the running max is only raised when a tile's max exceeds it
//     by more than 2^8, so exp2(s - m) <= 256 stays exact in fp32/bf16 and
//     the O rescale (a TMEM read-modify-write by the softmax warp, between
//     the S load and the next PV) is rare; the result is the same softmax.
//     This replaces the page's subtiled alpha scaling of the register
//     accumulator: with O in TMEM the rescale leaves the register file and
//     the PV critical path entirely on most steps.
//   * Every wait is bounded (globaltimer); on timeout the CTA records
//     FLEX_ERR_DEVICE_TIMEOUT, drains its copies and MMAs, frees TMEM, exits.
#pragma once

#include <cfloat>
#include <cstddef>

#include <cuda_bf16.h>

#include "flex_internal.h"
#include "ptx.cuh"
#include "tilelist.cuh"

namespace flex {

constexpr int kAttnThreads = 384;
constexpr int kTmaWarp = 8;   // Q and K loads
constexpr int kTmaVWarp = 10; // V loads
constexpr int kMmaWarp = 9;
constexpr int kSchedWarp = 11; // work items: union lists, Q loads, next item by launch control
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kHeadGroup = 4;              // fewest (batch, head) pairs scheduled together
constexpr float kRescaleThreshold = 8.0f;  // raise the running max only beyond 2^8
// P_i is handed to the MMA warp whole (one mbarrier per tile), not in column
// chunks: the thread that issues the MMAs spends ~46 cycles issuing each
// 64-cycle 128x128x16 MMA, so an extra wait and fence per chunk costs more
// tensor-core time than starting the PV on the first chunk early gains.
// Register split.  Three warps share each SM sub-partition's 64 KB register
// file, so the kernel is compiled to kRegsAtLaunch (168) registers per thread.
// The softmax warpgroups then raise their budget to kRegsSoftmax while the
// scheduler/TMA/MMA warpgroup lowers its own to kRegsControl (enough for its
// loop state without spilling); per sub-partition this is 2 * 216 + 72 =
// 3 * 168 registers per lane, the registers the CTA was launched with, so the
// increase never waits on registers that are not released.  The launcher
// checks the compiled count.
constexpr uint32_t kRegsAtLaunch = 168;
constexpr uint32_t kRegsSoftmax = 216;
constexpr uint32_t kRegsControl = 72;
static_assert(2 * kRegsSoftmax + kRegsControl == 3 * kRegsAtLaunch, "register split");

struct Bf16Params {
    int B, H, q_len, kv_len, nqt, nkvt, npairs;  // nqt, nkvt: 128-tiles along q and kv
    int bh_begin, nbh;  // the (b, h) pairs b * H + h in [bh_begin, bh_begin + nbh) are computed
    int head_group;     // (b, h) pairs scheduled together (at least kHeadGroup)
    TileLists lists;    // the BlockMask's kv side (any Q_BLOCK, KV_BLOCK), read as 128-tiles
    MaskDesc mask;
    float scale, score_param;
    float prescale;   // PRESCALE_QK: 0 = off, else Q is multiplied by it in shared memory (scale is then 1)
    uint16_t *out;    // bf16 bits, contiguous [B, H, q_len, D]
    float *lse;       // [B, H, q_len]
    float *row_max;   // OUTPUT_MAX: [B, H, q_len] or null
    int *status;
};

// One work item (two consecutive q blocks of one (batch, head)) as the
// scheduler warp publishes it.
struct ItemSlot {
    int nu;                                    // union length; -1: no more work for this CTA
    int b, h, qb0, has1;
    int pad[3];
    alignas(16) uint32_t ulist[kMaxKvBlocks];  // union, descending kv: kv block | flags << 16
};

// Shared-memory bookkeeping that follows the Q/K/V tiles.
struct AttnMisc {
    uint64_t q_full, q_empty;
    uint64_t q_loaded;                         // PRESCALE_QK: the Q copies landed (q_full follows the scaling)
    uint64_t near_end;                         // the K producer has issued an item's last K tile
    uint64_t k_full[4], v_full[4], k_empty[4], v_empty[4];
    uint64_t s_full[2], p_full[2];             // p_full[i]: all of P_i is in TMEM
    uint64_t s_free[2], pv_done[2];            // D = 64: S_i read by the softmax / PV_i complete
    uint64_t o_full[2], drain[2];              // o_full[i]: O_i final (kSepP: per tile; else [0] for both)
    uint64_t item_ready[2], item_free[2];      // per item slot
    uint64_t clc_bar;                          // cluster-launch-control response landed
    uint32_t tmem_base;
    int abort;
    alignas(16) uint32_t clc_resp[4];
    alignas(16) int32_t stage_doc[4][128];     // document ids of each stage's kv tile (bulk-copy target)
    alignas(16) uint32_t flags[kMaxKvBlocks];  // per kv tile: listed / full-pair counts of Q tiles 0 and 1
    ItemSlot slot[2];
};
// bulk copies and the launch-control response need 16-byte aligned destinations
static_assert(offsetof(AttnMisc, clc_resp) % 16 == 0, "clc_resp alignment");
static_assert(offsetof(AttnMisc, stage_doc) % 16 == 0, "stage_doc alignment");
static_assert(sizeof(AttnMisc::stage_doc[0]) % 16 == 0, "stage_doc row size");
static_assert(offsetof(AttnMisc, slot) % 16 == 0 && sizeof(ItemSlot) % 16 == 0, "item slot alignment");
// arrivals that free an item slot: 8 softmax warps and three control warps
// (K and V producers and the MMA thread; at D = 64 one producer, two MMA threads)
constexpr uint32_t kItemConsumers = 11;

template <int D>
struct Bf16Cfg {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kAtoms = D / 64;                  // 128-byte swizzle atoms along D
    static constexpr uint32_t kAtomBytes = 128 * 128;      // 128 rows x 128 bytes
    static constexpr uint32_t kTileBytes = 128 * D * 2;    // one 128 x D bf16 tile
    static constexpr int kStages = D == 128 ? 2 : 4;
    static constexpr uint32_t kQOff = 0;
    static constexpr uint32_t kKvOff = 2 * kTileBytes;
    static constexpr uint32_t kStageBytes = 2 * kTileBytes;  // K then V
    static constexpr uint32_t kMiscOff = kKvOff + kStages * kStageBytes;
    static constexpr uint32_t kSmemBytes = kMiscOff + sizeof(AttnMisc) + 1024;
    // TMEM columns: S0 | S1 | O0 | O1, and P_i (64 columns of bf16 pairs).
    // D = 128: P_i overwrites the first 64 columns of S_i, so the next S_i
    // waits for the PV MMA that reads P_i.  D = 64: P0 | P1 in the last 128
    // columns (kSepP), so the next S_i only waits for the softmax to have
    // read S_i and is computed while the softmax still works on the tile.
    static constexpr bool kSepP = D == 64;
    // kSepP: one MMA-issuing thread per Q tile (warps 9 and 10), the K and V
    // tiles loaded by one producer (warp 8); otherwise one issuer (warp 9)
    // and one producer each for K (warp 8) and V (warp 10)
    static constexpr uint32_t kIssuers = kSepP ? 2u : 1u;
    __host__ __device__ static constexpr uint32_t s_col(int i) { return i ? 128u : 0u; }
    __host__ __device__ static constexpr uint32_t o_col(int i) { return i ? 256u + D : 256u; }
    __host__ __device__ static constexpr uint32_t p_col(int i) { return kSepP ? 384u + 64u * i : s_col(i); }
};

__device__ __forceinline__ void record_failure(AttnMisc &ms, int *status) {
    *reinterpret_cast<volatile int *>(&ms.abort) = 1;
    atomicCAS(status, 0, kDeviceTimeout);
}

// A wait taken by all 32 lanes of a warp with one outcome for the warp.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        const int stop = (*abort != 0) || (global_timer_ns() - t0 > kWaitLimitNs);
        if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
    int never = 0;
    (void)mbar_wait(bar, parity, &never);
}

// TMEM read of 128 columns of this thread's lane as four 32-column loads
// (smaller register vectors than one x128) with a single wait.
__device__ __forceinline__ void tmem_ld128_sync(uint32_t taddr, uint32_t (&r)[128]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%128];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%129];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95}, [%130];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%131];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
        : "r"(taddr), "r"(taddr + 32), "r"(taddr + 64), "r"(taddr + 96)
        : "memory");
}

// TMEM read of 32 columns of this thread's lane, completed before returning.
__device__ __forceinline__ void tmem_ld32_sync(uint32_t taddr, uint32_t (&r)[32]) {
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

// score_mod in base-2 units, two columns (c, c+1) at a time on packed fp32x2,
// plus a per-tile addend A (the softmax folds its running-max shift into it):
//   identity : x = k0 s + A                          k0 = scale log2(e)
//   softcap  : x = k1 tanh(k0 s) + A                 k0 = scale / cap, k1 = log2(e) cap
//   ALiBi    : x = k0 s + slope2 c + A               slope2 = log2(e) slope_h
// The softcap's tanh is the hardware's single-instruction approximation
// (tanh.approx.f32, relative error about 2^-11), one special-function
// operation per score beside the softmax's exponential.
// For ALiBi the per-tile term slope2 (kv0 - q) is kept out of x as `offset`:
// it shifts the whole row, so it is added to the row max and subtracted in
// the exponent instead of being added to every element.  The column term
// slope2 c comes from eight interleaved add chains (step 16 slope2, at most
// seven adds each, error below 1e-4 in base-2 units on the tile's columns).
template <int SCORE>
struct ScoreLog2 {
    uint64_t k0, k1, add2;
    float slope2, offset;
    uint64_t bias[8];  // ALiBi: slope2 * (2j, 2j+1) for the next pair j of each of 8 chains
    uint64_t step;     // ALiBi: 16 slope2 in both lanes (8 pairs further on)
    __device__ __forceinline__ void init(const Bf16Params &p, int h) {
        float a0, a1 = 0.f;
        if constexpr (SCORE == FLEX_SCORE_SOFTCAP) {
            a0 = p.scale / p.score_param;
            a1 = p.score_param * kLog2e;
        } else {
            a0 = p.scale * kLog2e;
        }
        k0 = f2_pack(a0, a0);
        k1 = f2_pack(a1, a1);
        slope2 = SCORE == FLEX_SCORE_ALIBI ? kLog2e * exp2f(-8.f * (float)(h + 1) / (float)p.H) : 0.f;
        step = f2_pack(16.f * slope2, 16.f * slope2);
        offset = 0.f;
    }
    // row offset of a tile (ALiBi: slope2 (kv0 - q); 0 otherwise)
    __device__ __forceinline__ float tile_offset(int kv0, int q) const {
        return SCORE == FLEX_SCORE_ALIBI ? slope2 * (float)(kv0 - q) : 0.f;
    }
    // start of a tile: its row offset, the addend A, and the eight bias chains
    __device__ __forceinline__ void tile(int kv0, int q, float a) {
        if constexpr (SCORE == FLEX_SCORE_ALIBI) {
            offset = slope2 * (float)(kv0 - q);
#pragma unroll
            for (int t = 0; t < 8; ++t)
                bias[t] = f2_pack(fmaf(slope2, (float)(2 * t), a), fmaf(slope2, (float)(2 * t + 1), a));
        } else {
            add2 = f2_pack(a, a);
        }
    }
    // columns 2j, 2j+1 (called for j = 0, 1, ..., 63 in order)
    __device__ __forceinline__ uint64_t pair(uint64_t s2, int j) {
        if constexpr (SCORE == FLEX_SCORE_SOFTCAP) {
            float t0, t1;
            f2_unpack(f2_mul(s2, k0), t0, t1);
            return f2_fma(f2_pack(tanh_approx(t0), tanh_approx(t1)), k1, add2);
        } else if constexpr (SCORE == FLEX_SCORE_ALIBI) {
            const uint64_t x = f2_fma(s2, k0, bias[j & 7]);
            bias[j & 7] = f2_add(bias[j & 7], step);
            return x;
        } else {
            return f2_fma(s2, k0, add2);
        }
    }
};

// PRESCALE_QK on the Q tiles in shared memory: every bf16 element q becomes
// bf16(s q), rounded once.  The float product is taken toward zero and its
// last bit set when it was inexact (rounding to odd at 24 bits); rounding that
// to nearest even at bf16's 8 bits gives the correctly rounded product, since
// the float keeps at least two extra bits (S. Boldo, G. Melquiond, "Emulation
// of FMA and correctly rounded sums: proved algorithms using rounding to odd",
// IEEE Trans. Computers 57(4), 2008).  The 128-byte swizzle does not matter:
// every element gets the same factor.
__device__ __forceinline__ void prescale_q(uint4 *q, int n16, float s, int lane) {
    const uint64_t s2 = f2_pack(s, s), ns2 = f2_pack(-s, -s);
#pragma unroll 2
    for (int i = lane; i < n16; i += 32) {
        uint4 w = q[i];
        uint32_t e[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint64_t x2 = f2_pack(__uint_as_float(e[j] << 16), __uint_as_float(e[j] & 0xFFFF0000u));
            const uint64_t p2 = f2_mul_rz(x2, s2);
            float p0, p1, r0, r1;
            f2_unpack(p2, p0, p1);
            f2_unpack(f2_fma(x2, ns2, p2), r0, r1);  // p - x s exactly: nonzero iff the product was inexact
            p0 = __uint_as_float(__float_as_uint(p0) | (r0 != 0.f ? 1u : 0u));
            p1 = __uint_as_float(__float_as_uint(p1) | (r1 != 0.f ? 1u : 0u));
            e[j] = pack_bf16x2(p0, p1);
        }
        q[i] = make_uint4(e[0], e[1], e[2], e[3]);
    }
}

// mask_mod on a partial tile for row q (columns kv0 .. kv0 + 127), on the
// packed score pairs.
__device__ __forceinline__ uint64_t keep_pair(uint64_t v, bool k0, bool k1) {
    float a, b;
    f2_unpack(v, a, b);
    return f2_pack(k0 ? a : -INFINITY, k1 ? b : -INFINITY);
}

// Interval mask_mods (causal, sliding window, causal + prefix, all): the row
// keeps exactly the kv in [lo, hi], and nothing at or past KV_LEN (the zero
// rows that fill a tail tile).
__device__ __forceinline__ void apply_interval_mask(const MaskDesc &m, int q, int kv0, uint64_t (&x2)[64]) {
    int lo, hi;
    mask_row_interval(m, q, lo, hi);
    const int clo = lo - kv0, chi = min(hi, m.kv_len - 1) - kv0;
#pragma unroll
    for (int j = 0; j < 64; ++j)
        x2[j] = keep_pair(x2[j], 2 * j >= clo && 2 * j <= chi, 2 * j + 1 >= clo && 2 * j + 1 <= chi);
}

// Document mask_mod: same document id (the tile's ids staged in shared
// memory) and kv <= q.
__device__ __forceinline__ void apply_document_mask(int q, int kv0, int doc_q, const int32_t *tile_doc,
                                                    uint64_t (&x2)[64]) {
    const int lim = q - kv0;
    const int4 *dk = reinterpret_cast<const int4 *>(tile_doc);
    // keep-bits of the 128 columns in four words, then one fully unrolled
    // pass so the scores stay in registers
    uint32_t keep[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint32_t bits = 0u;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int4 d = dk[w * 8 + j];
            const int c = w * 32 + j * 4;
            const uint32_t nib = (uint32_t)(d.x == doc_q && c + 0 <= lim) | ((uint32_t)(d.y == doc_q && c + 1 <= lim) << 1) |
                                 ((uint32_t)(d.z == doc_q && c + 2 <= lim) << 2) |
                                 ((uint32_t)(d.w == doc_q && c + 3 <= lim) << 3);
            bits |= nib << (4 * j);
        }
        keep[w] = bits;
    }
#pragma unroll
    for (int j = 0; j < 64; ++j)
        x2[j] = keep_pair(x2[j], (keep[j / 16] >> ((2 * j) % 32)) & 1u, (keep[j / 16] >> ((2 * j + 1) % 32)) & 1u);
}

// Decode work item `item` (a CTA index of the launch grid): heads in groups of
// p.head_group (their K/V stay in L2 while in flight); inside a group, q-block
// pairs from the last (the longest kv lists for causal-like masks) to the
// first, the group's heads innermost, so the heaviest items of each group come
// first and the last items of the grid are light.
__device__ __forceinline__ void decode_item(const Bf16Params &p, int item, int &b, int &h, int &qb0, int &has1) {
    const int nbh = p.nbh;
    const int group_items = p.head_group * p.npairs;
    const int g0 = (item / group_items) * p.head_group;
    const int gsize = min(p.head_group, nbh - g0);
    const int r = item - (item / group_items) * group_items;
    const int pair = p.npairs - 1 - r / gsize;
    const int bh = p.bh_begin + g0 + r % gsize;
    b = bh / p.H;
    h = bh % p.H;
    qb0 = 2 * pair;
    has1 = qb0 + 1 < p.nqt ? 1 : 0;
}

// Build an item's union list into `sl` with the 32 lanes of one warp:
// mark every kv tile of both q blocks (bounds-checked: a malformed BlockMask
// cannot write outside the flag array), then compact the marked tiles in
// descending kv order with their present / full bits (1, 2 for tile 0; 4, 8
// for tile 1).  The index loads of a chunk are all issued before any of them
// is used, so the build costs a couple of memory latencies rather than one
// per 32 entries.  BLOCKS128: the lists hold 128-tiles directly (the code the
// MMA-issuing warpgroup's register budget was tuned with); otherwise they
// are read as 128-tiles through the general mapping (tilelist.cuh).
template <bool BLOCKS128>
__device__ __forceinline__ void build_item(const Bf16Params &p, AttnMisc &ms, ItemSlot &sl, int item, int lane) {
    int b, h, qb0, has1;
    decode_item(p, item, b, h, qb0, has1);
    const int nkvt = p.nkvt;
    const unsigned lt = (1u << lane) - 1u;
    int count = 0;
    if constexpr (BLOCKS128) {
        const int nkvb = nkvt;
        const int64_t row0 = ((int64_t)b * p.H + h) * p.nqt + qb0;
        const int32_t *pidx = p.lists.idx + row0 * nkvb, *fidx = p.lists.fidx + row0 * nkvb;
        const int np0 = min(max(__ldg(p.lists.num + row0), 0), nkvb);
        const int nf0 = min(max(__ldg(p.lists.fnum + row0), 0), nkvb);
        const int np1 = has1 ? min(max(__ldg(p.lists.num + row0 + 1), 0), nkvb) : 0;
        const int nf1 = has1 ? min(max(__ldg(p.lists.fnum + row0 + 1), 0), nkvb) : 0;
        for (int j = lane; j < nkvb; j += 32) ms.flags[j] = 0u;
        __syncwarp();
        constexpr int kUnroll = 4;
        for (int base = 0; base < nkvb; base += 32 * kUnroll) {
            int jj[4][kUnroll];
#pragma unroll
            for (int r = 0; r < kUnroll; ++r) {
                // the first chunk is read whole (every entry below nkvb lies
                // in its row), so its loads do not wait for the counts and a
                // short list costs one memory latency; entries past a count
                // are dropped below
                const int x = base + 32 * r + lane;
                const bool any = base == 0 && x < nkvb;
                jj[0][r] = x < np0 || any ? __ldg(pidx + x) : -1;
                jj[1][r] = x < nf0 || any ? __ldg(fidx + x) : -1;
                jj[2][r] = x < np1 || (any && has1) ? __ldg(pidx + nkvb + x) : -1;
                jj[3][r] = x < nf1 || (any && has1) ? __ldg(fidx + nkvb + x) : -1;
            }
#pragma unroll
            for (int r = 0; r < kUnroll; ++r) {
                const int x = base + 32 * r + lane;
                if (x >= np0) jj[0][r] = -1;
                if (x >= nf0) jj[1][r] = -1;
                if (x >= np1) jj[2][r] = -1;
                if (x >= nf1) jj[3][r] = -1;
            }
            constexpr uint32_t kBits[4] = {1u, 3u, 4u, 12u};  // present / full, tile 0 then tile 1
#pragma unroll
            for (int l = 0; l < 4; ++l)
#pragma unroll
                for (int r = 0; r < kUnroll; ++r)
                    if ((unsigned)jj[l][r] < (unsigned)nkvb) atomicOr(&ms.flags[jj[l][r]], kBits[l]);
        }
        __syncwarp();
        for (int base = 0; base < nkvb; base += 32) {
            const int c = nkvb - 1 - (base + lane);
            const uint32_t f = c >= 0 ? ms.flags[c] : 0u;
            const unsigned bal = __ballot_sync(0xffffffffu, f != 0u);
            if (f != 0u) sl.ulist[count + __popc(bal & lt)] = (uint32_t)c | (f << 16);
            count += __popc(bal);
        }
    } else {
        for (int j = lane; j < nkvt; j += 32) ms.flags[j] = 0u;
        __syncwarp();
        const int64_t bh = (int64_t)b * p.H + h;
        tl_mark_warp(p.lists, bh, qb0, 0, ms.flags, 0, nkvt, lane);
        if (has1) tl_mark_warp(p.lists, bh, qb0 + 1, 1, ms.flags, 0, nkvt, lane);
        __syncwarp();
        const uint32_t expect = tl_expect(p.lists);
        for (int base = 0; base < nkvt; base += 32) {
            const int c = nkvt - 1 - (base + lane);
            uint32_t f = 0u;
            if (c >= 0) {
                const uint32_t w = ms.flags[c];
                f = (tl_listed(w, 0) ? 1u : 0u) | (tl_full(expect, w, 0) ? 2u : 0u) | (tl_listed(w, 1) ? 4u : 0u) |
                    (tl_full(expect, w, 1) ? 8u : 0u);
            }
            const unsigned bal = __ballot_sync(0xffffffffu, f != 0u);
            if (f != 0u) sl.ulist[count + __popc(bal & lt)] = (uint32_t)c | (f << 16);
            count += __popc(bal);
        }
    }
    if (lane == 0) {
        sl.nu = count;
        sl.b = b;
        sl.h = h;
        sl.qb0 = qb0;
        sl.has1 = has1;
    }
    __syncwarp();
}

// DOC: the BlockMask's mask_mod is the document mask (its partial tiles read
// per-tile document ids staged next to V); other kinds are interval masks.
// BLOCKS128: the BlockMask's blocks are 128 x 128 (else any Q_BLOCK, KV_BLOCK,
// read as 128-tiles when the scheduler builds an item).
//
// Persistent over work items: each CTA starts with the item of its own index
// and then takes items from CTAs of the grid that have not started yet
// (cluster launch control), so one CTA stays on each SM and the next item's
// union list, Q tiles and first K/V tiles load while the current item
// computes.  Every role walks the same sequence of published items; all
// barrier phases (K/V ring, S/P hand-off, Q, O) continue across items.
template <int D, int SCORE, bool DOC, bool BLOCKS128>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_bf16_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
                     const __grid_constant__ CUtensorMap tmap_v, const Bf16Params p) {
    using C = Bf16Cfg<D>;
    constexpr int NS = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    AttnMisc &ms = *reinterpret_cast<AttnMisc *>(smem + C::kMiscOff);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        mbar_init(&ms.q_full, 1);
        mbar_init(&ms.q_empty, C::kIssuers);
        mbar_init(&ms.q_loaded, 1);
        mbar_init(&ms.near_end, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&ms.k_full[s], 1);
            mbar_init(&ms.v_full[s], 1);
            mbar_init(&ms.k_empty[s], C::kIssuers);
            mbar_init(&ms.v_empty[s], C::kIssuers);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ms.s_full[i], 1);
            mbar_init(&ms.p_full[i], 128);
            mbar_init(&ms.s_free[i], 128);
            mbar_init(&ms.pv_done[i], 1);
            mbar_init(&ms.item_ready[i], 1);
            mbar_init(&ms.item_free[i], kItemConsumers);
        }
        mbar_init(&ms.o_full[0], 1);
        mbar_init(&ms.o_full[1], 1);
        mbar_init(&ms.drain[0], 1);
        mbar_init(&ms.drain[1], 1);
        mbar_init(&ms.clc_bar, 1);
        ms.abort = 0;
        fence_barrier_init();
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

    if (warp >= 8) {
        regs_decrease<kRegsControl>();
    }
    if (warp == kSchedWarp) {
        // ----------------------------------------------------------- scheduler
        // Item n goes to slot n % 2 once every consumer has released that
        // slot's item n - 2.  The next item is taken from the grid when the
        // current one has its last K tile on the way (near_end, about one
        // ring depth before its end): late enough that no item sits claimed
        // behind much work while other SMs run dry at the end of the grid,
        // early enough that the next item's list is published (the K/V
        // producers run on into it) and its Q tiles are prefetched into L2
        // before the current item ends.  Q is loaded into shared memory as
        // soon as the current item's last S MMAs are done with it (q_empty).
        int item = blockIdx.x;
        uint32_t nq = 0;    // Q loads issued
        uint32_t nne = 0;   // near_end phases consumed
        uint32_t nclc = 0;  // launch-control responses consumed
        bool ok = true;
        // the Q copies complete on q_full, or with PRESCALE_QK on q_loaded
        const bool prescale = p.prescale != 0.f;
        uint64_t *q_bar = prescale ? &ms.q_loaded : &ms.q_full;
        if (lane == 0) prefetch_tensormap(&tmap_q);
        for (uint32_t n = 0;; ++n) {
            const int k = (int)(n & 1u);
            ItemSlot &sl = ms.slot[k];
            if (n >= 2 && !warp_wait(&ms.item_free[k], ((n - 2) >> 1) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            if (item >= 0) {
                build_item<BLOCKS128>(p, ms, sl, item, lane);
            } else if (lane == 0) {
                sl.nu = -1;
            }
            __threadfence_block();  // every lane's slot writes before the release below
            __syncwarp();
            const int nu = sl.nu;
            if (lane == 0) mbar_arrive(&ms.item_ready[k]);
            if (item < 0) break;
            if (nu > 0) {
                const int has1 = sl.has1;
                if (lane == 0)
                    for (int a = 0; a < C::kAtoms; ++a)
                        for (int i = 0; i <= has1; ++i) tma_prefetch_l2_4d(&tmap_q, 64 * a, (sl.qb0 + i) * kBlock, sl.h, sl.b);
                // the previous item with work has finished its S MMAs
                if (nq > 0 && !warp_wait(&ms.q_empty, (nq - 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(q_bar, (has1 ? 2u : 1u) * C::kTileBytes);
                    for (int a = 0; a < C::kAtoms; ++a) {
                        tma_load_4d(smem + C::kQOff + a * C::kAtomBytes, &tmap_q, q_bar, 64 * a, sl.qb0 * kBlock,
                                    sl.h, sl.b);
                        if (has1)
                            tma_load_4d(smem + C::kQOff + C::kTileBytes + a * C::kAtomBytes, &tmap_q, q_bar,
                                        64 * a, (sl.qb0 + 1) * kBlock, sl.h, sl.b);
                    }
                }
                ++nq;
                if (prescale) {
                    // PRESCALE_QK: scale Q in place once it has landed, then
                    // hand it to the MMA thread through q_full
                    if (!warp_wait(&ms.q_loaded, (nq - 1) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    prescale_q(reinterpret_cast<uint4 *>(smem + C::kQOff), (has1 ? 2 : 1) * (int)C::kTileBytes / 16,
                               p.prescale, lane);
                    fence_proxy_async_smem();  // the MMAs read these generic-proxy writes
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ms.q_full);
                }
                // wait until this item's last K tile is on the way
                if (!warp_wait(&ms.near_end, nne & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                ++nne;
            }
            if (lane == 0) {
                mbar_arrive_expect_tx(&ms.clc_bar, 16u);
                clc_try_cancel(ms.clc_resp, &ms.clc_bar);
            }
            if (!warp_wait(&ms.clc_bar, nclc & 1u, abort_flag)) {
                ok = false;
                break;
            }
            ++nclc;
            int next = 0;
            if (lane == 0) next = clc_cancelled_x(ms.clc_resp);
            item = __shfl_sync(0xffffffffu, next, 0);
        }
        if (!ok && lane == 0) record_failure(ms, p.status);
        // every Q copy issued above lands before the CTA exits (normally the
        // MMA thread has already consumed it)
        if (lane == 0 && nq > 0) drain_wait(q_bar, (nq - 1) & 1u);
        __syncwarp();
    } else if (warp == kTmaWarp || (!C::kSepP && warp == kTmaVWarp)) {
        // ----------------------------------------------------- TMA producers
        // warp 8 loads the K tiles, warp 10 the V tiles, into the stage ring
        // indexed by the CTA's global step count.  K of a stage is free once
        // its step's S MMAs are done, V once its PV MMAs are; with one
        // producer each, a late V release never holds back the next K.
        if (C::kSepP && lane == 0) {
            // one producer: K then V of every step (the V wait never holds
            // back a K that an S MMA is waiting for: V of a stage is freed
            // by the PV MMAs of kStages steps ago)
            const int32_t *doc_base = DOC ? p.mask.doc_ids : nullptr;
            prefetch_tensormap(&tmap_k);
            prefetch_tensormap(&tmap_v);
            uint32_t g = 0;
            bool ok = true;
            for (uint32_t n = 0; ok; ++n) {
                const int k = (int)(n & 1u);
                const ItemSlot &sl = ms.slot[k];
                if (!mbar_wait(&ms.item_ready[k], (n >> 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const int nu = sl.nu;
                if (nu < 0) break;
                const int b = sl.b, h = sl.h;
                for (int u = 0; u < nu; ++u, ++g) {
                    const int s = (int)(g % NS);
                    const uint32_t use = g / NS;
                    const int kv0 = (int)(sl.ulist[u] & 0xFFFFu) * kBlock;
                    uint8_t *dst = smem + C::kKvOff + s * C::kStageBytes;
                    if (use > 0 && !mbar_wait(&ms.k_empty[s], (use - 1) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&ms.k_full[s], C::kTileBytes);
                    for (int a = 0; a < C::kAtoms; ++a) tma_load_4d(dst + a * C::kAtomBytes, &tmap_k, &ms.k_full[s], 64 * a, kv0, h, b);
                    if (use > 0 && !mbar_wait(&ms.v_empty[s], (use - 1) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const uint32_t doc_bytes = DOC ? 4u * (uint32_t)min(kBlock, p.mask.doc_len - kv0) : 0u;
                    mbar_arrive_expect_tx(&ms.v_full[s], C::kTileBytes + doc_bytes);
                    for (int a = 0; a < C::kAtoms; ++a)
                        tma_load_4d(dst + C::kTileBytes + a * C::kAtomBytes, &tmap_v, &ms.v_full[s], 64 * a, kv0, h, b);
                    if (DOC) bulk_load(ms.stage_doc[s], doc_base + (int64_t)b * p.mask.doc_len + kv0, doc_bytes, &ms.v_full[s]);
                }
                if (ok && nu > 0) mbar_arrive(&ms.near_end);
                if (ok) mbar_arrive(&ms.item_free[k]);
            }
            if (!ok) record_failure(ms, p.status);
            for (uint32_t s = 0; s < (uint32_t)NS && s < g; ++s) {
                const uint32_t last = s + ((g - 1 - s) / NS) * NS;
                drain_wait(&ms.k_full[s], (last / NS) & 1u);
                drain_wait(&ms.v_full[s], (last / NS) & 1u);
            }
        } else if (lane == 0) {
            const bool is_k = warp == kTmaWarp;
            const CUtensorMap *map = is_k ? &tmap_k : &tmap_v;
            uint64_t *full = is_k ? ms.k_full : ms.v_full;
            uint64_t *empty = is_k ? ms.k_empty : ms.v_empty;
            const uint32_t half = is_k ? 0u : C::kTileBytes;
            // the kv tile's document ids travel with V: V's stage is released
            // only after both softmax groups are done with the tile
            const bool with_doc = DOC && !is_k;
            prefetch_tensormap(map);
            uint32_t g = 0;  // steps issued over all items
            bool ok = true;
            for (uint32_t n = 0; ok; ++n) {
                const int k = (int)(n & 1u);
                const ItemSlot &sl = ms.slot[k];
                if (!mbar_wait(&ms.item_ready[k], (n >> 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const int nu = sl.nu;
                if (nu < 0) break;
                const int b = sl.b, h = sl.h;
                const int32_t *doc_row = DOC ? p.mask.doc_ids + (int64_t)b * p.mask.doc_len : nullptr;
                for (int u = 0; u < nu; ++u, ++g) {
                    const int s = (int)(g % NS);
                    const uint32_t use = g / NS;
                    const int kv0 = (int)(sl.ulist[u] & 0xFFFFu) * kBlock;
                    uint8_t *dst = smem + C::kKvOff + s * C::kStageBytes + half;
                    if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    // a tail tile's ids end at the length (a multiple of 4, so
                    // whole 16-byte words); the columns past it are masked
                    // by causality, since document masks have Q_LEN == KV_LEN
                    const uint32_t doc_bytes =
                        with_doc ? 4u * (uint32_t)min(kBlock, p.mask.doc_len - kv0) : 0u;
                    mbar_arrive_expect_tx(&full[s], C::kTileBytes + doc_bytes);
                    for (int a = 0; a < C::kAtoms; ++a) tma_load_4d(dst + a * C::kAtomBytes, map, &full[s], 64 * a, kv0, h, b);
                    if (with_doc) bulk_load(ms.stage_doc[s], doc_row + kv0, doc_bytes, &full[s]);
                }
                // The last K tile of the item is issued once its stage is free,
                // about one ring depth (kStages steps) before the item ends:
                // the scheduler takes the next item now.
                if (ok && is_k && nu > 0) mbar_arrive(&ms.near_end);
                if (ok) mbar_arrive(&ms.item_free[k]);
            }
            if (!ok) record_failure(ms, p.status);
            // Drain: every copy issued above lands before the CTA exits.
            for (uint32_t s = 0; s < (uint32_t)NS && s < g; ++s) {
                const uint32_t last = s + ((g - 1 - s) / NS) * NS;
                drain_wait(&full[s], (last / NS) & 1u);
            }
        }
        __syncwarp();
    } else if (C::kSepP && (warp == kMmaWarp || warp == kTmaVWarp)) {
        // ------------------------------------------- MMA issuers (kSepP)
        // One thread per Q tile ti, each walking every item and step: S runs
        // two steps ahead (S_ti(u + 2) replaces S_ti(u + 1) once the softmax
        // has read it, and is issued right after PV_ti(u)), so the softmax
        // never waits for an S MMA, and neither tile's MMAs wait behind the
        // other tile's barriers.  The ring, Q and O barriers take one commit
        // from each thread per step or item, tile present or not.
        if (lane == 0) {
            const int ti = warp == kMmaWarp ? 0 : 1;
            const uint32_t present = ti ? 4u : 1u;
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, 0, 1);
            constexpr uint32_t kHi = smem_desc_hi_sw128(1024);
            const uint32_t kv_lo0 = smem_desc_lo(smem_u32(smem + C::kKvOff), 16);
            const uint32_t v_lo0 = smem_desc_lo(smem_u32(smem + C::kKvOff + C::kTileBytes), C::kAtomBytes);
            const uint32_t qa = smem_desc_lo(smem_u32(smem + C::kQOff + ti * C::kTileBytes), 16);
            uint32_t s_total = 0, pv_total = 0;  // this tile's S and PV groups over all items
            auto issue_s = [&](int s) -> bool {
                if (s_total > 0 && !mbar_wait(&ms.s_free[ti], (s_total - 1) & 1u, abort_flag)) return false;
                tc_fence_after_sync();
                ++s_total;
                const uint32_t ka = kv_lo0 + ((s * C::kStageBytes) >> 4);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = ((k / 4) * C::kAtomBytes + (k % 4) * 32) >> 4;
                    mma_ss_lo<kHi, kHi>(tmem + C::s_col(ti), qa + off, ka + off, idesc_s, k > 0 ? 1u : 0u);
                }
                mma_commit(&ms.s_full[ti]);
                return true;
            };
            auto issue_pv = [&](int s, bool acc) -> bool {
                if (!mbar_wait(&ms.p_full[ti], pv_total & 1u, abort_flag)) return false;
                tc_fence_after_sync();
                const uint32_t va = v_lo0 + ((s * C::kStageBytes) >> 4);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_ts_lo<kHi>(tmem + C::o_col(ti), tmem + C::p_col(ti) + k * 8, va + ((k * 2048) >> 4), idesc_o,
                                   (k > 0 || acc) ? 1u : 0u);
                mma_commit(&ms.pv_done[ti]);
                ++pv_total;
                return true;
            };
            uint32_t g = 0, nq = 0;
            bool ok = true;
            for (uint32_t n = 0; ok; ++n) {
                const int k = (int)(n & 1u);
                const ItemSlot &sl = ms.slot[k];
                if (!mbar_wait(&ms.item_ready[k], (n >> 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const int nu = sl.nu;
                if (nu < 0) break;
                if (nu > 0) {
                    ok = mbar_wait(&ms.q_full, nq & 1u, abort_flag);
                    tc_fence_after_sync();
                    // S of the first two steps
                    for (int u = 0; ok && u < min(nu, 2); ++u) {
                        const uint32_t gu = g + (uint32_t)u;
                        const int s = (int)(gu % NS);
                        ok = mbar_wait(&ms.k_full[s], (gu / NS) & 1u, abort_flag) &&
                             (!((sl.ulist[u] >> 16) & present) || issue_s(s));
                        mma_commit(&ms.k_empty[s]);
                        if (u + 1 == nu) mma_commit(&ms.q_empty);  // the item's last S is issued
                    }
                    uint32_t pv_item = 0;
                    for (int u = 0; ok && u < nu; ++u) {
                        const uint32_t gu = g + (uint32_t)u;
                        const int s = (int)(gu % NS);
                        if (!mbar_wait(&ms.v_full[s], (gu / NS) & 1u, abort_flag)) {
                            ok = false;
                            break;
                        }
                        if ((sl.ulist[u] >> 16) & present) {
                            if (!issue_pv(s, pv_item > 0)) {
                                ok = false;
                                break;
                            }
                            ++pv_item;
                        }
                        mma_commit(&ms.v_empty[s]);
                        if (u + 2 < nu) {
                            const uint32_t g2 = gu + 2;
                            const int s2 = (int)(g2 % NS);
                            if (!mbar_wait(&ms.k_full[s2], (g2 / NS) & 1u, abort_flag) ||
                                (((sl.ulist[u + 2] >> 16) & present) && !issue_s(s2))) {
                                ok = false;
                                break;
                            }
                            mma_commit(&ms.k_empty[s2]);
                            if (u + 3 == nu) mma_commit(&ms.q_empty);
                        }
                    }
                    if (!ok) break;
                    mma_commit(&ms.o_full[ti]);
                    g += (uint32_t)nu;
                    ++nq;
                }
                mbar_arrive(&ms.item_free[k]);
            }
            if (!ok) record_failure(ms, p.status);
            mma_commit(&ms.drain[ti]);  // every MMA issued above completes before TMEM is freed
            drain_wait(&ms.drain[ti], 0);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t idesc_o = idesc_bf16_f32(128, D, 0, 1);
            const uint32_t q_addr0 = smem_u32(smem + C::kQOff);
            uint32_t pv_total[2] = {0u, 0u};  // PV groups issued per tile, over all items
            uint32_t pv_item[2] = {0u, 0u};   // ... within the current item
            // Q and K are K-major (rows of 64 elements per 128-byte swizzle
            // atom, 8-row groups 1024 bytes apart); V is MN-major (kv rows of
            // 64 head-dim elements, the two 64-wide halves 16 KB apart).
            constexpr uint32_t kHi = smem_desc_hi_sw128(1024);
            const uint32_t kv_lo0 = smem_desc_lo(smem_u32(smem + C::kKvOff), 16);
            const uint32_t v_lo0 = smem_desc_lo(smem_u32(smem + C::kKvOff + C::kTileBytes), C::kAtomBytes);
            const uint32_t q_lo0 = smem_desc_lo(q_addr0, 16);
            auto issue_s = [&](int i, int s) {
                const uint32_t qa = q_lo0 + ((i * C::kTileBytes) >> 4);
                const uint32_t ka = kv_lo0 + ((s * C::kStageBytes) >> 4);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = ((k / 4) * C::kAtomBytes + (k % 4) * 32) >> 4;
                    mma_ss_lo<kHi, kHi>(tmem + C::s_col(i), qa + off, ka + off, idesc_s, k > 0 ? 1u : 0u);
                }
                mma_commit(&ms.s_full[i]);
            };
            // O_i += P_i V once all of P_i is in TMEM; the first PV of an item
            // overwrites O_i (its epilogue read of the previous item came
            // before this P in the softmax warps' program order)
            auto issue_pv = [&](int i, int s) -> bool {
                const uint32_t va = v_lo0 + ((s * C::kStageBytes) >> 4);
                const uint32_t acc = pv_item[i] > 0 ? 1u : 0u;
                if (!mbar_wait(&ms.p_full[i], pv_total[i] & 1u, abort_flag)) return false;
                tc_fence_after_sync();
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_ts_lo<kHi>(tmem + C::o_col(i), tmem + C::s_col(i) + k * 8, va + ((k * 2048) >> 4), idesc_o,
                                   (k > 0 || acc) ? 1u : 0u);
                ++pv_total[i];
                ++pv_item[i];
                return true;
            };
            uint32_t g = 0;   // global step of the item's first union entry
            uint32_t nq = 0;  // items with work so far (Q loads, o_full commits)
            bool ok = true;
            for (uint32_t n = 0; ok; ++n) {
                const int k = (int)(n & 1u);
                const ItemSlot &sl = ms.slot[k];
                if (!mbar_wait(&ms.item_ready[k], (n >> 1) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                const int nu = sl.nu;
                if (nu < 0) break;
                if (nu > 0) {
                    pv_item[0] = pv_item[1] = 0u;
                    const int s0 = (int)(g % NS);
                    ok = mbar_wait(&ms.q_full, nq & 1u, abort_flag) &&
                         mbar_wait(&ms.k_full[s0], (g / NS) & 1u, abort_flag);
                    tc_fence_after_sync();
                    if (ok) {
                        const uint32_t f = sl.ulist[0] >> 16;
                        if (f & 1u) issue_s(0, s0);
                        if (f & 4u) issue_s(1, s0);
                        mma_commit(&ms.k_empty[s0]);
                        if (nu == 1) mma_commit(&ms.q_empty);  // Q no longer read
                    }
                    for (int u = 0; ok && u < nu; ++u) {
                        const uint32_t gu = g + (uint32_t)u;
                        const int s = (int)(gu % NS);
                        const uint32_t f = sl.ulist[u] >> 16;
                        const bool nxt = u + 1 < nu;
                        const int s1 = (int)((gu + 1) % NS);
                        const uint32_t f1 = nxt ? (sl.ulist[u + 1] >> 16) : 0u;
                        // V of this step and K of the next arrive by TMA (the
                        // mbarriers alone order them for the MMA); both are
                        // waited for before P_0, which is usually last to come
                        if (!mbar_wait(&ms.v_full[s], (gu / NS) & 1u, abort_flag) ||
                            (nxt && !mbar_wait(&ms.k_full[s1], ((gu + 1) / NS) & 1u, abort_flag))) {
                            ok = false;
                            break;
                        }
                        if ((f & 1u) && !issue_pv(0, s)) {
                            ok = false;
                            break;
                        }
                        if (nxt && (f1 & 1u)) issue_s(0, s1);
                        if ((f & 4u) && !issue_pv(1, s)) {
                            ok = false;
                            break;
                        }
                        mma_commit(&ms.v_empty[s]);
                        if (nxt) {
                            if (f1 & 4u) issue_s(1, s1);
                            mma_commit(&ms.k_empty[s1]);
                            if (u + 2 == nu) mma_commit(&ms.q_empty);  // the item's last S is issued
                        }
                    }
                    if (!ok) break;
                    mma_commit(&ms.o_full[0]);
                    g += (uint32_t)nu;
                    ++nq;
                }
                mbar_arrive(&ms.item_free[k]);
            }
            if (!ok) record_failure(ms, p.status);
            mma_commit(&ms.drain[0]);  // every MMA issued above completes before TMEM is freed
            drain_wait(&ms.drain[0], 0);
        }
        __syncwarp();
    } else if (warp < 8) {
        // ----------------------------------------------------------- softmax
        regs_increase<kRegsSoftmax>();
        const int i = warp / 4;
        const int t = threadIdx.x % 128;
        const uint32_t lane_base = (uint32_t)((warp % 4) * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + C::s_col(i);
        const uint32_t p_addr = tmem + lane_base + C::p_col(i);
        const uint32_t o_addr = tmem + lane_base + C::o_col(i);
        const uint32_t present = i ? 4u : 1u, fullbit = i ? 8u : 2u;
        uint32_t cnt_total = 0;  // S_i tiles consumed over all items (s_full parity)
        uint32_t g = 0;          // global step of the item's first union entry
        uint32_t nq = 0;         // items with work so far (o_full parity)
        bool ok = true;
        for (uint32_t n = 0; ok; ++n) {
          const int k = (int)(n & 1u);
          const ItemSlot &sl = ms.slot[k];
          if (!warp_wait(&ms.item_ready[k], (n >> 1) & 1u, abort_flag)) {
              ok = false;
              break;
          }
          const int nu = sl.nu;
          if (nu < 0) break;
          const int b = sl.b, h = sl.h;
          const bool valid = i == 0 || sl.has1;
          const int q = (sl.qb0 + i) * kBlock + t;
          const int64_t bh = (int64_t)b * p.H + h;
          ScoreLog2<SCORE> score;
          score.init(p, h);
          int doc_q = 0;
          if constexpr (DOC) {
              if (valid && q < p.q_len) doc_q = __ldg(p.mask.doc_ids + (int64_t)b * p.mask.doc_len + q);
          }
          // The running max starts at a finite floor, so a tile whose scores
          // are all masked for this row gives exp2(-inf - floor) = 0 with no
          // special case, and the first live tile rescales by exp2(floor - m)
          // = 0.  Only the epilogue tells empty rows apart (l_run == 0).
          float m_run = -FLT_MAX, l_run = 0.f;
          float m_max = -INFINITY;  // exact row max (OUTPUT_MAX); m_run may lag it by < kRescaleThreshold
          uint32_t cnt = 0;  // tiles of this item
          if (valid) {
            for (int u = 0; u < nu; ++u) {
                const uint32_t e = sl.ulist[u];
                const uint32_t f = e >> 16;
                if (!(f & present)) continue;
                const int kv0 = (int)(e & 0xFFFFu) * kBlock;
                if (!warp_wait(&ms.s_full[i], cnt_total & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                // The scores come out shifted by A: by the running max's
                // shift (offset - m_run) once the row has a finite running
                // max, so that most tiles need no separate subtraction pass;
                // by nothing before that.
                const float a_shift = m_run > -FLT_MAX ? score.tile_offset(kv0, q) - m_run : 0.f;
                uint64_t x2[64];
                {
                    uint32_t r[128];
                    tmem_ld128_sync(s_addr, r);
                    if constexpr (C::kSepP) {
                        tc_fence_before_sync();
                        mbar_arrive(&ms.s_free[i]);  // S_i may be overwritten by the next S MMA
                    }
                    score.tile(kv0, q, a_shift);
#pragma unroll
                    for (int j = 0; j < 64; ++j)
                        x2[j] = score.pair(f2_pack(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), j);
                }
                if (!(f & fullbit)) {
                    if constexpr (DOC) {
                        const uint32_t gu = g + (uint32_t)u;
                        const int stage = (int)(gu % NS);
                        if (!warp_wait(&ms.v_full[stage], (gu / NS) & 1u, abort_flag)) {
                            ok = false;
                            break;
                        }
                        apply_document_mask(q, kv0, doc_q, ms.stage_doc[stage], x2);
                    } else {
                        apply_interval_mask(p.mask, q, kv0, x2);
                    }
                }

                float mx[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    float lo, hi;
                    f2_unpack(x2[k], lo, hi);
                    mx[k] = fmaxf(lo, hi);
                }
#pragma unroll
                for (int j = 8; j < 64; ++j) {
                    float lo, hi;
                    f2_unpack(x2[j], lo, hi);
                    mx[j & 7] = fmax3(mx[j & 7], lo, hi);
                }
                const float m_tile = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])) -
                                     a_shift + score.offset;
                m_max = fmaxf(m_max, m_tile);
                float alpha = 1.f;
                if (m_tile > m_run + kRescaleThreshold) {  // always taken at the row's first live tile
                    alpha = ex2_approx(m_run - m_tile);
                    m_run = m_tile;
                }
                // the exponent is s - m_run: what the scores already carry
                // unless this tile raised the running max (or it was not
                // finite when the tile started); one pass over the tile then
                const float shift = (score.offset - m_run) - a_shift;
                if (__any_sync(0xffffffffu, shift != 0.f)) {
                    const uint64_t shift2 = f2_pack(shift, shift);
#pragma unroll
                    for (int j = 0; j < 64; ++j) x2[j] = f2_add(x2[j], shift2);
                }
                // O rescale (rare) before P is handed over: the PV MMA of
                // this step accumulates into the rescaled O
                auto rescale_o = [&]() {
                    if (cnt > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
                        for (int c0 = 0; c0 < D; c0 += 32) {
                            uint32_t o[32];
                            tmem_ld32_sync(o_addr + c0, o);
                            const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                float lo, hi;
                                f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * j]), __uint_as_float(o[2 * j + 1])), a2),
                                          lo, hi);
                                o[2 * j] = __float_as_uint(lo);
                                o[2 * j + 1] = __float_as_uint(hi);
                            }
                            tmem_st32(o_addr + c0, o);
                        }
                    }
                };
                // the row sum takes the bf16 weights the PV MMA reads, so
                // each row's weights sum to l exactly
                float rsum4[4] = {0.f, 0.f, 0.f, 0.f};
                if constexpr (C::kSepP) {
                    // all of P in registers first; P_i and O_i are written
                    // once the previous PV MMA of this tile has read P_i and
                    // accumulated into O_i
                    uint32_t pk[64];
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        float d0, d1;
                        f2_unpack(x2[j], d0, d1);
                        pk[j] = pack_bf16x2(ex2_approx(d0), ex2_approx(d1));
                    }
#pragma unroll
                    for (int j = 0; j < 64; ++j) add_bf16x2_to_f32(rsum4[2 * (j & 1)], rsum4[2 * (j & 1) + 1], pk[j]);
                    if (cnt_total > 0 && !warp_wait(&ms.pv_done[i], (cnt_total - 1) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    rescale_o();
#pragma unroll
                    for (int gq = 0; gq < 4; ++gq)
                        tmem_st16(p_addr + 16 * gq, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16 * gq]));
                } else {
                    rescale_o();
#pragma unroll
                    for (int gq = 0; gq < 4; ++gq) {
                        uint32_t pk[16];
#pragma unroll
                        for (int t2 = 0; t2 < 16; ++t2) {
                            const int j = 16 * gq + t2;
                            float d0, d1;
                            f2_unpack(x2[j], d0, d1);
                            pk[t2] = pack_bf16x2(ex2_approx(d0), ex2_approx(d1));
                        }
                        tmem_st16(p_addr + 16 * gq, pk);
#pragma unroll
                        for (int t2 = 0; t2 < 16; ++t2)
                            add_bf16x2_to_f32(rsum4[2 * (t2 & 1)], rsum4[2 * (t2 & 1) + 1], pk[t2]);
                    }
                }
                tmem_wait_st();
                tc_fence_before_sync();
                mbar_arrive(&ms.p_full[i]);
                const float rsum = (rsum4[0] + rsum4[1]) + (rsum4[2] + rsum4[3]);
                l_run = fmaf(l_run, alpha, rsum);
                ++cnt;
                ++cnt_total;
            }
            // ---------------------------------------------------- epilogue
            bool have = ok && cnt > 0;
            // kSepP: this tile's own issuer signals its O; else one barrier for both
            if (have && !warp_wait(&ms.o_full[C::kSepP ? i : 0], nq & 1u, abort_flag)) {
                have = false;
                ok = false;
            }
            if (!ok) record_failure(ms, p.status);
            if (ok) {
                tc_fence_after_sync();
                const int64_t orow = bh * p.q_len + q;
                uint16_t *dst = p.out + orow * D;
                const bool store = q < p.q_len;  // rows of a tail tile past Q_LEN are padding
                const bool live = have && l_run > 0.f;
                const float inv = live ? 1.f / l_run : 0.f;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    if (have) {
                        tmem_ld32_sync(o_addr + c0, o);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) o[j] = 0u;
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        pk[j] = pack_bf16x2(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
                    // whole 32-byte sectors per store (the row's 16 values)
                    if (store) {
                        st_global_32B(dst + c0, &pk[0]);
                        st_global_32B(dst + c0 + 16, &pk[8]);
                    }
                }
                if (store) {
                    p.lse[orow] = live ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
                    if (p.row_max) p.row_max[orow] = m_max * kLn2;
                }
            }
          }
          if (nu > 0) {
              g += (uint32_t)nu;
              ++nq;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&ms.item_free[k]);
        }
        if (!ok) record_failure(ms, p.status);
    }

    // ---------------------------------------------------------- teardown
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace flex
