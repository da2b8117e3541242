// Helpers of the float32 kernels that run on the bf16 tensor-core datapath:
// the three-way bf16 split of a float32 value, the 128-byte swizzled row
// layout the split parts are stored in, a warp-wide bounded mbarrier wait
// and the TMEM row loads and stores those kernels use.
#pragma once

#include <cstdint>

#include "flex_internal.h"
#include "ptx.cuh"

namespace flex {

// Offset of 16-byte chunk c (8 bf16) of row r in a row-major tile with
// 128-byte swizzled rows: atoms of 64 bf16 along the row, each atom all rows
// x 128 bytes; 8-row groups 1024 bytes apart; the chunk index XORed with the
// row's index within its 8-row group.
__device__ __forceinline__ uint32_t sw128_chunk(int r, int c, uint32_t atom_bytes) {
    return (uint32_t)(c / 8) * atom_bytes + (uint32_t)(r / 8) * 1024u + (uint32_t)(r % 8) * 128u +
           (uint32_t)(((c % 8) ^ (r % 8)) * 16);
}

__device__ __forceinline__ float bf16lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// The three bf16 parts of two floats, as packed pairs (a in bits 0-15).
__device__ __forceinline__ void split3(float a, float b, uint32_t &w1, uint32_t &w2, uint32_t &w3) {
    w1 = pack_bf16x2(a, b);
    const float ra = a - bf16lo_f(w1), rb = b - bf16hi_f(w1);
    w2 = pack_bf16x2(ra, rb);
    w3 = pack_bf16x2(ra - bf16lo_f(w2), rb - bf16hi_f(w2));
}

__device__ __forceinline__ float f4_at(const float4 &v, int e) {
    return e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
}

// A wait taken by all 32 lanes of a warp, with one outcome for the warp.
__device__ __forceinline__ bool f32_warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        const int stop = (*abort != 0) || (global_timer_ns() - t0 > kWaitLimitNs);
        if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
}

__device__ __forceinline__ void f32_ld32(uint32_t taddr, uint32_t (&r)[32]) {
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

// Each thread of the warp writes 8 consecutive 32-bit columns of its own lane.
__device__ __forceinline__ void f32_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

}  // namespace flex
