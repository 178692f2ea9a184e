// Helpers shared by the tcgen05 kernels: bounded mbarrier waits that also give up when
// another role of the CTA has aborted, a loop-counter barrier for the optimiser, and the
// bf16 hi/lo operand split.
#pragma once

#include "ptx.cuh"

namespace efla {
namespace tc {
namespace {  // internal to each kernel's translation unit
using namespace ptx;

// Bounded wait that also gives up when another role has aborted.  The slow
// path is out of line: it is reached rarely and the kernel's code must stay
// small enough for the instruction cache.
__device__ __noinline__ bool wait_bar_slow(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                           uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 20000)) return true;  // sleeps instead of spinning
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *abort_flag = 1;
            return false;
        }
    }
}
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(bar, parity, abort_flag, limit_ns);
}
// The same for all 32 lanes of a warp, with one outcome for the whole warp: every lane
// waits, and the warp proceeds only if every lane's wait succeeded (the warp-collective
// TMEM loads and stores that follow need all lanes together).
__device__ __forceinline__ bool wait_bar_warp(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              uint64_t limit_ns) {
    const bool ok = wait_bar(bar, parity, abort_flag, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

// Hides a loop counter from the optimiser so that the loop stays rolled (the
// kernel's per-chunk code must fit the instruction cache).
__device__ __forceinline__ int opaque(int i) {
    asm volatile("" : "+r"(i));
    return i;
}

// Splits pairs x[2c], x[2c+1] into packed bf16 hi and lo words with
// x = hi + lo + e, |e| < 2^-14 |x|: hi is x truncated to bf16 (its upper 16
// bits), lo is the exact fp32 remainder x - hi truncated the same way.  Bit
// operations only (one byte permute per packed pair).
template <int NP>
__device__ __forceinline__ void split_pack(const float *x, uint32_t *hi, uint32_t *lo) {
#pragma unroll
    for (int c = 0; c < NP; ++c) {
        const uint32_t b0 = __float_as_uint(x[2 * c]), b1 = __float_as_uint(x[2 * c + 1]);
        hi[c] = __byte_perm(b0, b1, 0x7632);
        // the two remainders x - hi (exact) in one packed fp32x2 fma: hi * (-1) + x
        const float2 r = __ffma2_rn(make_float2(__uint_as_float(b0 & 0xffff0000u), __uint_as_float(b1 & 0xffff0000u)),
                                    make_float2(-1.f, -1.f), make_float2(x[2 * c], x[2 * c + 1]));
        lo[c] = __byte_perm(__float_as_uint(r.x), __float_as_uint(r.y), 0x7632);
    }
}

// Rows row0 .. row0 + 31 of column j (this lane) of a 128 x 128 fp32 matrix, x[i] = M[row0 + i][j],
// into the operand-tile layout the backward kernels load whole: bf16 hi (truncated) in the first
// 32 KB and lo (the remainder, truncated) in the next, each as 2 column blocks of [128 rows][64]
// with the 128-byte swizzle.  Lanes j and j ^ 1 of a warp (consecutive columns) pair up: each
// shuffle hands one half to the partner, the even lane stores the hi word, the odd lane the lo
// word.  All 32 lanes take part.
__device__ __forceinline__ void put_col_split_tile(uint8_t *tile, int row0, int j, const float (&x)[32]) {
    const bool odd = (j & 1) != 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t b = __float_as_uint(x[i]);
        const uint32_t h16 = b >> 16;
        const uint32_t l16 = __float_as_uint(x[i] - __uint_as_float(b & 0xffff0000u)) >> 16;
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, odd ? h16 : l16, 1);
        const uint32_t word = odd ? (recv | (l16 << 16)) : (h16 | (recv << 16));
        *reinterpret_cast<uint32_t *>(tile + swz_offset(row0 + i, j & ~1, 16384) + (odd ? 32768u : 0u)) = word;
    }
}

// Tokens t0 .. t0 + 31 (x) of column j (this lane) of a [token][128] block, times `sign`, as
// bf16 hi and lo (the split above) into two arrays of that shape whose token rows are `stride`
// elements apart (hi and lo point at token 0, column 0); tokens at or past `valid` are not
// written.  Lanes j and j ^ 1 pair up as in put_col_split_tile: the even lane stores the hi
// word, the odd lane the lo word.
__device__ __forceinline__ void put_col_split_rows(__nv_bfloat16 *hi, __nv_bfloat16 *lo, size_t stride, int valid,
                                                   int t0, int j, float sign, const float (&x)[32]) {
    const bool odd = (j & 1) != 0;
    uint32_t *dst = reinterpret_cast<uint32_t *>(odd ? lo + (j - 1) : hi + j);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const float v = sign * x[i];
        const uint32_t b = __float_as_uint(v);
        const uint32_t h16 = b >> 16;
        const uint32_t l16 = __float_as_uint(v - __uint_as_float(b & 0xffff0000u)) >> 16;
        const uint32_t recv = __shfl_xor_sync(0xffffffffu, odd ? h16 : l16, 1);
        if (t0 + i < valid) dst[(size_t)(t0 + i) * stride / 2] = odd ? (recv | (l16 << 16)) : (h16 | (recv << 16));
    }
}

}  // namespace
}  // namespace tc
}  // namespace efla
