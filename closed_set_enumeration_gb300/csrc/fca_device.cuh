// Device helpers shared by the kernels of libfca: bitset masks, popcounts, queue entry sizes and
// the per-device cache of a kernel's launch shape.
#pragma once

#include <cuda_runtime.h>

#include "fca_internal.cuh"

namespace fca {

constexpr unsigned FULL = 0xffffffffu;
constexpr int OUTBUF = 16;          // intents buffered per warp before one atomicAdd
constexpr int MAX_SLICES = 32;      // most work items one subtree root is split into
constexpr int WARPS_PER_BLOCK = 8;

__device__ __forceinline__ unsigned popc4(const uint4 &x)
{
    return __popc(x.x) + __popc(x.y) + __popc(x.z) + __popc(x.w);
}

// Bits >= b of 32-bit word `w` of a bitset (b is a bit index of the whole set).
__device__ __forceinline__ uint32_t ge_mask(int w, int b)
{
    const int bw = b >> 5;
    if (w < bw) return 0u;
    if (w > bw) return FULL;
    return FULL << (b & 31);
}

// Bits < b of word `w`.
__device__ __forceinline__ uint32_t lt_mask(int w, int b) { return ~ge_mask(w, b); }

// Transpose of a 32 x 32 bit matrix held one row per lane (bit j of lane i is entry (i, j)): on
// return bit i of lane j is entry (i, j). Five exchange rounds: the two off-diagonal 16 x 16 blocks
// trade places, then the off-diagonal 8 x 8 blocks inside each diagonal block, and so on down to
// single bits; each round is one shuffle and a masked merge.
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x)
{
    const unsigned lane = threadIdx.x & 31;
    constexpr uint32_t lo[5] = {0x0000ffffu, 0x00ff00ffu, 0x0f0f0f0fu, 0x33333333u, 0x55555555u};
#pragma unroll
    for (int r = 0; r < 5; ++r) {
        const int s = 16 >> r;
        const uint32_t m = lo[r];
        const uint32_t y = __shfl_xor_sync(FULL, x, s);
        x = (lane & (unsigned)s) ? ((x & ~m) | ((y >> s) & m)) : ((x & m) | ((y & m) << s));
    }
    return x;
}

// Largest number of restricted-column words (x32 attributes) a lane keeps in registers, by M: 8 (up
// to 256 relevant attributes) when M > 128, 4 when M > 64, else 2 (R <= M). The narrower kernels
// stay within 64 registers.
constexpr int REG_WORDS_MAX = 8;
constexpr int reg_words_for(int m) { return m > 128 ? 8 : (m > 64 ? 4 : 2); }

// Entry size in 32-bit words of an object-list queue root holding `cnt` objects (counting only).
__device__ __forceinline__ unsigned queue_entry_words(unsigned cnt, int wm)
{
    const unsigned per = cnt <= 32u ? 32u : 64u;
    return per + (unsigned)wm + 2u;
}

// A launch shape computed once per device and shared-memory size.
struct ShapeCache {
    int dev = -1;
    size_t smem = 0;
    int wpb = 0;
    int per_sm = 1;
};

}  // namespace fca
