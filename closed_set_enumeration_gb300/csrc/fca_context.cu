// Context build kernels of libfca (sm_103a).
//
//  mask_rows_kernel      clears the padding bits past M of every row.
//  transpose_kernel      ctxRows -> ctxCols, 32x32 bit tiles by warp ballots
//                        (the Parallel FCBO article, section 3.1, builds the
//                        same column bitmaps with one atomicOr per set bit).
//  top_kernel            top intent G' = AND of all rows, and whether some
//                        row holds every attribute (then the bottom concept
//                        has a non-empty extent and the search reaches it).
//  append_bottom_kernel  the bottom concept (intent M) when its extent is empty.
#include <cuda_runtime.h>

#include "fca_device.cuh"

namespace fca {
namespace {


// Clear the padding bits past M in the last word of every row (they are ignored on input).
__global__ void mask_rows_kernel(uint32_t *rows, Dims d)
{
    const long long o = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (o < d.n) rows[o * d.wm + d.wm - 1] &= (1u << (d.m & 31)) - 1u;
}

__global__ void transpose_kernel(const uint32_t *__restrict__ rows, uint32_t *__restrict__ cols,
                                 Dims d)
{
    const int wpb = blockDim.x >> 5;
    const long long tile = (long long)blockIdx.x * wpb + (threadIdx.x >> 5);
    if (tile >= d.wn * (long long)d.wm) return;  // uniform per warp
    const unsigned lane = threadIdx.x & 31;
    const long long ot = tile / d.wm;             // 32 objects
    const int aw = (int)(tile % d.wm);            // 32 attributes
    const long long o = ot * 32 + lane;
    uint32_t v = (o < d.n) ? rows[o * d.wm + aw] : 0u;
    const int valid = d.m - aw * 32;
    if (valid < 32) v &= (1u << valid) - 1u;      // ignore padding bits
    uint32_t mine = 0;
#pragma unroll
    for (int b = 0; b < 32; ++b) {
        const uint32_t bal = __ballot_sync(FULL, (v >> b) & 1u);
        if (lane == (unsigned)b) mine = bal;
    }
    const int a = aw * 32 + (int)lane;
    if (a < d.m) cols[(size_t)a * d.wnp + ot] = mine;
}

__global__ void top_kernel(const uint32_t *__restrict__ rows, uint32_t *top, uint32_t *flag, Dims d)
{
    __shared__ uint32_t red[32];
    const long long o = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const bool valid = o < d.n;
    bool full_row = valid;
    for (int w = 0; w < d.wm; ++w) {
        const int vb = d.m - w * 32;
        const uint32_t mask = vb >= 32 ? FULL : ((1u << vb) - 1u);
        uint32_t v = valid ? (rows[o * d.wm + w] & mask) : FULL;
        if (valid && v != mask) full_row = false;
        v = __reduce_and_sync(FULL, v);
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
        __syncthreads();
        if (threadIdx.x < 32) {
            uint32_t x = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : FULL;
            x = __reduce_and_sync(FULL, x);
            if (threadIdx.x == 0) atomicAnd(&top[w], x);
        }
        __syncthreads();
    }
    if (full_row) atomicOr(flag, 1u);
}

// The bottom concept when its extent is empty (no row holds every attribute): one more row.
__global__ void append_bottom_kernel(const uint32_t *flag, const uint32_t *full_mask, uint32_t *out,
                                     unsigned long long capacity, Counters *ctr, int wm, int guard)
{
    if (guard && (ctr->error != 0u || ctr->next_count != 0ull)) return;   // the search did not end here
    if (*flag) return;   // some object holds every attribute: the search has output it
    const unsigned lane = threadIdx.x & 31;
    unsigned long long slot = 0;
    if (lane == 0) slot = atomicAdd(&ctr->out_count, 1ull);
    slot = __shfl_sync(FULL, slot, 0);
    if (slot < capacity)
        for (int w = (int)lane; w < wm; w += 32) out[slot * wm + w] = full_mask[w];
}

// Counter set-up before a bitmap-tier launch: the next level's current fill, a zero work cursor and
// error word; then a copy of the counters, restored if the launch has to be rolled back.
__global__ void prepare_expand_kernel(Counters *ctr, Counters *snap, unsigned long long next_fill)
{
    if (threadIdx.x == 0) {
        ctr->next_count = next_fill;
        ctr->work_head = 0ull;
        ctr->error = 0u;
    }
    __syncthreads();
    const uint32_t *src = reinterpret_cast<const uint32_t *>(ctr);
    uint32_t *dst = reinterpret_cast<uint32_t *>(snap);
    for (int i = (int)threadIdx.x; i < (int)(sizeof(Counters) / 4); i += (int)blockDim.x) dst[i] = src[i];
}

// Before launch i of a chain of bitmap-tier launches (see ChainSlots).
__global__ void prepare_chain_kernel(Counters *ctr, ChainSlots *cs, int i, unsigned long long n0)
{
    if (threadIdx.x == 0) {
        unsigned long long pc = i == 0 ? n0 : ctr->next_count;
        if (i == 0) ctr->error = 0u;
        else if (ctr->error) pc = 0ull;     // an earlier launch of the chain overflowed: no work
        cs->counts[i] = pc;
        cs->pcount = pc;
        ctr->next_count = 0ull;
        ctr->work_head = 0ull;
    }
    __syncthreads();
    const uint32_t *src = reinterpret_cast<const uint32_t *>(ctr);
    uint32_t *dst = reinterpret_cast<uint32_t *>(&cs->snaps[i]);
    for (int w = (int)threadIdx.x; w < (int)(sizeof(Counters) / 4); w += (int)blockDim.x) dst[w] = src[w];
}

// Start of an enumeration: zero counters with the top intent in output row 0 (when capacity allows)
// and the root node (G, G', 0), either as entry 0 of bitmap level 0 (qi < 0) or as the first root of
// object-list queue qi.
__global__ void start_kernel(Counters *ctr, const uint32_t *top, const uint32_t *root_ext, Dims d,
                             uint32_t *out, unsigned long long capacity, Level L0, Queue Q, int qi)
{
    const int t = (int)threadIdx.x;
    uint32_t *c = reinterpret_cast<uint32_t *>(ctr);
    for (int i = t; i < (int)(sizeof(Counters) / 4); i += (int)blockDim.x) c[i] = 0u;
    __syncthreads();
    if (t == 0) {
        ctr->out_count = 1ull;
        if (qi >= 0) ctr->q_count[qi] = 1ull;
    }
    for (int w = t; w < d.wm; w += (int)blockDim.x) {
        if (capacity >= 1ull) out[w] = top[w];
        if (qi < 0) L0.itt[w] = top[w];
        else Q.itt[w] = top[w];
    }
    if (qi < 0) {
        for (long long q = t; q < d.wnp; q += blockDim.x) L0.ext[q] = root_ext[q];
        if (t == 0) {
            L0.y[0] = 0;
            L0.n[0] = (int32_t)d.n;
        }
    } else {
        const int per = 32 << qi;
        for (int i = t; i < per; i += (int)blockDim.x) Q.ids[i] = i < d.n ? (uint32_t)i : 0u;
        if (t == 0) {
            Q.y[0] = 0;
            Q.n[0] = (int32_t)d.n;
        }
    }
}

}  // namespace

int launch_prepare_expand(Counters *ctr, Counters *snap, uint64_t next_fill, void *stream)
{
    prepare_expand_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(ctr, snap, next_fill);
    return (int)cudaGetLastError();
}

int launch_prepare_chain(Counters *ctr, ChainSlots *cs, int i, uint64_t n0, void *stream)
{
    prepare_chain_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(ctr, cs, i, n0);
    return (int)cudaGetLastError();
}

int launch_start(Counters *ctr, const uint32_t *top, const uint32_t *root_ext, const Dims &d, uint32_t *out,
                 uint64_t capacity, const Level &L0, const Queue &Q, int qi, void *stream)
{
    start_kernel<<<1, 256, 0, (cudaStream_t)stream>>>(ctr, top, root_ext, d, out, capacity, L0, Q, qi);
    return (int)cudaGetLastError();
}

int launch_mask_rows(uint32_t *rows, const Dims &d, void *stream)
{
    if ((d.m & 31) == 0) return (int)cudaSuccess;
    const int tpb = 256;
    mask_rows_kernel<<<(unsigned)((d.n + tpb - 1) / tpb), tpb, 0, (cudaStream_t)stream>>>(rows, d);
    return (int)cudaGetLastError();
}

int launch_transpose(const uint32_t *rows, uint32_t *cols, const Dims &d, void *stream)
{
    const long long tiles = d.wn * (long long)d.wm;
    const int wpb = 8;
    const long long blocks = (tiles + wpb - 1) / wpb;
    transpose_kernel<<<(unsigned)blocks, wpb * 32, 0, (cudaStream_t)stream>>>(rows, cols, d);
    return (int)cudaGetLastError();
}

int launch_append_bottom(const uint32_t *flag, const uint32_t *full_mask, uint32_t *out, uint64_t capacity,
                         Counters *ctr, const Dims &d, void *stream, int guard)
{
    append_bottom_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(flag, full_mask, out, capacity, ctr, d.wm, guard);
    return (int)cudaGetLastError();
}

int launch_top(const uint32_t *rows, uint32_t *top, uint32_t *flag, const Dims &d, void *stream)
{
    const int tpb = 256;
    const long long blocks = (d.n + tpb - 1) / tpb;
    top_kernel<<<(unsigned)blocks, tpb, 0, (cudaStream_t)stream>>>(rows, top, flag, d);
    return (int)cudaGetLastError();
}

}  // namespace fca
