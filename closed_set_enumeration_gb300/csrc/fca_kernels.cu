// Kernels of libfca (sm_103a). Bitwise set algebra only: no tensor cores.
//
//  mask_rows_kernel      clears the padding bits past M of every row.
//  transpose_kernel      ctxRows -> ctxCols, 32x32 bit tiles by warp ballots
//                        (the Parallel FCBO article, section 3.1, builds the
//                        same column bitmaps with one atomicOr per set bit).
//  top_kernel            top intent G' = AND of all rows, and whether some
//                        row holds every attribute (then the bottom concept
//                        has a non-empty extent and the search reaches it).
//  expand_bitmap_kernel  bitmap tier: one warp per (parent, j) candidate:
//                        extent intersection, closure, canonical test,
//                        compaction of the child (FCbO-to-CUDA article,
//                        sections 2.1-2.3, 4.2-4.4; Parallel FCBO article,
//                        sections 2.1, 3.2).
//  subtree_kernel<NW>    object-list tier: one warp runs a whole subtree whose
//                        root extent holds at most 32*NW objects.
#include <cuda_runtime.h>

#include <algorithm>

#include "fca_internal.cuh"

namespace fca {
namespace {

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

// Largest number of restricted-column words (x32 attributes) a lane keeps in registers: 8 (up to
// 256 relevant attributes) when M > 128, else 4, which keeps the kernel within 64 registers.
constexpr int REG_WORDS_MAX = 8;
constexpr int reg_words_for(int m) { return m > 128 ? 8 : 4; }

// Entry size in 32-bit words of an object-list queue root holding `cnt` objects (counting only).
__device__ __forceinline__ unsigned queue_entry_words(unsigned cnt, int wm)
{
    const unsigned per = cnt <= 32u ? 32u : 64u;
    return per + (unsigned)wm + 2u;
}

// ------------------------------------------------------------------ context build

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
                                     unsigned long long capacity, Counters *ctr, int wm)
{
    if (*flag) return;   // some object holds every attribute: the search has output it
    const unsigned lane = threadIdx.x & 31;
    unsigned long long slot = 0;
    if (lane == 0) slot = atomicAdd(&ctr->out_count, 1ull);
    slot = __shfl_sync(FULL, slot, 0);
    if (slot < capacity)
        for (int w = (int)lane; w < wm; w += 32) out[slot * wm + w] = full_mask[w];
}

// ------------------------------------------------------------------ bitmap tier

// C subset of column K, with C = A & J on the staged chunks of A (values av[i] at uint4 index
// idx[i]) and J the candidate's column: early exit at the first block of 64 chunks that disagrees.
// `loads` counts the column uint4 read.
__device__ __forceinline__ bool subset_of_column(const uint4 *av, const uint32_t *idx, int nnz,
                                                 const uint4 *__restrict__ J, const uint4 *__restrict__ K,
                                                 unsigned lane, unsigned &loads)
{
    for (int base = 0; base < nnz; base += 64) {
        bool bad = false;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = base + h * 32 + (int)lane;
            if (i < nnz) {
                const uint4 a4 = av[i], j4 = __ldg(J + idx[i]);
                const uint4 c = make_uint4(a4.x & j4.x, a4.y & j4.y, a4.z & j4.z, a4.w & j4.w);
                loads += 1;
                if (c.x | c.y | c.z | c.w) {
                    const uint4 k = __ldg(K + idx[i]);
                    ++loads;
                    bad |= ((c.x & ~k.x) | (c.y & ~k.y) | (c.z & ~k.z) | (c.w & ~k.w)) != 0u;
                }
            }
        }
        if (__any_sync(FULL, bad)) return false;
    }
    return true;
}

// Largest parent extent (objects) whose columns the block rebuilds restricted to its objects,
// limited by shared memory: M restricted columns of TR/32 words plus the object list.
constexpr int RESTRICT_CAP = 4096;
constexpr int RPL = RESTRICT_CAP / 1024;   // restricted-column words per lane
constexpr int ROW_BOUND = 8;               // rows ANDed for the closure's upper bound (restricted path)

// Shared memory of expand_bitmap_kernel. Both paths first stage the parent's non-zero extent
// chunks (uint4 index and value). The gather path then keeps, per warp, up to SMALL_MAX object
// ids (C itself is recomputed from the staged chunks and column j when needed); the restricted
// path keeps the parent's object list, its columns restricted to those objects (M x TR/32 words)
// and per-warp object ids.
struct ExpandLayout {
    size_t o_aidx, o_aval, o_wbase, per_warp, o_oid, o_colr, o_rids, o_blk, bytes;
    __host__ __device__ ExpandLayout(const Dims &d, int wpb, int tr)
    {
        const size_t wq = (size_t)(d.wnp >> 2);
        o_aval = 0;                                        // wq uint4
        o_aidx = o_aval + wq * 16;                         // wq uint32
        o_wbase = (o_aidx + wq * 4 + 15) & ~(size_t)15;
        per_warp = SMALL_MAX * 4;                          // ids
        const size_t gather_end = o_wbase + per_warp * wpb;
        o_oid = o_wbase;                                   // tr uint32
        o_colr = o_oid + (size_t)tr * 4;                   // m x tr/32 uint32
        o_rids = o_colr + (size_t)d.m * (size_t)(tr / 32) * 4;
        const size_t restrict_end = o_rids + (size_t)wpb * SMALL_MAX * 4;
        o_blk = ((gather_end > restrict_end ? gather_end : restrict_end) + 15) & ~(size_t)15;
        bytes = o_blk + 32 * 4;                            // block scratch: counts and sums
    }
};

// Block-wide exclusive prefix sum of one value per thread (all threads call it); returns the
// thread's offset and writes the block total to *total. `scratch` holds 2 x 32 ints.
__device__ __forceinline__ int block_exclusive_sum(int v, int *scratch, int *total)
{
    const unsigned lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5, wpb = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(FULL, incl, off);
        if (lane >= (unsigned)off) incl += t;
    }
    if (lane == 31) scratch[wib] = incl;
    __syncthreads();
    int before = 0, all = 0;
    for (int w = 0; w < wpb; ++w) {
        const int s = scratch[w];
        if (w < wib) before += s;
        all += s;
    }
    __syncthreads();
    *total = all;
    return before + incl - v;
}

// The rest of a candidate once |C| and the first `need` object ids of C are known: the closure
// (the AND of their rows: exact when need == |C|, else an upper bound whose extra attributes are
// decided by `subset(k)` in ascending order, so a violation below j ends the candidate early),
// the canonical test, the intent and the child. `write_ext(dst)` writes C as a dense bitmap for a
// child of the next level; `all_ids()` completes the id list of a small child (need < |C|).
template <bool COUNT, class Subset, class WriteExt, class AllIds>
__device__ __forceinline__ void finish_candidate(const ExpandArgs &a, const Dims &d, const uint32_t *B, int j,
                                                 unsigned cnt, const uint32_t *ids, unsigned need, Subset &&subset,
                                                 WriteExt &&write_ext, AllIds &&all_ids,
                                                 unsigned long long &my_bytes)
{
    const unsigned lane = threadIdx.x & 31;
    uint32_t U = 0;
    for (int w = 0; w < d.wm; ++w) {
        uint32_t acc = FULL;
        for (unsigned i = lane; i < need; i += 32) acc &= __ldg(a.rows + (size_t)ids[i] * d.wm + w);
        acc = __reduce_and_sync(FULL, acc);
        if ((int)lane == w) U = acc;
    }
    if (COUNT && lane == 0) my_bytes += (unsigned long long)need * d.wm * 4;   // rows read
    const uint32_t Bw = lane < (unsigned)d.wm ? B[lane] : 0u;
    const int ju = j >> 5;
    const uint32_t jbit = 1u << (j & 31);
    const uint32_t pm = lt_mask((int)lane, j);   // attributes below j
    uint32_t Dw;
    if (need == cnt) {
        Dw = U;
        if (__any_sync(FULL, (U & ~Bw & pm) != 0u)) return;
    } else {
        // attributes that may still join: in U, not in B, not j; tested in ascending order
        uint32_t X = U & ~Bw;
        if ((int)lane == ju) X &= ~jbit;
        Dw = Bw | ((int)lane == ju ? jbit : 0u);
        for (;;) {
            const unsigned bal = __ballot_sync(FULL, X != 0u);
            if (!bal) break;
            const int u = __ffs(bal) - 1;
            const uint32_t xw = __shfl_sync(FULL, X, u);
            const int b = __ffs(xw) - 1;
            const int k = u * 32 + b;
            if ((int)lane == u) X &= ~(1u << b);
            if (subset(k)) {
                if (k < j) return;                      // not canonical
                if ((int)lane == u) Dw |= 1u << b;
            }
        }
    }

    if (COUNT && lane == 0) {   // the intent row and the child entry written
        my_bytes += (unsigned long long)d.wm * 4;
        my_bytes += cnt <= (unsigned)SMALL_MAX ? 4ull * queue_entry_words(cnt, d.wm)
                                               : (unsigned long long)(4 * d.wnp + 4 * d.wm + 4);
    }
    // emit the intent
    unsigned long long slot = 0;
    if (lane == 0) slot = atomicAdd(&a.ctr->out_count, 1ull);
    slot = __shfl_sync(FULL, slot, 0);
    if (slot < a.capacity && lane < (unsigned)d.wm) a.out[slot * d.wm + lane] = Dw;

    // the child (C, D, j+1): an object-list root, or an entry of the next bitmap level.
    // A destination that is full only counts; the driver rolls the launch back and retries.
    if (cnt <= (unsigned)SMALL_MAX) {
        const int qi = cnt <= 32u ? 0 : 1;
        const Queue &Q = a.q[qi];
        const int per = 32 << qi;
        unsigned long long s = 0;
        if (lane == 0) s = atomicAdd(&a.ctr->q_count[qi], 1ull);
        s = __shfl_sync(FULL, s, 0);
        if (s >= Q.cap) {
            if (lane == 0) atomicOr(&a.ctr->error, ERR_QUEUE0 << qi);
            return;
        }
        if (need < cnt) all_ids();
        __syncwarp();
        for (int i = (int)lane; i < per; i += 32) Q.ids[s * per + i] = i < (int)cnt ? ids[i] : 0u;
        if (lane < (unsigned)d.wm) Q.itt[s * d.wm + lane] = Dw;
        if (lane == 0) { Q.y[s] = j + 1; Q.n[s] = (int)cnt; }
    } else {
        unsigned long long s = 0;
        if (lane == 0) s = atomicAdd(&a.ctr->next_count, 1ull);
        s = __shfl_sync(FULL, s, 0);
        if (s >= a.next.cap) {
            if (lane == 0) atomicOr(&a.ctr->error, ERR_NEXT);
            return;
        }
        write_ext(a.next.ext + s * (size_t)d.wnp);
        if (lane < (unsigned)d.wm) a.next.itt[s * d.wm + lane] = Dw;
        if (lane == 0) { a.next.y[s] = j + 1; a.next.n[s] = (int)cnt; }
    }
}

// Bitmap tier. A work item is (parent, part of the attribute range). The block stages the parent's
// non-zero extent chunks once. Extents of at most `a.restrict_max` objects are then turned into an
// object list, and the rows of those objects are transposed into columns restricted to them (one
// ballot per attribute and 32 objects); each candidate's C is read from those columns without any
// global column access. Larger extents keep the chunk list: each warp gathers column j on the
// parent's non-zero chunks. Either way the warps of the block take the part's candidates j in turn.
template <bool COUNT>
__global__ void __launch_bounds__(256) expand_bitmap_kernel(ExpandArgs a)
{
    extern __shared__ __align__(16) unsigned char smem[];
    const Dims d = a.d;
    const int wq = (int)(d.wnp >> 2);
    const unsigned lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int wpb = blockDim.x >> 5;
    const int tr = a.restrict_max;
    const ExpandLayout L(d, wpb, tr);
    uint4 *aval = reinterpret_cast<uint4 *>(smem + L.o_aval);
    uint32_t *aidx = reinterpret_cast<uint32_t *>(smem + L.o_aidx);
    uint32_t *gids = reinterpret_cast<uint32_t *>(smem + L.o_wbase + L.per_warp * wib);
    uint32_t *oid = reinterpret_cast<uint32_t *>(smem + L.o_oid);
    uint32_t *colr = reinterpret_cast<uint32_t *>(smem + L.o_colr);
    uint32_t *rids = reinterpret_cast<uint32_t *>(smem + L.o_rids) + (size_t)wib * SMALL_MAX;
    int *blk = reinterpret_cast<int *>(smem + L.o_blk);   // [0..31] scan scratch
    const uint4 *cols4 = reinterpret_cast<const uint4 *>(a.cols);
    const uint4 *ext4 = reinterpret_cast<const uint4 *>(a.in.ext);

    unsigned long long my_closures = 0, my_bytes = 0;
    unsigned loads = 0;   // uint4 loads of columns by this lane (counting only)
    const int parts = a.parts;
    const int span = (d.m + parts - 1) / parts;
    const unsigned long long items = a.p_count * (unsigned long long)parts;
    for (unsigned long long item = blockIdx.x; item < items; item += gridDim.x) {
        const unsigned long long p = a.p_begin + item / (unsigned)parts;
        const int part = (int)(item % (unsigned)parts);
        const int y = a.in.y[p];
        // a parent small enough for restricted columns is expanded whole by its first part (the
        // transposition is paid once), when its candidates make that cheaper than gathering
        const int np = a.in.n[p];
        const int gw = (np + 31) >> 5;
        const bool restricted = np <= tr && (long long)(d.m - y) * min(wq, np) >= 4ll * gw * d.wm;
        if (restricted && part > 0) continue;
        const int j_lo = restricted ? y : max(y, part * span);
        const int j_hi = restricted ? d.m : min(d.m, (part + 1) * span);
        if (j_lo >= j_hi) continue;                       // uniform over the block
        const uint32_t *B = a.in.itt + p * d.wm;

        // ---- stage the non-zero chunks of A in order (block-wide compaction), and |A|
        const uint4 *A4 = ext4 + p * wq;
        __syncthreads();
        int nnz = 0, na = 0;
        for (int base = 0; base < wq; base += blockDim.x) {
            const int q = base + (int)threadIdx.x;
            uint4 x = make_uint4(0u, 0u, 0u, 0u);
            if (q < wq) x = A4[q];
            const bool nz = (x.x | x.y | x.z | x.w) != 0u;
            int round_nnz = 0, round_na = 0;
            const int off = block_exclusive_sum(nz ? 1 : 0, blk, &round_nnz);
            (void)block_exclusive_sum((int)popc4(x), blk, &round_na);
            if (nz) { aval[nnz + off] = x; aidx[nnz + off] = (uint32_t)q; }
            nnz += round_nnz;
            na += round_na;
        }
        __syncthreads();
        if (COUNT && threadIdx.x == 0) my_bytes += (unsigned long long)d.wnp * 4;   // the parent extent

        if (restricted) {
            // ---- restricted path: object list, then the columns restricted to these objects
            int base_id = 0;
            for (int base = 0; base < nnz; base += blockDim.x) {
                const int i = base + (int)threadIdx.x;
                const uint4 x = i < nnz ? aval[i] : make_uint4(0u, 0u, 0u, 0u);
                int round = 0;
                int pos = base_id + block_exclusive_sum((int)popc4(x), blk, &round);
                if (i < nnz) {
                    const uint32_t q = aidx[i];
                    const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        uint32_t bits = w4[t];
                        while (bits) {
                            const int b = __ffs(bits) - 1;
                            bits &= bits - 1u;
                            oid[pos++] = (4 * q + t) * 32 + b;
                        }
                    }
                }
                base_id += round;
            }
            __syncthreads();
            const int G = (na + 31) >> 5;                  // restricted-column words
            for (int unit = wib; unit < G * d.wm; unit += wpb) {
                const int g = unit / d.wm, w = unit % d.wm;
                const int pidx = 32 * g + (int)lane;
                const uint32_t v = pidx < na ? __ldg(a.rows + (size_t)oid[pidx] * d.wm + w) : 0u;
                uint32_t mine = 0;
#pragma unroll
                for (int b = 0; b < 32; ++b) {
                    const uint32_t bal = __ballot_sync(FULL, (v >> b) & 1u);
                    if (lane == (unsigned)b) mine = bal;
                }
                const int k = 32 * w + (int)lane;
                if (k < d.m) colr[(size_t)k * G + g] = mine;
            }
            __syncthreads();
            if (COUNT && threadIdx.x == 0) my_bytes += (unsigned long long)na * d.wm * 4;   // rows of A

            for (int j = j_lo + wib; j < j_hi; j += wpb) {
                if ((B[j >> 5] >> (j & 31)) & 1u) continue;   // saturation: A inside column j
                ++my_closures;
                uint32_t c[RPL];
                unsigned cnt = 0;
#pragma unroll
                for (int r = 0; r < RPL; ++r) {
                    const int g = 32 * r + (int)lane;
                    c[r] = g < G ? colr[(size_t)j * G + g] : 0u;
                    cnt += __popc(c[r]);
                }
                cnt = __reduce_add_sync(FULL, cnt);
                if (cnt == 0) continue;   // empty extent: its closure is the bottom, added by the host

                // the first object ids of C in ascending order: the closure is bounded by their rows and
                // completed on the restricted columns
                auto collect = [&](unsigned want) {
                    unsigned got = 0;
#pragma unroll
                    for (int r = 0; r < RPL; ++r) {
                        if (got >= want) break;
                        const unsigned pc = __popc(c[r]);
                        unsigned incl = pc;
#pragma unroll
                        for (int off = 1; off < 32; off <<= 1) {
                            const unsigned t = __shfl_up_sync(FULL, incl, off);
                            if (lane >= (unsigned)off) incl += t;
                        }
                        unsigned pos = got + incl - pc;
                        uint32_t bits = c[r];
                        const int g = 32 * r + (int)lane;
                        while (bits && pos < want) {
                            const int b = __ffs(bits) - 1;
                            bits &= bits - 1u;
                            rids[pos++] = oid[32 * g + b];
                        }
                        got += __shfl_sync(FULL, incl, 31);
                    }
                };
                const unsigned need = cnt < (unsigned)ROW_BOUND ? cnt : (unsigned)ROW_BOUND;
                collect(need);
                __syncwarp();
                finish_candidate<COUNT>(
                    a, d, B, j, cnt, rids, need,
                    [&](int k) {
                        bool bad = false;
#pragma unroll
                        for (int r = 0; r < RPL; ++r) {
                            const int g = 32 * r + (int)lane;
                            if (g < G) bad |= (c[r] & ~colr[(size_t)k * G + g]) != 0u;
                        }
                        return !__any_sync(FULL, bad);
                    },
                    [&](uint32_t *dst) {
                        for (int q = (int)lane; q < (int)d.wnp; q += 32) dst[q] = 0u;
                        __syncwarp();
#pragma unroll
                        for (int r = 0; r < RPL; ++r) {
                            uint32_t bits = c[r];
                            const int g = 32 * r + (int)lane;
                            while (bits) {
                                const int b = __ffs(bits) - 1;
                                bits &= bits - 1u;
                                const uint32_t o = oid[32 * g + b];
                                atomicOr(dst + (o >> 5), 1u << (o & 31));
                            }
                        }
                    },
                    [&]() { collect(cnt); },
                    my_bytes);
                __syncwarp();
            }
            continue;
        }

        // ---- gather path: candidates j of this part, warps in turn
        for (int j = j_lo + wib; j < j_hi; j += wpb) {
            if ((B[j >> 5] >> (j & 31)) & 1u) continue;   // saturation: A inside column j
            ++my_closures;

            // |C| for C = A & column j on the chunks of A (C itself is recomputed when needed)
            const uint4 *J4 = cols4 + (size_t)j * wq;
            unsigned cnt = 0;
            for (int i = (int)lane; i < nnz; i += 32) {
                const uint4 x = aval[i], cc = __ldg(J4 + aidx[i]);
                if (COUNT) ++loads;
                cnt += __popc(x.x & cc.x) + __popc(x.y & cc.y) + __popc(x.z & cc.z) + __popc(x.w & cc.w);
            }
            cnt = __reduce_add_sync(FULL, cnt);
            if (cnt == 0) continue;   // empty extent: its closure is the bottom, added by the host

            // object ids of C in ascending order: all of them when |C| <= SMALL_MAX, else the first 32
            const unsigned need = cnt <= (unsigned)SMALL_MAX ? cnt : 32u;
            unsigned got = 0;
            for (int base = 0; base < nnz && got < need; base += 32) {
                const int i = base + (int)lane;
                uint4 x = make_uint4(0u, 0u, 0u, 0u);
                uint32_t q = 0u;
                if (i < nnz) {
                    const uint4 av = aval[i];
                    q = aidx[i];
                    const uint4 cc = __ldg(J4 + q);
                    if (COUNT) ++loads;
                    x = make_uint4(av.x & cc.x, av.y & cc.y, av.z & cc.z, av.w & cc.w);
                }
                const unsigned pc = popc4(x);
                unsigned incl = pc;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const unsigned t = __shfl_up_sync(FULL, incl, off);
                    if (lane >= (unsigned)off) incl += t;
                }
                unsigned pos = got + incl - pc;
                const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    uint32_t bits = w4[t];
                    while (bits && pos < need) {
                        const int b = __ffs(bits) - 1;
                        bits &= bits - 1u;
                        gids[pos++] = (uint32_t)((4 * q + t) * 32 + b);
                    }
                }
                got += __shfl_sync(FULL, incl, 31);
            }
            __syncwarp();
            finish_candidate<COUNT>(
                a, d, B, j, cnt, gids, need,
                [&](int k) { return subset_of_column(aval, aidx, nnz, J4, cols4 + (size_t)k * wq, lane, loads); },
                [&](uint32_t *dst) {
                    uint4 *dst4 = reinterpret_cast<uint4 *>(dst);
                    for (int q = (int)lane; q < wq; q += 32) dst4[q] = make_uint4(0u, 0u, 0u, 0u);
                    __syncwarp();
                    for (int i = (int)lane; i < nnz; i += 32) {
                        const uint4 av = aval[i], cc = __ldg(J4 + aidx[i]);
                        const uint4 x = make_uint4(av.x & cc.x, av.y & cc.y, av.z & cc.z, av.w & cc.w);
                        if (x.x | x.y | x.z | x.w) dst4[aidx[i]] = x;
                    }
                },
                [&]() {},
                my_bytes);
            __syncwarp();
        }
    }
    if (COUNT) {
        const unsigned tl = __reduce_add_sync(FULL, loads);
        if (lane == 0) atomicAdd(&a.ctr->bytes, my_bytes + 16ull * tl);
    }
    if (lane == 0 && my_closures) atomicAdd(&a.ctr->closures, my_closures);
}

// ------------------------------------------------------------------ object-list tier

// Shared-memory layout of one warp of subtree_kernel<NW> (32-bit words).
struct SubtreeLayout {
    int mp, wm, fr, fs;
    size_t o_rmap, o_rootb, o_rm, o_rlo, o_sufb, o_dsc, o_stack, o_outbuf, words;
    __host__ __device__ SubtreeLayout(const Dims &d, int nw)
    {
        mp = (d.m + 31) & ~31;
        wm = d.wm;
        fr = (32 * nw < d.m ? 32 * nw : d.m) + 1;     // depth <= |extent| and <= |R|
        // frame: extent mask, then cursor + intent (shared-memory search) or candidates + intent
        fs = nw + (1 + wm > 2 * REG_WORDS_MAX ? 1 + wm : 2 * REG_WORDS_MAX);
        o_rmap = (size_t)nw * mp;
        o_rootb = o_rmap + mp / 2;
        o_rm = o_rootb + 32;
        o_rlo = o_rm + 32;
        o_sufb = o_rlo + 34;
        o_dsc = o_sufb + 32;
        o_stack = o_dsc + 34;
        o_outbuf = o_stack + (size_t)fr * fs;
        words = o_outbuf + (size_t)OUTBUF * wm;
        words = (words + 3) & ~(size_t)3;
    }
};

// Per-warp state of the object-list tier: shared-memory areas of the current subtree root,
// the output buffer and the warp's counters.
struct SubtreeWarp {
    uint32_t *cR;       // restricted columns, NW planes x mp (compact attribute index)
    uint16_t *rmap;     // compact index -> attribute
    uint32_t *rootB;    // root intent (full attribute space), 32 words
    uint32_t *Rm;       // relevant attributes per full word
    uint32_t *rlo;      // first compact index of each full word (wm + 1 entries)
    uint32_t *sufB;     // root-intent attributes in the words above each word
    uint32_t *dsc;      // compact intent of the child being written
    uint32_t *stk;      // search stack
    uint32_t *ob;       // output buffer, OUTBUF x wm
    int mp, wm, fs, m;
    uint32_t *out;
    unsigned long long capacity;
    Counters *ctr;
    int nb;             // intents waiting in the output buffer
    unsigned long long closures, ops;

    __device__ void flush()
    {
        const unsigned lane = threadIdx.x & 31;
        unsigned long long b0 = 0;
        if (lane == 0) b0 = atomicAdd(&ctr->out_count, (unsigned long long)nb);
        b0 = __shfl_sync(FULL, b0, 0);
        __syncwarp();
        for (int i = (int)lane; i < nb * wm; i += 32)
            if (b0 + (unsigned long long)(i / wm) < capacity) out[b0 * wm + i] = ob[i];
        __syncwarp();
        nb = 0;
    }

    // Write the full intent of a canonical child whose compact intent is in dsc[]:
    // root intent plus the compact bits mapped back to their attributes.
    template <bool COUNT>
    __device__ void emit()
    {
        const unsigned lane = threadIdx.x & 31;
        __syncwarp();
        if (lane < (unsigned)wm) {
            const int w = (int)lane;
            const int lo = (int)rlo[w], hi = (int)rlo[w + 1];
            const int su = lo >> 5, sh = lo & 31;
            const uint32_t s0 = dsc[su];
            const uint32_t s1 = sh ? dsc[su + 1] : 0u;
            uint32_t seg = sh ? ((s0 >> sh) | (s1 << (32 - sh))) : s0;
            const int len = hi - lo;
            if (len < 32) seg &= (1u << len) - 1u;
            uint32_t res = rootB[w];
            while (seg) {                      // each compact attribute of D in this word
                const int i = __ffs(seg) - 1;
                seg &= seg - 1u;
                res |= 1u << (rmap[lo + i] & 31);
            }
            ob[nb * wm + w] = res;
        }
        ++nb;
        if (COUNT) ops += (unsigned)wm;   // the intent words written
        __syncwarp();
        if (nb == OUTBUF) flush();
    }

    // Candidates of a child created at compact candidate j whose compact intent has `above`
    // attributes after j: the attributes after rmap[j] outside its full intent.
    __device__ void count_child(int j, int above)
    {
        const int rj = rmap[j];
        const int rw = rj >> 5, rb = rj & 31;
        const uint32_t hi = rb == 31 ? 0u : (rootB[rw] >> (rb + 1));
        closures += (unsigned long long)(m - rj - 1 - (int)sufB[rw] - __popc(hi) - above);
    }
};

// Depth-first search of one subtree with the restricted columns in registers: lane l holds the
// columns of compact attributes 32u + l, u < WRT (R <= 32 * WRT). Extent, intent and remaining
// candidates of the current node are warp-uniform registers; the stack of ancestors is in shared
// memory. A node's candidates are filtered once, when the node is entered, to the attributes
// whose column meets its extent (the others give an empty extent, whose closure is the bottom
// concept the host adds), so the loop only visits candidates with a non-empty C.
template <int NW, int WRT, bool COUNT>
__device__ void dfs_regs(SubtreeWarp &S, int R, int n, int jn, int slices, int slice)
{
    const unsigned lane = threadIdx.x & 31;
    uint32_t col[WRT][NW];
#pragma unroll
    for (int u = 0; u < WRT; ++u) {
        const int k = 32 * u + (int)lane;
#pragma unroll
        for (int t = 0; t < NW; ++t) col[u][t] = k < R ? S.cR[t * S.mp + k] : 0u;
    }
    uint32_t B[WRT], cand[WRT];
    uint32_t ext[NW];
#pragma unroll
    for (int t = 0; t < NW; ++t) {
        const int k = n - 32 * t;
        ext[t] = k >= 32 ? FULL : (k > 0 ? ((1u << k) - 1u) : 0u);
    }
    // the root: empty compact intent; candidates from jn on, in this slice, meeting the extent
#pragma unroll
    for (int u = 0; u < WRT; ++u) {
        bool meets = false;
#pragma unroll
        for (int t = 0; t < NW; ++t) meets = meets || (ext[t] & col[u][t]) != 0u;
        const int k = 32 * u + (int)lane;
        const bool mine = slices <= 1 || k % slices == slice;
        cand[u] = __ballot_sync(FULL, meets && mine) & ge_mask(u, jn);
        B[u] = 0u;
        if (COUNT) S.ops += 2ull * NW * (unsigned)max(0, min(32, R - 32 * u));
    }
    int depth = 0;
    for (;;) {
        int j = -1;
#pragma unroll
        for (int u = 0; u < WRT; ++u)
            if (j < 0 && cand[u]) j = 32 * u + __ffs(cand[u]) - 1;
        if (j < 0) {
            if (depth == 0) break;
            --depth;
            const uint32_t *f = S.stk + (size_t)depth * S.fs;
#pragma unroll
            for (int t = 0; t < NW; ++t) ext[t] = f[t];
#pragma unroll
            for (int u = 0; u < WRT; ++u) {
                cand[u] = f[NW + u];
                B[u] = f[NW + WRT + u];
            }
            __syncwarp();
            continue;
        }
        const int ju = j >> 5;
#pragma unroll
        for (int u = 0; u < WRT; ++u)
            if (u == ju) cand[u] &= cand[u] - 1u;     // j is the lowest remaining candidate
        uint32_t C[NW];
#pragma unroll
        for (int t = 0; t < NW; ++t) C[t] = ext[t] & S.cR[t * S.mp + j];
        if (COUNT) S.ops += NW;            // the extent intersection

        // closure over the relevant attributes, canonical prefix first
        const uint32_t jm = (1u << (j & 31)) - 1u;
        uint32_t D[WRT];
        bool canon = true;
#pragma unroll
        for (int u = 0; u < WRT; ++u) {
            bool in = true;
#pragma unroll
            for (int t = 0; t < NW; ++t) in = in && ((C[t] & ~col[u][t]) == 0u);
            D[u] = __ballot_sync(FULL, in);   // columns past R are 0, so those bits stay clear
            if (COUNT) S.ops += 2ull * NW * (unsigned)max(0, min(32, R - 32 * u)) + (u <= ju ? 2 : 0);
            if (u <= ju && (D[u] & ~B[u] & (u < ju ? FULL : jm))) { canon = false; break; }
        }
        if (!canon) continue;

        // canonical child (C, D, j+1): write its intent, count its candidates, descend
        if (lane == 0) {
#pragma unroll
            for (int u = 0; u < WRT; ++u) S.dsc[u] = D[u];
            S.dsc[WRT] = 0u;
        }
        S.emit<COUNT>();
        int above = 0;
#pragma unroll
        for (int u = 0; u < WRT; ++u) above += __popc(D[u] & ge_mask(u, j + 1));
        S.count_child(j, above);
        if (lane == 0) {
            uint32_t *f = S.stk + (size_t)depth * S.fs;
#pragma unroll
            for (int t = 0; t < NW; ++t) f[t] = ext[t];
#pragma unroll
            for (int u = 0; u < WRT; ++u) {
                f[NW + u] = cand[u];
                f[NW + WRT + u] = B[u];
            }
        }
        __syncwarp();
        ++depth;
#pragma unroll
        for (int t = 0; t < NW; ++t) ext[t] = C[t];
#pragma unroll
        for (int u = 0; u < WRT; ++u) {
            bool meets = false;
#pragma unroll
            for (int t = 0; t < NW; ++t) meets = meets || (C[t] & col[u][t]) != 0u;
            B[u] = D[u];
            cand[u] = __ballot_sync(FULL, meets) & ~D[u] & ge_mask(u, j + 1);
            if (COUNT) S.ops += 2ull * NW * (unsigned)max(0, min(32, R - 32 * u));
        }
    }
}

// Same search with the restricted columns read from shared memory, for any R <= M: lane u of the
// warp holds word u of the current compact intent.
template <int NW, bool COUNT>
__device__ void dfs_smem(SubtreeWarp &S, int R, int n, int jn, int slices, int slice)
{
    const unsigned lane = threadIdx.x & 31;
    const uint32_t validR = lt_mask((int)lane, R);
    const int WR = (R + 31) >> 5;
    uint32_t myB = 0;
    uint32_t ext[NW];
#pragma unroll
    for (int t = 0; t < NW; ++t) {
        const int k = n - 32 * t;
        ext[t] = k >= 32 ? FULL : (k > 0 ? ((1u << k) - 1u) : 0u);
    }
    int depth = 0;
    for (;;) {
        const uint32_t cw = ~myB & validR & ge_mask((int)lane, jn);
        const unsigned bal = __ballot_sync(FULL, cw != 0u);
        if (bal == 0u) {
            if (depth == 0) break;
            --depth;
            const uint32_t *f = S.stk + (size_t)depth * S.fs;
#pragma unroll
            for (int t = 0; t < NW; ++t) ext[t] = f[t];
            jn = (int)f[NW];
            myB = lane < (unsigned)S.wm ? f[NW + 1 + lane] : 0u;
            __syncwarp();
            continue;
        }
        const int u0 = __ffs(bal) - 1;
        const uint32_t cwu = __shfl_sync(FULL, cw, u0);
        const int j = u0 * 32 + __ffs(cwu) - 1;
        jn = j + 1;
        if (depth == 0 && slices > 1 && j % slices != slice) continue;   // another slice's child

        uint32_t C[NW];
        bool nonempty = false;
#pragma unroll
        for (int t = 0; t < NW; ++t) {
            C[t] = ext[t] & S.cR[t * S.mp + j];
            nonempty |= C[t] != 0u;
        }
        if (COUNT) S.ops += NW;
        if (!nonempty) continue;

        const int ju = j >> 5;
        const uint32_t jm = (1u << (j & 31)) - 1u;
        bool canon = true;
        uint32_t myD = 0;
        for (int u = 0; u < WR; ++u) {
            const int k = u * 32 + (int)lane;
            bool in = k < R;
            if (in) {
#pragma unroll
                for (int t = 0; t < NW; ++t) in = in && ((C[t] & ~S.cR[t * S.mp + k]) == 0u);
            }
            const uint32_t Du = __ballot_sync(FULL, in);
            if (COUNT) S.ops += 2ull * NW * (unsigned)min(32, R - 32 * u) + (u <= ju ? 2 : 0);
            if (u <= ju) {
                const uint32_t Bu = __shfl_sync(FULL, myB, u);
                const uint32_t pm = u < ju ? FULL : jm;
                if (Du & ~Bu & pm) { canon = false; break; }
            }
            if ((int)lane == u) myD = Du;
        }
        if (!canon) continue;

        if (lane <= (unsigned)WR) S.dsc[lane] = lane < (unsigned)WR ? myD : 0u;
        S.emit<COUNT>();
        unsigned c = __popc(myD & ge_mask((int)lane, j + 1) & validR);
        c = __reduce_add_sync(FULL, c);
        S.count_child(j, (int)c);
        {
            uint32_t *f = S.stk + (size_t)depth * S.fs;
#pragma unroll
            for (int t = 0; t < NW; ++t)
                if ((int)lane == t) f[t] = ext[t];
            if (lane == 0) f[NW] = (uint32_t)jn;
            if (lane < (unsigned)S.wm) f[NW + 1 + lane] = myB;
            __syncwarp();
            ++depth;
#pragma unroll
            for (int t = 0; t < NW; ++t) ext[t] = C[t];
            myB = myD;
        }
    }
}

template <int NW, bool COUNT, int RW>
__global__ void __launch_bounds__(256, RW > 4 ? 3 : 4) subtree_kernel(SubtreeArgs a)
{
    extern __shared__ uint32_t smw[];
    const Dims d = a.d;
    const SubtreeLayout L(d, NW);
    const unsigned lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    uint32_t *base = smw + (size_t)wib * L.words;
    SubtreeWarp S;
    S.cR = base;
    S.rmap = reinterpret_cast<uint16_t *>(base + L.o_rmap);
    S.rootB = base + L.o_rootb;
    S.Rm = base + L.o_rm;
    S.rlo = base + L.o_rlo;
    S.sufB = base + L.o_sufb;
    S.dsc = base + L.o_dsc;
    S.stk = base + L.o_stack;
    S.ob = base + L.o_outbuf;
    S.mp = L.mp;
    S.wm = d.wm;
    S.fs = L.fs;
    S.m = d.m;
    S.out = a.out;
    S.capacity = a.capacity;
    S.ctr = a.ctr;
    S.nb = 0;
    S.closures = 0;
    S.ops = 0;
    const int mp = L.mp, WM = d.wm, PER = 32 * NW;

    const unsigned long long items = a.q_count * (unsigned long long)a.slices;
    for (;;) {
        unsigned long long item = 0;
        if (lane == 0) item = atomicAdd(&a.ctr->q_head[a.q_index], 1ull);
        item = __shfl_sync(FULL, item, 0);
        if (item >= items) break;
        // work item = (root, slice): the slice takes the root's children j with j % slices == slice
        const unsigned long long r = item / (unsigned)a.slices;
        const int slice = (int)(item % (unsigned)a.slices);

        // ---- root: object ids, intent, cursor
        const int n = a.q.n[r];
        const int y0 = a.q.y[r];
        uint32_t id[NW];
#pragma unroll
        for (int t = 0; t < NW; ++t) {
            const int o = 32 * t + (int)lane;
            id[t] = o < n ? a.q.ids[r * PER + o] : 0u;
        }
        const uint32_t myRootB = lane < (unsigned)WM ? a.q.itt[r * WM + lane] : 0u;
        __syncwarp();
        S.rootB[lane] = myRootB;

        // ---- relevant attributes R (held by some but not all objects), compact index order =
        //      attribute order, and the columns restricted to the subtree's objects
        int R = 0;
        for (int w = 0; w < WM; ++w) {
            uint32_t rw[NW];
            uint32_t uni = 0;
#pragma unroll
            for (int t = 0; t < NW; ++t) {
                rw[t] = (32 * t + (int)lane < n) ? __ldg(a.rows + (size_t)id[t] * WM + w) : 0u;
                uni |= rw[t];
            }
            uni = __reduce_or_sync(FULL, uni);
            const uint32_t rm = uni & ~__shfl_sync(FULL, myRootB, w);
            if (lane == 0) { S.Rm[w] = rm; S.rlo[w] = (uint32_t)R; }
            uint32_t bits = rm;
            while (bits) {
                const int b = __ffs(bits) - 1;
                bits &= bits - 1u;
#pragma unroll
                for (int t = 0; t < NW; ++t) {
                    const uint32_t bal = __ballot_sync(FULL, (rw[t] >> b) & 1u);
                    if (lane == 0) S.cR[t * mp + R] = bal;
                }
                if (lane == 0) S.rmap[R] = (uint16_t)(32 * w + b);
                ++R;
            }
        }
        if (lane == 0) S.rlo[WM] = (uint32_t)R;
        {
            // sufB[w] = number of root-intent attributes in words above w
            const unsigned pc = lane < (unsigned)WM ? __popc(myRootB) : 0u;
            unsigned incl = pc;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const unsigned t = __shfl_up_sync(FULL, incl, off);
                if (lane >= (unsigned)off) incl += t;
            }
            const unsigned tot = __shfl_sync(FULL, incl, 31);
            S.sufB[lane] = tot - incl;
        }
        __syncwarp();

        // ---- candidates of the root: attributes >= y0 outside its intent (counted by slice 0)
        {
            unsigned c = lane < (unsigned)WM ? __popc(myRootB & ge_mask((int)lane, y0)) : 0u;
            c = __reduce_add_sync(FULL, c);
            if (slice == 0) S.closures += (unsigned long long)(d.m - y0 - (int)c);
        }
        int jn;   // compact cursor: relevant attributes below y0 are not candidates
        {
            const unsigned c = lane < (unsigned)WM ? __popc(S.Rm[lane] & lt_mask((int)lane, y0)) : 0u;
            jn = (int)__reduce_add_sync(FULL, c);
        }

        // ---- depth-first search of the subtree
        const int sl = a.slices;
        if (R <= 32) dfs_regs<NW, 1, COUNT>(S, R, n, jn, sl, slice);
        else if (R <= 64) dfs_regs<NW, 2, COUNT>(S, R, n, jn, sl, slice);
        else if (R <= 128) dfs_regs<NW, 4, COUNT>(S, R, n, jn, sl, slice);
        else if (RW > 4 && R <= 32 * RW) dfs_regs<NW, RW, COUNT>(S, R, n, jn, sl, slice);
        else dfs_smem<NW, COUNT>(S, R, n, jn, sl, slice);
        __syncwarp();
    }
    if (S.nb) S.flush();
    if (lane == 0 && S.closures) atomicAdd(&a.ctr->closures, S.closures);
    if (COUNT && lane == 0 && S.ops) atomicAdd(&a.ctr->word_ops, S.ops);
}

}  // namespace

// ------------------------------------------------------------------ launch wrappers

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
                         Counters *ctr, const Dims &d, void *stream)
{
    append_bottom_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(flag, full_mask, out, capacity, ctr, d.wm);
    return (int)cudaGetLastError();
}

int launch_top(const uint32_t *rows, uint32_t *top, uint32_t *flag, const Dims &d, void *stream)
{
    const int tpb = 256;
    const long long blocks = (d.n + tpb - 1) / tpb;
    top_kernel<<<(unsigned)blocks, tpb, 0, (cudaStream_t)stream>>>(rows, top, flag, d);
    return (int)cudaGetLastError();
}

size_t expand_smem_per_warp(const Dims &d) { return ExpandLayout(d, 1, 0).bytes; }

// A launch shape computed once per device and shared-memory size.
struct ShapeCache {
    int dev = -1;
    size_t smem = 0;
    int wpb = 0;
    int per_sm = 1;
};

static int warps_for(size_t per_warp)
{
    const size_t budget = 200 * 1024;
    int w = WARPS_PER_BLOCK;
    while (w > 1 && (size_t)w * per_warp > budget) --w;
    return w;
}

template <bool COUNT>
static int launch_expand_t(const ExpandArgs &a, int sm_count, void *stream)
{
    int wpb = WARPS_PER_BLOCK;
    while (wpb > 1 && ExpandLayout(a.d, wpb, 0).bytes > 200 * 1024) --wpb;
    // the largest restricted extent whose columns fit in the shared memory of three blocks per SM
    // (or next to the gather path's own, when that is larger)
    const size_t budget = std::max<size_t>(ExpandLayout(a.d, wpb, 0).bytes, 72 * 1024);
    int tr = RESTRICT_CAP;
    while (tr > 0 && ExpandLayout(a.d, wpb, tr).bytes > budget) tr -= 32;
    const size_t smem = ExpandLayout(a.d, wpb, tr).bytes;
    // the shared-memory attribute and the occupancy query, once per device and size (per thread)
    static thread_local ShapeCache cache;
    int dev = 0;
    cudaGetDevice(&dev);
    if (cache.dev != dev || cache.smem != smem || cache.wpb != wpb) {
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(expand_bitmap_kernel<COUNT>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return (int)e;
        }
        int ps = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ps, expand_bitmap_kernel<COUNT>, wpb * 32, smem);
        cache = ShapeCache{dev, smem, wpb, ps < 1 ? 1 : ps};
    }
    const int per_sm = cache.per_sm;
    // split each parent's attribute range into parts when there are too few parents to fill the GPU
    // (at least one candidate per warp in every part)
    ExpandArgs b = a;
    b.restrict_max = tr;
    const unsigned long long resident = (unsigned long long)sm_count * per_sm;
    const unsigned long long pc = std::max<unsigned long long>(1, a.p_count);
    const int max_parts = std::max(1, a.d.m / wpb);
    b.parts = (int)std::min<unsigned long long>(max_parts, std::max<unsigned long long>(1, (2 * resident + pc - 1) / pc));
    const unsigned long long items = a.p_count * (unsigned long long)b.parts;
    unsigned long long blocks = std::min<unsigned long long>(items, resident * 2);
    if (blocks < 1) blocks = 1;
    expand_bitmap_kernel<COUNT><<<(unsigned)blocks, wpb * 32, smem, (cudaStream_t)stream>>>(b);
    return (int)cudaGetLastError();
}

int launch_expand(const ExpandArgs &a, int sm_count, void *stream)
{
    return a.count_work ? launch_expand_t<true>(a, sm_count, stream) : launch_expand_t<false>(a, sm_count, stream);
}

// Block shape of the subtree kernel (persistent: at most one block per resident slot).
template <int NW, bool COUNT, int RW>
static int subtree_shape(const Dims &d, int *wpb_out, size_t *smem_out, int *per_sm_out)
{
    const size_t pw = SubtreeLayout(d, NW).words * 4;
    const int wpb = warps_for(pw);
    const size_t smem = pw * wpb;
    static thread_local ShapeCache cache;
    int dev = 0;
    cudaGetDevice(&dev);
    if (cache.dev != dev || cache.smem != smem || cache.wpb != wpb) {
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(subtree_kernel<NW, COUNT, RW>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return (int)e;
        }
        int ps = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ps, subtree_kernel<NW, COUNT, RW>, wpb * 32, smem);
        if (e != cudaSuccess) return (int)e;
        cache = ShapeCache{dev, smem, wpb, ps < 1 ? 1 : ps};
    }
    *wpb_out = wpb;
    *smem_out = smem;
    *per_sm_out = cache.per_sm;
    return (int)cudaSuccess;
}

template <int NW, bool COUNT, int RW>
static int launch_subtree_nw(const SubtreeArgs &a, int sm_count, void *stream)
{
    int wpb = 0, per_sm = 0;
    size_t smem = 0;
    int e = subtree_shape<NW, COUNT, RW>(a.d, &wpb, &smem, &per_sm);
    if (e != (int)cudaSuccess) return e;
    // split roots into slices when there are too few roots to keep every resident warp busy
    SubtreeArgs b = a;
    const unsigned long long resident = (unsigned long long)sm_count * per_sm * wpb;
    const unsigned long long want = 4 * resident;
    const unsigned long long qn = std::max<unsigned long long>(1, a.q_count);
    b.slices = (int)std::min<unsigned long long>(MAX_SLICES, std::max<unsigned long long>(1, (want + qn - 1) / qn));
    unsigned long long blocks = (a.q_count * b.slices + wpb - 1) / wpb;
    const unsigned long long cap = (unsigned long long)sm_count * per_sm;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    subtree_kernel<NW, COUNT, RW><<<(unsigned)blocks, wpb * 32, smem, (cudaStream_t)stream>>>(b);
    return (int)cudaGetLastError();
}

int launch_subtree(const SubtreeArgs &a, int nw, int sm_count, void *stream)
{
    const bool wide = reg_words_for(a.d.m) > 4;
    if (a.count_work) {
        if (wide) return nw == 1 ? launch_subtree_nw<1, true, 8>(a, sm_count, stream)
                                 : launch_subtree_nw<2, true, 8>(a, sm_count, stream);
        return nw == 1 ? launch_subtree_nw<1, true, 4>(a, sm_count, stream) : launch_subtree_nw<2, true, 4>(a, sm_count, stream);
    }
    if (wide) return nw == 1 ? launch_subtree_nw<1, false, 8>(a, sm_count, stream)
                             : launch_subtree_nw<2, false, 8>(a, sm_count, stream);
    return nw == 1 ? launch_subtree_nw<1, false, 4>(a, sm_count, stream) : launch_subtree_nw<2, false, 4>(a, sm_count, stream);
}

}  // namespace fca
