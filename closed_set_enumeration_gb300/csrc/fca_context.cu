// Context build kernels of libfca (sm_103a).
//
//  table_init_kernel     top intent and bottom extent set to every attribute / every object.
//  table_kernel          ctxRows (padding bits cleared, copied from the caller's rows) -> ctxCols
//                        by 32x32 register transposes of bit tiles (the Parallel FCBO article,
//                        section 3.1, builds the same column bitmaps with one atomicOr per set bit),
//                        and by AND-reductions the top intent G' (AND of all rows) and the bottom
//                        extent M' (AND of all columns: the objects holding every attribute; when it
//                        is not empty the search reaches the bottom concept).
//  append_bottom_kernel  the bottom concept (intent M) when its extent is empty.
#include <cuda_runtime.h>

#include "fca_device.cuh"

namespace fca {
namespace {


// Start of a table build: the top intent (AND of all rows) starts as every attribute and the
// bottom extent (objects holding every attribute) as every object; table_kernel narrows both.
__global__ void table_init_kernel(uint32_t *top, const uint32_t *full_mask, uint32_t *botext, uint32_t *sup, Dims d)
{
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t < d.wm) top[t] = full_mask[t];
    if (t < d.wn) botext[t] = FULL;
    if (sup && t < d.m) sup[t] = 0u;
}

// The context's tables from the caller's rows, one warp per tile of 32 objects x 32 attributes:
// padding bits past M cleared (they are ignored on input) in the context's row copy (which the
// rows are copied into when `src` is another buffer), the columns as the tile's transpose (one
// 32 x 32 register transpose), and the tile's share of the top intent and of the bottom extent by
// AND-reductions and one atomicAnd each.
__global__ void table_kernel(const uint32_t *__restrict__ src, uint32_t *rows, uint32_t *__restrict__ cols,
                             uint32_t *top, uint32_t *botext, uint32_t *sup, Dims d)
{
    const int wpb = blockDim.x >> 5;
    const long long tile = (long long)blockIdx.x * wpb + (threadIdx.x >> 5);
    if (tile >= d.wn * (long long)d.wm) return;  // uniform per warp
    const unsigned lane = threadIdx.x & 31;
    const long long ot = tile / d.wm;             // 32 objects
    const int aw = (int)(tile % d.wm);            // 32 attributes
    const long long o = ot * 32 + lane;
    const bool obj = o < d.n;
    uint32_t v = obj ? src[o * d.wm + aw] : 0u;
    const int valid = d.m - aw * 32;
    if (valid < 32) v &= (1u << valid) - 1u;      // ignore padding bits
    if (obj && (src != rows || valid < 32)) rows[o * d.wm + aw] = v;
    const uint32_t col = warp_transpose32(v);     // lane b: attribute 32 aw + b over the tile's objects
    const int a = aw * 32 + (int)lane;
    if (a < d.m) {
        cols[(size_t)a * d.wnp + ot] = col;
        if (sup) atomicAdd(&sup[a], (uint32_t)__popc(col));   // the attribute's support
    }
    const uint32_t t_and = __reduce_and_sync(FULL, obj ? v : FULL);
    const uint32_t b_and = __reduce_and_sync(FULL, a < d.m ? col : FULL);
    if (lane == 0) {
        atomicAnd(&top[aw], t_and);
        atomicAnd(&botext[ot], b_and);
    }
}

// Processing order of the attributes: ascending support, ties by index (a stable sort). perm[a] is
// the position of attribute a, inv[r] the attribute at position r. One block; the supports are
// staged in shared memory and each thread ranks its attributes by counting (M <= 1024).
__global__ void order_kernel(const uint32_t *sup, int32_t *perm, int32_t *inv, int m)
{
    __shared__ uint32_t s[MAX_ATTRS];
    for (int a = (int)threadIdx.x; a < m; a += (int)blockDim.x) s[a] = sup[a];
    __syncthreads();
    for (int a = (int)threadIdx.x; a < m; a += (int)blockDim.x) {
        const uint32_t v = s[a];
        int r = 0;
        for (int b = 0; b < m; ++b) r += (s[b] < v) || (s[b] == v && b < a);
        perm[a] = r;
        inv[r] = a;
    }
}

// The tables in processing order, one warp per tile of 32 objects x 32 positions: lane b of tile
// (ot, aw) gathers word ot of the column of attribute inv[32 aw + b] into position 32 aw + b of
// cols2; one register transpose turns the tile into words aw of the rows of its 32 objects; the
// tiles of object word 0 also write word aw of the permuted top intent.
__global__ void permute_kernel(const uint32_t *__restrict__ cols, uint32_t *__restrict__ cols2, uint32_t *rows,
                               const int32_t *inv, const uint32_t *top, uint32_t *top2, Dims d)
{
    const int wpb = blockDim.x >> 5;
    const long long tile = (long long)blockIdx.x * wpb + (threadIdx.x >> 5);
    if (tile >= d.wn * (long long)d.wm) return;  // uniform per warp
    const unsigned lane = threadIdx.x & 31;
    const long long ot = tile / d.wm;
    const int aw = (int)(tile % d.wm);
    const int r = aw * 32 + (int)lane;
    const int a = r < d.m ? inv[r] : 0;
    uint32_t col = 0u;
    if (r < d.m) {
        col = cols[(size_t)a * d.wnp + ot];
        cols2[(size_t)r * d.wnp + ot] = col;
    }
    const uint32_t v = warp_transpose32(col);   // lane l: positions 32 aw .. of object 32 ot + l
    const long long o = ot * 32 + lane;
    if (o < d.n) rows[o * d.wm + aw] = v;
    if (ot == 0) {
        const bool bit = r < d.m && ((top[a >> 5] >> (a & 31)) & 1u);
        const uint32_t w = __ballot_sync(FULL, bit);
        if (lane == 0) top2[aw] = w;
    }
}

// Output rows [start, min(out_count, capacity)) mapped back from processing order to attribute order:
// bit a of a row becomes bit a of the result when it was at position perm[a]. Each warp takes runs
// of UNPERM_ROWS consecutive rows (contiguous words, loaded and stored coalesced through shared
// memory, so one memory latency serves the run) and forms each result word with one ballot;
// `guard` as for the guarded launches (SubtreeArgs::guard).
constexpr int UNPERM_ROWS = 8;
__global__ void unpermute_kernel(uint32_t *out, unsigned long long start, unsigned long long capacity,
                                 const Counters *ctr, const int32_t *perm, int wm, int m, int guard)
{
    if (guard && (ctr->error != 0u || ctr->next_count != 0ull)) return;
    __shared__ int32_t p[MAX_ATTRS];
    __shared__ uint32_t stage[8][UNPERM_ROWS * 32];
    __shared__ uint32_t res[8][UNPERM_ROWS * 32];
    for (int a = (int)threadIdx.x; a < m; a += (int)blockDim.x) p[a] = perm[a];
    __syncthreads();
    const unsigned lane = threadIdx.x & 31;
    const int wib = (int)(threadIdx.x >> 5);
    const unsigned long long total = ctr->out_count < capacity ? ctr->out_count : capacity;
    const unsigned long long step = (unsigned long long)gridDim.x * (blockDim.x >> 5) * UNPERM_ROWS;
    for (unsigned long long r0 = start + ((unsigned long long)blockIdx.x * (blockDim.x >> 5) + wib) * UNPERM_ROWS;
         r0 < total; r0 += step) {
        const int nr = (int)(total - r0 < (unsigned long long)UNPERM_ROWS ? total - r0 : UNPERM_ROWS);
        const int words = nr * wm;
        uint32_t *src = out + r0 * (unsigned long long)wm;
        for (int i = (int)lane; i < words; i += 32) stage[wib][i] = src[i];
        __syncwarp();
        if (wm <= 16) {
            // each lane's source word and bit for the up to 16 result words, held in registers
            int qw[16];
            uint32_t qb[16];
#pragma unroll
            for (int w = 0; w < 16; ++w) {
                const int a = 32 * w + (int)lane;
                const int q = w < wm && a < m ? p[a] : -1;
                qw[w] = q < 0 ? 0 : q >> 5;
                qb[w] = q < 0 ? 32u : (uint32_t)(q & 31);
            }
            for (int r = 0; r < nr; ++r) {
                const uint32_t *row = stage[wib] + r * wm;
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    if (w >= wm) break;
                    const bool bit = qb[w] < 32u && ((row[qw[w]] >> qb[w]) & 1u);
                    const uint32_t word = __ballot_sync(FULL, bit);
                    if (lane == 0) res[wib][r * wm + w] = word;
                }
            }
        } else {
            for (int r = 0; r < nr; ++r) {
                const uint32_t *row = stage[wib] + r * wm;
                for (int w = 0; w < wm; ++w) {
                    const int a = 32 * w + (int)lane;
                    bool bit = false;
                    if (a < m) {
                        const int q = p[a];
                        bit = (row[q >> 5] >> (q & 31)) & 1u;
                    }
                    const uint32_t word = __ballot_sync(FULL, bit);
                    if (lane == 0) res[wib][r * wm + w] = word;
                }
            }
        }
        __syncwarp();
        for (int i = (int)lane; i < words; i += 32) src[i] = res[wib][i];
        __syncwarp();
    }
}

// The same map for rows of at most WMAX words (M <= 32 WMAX), a tile of 32 rows per warp: lane l
// loads row l of the tile (all its words in flight), and each 32 x 32 bit block (32 rows x one word)
// is transposed in registers, so that lane b holds position 32q + b of every row of the tile as one
// word. Permuting the attributes is then a gather of those columns (lane l of result word w takes
// column perm[32w + l], by one shuffle per source word), and transposing back gives each lane its
// row in attribute order. About 15 instructions per row against some 64 for a ballot per result word.
template <int WMAX>
__global__ void __launch_bounds__(256) unpermute_tiles_kernel(uint32_t *out, unsigned long long start,
                                                              unsigned long long capacity, const Counters *ctr,
                                                              const int32_t *perm, int wm, int m, int guard)
{
    if (guard && (ctr->error != 0u || ctr->next_count != 0ull)) return;
    const unsigned lane = threadIdx.x & 31;
    // this lane's source word and bit for each result word (bit 32: past M, left clear)
    int pq[WMAX];
    uint32_t pb[WMAX];
#pragma unroll
    for (int w = 0; w < WMAX; ++w) {
        const int a = 32 * w + (int)lane;
        const int q = w < wm && a < m ? perm[a] : -1;
        pq[w] = q < 0 ? -1 : q >> 5;
        pb[w] = q < 0 ? 0u : (uint32_t)(q & 31);
    }
    const unsigned long long total = ctr->out_count < capacity ? ctr->out_count : capacity;
    const unsigned long long nwarps = (unsigned long long)gridDim.x * (blockDim.x >> 5);
    // rows of a multiple of 4 words in a 16-byte aligned buffer move as uint4
    const bool vec = (wm & 3) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0;
    for (unsigned long long r0 = start + 32ull * ((unsigned long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5));
         r0 < total; r0 += 32ull * nwarps) {
        const unsigned long long r = r0 + lane;
        const bool mine = r < total;
        uint32_t *row = out + r * (unsigned long long)wm;
        uint32_t t[WMAX];
        if (vec) {
            // whole rows of 4-word groups, 16-byte aligned: one vector load per group
#pragma unroll
            for (int q = 0; q < WMAX; q += 4) {
                uint4 x = make_uint4(0u, 0u, 0u, 0u);
                if (mine && q < wm) x = *reinterpret_cast<const uint4 *>(row + q);
                t[q] = x.x; t[q + 1] = x.y; t[q + 2] = x.z; t[q + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int q = 0; q < WMAX; ++q) t[q] = (mine && q < wm) ? row[q] : 0u;
        }
#pragma unroll
        for (int q = 0; q < WMAX; ++q)
            if (q < wm) t[q] = warp_transpose32(t[q]);
        uint32_t o[WMAX];
#pragma unroll
        for (int w = 0; w < WMAX; ++w) {
            uint32_t v = 0u;
            if (w < wm) {
#pragma unroll
                for (int q = 0; q < WMAX; ++q) {
                    if (q >= wm) break;
                    const uint32_t x = __shfl_sync(FULL, t[q], pb[w]);
                    if (q == pq[w]) v = x;
                }
            }
            o[w] = v;
        }
#pragma unroll
        for (int w = 0; w < WMAX; ++w)
            if (w < wm) o[w] = warp_transpose32(o[w]);
        if (vec) {
#pragma unroll
            for (int w = 0; w < WMAX; w += 4)
                if (mine && w < wm) *reinterpret_cast<uint4 *>(row + w) = make_uint4(o[w], o[w + 1], o[w + 2], o[w + 3]);
        } else {
#pragma unroll
            for (int w = 0; w < WMAX; ++w)
                if (mine && w < wm) row[w] = o[w];
        }
    }
}

// The bottom concept when its extent is empty (no row holds every attribute): one more row.
__global__ void append_bottom_kernel(const uint32_t *botext, long long wn, const uint32_t *full_mask, uint32_t *out,
                                     unsigned long long capacity, Counters *ctr, int wm, int guard)
{
    if (guard && (ctr->error != 0u || ctr->next_count != 0ull)) return;   // the search did not end here
    const unsigned lane = threadIdx.x & 31;
    uint32_t any = 0;
    for (long long q = lane; q < wn; q += 32) any |= botext[q];
    if (__any_sync(FULL, any != 0u)) return;   // some object holds every attribute: the search output it
    unsigned long long slot = 0;
    if (lane == 0) slot = atomicAdd(&ctr->out_count, 1ull);
    slot = __shfl_sync(FULL, slot, 0);
    if (slot < capacity)
        for (int w = (int)lane; w < wm; w += 32) out[slot * wm + w] = full_mask[w];
}

// Counter set-up before a level launch: the next level's current fills, zero work cursors and
// error word; then a copy of the counters, restored if the launch has to be rolled back.
__global__ void prepare_expand_kernel(Counters *ctr, Counters *snap, unsigned long long next_fill,
                                      unsigned long long next_mid_fill)
{
    if (threadIdx.x == 0) {
        ctr->next_count = next_fill;
        ctr->next_mid = next_mid_fill;
        ctr->work_head = 0ull;
        ctr->mid_head = 0ull;
        ctr->error = 0u;
    }
    __syncthreads();
    const uint32_t *src = reinterpret_cast<const uint32_t *>(ctr);
    uint32_t *dst = reinterpret_cast<uint32_t *>(snap);
    for (int i = (int)threadIdx.x; i < (int)(sizeof(Counters) / 4); i += (int)blockDim.x) dst[i] = src[i];
}

// Before launch i of a chain of level launches (see ChainSlots).
__global__ void prepare_chain_kernel(Counters *ctr, ChainSlots *cs, int i, unsigned long long n0,
                                     unsigned long long n0_mid)
{
    if (threadIdx.x == 0) {
        unsigned long long pc = i == 0 ? n0 : ctr->next_count;
        unsigned long long pm = i == 0 ? n0_mid : ctr->next_mid;
        if (i == 0) ctr->error = 0u;
        else if (ctr->error) pc = pm = 0ull;   // an earlier launch of the chain overflowed: no work
        cs->counts[i] = pc;
        cs->mcounts[i] = pm;
        cs->pcount = pc;
        cs->pcount_mid = pm;
        ctr->next_count = 0ull;
        ctr->next_mid = 0ull;
        ctr->work_head = 0ull;
        ctr->mid_head = 0ull;
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
        // the root inherits no failures (the entry's words past its extent, when kept)
        for (long long q = d.wnp + t; q < L0.stride; q += blockDim.x) L0.ext[q] = 0xffffffffu;
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

int launch_prepare_expand(Counters *ctr, Counters *snap, uint64_t next_fill, uint64_t next_mid_fill, void *stream)
{
    prepare_expand_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(ctr, snap, next_fill, next_mid_fill);
    return (int)cudaGetLastError();
}

int launch_prepare_chain(Counters *ctr, ChainSlots *cs, int i, uint64_t n0, uint64_t n0_mid, void *stream)
{
    prepare_chain_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(ctr, cs, i, n0, n0_mid);
    return (int)cudaGetLastError();
}

int launch_start(Counters *ctr, const uint32_t *top, const uint32_t *root_ext, const Dims &d, uint32_t *out,
                 uint64_t capacity, const Level &L0, const Queue &Q, int qi, void *stream)
{
    start_kernel<<<1, 256, 0, (cudaStream_t)stream>>>(ctr, top, root_ext, d, out, capacity, L0, Q, qi);
    return (int)cudaGetLastError();
}

int launch_table(const uint32_t *src, uint32_t *rows, uint32_t *cols, uint32_t *top, const uint32_t *full_mask,
                 uint32_t *botext, uint32_t *sup, const Dims &d, void *stream)
{
    long long init = d.wn > d.wm ? d.wn : d.wm;
    if (init < d.m) init = d.m;
    table_init_kernel<<<(unsigned)((init + 255) / 256), 256, 0, (cudaStream_t)stream>>>(top, full_mask, botext, sup, d);
    const long long tiles = d.wn * (long long)d.wm;
    const int wpb = 8;
    table_kernel<<<(unsigned)((tiles + wpb - 1) / wpb), wpb * 32, 0, (cudaStream_t)stream>>>(src, rows, cols, top,
                                                                                           botext, sup, d);
    return (int)cudaGetLastError();
}

int launch_order(const uint32_t *sup, int32_t *perm, int32_t *inv, const uint32_t *cols, uint32_t *cols2,
                 uint32_t *rows, const uint32_t *top, uint32_t *top2, const Dims &d, void *stream)
{
    order_kernel<<<1, 1024, 0, (cudaStream_t)stream>>>(sup, perm, inv, d.m);
    const long long tiles = d.wn * (long long)d.wm;
    const int wpb = 8;
    permute_kernel<<<(unsigned)((tiles + wpb - 1) / wpb), wpb * 32, 0, (cudaStream_t)stream>>>(cols, cols2, rows, inv,
                                                                                             top, top2, d);
    return (int)cudaGetLastError();
}

int launch_unpermute(uint32_t *out, uint64_t capacity, const Counters *ctr, const int32_t *perm, const Dims &d,
                     int sm_count, void *stream, int guard, uint64_t start)
{
    cudaStream_t st = (cudaStream_t)stream;
    if (d.wm <= 8)
        unpermute_tiles_kernel<8><<<(unsigned)(8 * sm_count), 256, 0, st>>>(out, start, capacity, ctr, perm, d.wm, d.m, guard);
    else if (d.wm <= 16)
        unpermute_tiles_kernel<16><<<(unsigned)(8 * sm_count), 256, 0, st>>>(out, start, capacity, ctr, perm, d.wm, d.m, guard);
    else
        unpermute_kernel<<<(unsigned)(4 * sm_count), 256, 0, st>>>(out, start, capacity, ctr, perm, d.wm, d.m, guard);
    return (int)cudaGetLastError();
}

int launch_append_bottom(const uint32_t *botext, const uint32_t *full_mask, uint32_t *out, uint64_t capacity,
                         Counters *ctr, const Dims &d, void *stream, int guard)
{
    append_bottom_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(botext, d.wn, full_mask, out, capacity, ctr, d.wm, guard);
    return (int)cudaGetLastError();
}

}  // namespace fca
