// Bitmap tier of libfca (sm_103a): expand_bitmap_kernel expands the concepts of one level whose
// extents hold more than 64 objects. Per (parent, j) candidate it forms the extent intersection,
// the closure, the canonical test and the child (FCbO-to-CUDA article, sections 2.1-2.3, 4.2-4.4;
// Parallel FCBO article, sections 2.1, 3.2). Bitwise set algebra only: no tensor cores.
#include <cuda_runtime.h>

#include <algorithm>

#include "fca_device.cuh"

namespace fca {
namespace {


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
// Two block shapes. The warps of a block share one parent's staged extent, restricted columns and
// rows. With many attributes (many candidates per parent) blocks of 16 warps, two per SM, hide more
// latency per byte of shared memory, and so do levels with too few parents to fill the GPU; on
// large levels with fewer attributes the per-parent set-up dominates and blocks of 8 warps, three per
// SM, keep more parents in flight. Measured with 16 warps throughout: zipf (M = 400) 2.95 -> 2.35 ms
// per enumeration, sparse (small levels) 0.095 -> 0.073 ms; skewed (M = 128) 94 -> 107 ms and
// biclusters (M = 256) 3.3 -> 4.2 s.
constexpr int WIDE_EXPAND_MIN_ATTRS = 320;
template <int WARPS> struct ExpandShape;
template <> struct ExpandShape<8> {
    static constexpr int blocks_per_sm = 3;
    static constexpr size_t smem_budget = 72 * 1024;
};
template <> struct ExpandShape<16> {
    static constexpr int blocks_per_sm = 2;
    static constexpr size_t smem_budget = 108 * 1024;
};
constexpr int ROWS_KEPT = 256;             // restricted extents up to this size keep their rows in shared memory
constexpr int CHILD_SLOTS = 64;            // level children of one work item that inherit its failures
constexpr int WIT_WORDS_MAX = 64;          // failure witnesses of one parent (M <= 256: a byte each)

// Shared memory of expand_bitmap_kernel. Both paths first stage the parent's non-zero extent
// chunks (uint4 index and value). The gather path then keeps, per warp, up to SMALL_MAX object
// ids (C itself is recomputed from the staged chunks and column j when needed); the restricted
// path keeps the parent's object list, its columns restricted to those objects (M x TR/32 words)
// and per-warp positions in that list; parents of at most min(TR, ROWS_KEPT) objects also keep
// their rows (positions x W_M words).
struct ExpandLayout {
    size_t o_aidx, o_aval, o_wbase, per_warp, o_oid, o_colr, o_rowr, o_rids, o_blk, bytes;
    int rk;   // rows kept: largest restricted extent whose rows are in shared memory
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
        rk = tr < ROWS_KEPT ? tr : ROWS_KEPT;
        o_rowr = o_colr + (size_t)d.m * (size_t)(tr / 32) * 4;     // rk x wm uint32
        o_rids = o_rowr + (size_t)rk * (size_t)d.wm * 4;
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

// The rest of a candidate once |C| and the first `need` objects of C are known: the closure
// (the AND of their rows: exact when need == |C|, else an upper bound whose extra attributes are
// decided by `subset(k)` in ascending order, so a violation below j ends the candidate early),
// the canonical test, the intent and the child. `row_word(i, w)` is word w of the row of the i-th
// object of C and `obj_id(i)` its object id; `write_ext(dst)` writes C as a dense bitmap for a
// child of the next level, `write_list(dst)` as its ascending object ids (a child of at most
// list_max objects); `all_ids()` completes the list of a small child (need < |C|).
template <bool COUNT, bool INHERIT, class RowWord, class ObjId, class Subset, class WriteExt, class WriteList,
          class AllIds>
__device__ __forceinline__ int finish_candidate(const ExpandArgs &a, const Dims &d, const uint32_t *B, int j,
                                                unsigned cnt, unsigned need, RowWord &&row_word, ObjId &&obj_id,
                                                Subset &&subset, WriteExt &&write_ext, WriteList &&write_list,
                                                AllIds &&all_ids, unsigned long long &my_bytes, uint32_t *cslots,
                                                int *ccount)
{
    const unsigned lane = threadIdx.x & 31;
    // AND of the rows: lanes take (object, word) pairs with the words padded to a power of two W2
    // (so a lane always holds the same word), issue all their loads at once, then AND across the
    // lanes holding the same word; lane w ends with word w.
    const int w2 = d.wm <= 1 ? 1 : 1 << (32 - __clz(d.wm - 1));
    const int my_w = (int)lane & (w2 - 1);
    uint32_t U = FULL;
    if (my_w < d.wm)
        for (unsigned pidx = lane; pidx < need * (unsigned)w2; pidx += 32)
            U &= row_word(pidx / (unsigned)w2, my_w);
    for (int sft = w2; sft < 32; sft <<= 1) U &= __shfl_xor_sync(FULL, U, sft);
    if ((int)lane >= d.wm) U = 0u;
    if (COUNT && lane == 0) my_bytes += (unsigned long long)need * d.wm * 4;   // rows read
    const uint32_t Bw = lane < (unsigned)d.wm ? B[lane] : 0u;
    const int ju = j >> 5;
    const uint32_t jbit = 1u << (j & 31);
    const uint32_t pm = lt_mask((int)lane, j);   // attributes below j
    uint32_t Dw;
    if (need == cnt) {
        Dw = U;
        // not canonical: the lowest attribute below j in the closure is the failure's witness
        const uint32_t viol = U & ~Bw & pm;
        const unsigned vb = __ballot_sync(FULL, viol != 0u);
        if (vb) {
            const int vw = __ffs(vb) - 1;
            return 32 * vw + __ffs(__shfl_sync(FULL, viol, vw)) - 1;
        }
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
                if (k < j) return k;                    // not canonical, k its witness
                if ((int)lane == u) Dw |= 1u << b;
            }
        }
    }

    if (COUNT && lane == 0) {   // the intent row and the child entry written
        my_bytes += (unsigned long long)d.wm * 4;
        my_bytes += cnt <= (unsigned)SMALL_MAX ? 4ull * queue_entry_words(cnt, d.wm)
                    : (int)cnt <= a.list_max ? 4ull * (cnt + d.wm + 2)
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
            return -1;
        }
        if (need < cnt) all_ids();
        __syncwarp();
        for (int i = (int)lane; i < per; i += 32) Q.ids[s * per + i] = i < (int)cnt ? obj_id((unsigned)i) : 0u;
        if (lane < (unsigned)d.wm) Q.itt[s * d.wm + lane] = Dw;
        if (lane == 0) { Q.y[s] = j + 1; Q.n[s] = (int)cnt; }
    } else {
        // the next level: its mid pool (an id list of at most mid_max objects) or its big pool (an
        // id list up to list_max objects, a bitmap above)
        const bool mid = (int)cnt <= a.mid_max;
        const Level &X = mid ? a.next_mid : a.next;
        unsigned long long s = 0;
        if (lane == 0) s = atomicAdd(mid ? &a.ctr->next_mid : &a.ctr->next_count, 1ull);
        s = __shfl_sync(FULL, s, 0);
        if (s >= X.cap) {
            if (lane == 0) atomicOr(&a.ctr->error, mid ? ERR_NEXT_MID : ERR_NEXT);
            return -1;
        }
        if ((int)cnt <= a.list_max) write_list(X.ext + s * (size_t)X.stride);
        else write_ext(X.ext + s * (size_t)X.stride);
        if (lane < (unsigned)d.wm) X.itt[s * d.wm + lane] = Dw;
        if (lane == 0) { X.y[s] = j + 1; X.n[s] = (int)cnt; }
        if (INHERIT) {
            // the child's inherited failures are written when the work item is done (past
            // CHILD_SLOTS children of one item: none)
            int ci = 0;
            if (lane == 0) ci = atomicAdd(ccount, 1);
            ci = __shfl_sync(FULL, ci, 0);
            if (ci < CHILD_SLOTS) {
                if (lane == 0) cslots[ci] = (uint32_t)s | (mid ? 0x80000000u : 0u);
            } else {
                uint32_t *w = X.ext + s * (size_t)X.stride + (mid ? a.wit_off : a.wit_off_big);
                for (int i = (int)lane; i < a.wit_words; i += 32) w[i] = FULL;
            }
        }
    }
    return -1;
}

// Parts per parent: each parent's attribute range is split when there are too few parents to fill
// the GPU (two work items per resident block), with at least one candidate per warp in a part.
__host__ __device__ inline int expand_parts(unsigned long long p_count, unsigned long long resident, int max_parts)
{
    const unsigned long long pc = p_count > 0 ? p_count : 1;
    const unsigned long long want = (2 * resident + pc - 1) / pc;
    return (int)(want < 1 ? 1 : (want > (unsigned long long)max_parts ? (unsigned long long)max_parts : want));
}

// Bitmap tier. A work item is (parent, part of the attribute range). The block stages the parent's
// non-zero extent chunks once (an entry stored as an object-id list is read as such). Extents of at
// most `a.restrict_max` objects are then turned into an object list, and the rows of those objects
// are transposed into columns restricted to them (one 32 x 32 register transpose per row word and 32
// objects); each candidate's C is read from those columns without any global column access. Larger
// extents keep the chunk list: each warp gathers column j on the parent's non-zero chunks. Either
// way the warps of the block take the part's candidates j in turn.
template <bool COUNT, int WARPS, bool INHERIT>
__global__ void __launch_bounds__(32 * WARPS, ExpandShape<WARPS>::blocks_per_sm) expand_bitmap_kernel(ExpandArgs a)
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
    uint32_t *rowr = reinterpret_cast<uint32_t *>(smem + L.o_rowr);
    uint32_t *rids = reinterpret_cast<uint32_t *>(smem + L.o_rids) + (size_t)wib * SMALL_MAX;
    int *blk = reinterpret_cast<int *>(smem + L.o_blk);   // [0..31] scan scratch
    const uint4 *cols4 = reinterpret_cast<const uint4 *>(a.cols);

    unsigned long long my_closures = 0, my_bytes = 0;
    unsigned loads = 0;   // uint4 loads of columns by this lane (counting only)
    // the parent count: given, or (a launch queued behind the one producing this level) read from
    // the device; then the parts per parent, as the launcher would choose them
    const unsigned long long p_count1 = a.p_count_dev ? *a.p_count_dev : a.p_count;
    const unsigned long long p_count = p_count1 + (a.p_count2_dev ? *a.p_count2_dev : a.p_count2);
    const int parts = a.parts > 0 ? a.parts
                                  : expand_parts(p_count, a.resident, max(1, d.m / wpb));
    const int span = (d.m + parts - 1) / parts;
    const unsigned long long items = p_count * (unsigned long long)parts;
    __shared__ unsigned long long next_item;
    // the item's candidates are dealt to its warps one at a time (a fixed stride over the warps left
    // the block waiting at the next item for the warps that drew the expensive candidates)
    __shared__ int jclaim;
    // inherited failures (the Fast Close-by-One rule): the parent's witness byte per attribute
    // (0xff: none), updated by the item's own failures, and the level children that receive it
    __shared__ uint32_t bwit[INHERIT ? WIT_WORDS_MAX : 1];
    __shared__ uint32_t cslots[INHERIT ? CHILD_SLOTS : 1];
    __shared__ int ccount;
    const uint8_t *bwitb = reinterpret_cast<const uint8_t *>(bwit);
    if (INHERIT && threadIdx.x == 0) ccount = 0;
    for (;;) {
        // work items are dealt one at a time from a launch-wide cursor, so the blocks that draw
        // large parents do not hold back the rest
        __syncthreads();
        if (INHERIT) {
            // the previous item's level children get its failures, now that all its candidates are done
            const int nc = min(ccount, CHILD_SLOTS);
            for (int e = (int)threadIdx.x; e < nc * a.wit_words; e += (int)blockDim.x) {
                const int ci = e / a.wit_words, wi = e - ci * a.wit_words;
                const uint32_t v = cslots[ci];
                const bool to_mid = (v >> 31) != 0u;
                const Level &X = to_mid ? a.next_mid : a.next;
                X.ext[(size_t)(v & 0x7fffffffu) * X.stride + (to_mid ? a.wit_off : a.wit_off_big) + wi] = bwit[wi];
            }
            __syncthreads();
            if (threadIdx.x == 0) ccount = 0;
        }
        if (threadIdx.x == 0) {
            next_item = atomicAdd(&a.ctr->work_head, 1ull);
            jclaim = 0;
        }
        __syncthreads();
        const unsigned long long item = next_item;
        if (item >= items) break;
        const unsigned long long idx = item / (unsigned)parts;
        const bool second = idx >= p_count1;             // a parent of the second pool
        const Level &P = second ? a.in2 : a.in;
        const unsigned long long p = second ? a.p_begin2 + (idx - p_count1) : a.p_begin + idx;
        const int part = (int)(item % (unsigned)parts);
        const int y = P.y[p];
        // this part's candidates; a parent small enough for restricted columns is expanded on them
        // when its candidates in the part make that cheaper than gathering (the transposition is
        // paid by every part: parts exist only when a level is too small to fill the GPU, where
        // spreading a parent's candidates over blocks shortens the launch)
        const int np = P.n[p];
        const int gw = (np + 31) >> 5;
        const int j_lo = max(y, part * span);
        const int j_hi = min(d.m, (part + 1) * span);
        if (j_lo >= j_hi) continue;                       // uniform over the block
        const bool is_list = np <= a.list_max;             // the entry holds its object ids
        const bool restricted = is_list || (np <= tr && (long long)(j_hi - j_lo) * min(wq, np) >= 4ll * gw * d.wm);
        // the parent intent, read by every candidate, in shared memory
        __shared__ uint32_t sB[MAX_ATTRS / 32];
        if ((int)threadIdx.x < d.wm) sB[threadIdx.x] = P.itt[p * d.wm + threadIdx.x];
        const uint32_t *B = sB;
        if (INHERIT) {
            const uint32_t *ws = P.ext + p * (size_t)P.stride + (second ? a.wit_off : a.wit_off_big);
            for (int i = (int)threadIdx.x; i < a.wit_words; i += (int)blockDim.x) bwit[i] = ws[i];
        }

        // ---- stage the non-zero chunks of A in order (block-wide compaction), and |A|
        const uint4 *A4 = reinterpret_cast<const uint4 *>(P.ext + p * (size_t)P.stride);   // a bitmap entry: big pool
        __syncthreads();
        int nnz = 0, na = 0;
        for (int base = 0; base < (is_list ? 0 : wq); base += blockDim.x) {
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
        if (COUNT && threadIdx.x == 0) my_bytes += is_list ? 4ull * np : (unsigned long long)d.wnp * 4;   // the parent extent

        if (restricted) {
            // ---- restricted path: object list, then the columns restricted to these objects
            if (is_list) {
                const uint32_t *src = P.ext + p * (size_t)P.stride;
                for (int i = (int)threadIdx.x; i < np; i += blockDim.x) oid[i] = src[i];
                na = np;
            }
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
            const bool keep_rows = na <= L.rk;
            for (int unit = wib; unit < G * d.wm; unit += wpb) {
                const int g = unit / d.wm, w = unit % d.wm;
                const int pidx = 32 * g + (int)lane;
                const uint32_t v = pidx < na ? __ldg(a.rows + (size_t)oid[pidx] * d.wm + w) : 0u;
                if (keep_rows && pidx < na) rowr[(size_t)pidx * d.wm + w] = v;
                // lane b receives the column of attribute 32w + b over these 32 objects
                const uint32_t mine = warp_transpose32(v);
                const int k = 32 * w + (int)lane;
                if (k < d.m) colr[(size_t)k * G + g] = mine;
            }
            __syncthreads();
            if (COUNT && threadIdx.x == 0) my_bytes += (unsigned long long)na * d.wm * 4;   // rows of A

            for (;;) {
                int j = 0;
                if (lane == 0) j = j_lo + atomicAdd(&jclaim, 1);
                j = __shfl_sync(FULL, j, 0);
                if (j >= j_hi) break;
                if ((B[j >> 5] >> (j & 31)) & 1u) continue;   // saturation: A inside column j
                ++my_closures;
                if (INHERIT) {
                    // j failed at an ancestor with a witness k < j in its closure: while k stays
                    // outside B, the closure here (of a subset of that extent) holds k again
                    const unsigned w = bwitb[j];
                    if (w != 0xffu && !((B[w >> 5] >> (w & 31)) & 1u)) continue;
                }
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

                // the positions (in the object list) of the first objects of C in ascending order: the
                // closure is bounded by their rows and completed on the restricted columns
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
                            rids[pos++] = (uint32_t)(32 * g + b);
                        }
                        got += __shfl_sync(FULL, incl, 31);
                    }
                };
                const unsigned need = cnt < (unsigned)ROW_BOUND ? cnt : (unsigned)ROW_BOUND;
                collect(need);
                __syncwarp();
                const int wk = finish_candidate<COUNT, INHERIT>(
                    a, d, B, j, cnt, need,
                    [&](unsigned i, int w) {
                        const uint32_t p = rids[i];
                        return keep_rows ? rowr[(size_t)p * d.wm + w] : __ldg(a.rows + (size_t)oid[p] * d.wm + w);
                    },
                    [&](unsigned i) { return oid[rids[i]]; },
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
                    [&](uint32_t *dst) {
                        // positions 32 g + b of C in ascending order map to ascending object ids
                        unsigned got = 0;
#pragma unroll
                        for (int r = 0; r < RPL; ++r) {
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
                            while (bits) {
                                const int b = __ffs(bits) - 1;
                                bits &= bits - 1u;
                                dst[pos++] = oid[32 * g + b];
                            }
                            got += __shfl_sync(FULL, incl, 31);
                        }
                    },
                    [&]() { collect(cnt); },
                    my_bytes, cslots, &ccount);
                if (INHERIT && lane == 0) reinterpret_cast<uint8_t *>(bwit)[j] = wk >= 0 ? (uint8_t)wk : 0xffu;
                __syncwarp();
            }
            continue;
        }

        // ---- gather path: candidates j of this part, warps in turn
        for (;;) {
                int j = 0;
                if (lane == 0) j = j_lo + atomicAdd(&jclaim, 1);
                j = __shfl_sync(FULL, j, 0);
                if (j >= j_hi) break;
            if ((B[j >> 5] >> (j & 31)) & 1u) continue;   // saturation: A inside column j
            ++my_closures;
            if (INHERIT) {
                const unsigned w = bwitb[j];
                if (w != 0xffu && !((B[w >> 5] >> (w & 31)) & 1u)) continue;
            }

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
            const int wk = finish_candidate<COUNT, INHERIT>(
                a, d, B, j, cnt, need,
                [&](unsigned i, int w) { return __ldg(a.rows + (size_t)gids[i] * d.wm + w); },
                [&](unsigned i) { return gids[i]; },
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
                [&](uint32_t *dst) {
                    // the ids of C in ascending order, chunk by chunk
                    unsigned got = 0;
                    for (int base = 0; base < nnz; base += 32) {
                        const int i = base + (int)lane;
                        uint4 x = make_uint4(0u, 0u, 0u, 0u);
                        uint32_t q = 0u;
                        if (i < nnz) {
                            const uint4 av = aval[i];
                            q = aidx[i];
                            const uint4 cc = __ldg(J4 + q);
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
                            while (bits) {
                                const int b = __ffs(bits) - 1;
                                bits &= bits - 1u;
                                dst[pos++] = (uint32_t)((4 * q + t) * 32 + b);
                            }
                        }
                        got += __shfl_sync(FULL, incl, 31);
                    }
                },
                [&]() {},
                my_bytes, cslots, &ccount);
            if (INHERIT && lane == 0) reinterpret_cast<uint8_t *>(bwit)[j] = wk >= 0 ? (uint8_t)wk : 0xffu;
            __syncwarp();
        }
    }
    if (COUNT) {
        const unsigned tl = __reduce_add_sync(FULL, loads);
        if (lane == 0) atomicAdd(&a.ctr->bytes, my_bytes + 16ull * tl);
    }
    if (lane == 0 && my_closures) atomicAdd(&a.ctr->closures, my_closures);
}

}  // namespace

size_t expand_smem_per_warp(const Dims &d) { return ExpandLayout(d, 1, 0).bytes; }

// Largest extent whose columns a block of the WARPS shape rebuilds restricted to its objects (the
// launcher's choice below).
template <int WARPS>
static int restrict_max_of(const Dims &d)
{
    int wpb = WARPS;
    while (wpb > 1 && ExpandLayout(d, wpb, 0).bytes > 200 * 1024) --wpb;
    const size_t budget = std::max<size_t>(ExpandLayout(d, wpb, 0).bytes, ExpandShape<WARPS>::smem_budget);
    int tr = RESTRICT_CAP;
    while (tr > 0 && ExpandLayout(d, wpb, tr).bytes > budget) tr -= 32;
    return tr;
}

int list_max_for(const Dims &d)
{
    // a list is stored only where it is shorter than the bitmap (n < W_Np words) and where either
    // block shape can take it on its restricted path
    const long long lim = std::min<long long>(std::min(restrict_max_of<8>(d), restrict_max_of<16>(d)), d.wnp - 1);
    return lim > SMALL_MAX ? (int)lim : 0;
}

template <bool COUNT, int WARPS, bool INHERIT>
static int launch_expand_t(const ExpandArgs &a, int sm_count, void *stream)
{
    int wpb = WARPS;
    while (wpb > 1 && ExpandLayout(a.d, wpb, 0).bytes > 200 * 1024) --wpb;
    // the largest restricted extent whose columns fit in the shared memory of the shape's blocks per
    // SM (or next to the gather path's own, when that is larger)
    const int tr = restrict_max_of<WARPS>(a.d);
    const size_t smem = ExpandLayout(a.d, wpb, tr).bytes;
    // the shared-memory attribute and the occupancy query, once per device and size (per thread)
    static thread_local ShapeCache cache;
    int dev = 0;
    cudaGetDevice(&dev);
    if (cache.dev != dev || cache.smem != smem || cache.wpb != wpb) {
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(expand_bitmap_kernel<COUNT, WARPS, INHERIT>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return (int)e;
        }
        int ps = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ps, expand_bitmap_kernel<COUNT, WARPS, INHERIT>, wpb * 32, smem);
        cache = ShapeCache{dev, smem, wpb, ps < 1 ? 1 : ps};
    }
    const int per_sm = cache.per_sm;
    // split each parent's attribute range into parts when there are too few parents to fill the GPU
    // (at least one candidate per warp in every part)
    ExpandArgs b = a;
    b.restrict_max = tr;
    const unsigned long long resident = (unsigned long long)sm_count * per_sm;
    const int max_parts = std::max(1, a.d.m / wpb);
    b.resident = resident;
    // with the count on the device the kernel chooses the parts; the grid is sized by the count
    // the caller expects
    const bool on_device = a.p_count_dev || a.p_count2_dev;
    const unsigned long long pc = a.p_count + a.p_count2;   // both pools (the second one may be empty)
    b.parts = on_device ? 0 : expand_parts(pc, resident, max_parts);
    const unsigned long long items = pc * (unsigned long long)(b.parts > 0 ? b.parts : expand_parts(pc, resident, max_parts));
    // a launch that reads its count on the device gets the whole resident wave (blocks without work
    // leave at once)
    unsigned long long blocks = on_device ? resident : std::min<unsigned long long>(items, resident);
    if (blocks < 1) blocks = 1;
    expand_bitmap_kernel<COUNT, WARPS, INHERIT><<<(unsigned)blocks, wpb * 32, smem, (cudaStream_t)stream>>>(b);
    return (int)cudaGetLastError();
}

int launch_expand(const ExpandArgs &a, int sm_count, void *stream)
{
    // wide blocks for many attributes, or for levels too small to fill the GPU with narrow blocks
#define FCA_EXPAND(W)                                                                               \
    (a.wit_words > 0 ? (a.count_work ? launch_expand_t<true, W, true>(a, sm_count, stream)              \
                                     : launch_expand_t<false, W, true>(a, sm_count, stream))            \
                     : (a.count_work ? launch_expand_t<true, W, false>(a, sm_count, stream)             \
                                     : launch_expand_t<false, W, false>(a, sm_count, stream)))
    if (a.d.m >= WIDE_EXPAND_MIN_ATTRS || a.p_count + a.p_count2 < 2ull * 3 * (unsigned long long)sm_count)
        return FCA_EXPAND(16);
    return FCA_EXPAND(8);
#undef FCA_EXPAND
}

}  // namespace fca
