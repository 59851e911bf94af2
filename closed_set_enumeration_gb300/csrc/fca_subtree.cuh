// Object-list tier of libfca (sm_103a), device code: subtree_kernel<NW> runs whole Close-by-One
// subtrees whose root extent holds at most 32*NW objects, one warp per subtree, on the context's
// columns restricted to the root's objects (the recursive Close-by-One search of the FCbO-to-CUDA
// article, sections 2.1-2.3). Bitwise set algebra only: no tensor cores. Included by
// fca_subtree.cu (launches without work sharing) and fca_subtree_share.cu (with it), which compile
// in parallel.
#pragma once
#include <cuda_runtime.h>

#include <algorithm>

#include "fca_device.cuh"

namespace fca {
namespace {


// Shared-memory layout of one warp of subtree_kernel<NW> (32-bit words).
struct SubtreeLayout {
    static constexpr int ROOTB_W = 32, RM_W = 32, RLO_W = 34, SUFB_W = 32, IDS_W = 64, DSC_W = 34;
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
        o_rm = o_rootb + ROOTB_W;
        o_rlo = o_rm + RM_W;
        o_sufb = o_rlo + RLO_W;
        o_dsc = o_sufb + SUFB_W + IDS_W;
        o_stack = o_dsc + DSC_W;
        o_outbuf = o_stack + (size_t)fr * fs;
        words = o_outbuf + (size_t)OUTBUF * wm;
        words = (words + 3) & ~(size_t)3;
    }
};

// Per-warp state of the object-list tier: shared-memory areas of the current subtree root,
// the output buffer and the warp's counters.
struct SubtreeWarp {
    // Two base pointers and two offsets locate every area (the others are fixed offsets from them),
    // which keeps the search's register footprint small.
    uint32_t *own;      // this warp's area: dsc, stack, output buffer
    uint32_t *root;     // the root areas in use: this warp's, or a donor's
    int orm;            // word offset of the attribute map in a warp area
    int oob;            // word offset of the output buffer in a warp area
    using SL = SubtreeLayout;
    // restricted columns, NW planes x mp (compact attribute index)
    __device__ uint32_t *cR() const { return root; }
    // compact index -> attribute
    __device__ uint16_t *rmap() const { return reinterpret_cast<uint16_t *>(root + orm); }
    // root intent (full attribute space), 32 words
    __device__ uint32_t *rootB() const { return root + orm + mp / 2; }
    // relevant attributes per full word
    __device__ uint32_t *Rm() const { return rootB() + SL::ROOTB_W; }
    // first compact index of each full word (wm + 1 entries)
    __device__ uint32_t *rlo() const { return Rm() + SL::RM_W; }
    // root-intent attributes in the words above each word
    __device__ uint32_t *sufB() const { return rlo() + SL::RLO_W; }
    // compact intent of the child being written, or a handed-over node
    __device__ uint32_t *dsc() const
    {
        return own + orm + mp / 2 + SL::ROOTB_W + SL::RM_W + SL::RLO_W + SL::SUFB_W + SL::IDS_W;
    }
    // the root's object ids (32 * NW)
    __device__ uint32_t *ids() const { return sufB() + SL::SUFB_W; }
    // search stack
    __device__ uint32_t *stk() const { return dsc() + SL::DSC_W; }
    // output buffer, OUTBUF x wm
    __device__ uint32_t *ob() const { return own + oob; }
    int mp, wm, fs, m;
    const SubtreeArgs *args;   // the launch's arguments (spill queue, counters)
    long long deadline;        // clock64() past which the current search spills (0: none)
    uint32_t *out;
    unsigned long long capacity;
    Counters *ctr;
    int nb;             // intents waiting in the output buffer
    unsigned long long closures, ops;

    // Point the root areas (restricted columns, attribute map, root intent and its word tables) at
    // the per-warp area starting at `base`.
    __device__ void bind(uint32_t *base) { root = base; }

    __device__ void flush()
    {
        const unsigned lane = threadIdx.x & 31;
        unsigned long long b0 = 0;
        if (lane == 0) b0 = atomicAdd(&ctr->out_count, (unsigned long long)nb);
        b0 = __shfl_sync(FULL, b0, 0);
        __syncwarp();
        for (int i = (int)lane; i < nb * wm; i += 32)
            if (b0 + (unsigned long long)(i / wm) < capacity) out[b0 * wm + i] = ob()[i];
        __syncwarp();
        nb = 0;
    }

    // Write the full intent of a canonical child whose compact intent is in dsc()[]:
    // root intent plus the compact bits mapped back to their attributes.
    template <bool COUNT>
    __device__ void emit()
    {
        const unsigned lane = threadIdx.x & 31;
        __syncwarp();
        if (lane < (unsigned)wm) {
            const int w = (int)lane;
            const int lo = (int)rlo()[w], hi = (int)rlo()[w + 1];
            const int su = lo >> 5, sh = lo & 31;
            const uint32_t s0 = dsc()[su];
            const uint32_t s1 = sh ? dsc()[su + 1] : 0u;
            uint32_t seg = sh ? ((s0 >> sh) | (s1 << (32 - sh))) : s0;
            const int len = hi - lo;
            if (len < 32) seg &= (1u << len) - 1u;
            uint32_t res = rootB()[w];
            while (seg) {                      // each compact attribute of D in this word
                const int i = __ffs(seg) - 1;
                seg &= seg - 1u;
                res |= 1u << (rmap()[lo + i] & 31);
            }
            ob()[nb * wm + w] = res;
        }
        ++nb;
        if (COUNT) ops += (unsigned)wm;   // the intent words written
        __syncwarp();
        if (nb == OUTBUF) flush();
    }

    // Same for a compact intent held in warp-uniform registers (dfs_regs): lane l owns compact
    // attribute 32u + l of word u, and lane w collects full word w. Each full word that D touches
    // takes one OR-reduction of the bits of the lanes whose attribute lies in it.
    // Word `lane` (lane < wm) of the full intent: root intent plus the compact bits of D mapped back.
    template <int WRT>
    __device__ uint32_t full_word(const uint32_t (&D)[WRT])
    {
        const unsigned lane = threadIdx.x & 31;
        uint32_t acc = lane < (unsigned)wm ? rootB()[lane] : 0u;
#pragma unroll
        for (int u = 0; u < WRT; ++u) {
            uint32_t pend = D[u];
            if (pend == 0u) continue;
            const int a = ((pend >> lane) & 1u) ? (int)rmap()[32 * u + (int)lane] : -1;
            while (pend) {
                const int w = __shfl_sync(FULL, a, __ffs(pend) - 1) >> 5;
                const bool in = a >= 0 && (a >> 5) == w;
                const uint32_t v = __reduce_or_sync(FULL, in ? (1u << (a & 31)) : 0u);
                if (lane == (unsigned)w) acc |= v;
                pend &= ~__ballot_sync(FULL, in);
            }
        }
        return acc;
    }

    template <int WRT, bool COUNT>
    __device__ void emit_regs(const uint32_t (&D)[WRT])
    {
        const unsigned lane = threadIdx.x & 31;
        const uint32_t acc = full_word<WRT>(D);
        if (lane < (unsigned)wm) ob()[nb * wm + (int)lane] = acc;
        ++nb;
        if (COUNT) ops += (unsigned)wm;   // the intent words written
        __syncwarp();
        if (nb == OUTBUF) flush();
    }

    // Candidates of a child created at compact candidate j whose compact intent has `above`
    // attributes after j: the attributes after rmap()[j] outside its full intent.
    __device__ void count_child(int j, int above)
    {
        const int rj = rmap()[j];
        const int rw = rj >> 5, rb = rj & 31;
        const uint32_t hi = rb == 31 ? 0u : (rootB()[rw] >> (rb + 1));
        closures += (unsigned long long)(m - rj - 1 - (int)sufB()[rw] - __popc(hi) - above);
    }
};

// Work sharing inside a block. A warp that finds no more work items stays and searches candidate
// sets that busy warps of the block hand over through one mailbox in shared memory: the remaining
// candidates of a node of the donor's subtree, searched on the donor's restricted columns (which
// the donor no longer changes, as it has no work items left either).
constexpr int H_BUSY = 0;      // warps of the block with a work item or a handed-over node
constexpr int H_IDLE = 1;      // warps waiting for a hand-over
constexpr int H_MB = 2;        // mailbox state (MB_*)
constexpr int H_OWNER = 3;     // warp whose root areas the handed-over node uses
constexpr int H_R = 4;         // its relevant-attribute count
constexpr int H_EXT = 5;       // extent (NW words)
constexpr int H_B = 8;         // compact intent (WRT words)
constexpr int H_CAND = 16;     // candidates to search (WRT words)
constexpr int H_TAIL = 24;     // some warp of the block found no more work items (all kernels)
constexpr int HDR_WORDS = 32;
constexpr int MB_EMPTY = 0, MB_WRITING = 1, MB_FULL = 2, MB_TAKING = 3;
// Nodes a search visits before it may hand work over: short searches finish sooner than a hand-over
// would pay for itself.
constexpr int SHARE_AFTER = 24;

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ int vload(const int *p) { return *reinterpret_cast<const volatile int *>(p); }

// Dynamic shared memory of subtree_kernel: the block's work-sharing words (HDR_WORDS) first, then
// one area per warp. The header thus sits at a fixed address.
extern __shared__ uint32_t subtree_smem[];
__device__ __forceinline__ int *block_hdr() { return reinterpret_cast<int *>(subtree_smem); }

// Register width used for R relevant attributes (must match the dispatch in subtree_kernel): kernels
// with RW <= 4 take the narrowest of 1, 2 and 4 words; the wider kernels search every subtree of up
// to 32·RW relevant attributes at RW words, so that they hold one register search variant instead
// of four (their code then fits the instruction caches better, which measured faster than the
// narrower registers).
template <int RW>
__device__ __forceinline__ int regs_width(int R)
{
    if (RW > 4) return R <= 32 * RW ? RW : 0;
    return R <= 32 ? 1 : (R <= 64 ? 2 : (RW >= 4 && R <= 128 ? 4 : 0));
}

// Offer half of this warp's remaining search to an idle warp of the block: the remaining
// candidates of the shallowest stack frame that has any (else of the current node, when it has at
// least two), every other one in attribute order so both halves mix early (larger) and late
// (smaller) subtrees. Nothing happens when the mailbox is taken.
template <int NW, int WRT>
__device__ void offer(SubtreeWarp &S, int R, int depth, const uint32_t (&ext)[NW], const uint32_t (&B)[WRT],
                      uint32_t (&cand)[WRT])
{
    const unsigned lane = threadIdx.x & 31;
    int got = 0;
    if (lane == 0) got = atomicCAS(&block_hdr()[H_MB], MB_EMPTY, MB_WRITING) == MB_EMPTY;
    if (!__shfl_sync(FULL, got, 0)) return;
    int fd = -1;
    for (int d = 0; d < depth && fd < 0; ++d) {
        const uint32_t *f = S.stk() + (size_t)d * S.fs;
        uint32_t any = 0;
#pragma unroll
        for (int u = 0; u < WRT; ++u) any |= f[NW + u];
        if (any) fd = d;
    }
    uint32_t c[WRT], e[NW], b[WRT];
    uint32_t *f = S.stk() + (size_t)(fd < 0 ? 0 : fd) * S.fs;
#pragma unroll
    for (int t = 0; t < NW; ++t) e[t] = fd < 0 ? ext[t] : f[t];
    int tot = 0;
#pragma unroll
    for (int u = 0; u < WRT; ++u) {
        c[u] = fd < 0 ? cand[u] : f[NW + u];
        b[u] = fd < 0 ? B[u] : f[NW + WRT + u];
        tot += __popc(c[u]);
    }
    if (fd < 0 && tot < 2) {
        if (lane == 0) atomicExch(&block_hdr()[H_MB], MB_EMPTY);
        return;
    }
    // odd-ranked candidates (or the only one of a frame): a set bit has odd rank iff the parity of
    // the set bits up to and including it, carried across words, is even
    uint32_t give[WRT];
    bool odd_before = false;
#pragma unroll
    for (int u = 0; u < WRT; ++u) {
        uint32_t p = c[u];
        p ^= p << 1;
        p ^= p << 2;
        p ^= p << 4;
        p ^= p << 8;
        p ^= p << 16;
        give[u] = tot == 1 ? c[u] : c[u] & ~(odd_before ? ~p : p);
        odd_before ^= (__popc(c[u]) & 1) != 0;
    }
    __syncwarp();
    if (lane == 0) {
#pragma unroll
        for (int u = 0; u < WRT; ++u)
            if (fd >= 0) f[NW + u] = c[u] & ~give[u];
        block_hdr()[H_OWNER] = (int)(S.root - subtree_smem);
        block_hdr()[H_R] = R;
#pragma unroll
        for (int t = 0; t < NW; ++t) block_hdr()[H_EXT + t] = (int)e[t];
#pragma unroll
        for (int u = 0; u < WRT; ++u) {
            block_hdr()[H_B + u] = (int)b[u];
            block_hdr()[H_CAND + u] = (int)give[u];
        }
        __threadfence_block();
        atomicExch(&block_hdr()[H_MB], MB_FULL);
    }
    if (fd < 0) {
#pragma unroll
        for (int u = 0; u < WRT; ++u) cand[u] &= ~give[u];
    }
    __syncwarp();
}

// Candidate screening for dfs_regs (R <= 128): drops, from the remaining candidates of a node, those
// whose closure adds an attribute below j (not canonical), evaluating 32 candidates at once: lane l
// takes candidate j = 32u + l, forms C = ext & c_j from its own column, and ANDs the compact rows of
// the objects of C into words 0..u of D (broadcast by shuffles, one object at a time, over the
// objects that lie in some live candidate's C). A word of candidates is screened only when that
// costs fewer instructions than evaluating its candidates one by one (about 2u + 4 per object
// against about 40 + 6(u + 1) per candidate).
constexpr int SCREEN_PER_CAND = 40;

template <int NW, int WRT, bool COUNT>
__device__ __forceinline__ void screen(SubtreeWarp &S, uint32_t (&cand)[WRT], const uint32_t (&ext)[NW],
                                       const uint32_t (&B)[WRT], const uint32_t (&col)[WRT][NW],
                                       const uint32_t (&rowc)[NW][WRT])
{
    const unsigned lane = threadIdx.x & 31;
#pragma unroll
    for (int u = 0; u < WRT; ++u) {
        if (cand[u] == 0u) continue;
        // only objects in some candidate's C matter, and only the closure words up to u (the
        // canonical test of j = 32u + lane looks at attributes below j)
        const bool live = (cand[u] >> lane) & 1u;
        uint32_t C[NW], E[NW];
        int ne = 0;
#pragma unroll
        for (int t = 0; t < NW; ++t) {
            C[t] = ext[t] & col[u][t];
            E[t] = __reduce_or_sync(FULL, live ? C[t] : 0u);
            ne += __popc(E[t]);
        }
        if (ne * (2 * u + 4) >= (SCREEN_PER_CAND + 6 * (u + 1)) * __popc(cand[u])) continue;   // uniform
        uint32_t D[WRT];
#pragma unroll
        for (int w = 0; w <= u; ++w) D[w] = FULL;
#pragma unroll
        for (int t = 0; t < NW; ++t) {
            uint32_t e = E[t];
            while (e) {
                const int o = __ffs(e) - 1;
                e &= e - 1u;
                const bool in = (C[t] >> o) & 1u;
#pragma unroll
                for (int w = 0; w <= u; ++w) {
                    const uint32_t r = __shfl_sync(FULL, rowc[t][w], o);
                    if (in) D[w] &= r;
                }
            }
        }
        // canonical iff D adds no attribute below j = 32u + lane to B
        bool ok = true;
#pragma unroll
        for (int w = 0; w <= u; ++w) {
            const uint32_t below = w < u ? FULL : (1u << lane) - 1u;
            ok = ok && (D[w] & ~B[w] & below) == 0u;
        }
        cand[u] &= __ballot_sync(FULL, ok);
        if (COUNT) S.ops += (unsigned long long)ne * 2 * (u + 1);
    }
}

// A search that ran past its time budget in the tail of its launch: the nodes it has not finished
// (the current node and every ancestor on the stack from depth d_lo on with candidates left) are
// written to the spill queue as roots of their own: the root's object ids selected by the node's extent, the full intent, and the cursor
// at its first remaining candidate, stored as -(y + 1) because their candidates were counted when
// the nodes were created. Candidates that screening had already dropped come back with the cursor
// and fail again. Slots for all of them are taken with one atomicAdd; returns false (nothing
// written) when the spill queue cannot hold them.
template <int NW, int WRT>
__device__ bool spill_rest(SubtreeWarp &S, int d_lo, int depth, const uint32_t (&ext)[NW], const uint32_t (&B)[WRT],
                           const uint32_t (&cand)[WRT])
{
    const unsigned lane = threadIdx.x & 31;
    const SubtreeArgs &a = *S.args;
    int count = 0;
    for (int d = d_lo; d <= depth; ++d) {
        uint32_t any = 0;
        if (d == depth) {
#pragma unroll
            for (int u = 0; u < WRT; ++u) any |= cand[u];
        } else {
            const uint32_t *f = S.stk() + (size_t)d * S.fs;
#pragma unroll
            for (int u = 0; u < WRT; ++u) any |= f[NW + u];
        }
        count += any != 0u;
    }
    if (count == 0) return true;
    unsigned long long slot = 0;
    if (lane == 0) slot = atomicAdd(&a.ctr->spill[a.q_index], (unsigned long long)count);
    slot = __shfl_sync(FULL, slot, 0);
    if (slot + count > a.spill.cap) {
        // the queue is full: the reserved slots that exist become empty roots (no objects)
        for (unsigned long long k = slot + lane; k < a.spill.cap && k < slot + count; k += 32) {
            a.spill.n[k] = 0;
            a.spill.y[k] = -1;
        }
        return false;
    }
    const int per = 32 * NW;
    for (int d = d_lo; d <= depth; ++d) {
        uint32_t e[NW], b[WRT], c[WRT];
        if (d == depth) {
#pragma unroll
            for (int t = 0; t < NW; ++t) e[t] = ext[t];
#pragma unroll
            for (int u = 0; u < WRT; ++u) {
                b[u] = B[u];
                c[u] = cand[u];
            }
        } else {
            const uint32_t *f = S.stk() + (size_t)d * S.fs;
#pragma unroll
            for (int t = 0; t < NW; ++t) e[t] = f[t];
#pragma unroll
            for (int u = 0; u < WRT; ++u) {
                c[u] = f[NW + u];
                b[u] = f[NW + WRT + u];
            }
        }
        int first = -1;
#pragma unroll
        for (int u = 0; u < WRT; ++u)
            if (first < 0 && c[u]) first = 32 * u + __ffs(c[u]) - 1;
        if (first < 0) continue;
        int pos = 0;
#pragma unroll
        for (int t = 0; t < NW; ++t) {
            if ((e[t] >> lane) & 1u)
                a.spill.ids[slot * per + pos + __popc(e[t] & ((1u << lane) - 1u))] = S.ids()[32 * t + (int)lane];
            pos += __popc(e[t]);
        }
        const uint32_t w = S.full_word<WRT>(b);
        if (lane < (unsigned)S.wm) a.spill.itt[slot * S.wm + lane] = w;
        if (lane == 0) {
            a.spill.n[slot] = pos;
            a.spill.y[slot] = -((int)S.rmap()[first] + 1);
        }
        ++slot;
    }
    __syncwarp();
    return true;
}

// Depth-first search of one subtree with the restricted columns in registers: lane l holds the
// columns of compact attributes 32u + l, u < WRT (R <= 32 * WRT). Extent, intent and remaining
// candidates of the current node are warp-uniform registers; the stack of ancestors is in shared
// memory. A node's candidates are filtered once, when the node is entered, to the attributes
// whose column meets its extent (the others give an empty extent, whose closure is the bottom
// concept the host adds), so the loop only visits candidates with a non-empty C. With `handed`,
// the search starts instead from a node another warp handed over (extent, compact intent and the
// candidates to search, already screened, in this warp's dsc[] area).
template <int NW, int WRT, bool COUNT, bool SHARE, bool SPILL>
__device__ void dfs_regs(SubtreeWarp &S, int R, int n, int jn, int slices, int slice, bool handed)
{
    const unsigned lane = threadIdx.x & 31;
    uint32_t col[WRT][NW];
#pragma unroll
    for (int u = 0; u < WRT; ++u) {
        const int k = 32 * u + (int)lane;
#pragma unroll
        for (int t = 0; t < NW; ++t) col[u][t] = k < R ? S.cR()[t * S.mp + k] : 0u;
    }
    // compact rows of the root's objects (lane l holds object 32t + l), for candidate screening:
    // the transpose of the restricted columns, one 32 x 32 register transpose per word
    constexpr bool SCREEN = WRT <= 4;
    uint32_t rowc[NW][WRT];
#pragma unroll
    for (int t = 0; t < NW; ++t)
#pragma unroll
        for (int w = 0; w < WRT; ++w) rowc[t][w] = SCREEN ? warp_transpose32(col[w][t]) : 0u;
    uint32_t B[WRT], cand[WRT];
    uint32_t ext[NW];
    if (handed) {
#pragma unroll
        for (int t = 0; t < NW; ++t) ext[t] = S.dsc()[t];
#pragma unroll
        for (int u = 0; u < WRT; ++u) {
            B[u] = S.dsc()[NW + u];
            cand[u] = S.dsc()[NW + WRT + u];
        }
    } else {
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
        if (SCREEN) screen<NW, WRT, COUNT>(S, cand, ext, B, col, rowc);
    }
    // Candidate cursor: cu is the lowest word of cand[] with candidates left and cw its remaining
    // bits (cand[cu] itself is stale, words below cu are spent), so taking the next candidate costs
    // a few instructions whatever WRT is; cand[] is brought up to date only when a frame is pushed
    // or the candidates leave the search (spill, hand-over).
    int cu;
    uint32_t cw;
    auto cursor_from_cand = [&]() {
        cu = WRT;
        cw = 0u;
#pragma unroll
        for (int u = WRT - 1; u >= 0; --u)
            if (cand[u]) {
                cu = u;
                cw = cand[u];
            }
    };
    auto cand_from_cursor = [&]() {
#pragma unroll
        for (int u = 0; u < WRT; ++u) cand[u] = u < cu ? 0u : (u == cu ? cw : cand[u]);
    };
    cursor_from_cand();
    // Column prefetch (R <= 128, where the registers allow it; with 256 relevant attributes the two
    // extra registers per extent word cost more than the load latency they hide)
    constexpr bool PREFETCH = WRT <= 4;
    int pj = -1;        // compact index whose column pc[] holds
    uint32_t pc[NW];
    int depth = 0;
    int visits = 0;
    for (;;) {
        // past the time budget: the rest of the search goes to the spill queue (when it fits)
        // Past the time budget, once the block has run out of work items: the rest of the search
        // goes to the spill queue (when it fits). A node whose candidates are a subset of its
        // candidates from the cursor on (the root of a sliced item, a handed-over node, frames
        // that handed candidates over) cannot be restarted from a cursor, so work-sharing searches
        // never spill and a sliced or handed-over search keeps its depth-0 node and goes on there.
        ++visits;
        if (SPILL && !SHARE && S.deadline != 0 && (visits & 31) == 0 && clock64() > S.deadline &&
            vload(&block_hdr()[H_TAIL]) != 0) {
            const bool keep0 = handed || slices > 1;
            cand_from_cursor();
            if (!keep0) {
                if (spill_rest<NW, WRT>(S, 0, depth, ext, B, cand)) return;
                S.deadline = 0;
            } else if (depth > 0) {
                if (spill_rest<NW, WRT>(S, 1, depth, ext, B, cand)) {
                    depth = 0;
                    const uint32_t *f = S.stk();
#pragma unroll
                    for (int t = 0; t < NW; ++t) ext[t] = f[t];
#pragma unroll
                    for (int u = 0; u < WRT; ++u) {
                        cand[u] = f[NW + u];
                        B[u] = f[NW + WRT + u];
                    }
                    __syncwarp();
                    S.deadline = clock64() + S.args->budget;
                    cursor_from_cand();
                    continue;
                }
                S.deadline = 0;
            }
        }
        // an idle warp of the block is waiting and this search is long: hand it half of the rest
        if (SHARE && visits > SHARE_AFTER &&
            __any_sync(FULL, vload(&block_hdr()[H_IDLE]) > 0 && vload(&block_hdr()[H_MB]) == MB_EMPTY)) {
            cand_from_cursor();
            offer<NW, WRT>(S, R, depth, ext, B, cand);
            cursor_from_cand();
        }
        if (cw == 0u) {
            // the next word with candidates, or back up to the parent
            int nu = WRT;
            uint32_t nw = 0u;
#pragma unroll
            for (int u = WRT - 1; u >= 0; --u)
                if (u > cu && cand[u]) {
                    nu = u;
                    nw = cand[u];
                }
            cu = nu;
            cw = nw;
        }
        if (cw == 0u) {
            if (depth == 0) break;
            --depth;
            const uint32_t *f = S.stk() + (size_t)depth * S.fs;
#pragma unroll
            for (int t = 0; t < NW; ++t) ext[t] = f[t];
#pragma unroll
            for (int u = 0; u < WRT; ++u) {
                cand[u] = f[NW + u];
                B[u] = f[NW + WRT + u];
            }
            __syncwarp();
            cursor_from_cand();
            continue;
        }
        const int ju = cu;
        const int j = 32 * cu + __ffs(cw) - 1;   // the lowest remaining candidate
        cw &= cw - 1u;
        uint32_t C[NW];
        if (PREFETCH && j == pj) {
#pragma unroll
            for (int t = 0; t < NW; ++t) C[t] = ext[t] & pc[t];
        } else {
#pragma unroll
            for (int t = 0; t < NW; ++t) C[t] = ext[t] & S.cR()[t * S.mp + j];
        }
        if (PREFETCH) {
            // the column of the next candidate of this word, loaded while this one is evaluated
            pj = cw ? 32 * cu + __ffs(cw) - 1 : -1;
            if (pj >= 0) {
#pragma unroll
                for (int t = 0; t < NW; ++t) pc[t] = S.cR()[t * S.mp + pj];
            }
        }
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
        S.emit_regs<WRT, COUNT>(D);
        int above = 0;
#pragma unroll
        for (int u = 0; u < WRT; ++u) above += __popc(D[u] & ge_mask(u, j + 1));
        S.count_child(j, above);
        if (lane == 0) {
            uint32_t *f = S.stk() + (size_t)depth * S.fs;
#pragma unroll
            for (int t = 0; t < NW; ++t) f[t] = ext[t];
#pragma unroll
            for (int u = 0; u < WRT; ++u) {
                f[NW + u] = u < cu ? 0u : (u == cu ? cw : cand[u]);
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
        if (SCREEN) screen<NW, WRT, COUNT>(S, cand, ext, B, col, rowc);
        cursor_from_cand();
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
            const uint32_t *f = S.stk() + (size_t)depth * S.fs;
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
            C[t] = ext[t] & S.cR()[t * S.mp + j];
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
                for (int t = 0; t < NW; ++t) in = in && ((C[t] & ~S.cR()[t * S.mp + k]) == 0u);
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

        if (lane <= (unsigned)WR) S.dsc()[lane] = lane < (unsigned)WR ? myD : 0u;
        S.emit<COUNT>();
        unsigned c = __popc(myD & ge_mask((int)lane, j + 1) & validR);
        c = __reduce_add_sync(FULL, c);
        S.count_child(j, (int)c);
        {
            uint32_t *f = S.stk() + (size_t)depth * S.fs;
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

// SHARE: the block's warps hand parts of long searches to warps that have run out of work items
// (the block-shared header comes first in shared memory); without it a warp ends when the items do.
// Four blocks per SM (64 registers) except for the 33-64-object kernel with eight register words,
// which needs about 80 and whose shared memory allows three blocks anyway; the 1-32-object one fits
// four in shared memory and runs faster there in spite of a few spilled registers.
template <int NW, bool COUNT, int RW, bool SHARE>
__global__ void __launch_bounds__(256, (RW > 4 && NW > 1) ? 3 : 4) subtree_kernel(const __grid_constant__ SubtreeArgs a)
{
    // a launch queued before the host knew whether the bitmap search had ended cleanly
    if (a.guard && (a.ctr->error != 0u || a.ctr->next_count != 0ull)) return;
    uint32_t *const smw = subtree_smem + HDR_WORDS;
    // time-budgeted searches that spill in the tail: kernels of at most four register words (their
    // extra code costs the wider ones more than it saves)
    constexpr bool SPILLS = RW <= 4;
    const Dims d = a.d;
    const SubtreeLayout L(d, NW);
    const unsigned lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int nwb = (int)(blockDim.x >> 5);
    uint32_t *base = smw + (size_t)wib * L.words;
    int *const hdr = block_hdr();
    if (threadIdx.x == 0) {
        hdr[H_TAIL] = 0;
        if (SHARE) {
            hdr[H_BUSY] = nwb;
            hdr[H_IDLE] = 0;
            hdr[H_MB] = MB_EMPTY;
        }
    }
    __syncthreads();

    SubtreeWarp S;
    S.own = base;
    S.root = base;
    S.orm = (int)L.o_rmap;
    S.oob = (int)L.o_outbuf;
    S.mp = L.mp;
    S.wm = d.wm;
    S.fs = L.fs;
    S.m = d.m;
    S.args = &a;
    S.deadline = 0;
    S.out = a.out;
    S.capacity = a.capacity;
    S.ctr = a.ctr;
    S.nb = 0;
    S.closures = 0;
    S.ops = 0;
    const int mp = L.mp, WM = d.wm, PER = 32 * NW;

    const unsigned long long q_count = a.q_count_dev ? *a.q_count_dev : a.q_count;
    const unsigned long long items = q_count * (unsigned long long)a.slices;
    // Guided self-scheduling: a warp claims a run of consecutive items with one atomic, a quarter of
    // its share of what was left at its last claim (so claims shrink to single items near the end),
    // which keeps the launch-wide cursor from becoming a hot spot when items are short.
    const unsigned long long nwarps = (unsigned long long)gridDim.x * (blockDim.x >> 5);
    unsigned long long next = 0, end = 0, seen = 0;
    bool claiming = true;            // work items may be left
    unsigned long long t0 = 0;       // start of the current wait for a hand-over
    const unsigned long long wait_ns = a.wait_ns ? a.wait_ns : DEFAULT_WAIT_NS;
    for (;;) {
        bool handed = false, share = false;
        int R = 0, n = 0, jn = 0, slice = 0;
        if (claiming) {
            if (next >= end) {
                unsigned long long base = 0;
                const unsigned long long left = items > seen ? items - seen : 0;
                const unsigned long long k = min(32ull, max(1ull, left / (4 * nwarps)));
                if (lane == 0) base = atomicAdd(&a.ctr->q_head[a.q_index], k);
                base = __shfl_sync(FULL, base, 0);
                if (base >= items) {
                    claiming = false;
                    if (lane == 0) hdr[H_TAIL] = 1;   // the block's searches are now the tail
                    if (!SHARE) break;       // no work sharing in this launch: the warp is done
                    if (lane == 0) {
                        atomicSub(&hdr[H_BUSY], 1);
                        atomicAdd(&hdr[H_IDLE], 1);
                    }
                    t0 = global_ns();
                    continue;
                }
                next = base;
                end = min(items, base + k);
                seen = base + k;
            }
            const unsigned long long item = next++;
            // work item = (root, slice): the slice takes the root's children j with j % slices == slice
            const unsigned long long r = item / (unsigned)a.slices;
            slice = (int)(item % (unsigned)a.slices);

            // ---- root: object ids, intent, cursor
            n = a.q.n[r];
            // a negative cursor -(y + 1) marks a root spilled by a search that ran out of time: its
            // candidates were counted when it was created (cursor y)
            const int yr = a.q.y[r];
            const int y0 = yr < 0 ? -yr - 1 : yr;
            uint32_t id[NW];
#pragma unroll
            for (int t = 0; t < NW; ++t) {
                const int o = 32 * t + (int)lane;
                id[t] = o < n ? a.q.ids[r * PER + o] : 0u;
            }
            const uint32_t myRootB = lane < (unsigned)WM ? a.q.itt[r * WM + lane] : 0u;
            __syncwarp();
            S.rootB()[lane] = myRootB;
#pragma unroll
            for (int t = 0; t < NW; ++t) S.ids()[32 * t + (int)lane] = id[t];

            // ---- relevant attributes R (held by some but not all objects), compact index order =
            //      attribute order, and the columns restricted to the subtree's objects. Lane l holds
            //      the rows of objects 32t + l, loaded CH words at a time (independent loads); each
            //      32 x 32 block of a word is transposed in registers, so lane b then holds the column of
            //      attribute 32w + b, and the relevant lanes store theirs at their compact index.
            constexpr int CH = RW < 8 ? RW : 8;
            R = 0;
            for (int w0 = 0; w0 < WM; w0 += CH) {
                uint32_t rw[NW][CH];
#pragma unroll
                for (int t = 0; t < NW; ++t)
#pragma unroll
                    for (int i = 0; i < CH; ++i)
                        rw[t][i] = (w0 + i < WM && 32 * t + (int)lane < n)
                                       ? __ldg(a.rows + (size_t)id[t] * WM + w0 + i) : 0u;
#pragma unroll
                for (int i = 0; i < CH; ++i) {
                    const int w = w0 + i;
                    if (w >= WM) break;
                    uint32_t uni = 0;
#pragma unroll
                    for (int t = 0; t < NW; ++t) uni |= rw[t][i];
                    uni = __reduce_or_sync(FULL, uni);
                    const uint32_t rm = uni & ~__shfl_sync(FULL, myRootB, w);
                    if (lane == 0) { S.Rm()[w] = rm; S.rlo()[w] = (uint32_t)R; }
                    if (rm == 0u) continue;
                    const bool mine = (rm >> lane) & 1u;
                    const int k = R + __popc(rm & ((1u << lane) - 1u));
#pragma unroll
                    for (int t = 0; t < NW; ++t) {
                        const uint32_t c = warp_transpose32(rw[t][i]);
                        if (mine) S.cR()[t * mp + k] = c;
                    }
                    if (mine) S.rmap()[k] = (uint16_t)(32 * w + (int)lane);
                    R += __popc(rm);
                }
            }
            if (lane == 0) S.rlo()[WM] = (uint32_t)R;
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
                S.sufB()[lane] = tot - incl;
            }
            __syncwarp();

            // ---- candidates of the root: attributes >= y0 outside its intent (counted by slice 0)
            {
                unsigned c = lane < (unsigned)WM ? __popc(myRootB & ge_mask((int)lane, y0)) : 0u;
                c = __reduce_add_sync(FULL, c);
                if (slice == 0 && yr >= 0) S.closures += (unsigned long long)(d.m - y0 - (int)c);
            }
            // compact cursor jn: relevant attributes below y0 are not candidates
            {
                const unsigned c = lane < (unsigned)WM ? __popc(S.Rm()[lane] & lt_mask((int)lane, y0)) : 0u;
                jn = (int)__reduce_add_sync(FULL, c);
            }

            // with no claimed items left, part of the search may be handed to idle warps of the
            // block (this warp's root areas then stay as they are until the launch ends)
            share = SHARE && next >= end;
        } else if constexpr (SHARE) {
            // ---- no work items left: search what busy warps of the block hand over, until none
            //      is busy. Each wait is bounded (SubtreeArgs::wait_ns); past it FAULT_WAIT is
            //      recorded and the warp stops.
            int st = 0;   // 0: wait, 1: took a hand-over, 2: block done, 3: waited too long
            if (lane == 0) {
                const int mb = vload(&hdr[H_MB]);
                if (mb == MB_FULL && atomicCAS(&hdr[H_MB], MB_FULL, MB_TAKING) == MB_FULL) st = 1;
                else if (mb == MB_EMPTY && vload(&hdr[H_BUSY]) == 0) st = 2;
                else if (global_ns() - t0 > wait_ns) st = 3;
            }
            st = __shfl_sync(FULL, st, 0);
            if (st == 2) break;
            if (st == 3) {
                if (lane == 0) atomicOr(&a.ctr->fault, FAULT_WAIT);
                break;
            }
            if (st == 0) {
                __nanosleep(256);
                continue;
            }
            if (lane == 0) {
                atomicAdd(&hdr[H_BUSY], 1);
                atomicSub(&hdr[H_IDLE], 1);
            }
            __threadfence_block();
            const int owner = vload(&hdr[H_OWNER]);   // word offset of the donor's root areas
            R = vload(&hdr[H_R]);
            const int wr = regs_width<RW>(R);
            if (lane < (unsigned)NW) S.dsc()[lane] = (uint32_t)vload(&hdr[H_EXT + lane]);
            if (lane < (unsigned)wr) {
                S.dsc()[NW + lane] = (uint32_t)vload(&hdr[H_B + lane]);
                S.dsc()[NW + wr + lane] = (uint32_t)vload(&hdr[H_CAND + lane]);
            }
            __syncwarp();
            if (lane == 0) {
                __threadfence_block();
                atomicExch(&hdr[H_MB], MB_EMPTY);
            }
            S.bind(subtree_smem + owner);
            share = true;
            handed = true;
        }

        // ---- depth-first search of the subtree (or of the handed-over node), with its time budget
        S.deadline = SPILLS && a.budget ? clock64() + a.budget : 0;
        const int sl = handed ? 1 : a.slices;
        const int wr = regs_width<RW>(R);
        if (SHARE && share) {
            if (RW <= 4 && wr == 1) dfs_regs<NW, 1, COUNT, true, SPILLS>(S, R, n, jn, sl, slice, handed);
            else if (RW <= 4 && wr == 2) dfs_regs<NW, 2, COUNT, true, SPILLS>(S, R, n, jn, sl, slice, handed);
            else if (RW == 4 && wr == 4) dfs_regs<NW, 4, COUNT, true, SPILLS>(S, R, n, jn, sl, slice, handed);
            else if (RW > 4 && wr == RW) dfs_regs<NW, RW, COUNT, true, SPILLS>(S, R, n, jn, sl, slice, handed);
            else dfs_smem<NW, COUNT>(S, R, n, jn, sl, slice);
        } else {
            if (RW <= 4 && wr == 1) dfs_regs<NW, 1, COUNT, false, SPILLS>(S, R, n, jn, sl, slice, false);
            else if (RW <= 4 && wr == 2) dfs_regs<NW, 2, COUNT, false, SPILLS>(S, R, n, jn, sl, slice, false);
            else if (RW == 4 && wr == 4) dfs_regs<NW, 4, COUNT, false, SPILLS>(S, R, n, jn, sl, slice, false);
            else if (RW > 4 && wr == RW) dfs_regs<NW, RW, COUNT, false, SPILLS>(S, R, n, jn, sl, slice, false);
            else dfs_smem<NW, COUNT>(S, R, n, jn, sl, slice);
        }
        __syncwarp();
        if (SHARE && handed) {
            if (lane == 0) {
                atomicSub(&hdr[H_BUSY], 1);
                atomicAdd(&hdr[H_IDLE], 1);
            }
            t0 = global_ns();
        }
    }
    if (S.nb) S.flush();
    if (lane == 0 && S.closures) atomicAdd(&a.ctr->closures, S.closures);
    if (COUNT && lane == 0 && S.ops) atomicAdd(&a.ctr->word_ops, S.ops);
}

}  // namespace

static int warps_for(size_t per_warp, size_t header)
{
    const size_t budget = 200 * 1024;
    int w = WARPS_PER_BLOCK;
    while (w > 1 && (size_t)w * per_warp + header > budget) --w;
    return w;
}

// Block shape of the subtree kernel (persistent: at most one block per resident slot).
template <int NW, bool COUNT, int RW, bool SHARE>
static int subtree_shape(const Dims &d, int *wpb_out, size_t *smem_out, int *per_sm_out)
{
    const size_t pw = SubtreeLayout(d, NW).words * 4;
    const size_t header = HDR_WORDS * 4;
    const int wpb = warps_for(pw, header);
    const size_t smem = pw * wpb + header;
    static thread_local ShapeCache cache;
    int dev = 0;
    cudaGetDevice(&dev);
    if (cache.dev != dev || cache.smem != smem || cache.wpb != wpb) {
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(subtree_kernel<NW, COUNT, RW, SHARE>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return (int)e;
        }
        int ps = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &ps, subtree_kernel<NW, COUNT, RW, SHARE>, wpb * 32, smem);
        if (e != cudaSuccess) return (int)e;
        cache = ShapeCache{dev, smem, wpb, ps < 1 ? 1 : ps};
    }
    *wpb_out = wpb;
    *smem_out = smem;
    *per_sm_out = cache.per_sm;
    return (int)cudaSuccess;
}

// Launch over the b.q_count * b.slices work items of `b` (slices already set): one block per
// resident slot at most.
template <int NW, bool COUNT, int RW, bool SHARE>
static int launch_subtree_kernel(const SubtreeArgs &b, int sm_count, void *stream)
{
    int wpb = 0, per_sm = 0;
    size_t smem = 0;
    int e = subtree_shape<NW, COUNT, RW, SHARE>(b.d, &wpb, &smem, &per_sm);
    if (e != (int)cudaSuccess) return e;
    // a launch reading its root count on the device gets the whole resident wave
    unsigned long long blocks = b.q_count_dev ? ~0ull : (b.q_count * b.slices + wpb - 1) / wpb;
    const unsigned long long cap = (unsigned long long)sm_count * per_sm;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    subtree_kernel<NW, COUNT, RW, SHARE><<<(unsigned)blocks, wpb * 32, smem, (cudaStream_t)stream>>>(b);
    return (int)cudaGetLastError();
}

}  // namespace fca
