// Concept-lattice kernels of libfca (sm_103a): the extent of each intent and the cover relation of
// the lattice (FCbO-to-CUDA article, section 4.4: the concept pool keeps extents beside intents, and
// the lattice's edges are rebuilt afterwards by extent inclusion; Parallel FCBO article, section 3.4).
//
//  extents_kernel      A = B' for each given attribute set B: the AND of the columns of B's
//                      attributes (every object for the empty set). Short extents (W_N <= 16):
//                      a group of lanes per intent, one output word per lane; longer ones: a warp
//                      per intent, the rarest column first, then four columns per step over 128
//                      words at a time, until every lane holds zero words.
//  hash_insert_kernel  an open-addressing table from intent to row index (linear probing).
//  covers_kernel       the lower covers of each concept (A, B), one warp per concept. For k not in
//                      B let C_k = A & column k. The extents of the lower covers are exactly the
//                      maximal sets among the distinct C_k (a concept below (A, B) has an extent
//                      inside some C_k; a maximal C_k is closed, since C_k'' = A & (B + k)' = C_k), and
//                      the cover with extent C has intent D = B + {k : C_k = C}. Each cover is
//                      emitted once, by the smallest k with C_k = C, and its row index is looked up.
//                      With at most 64 objects in A, the sets C_k are 64-bit masks over A's objects
//                      (built from the rows by 32 x 32 bit transposes); above that they are words of
//                      the object bitmap, restricted to the words where A is not zero; there the
//                      supports are counted a few attributes per pass, and the containment tests read
//                      C_k's compacted words warp-wide and gather several column words at a time, so
//                      that the loads of one lane are not a chain of dependent round trips. In both
//                      forms the candidates with an empty C_k (most of them, on sparse tables) are
//                      settled by one vote: such a C_k is a cover's extent only when all are empty.
#include <cuda_runtime.h>

#include <algorithm>

#include "fca_device.cuh"

namespace fca {
namespace {

constexpr uint32_t EMPTY_SLOT = 0xffffffffu;

// Mask of the valid bits of word w of an n-bit set.
__device__ __forceinline__ uint32_t valid_bits(long long w, long long words, long long n)
{
    const int tail = (int)(n & 31);
    return (w == words - 1 && tail) ? ((1u << tail) - 1u) : FULL;
}

// The attributes of B in processing order, rarest first: lane w holds word w of B (attribute
// order); the positions (perm maps an attribute to its position, null: the identity) are written in
// ascending order to list[0..nb) and nb is returned to every lane. scratch (W_M words) receives B by
// position.
__device__ __forceinline__ int attr_list(uint32_t Bw, const int32_t *perm, uint16_t *list, uint32_t *scratch, int wm,
                                         unsigned lane)
{
    if (perm) {
        if ((int)lane < wm) scratch[lane] = 0u;
        __syncwarp();
        uint32_t bits = Bw;
        while (bits) {
            const int p = perm[32 * (int)lane + __ffs(bits) - 1];
            bits &= bits - 1u;
            atomicOr(scratch + (p >> 5), 1u << (p & 31));
        }
        __syncwarp();
        Bw = (int)lane < wm ? scratch[lane] : 0u;
    } else {
        if ((int)lane < wm) scratch[lane] = Bw;
        __syncwarp();
    }
    const unsigned c = __popc(Bw);
    unsigned pre = c;   // inclusive prefix sum over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(FULL, pre, o);
        if ((int)lane >= o) pre += y;
    }
    unsigned q = pre - c;
    while (Bw) {
        list[q++] = (uint16_t)(32 * lane + __ffs(Bw) - 1);
        Bw &= Bw - 1u;
    }
    __syncwarp();
    return (int)__shfl_sync(FULL, pre, 31);
}

// Words w0 + 32u + lane (u < U) of the extent of an attribute list: the AND of column words, the
// first (rarest) column alone, the rest four columns at a time (4U loads in flight per lane), until
// every lane of the warp holds zero words (warp-wide).
template <int U>
__device__ __forceinline__ void extent_words(uint32_t (&acc)[U], const uint16_t *list, int nb, const uint32_t *cols,
                                             long long wnp, long long w0, unsigned lane)
{
    if (nb > 0) {
        const uint32_t *c0 = cols + (size_t)list[0] * wnp + w0 + lane;
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (acc[u]) acc[u] &= __ldg(c0 + 32 * u);
    }
    for (int q = 1; q < nb; q += 4) {
        uint32_t any = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) any |= acc[u];
        if (!__any_sync(FULL, any != 0u)) break;
        const int p0 = list[q];
        const uint32_t *c0 = cols + (size_t)p0 * wnp + w0 + lane;
        const uint32_t *c1 = cols + (size_t)(q + 1 < nb ? list[q + 1] : p0) * wnp + w0 + lane;
        const uint32_t *c2 = cols + (size_t)(q + 2 < nb ? list[q + 2] : p0) * wnp + w0 + lane;
        const uint32_t *c3 = cols + (size_t)(q + 3 < nb ? list[q + 3] : p0) * wnp + w0 + lane;
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (acc[u]) acc[u] &= __ldg(c0 + 32 * u) & __ldg(c1 + 32 * u) & __ldg(c2 + 32 * u) & __ldg(c3 + 32 * u);
    }
}

constexpr int EXT_U = 4;   // extent words per lane and pass

// G lanes per row (G a power of two, the smallest at least W_N, at most 32). With G = 32 a warp takes
// one row, lists its attributes rarest first (columns in processing order) and walks the row 128
// words at a time (four per lane), so its stores are consecutive words; with G < 32 (W_N <= 16) a warp takes 32 / G
// rows and each lane ANDs the columns of its row's attributes in attribute order.
template <int G>
__global__ void __launch_bounds__(256) extents_kernel(const uint32_t *__restrict__ intents, unsigned long long count,
                                                      const uint32_t *__restrict__ cols,
                                                      const uint32_t *__restrict__ cols_p,
                                                      const int32_t *__restrict__ perm, Dims d,
                                                      uint32_t *__restrict__ extents)
{
    constexpr int RPW = 32 / G;
    const unsigned lane = threadIdx.x & 31;
    const unsigned long long warp = ((unsigned long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const unsigned long long warps = ((unsigned long long)gridDim.x * blockDim.x) >> 5;
    if constexpr (G == 32) {
        __shared__ uint16_t lists[8][MAX_ATTRS];
        __shared__ uint32_t scratch[8][32];
        uint16_t *list = lists[threadIdx.x >> 5];
        for (unsigned long long r = warp; r < count; r += warps) {
            const uint32_t Bw = (int)lane < d.wm ? intents[r * d.wm + lane] & valid_bits(lane, d.wm, d.m) : 0u;
            const int nb = attr_list(Bw, perm, list, scratch[threadIdx.x >> 5], d.wm, lane);
            uint32_t *o = extents + r * (unsigned long long)d.wn;
            for (long long w0 = 0; w0 < d.wn; w0 += 32 * EXT_U) {
                uint32_t acc[EXT_U];
#pragma unroll
                for (int u = 0; u < EXT_U; ++u) {
                    const long long w = w0 + 32 * u + lane;
                    acc[u] = w < d.wn ? valid_bits(w, d.wn, d.n) : 0u;
                }
                extent_words<EXT_U>(acc, list, nb, cols_p, d.wnp, w0, lane);
#pragma unroll
                for (int u = 0; u < EXT_U; ++u) {
                    const long long w = w0 + 32 * u + lane;
                    if (w < d.wn) o[w] = acc[u];
                }
            }
            __syncwarp();
        }
    } else {
        const int gl = (int)(lane % G);
        for (unsigned long long r0 = warp * RPW; r0 < count; r0 += warps * RPW) {
            const unsigned long long r = r0 + lane / G;
            const bool live = r < count && gl < d.wn;
            if (!live) continue;
            const uint32_t *b = intents + r * (unsigned long long)d.wm;
            uint32_t acc = valid_bits(gl, d.wn, d.n);
            for (int iw = 0; iw < d.wm && acc; ++iw) {
                uint32_t bits = __ldg(b + iw) & valid_bits(iw, d.wm, d.m);
                while (bits && acc) {
                    const int a = 32 * iw + __ffs(bits) - 1;
                    bits &= bits - 1u;
                    acc &= __ldg(cols + (size_t)a * d.wnp + gl);
                }
            }
            extents[r * (unsigned long long)d.wn + gl] = acc;
        }
    }
}

// Order-independent hash of an intent: the 64-bit sum over its words of a mixed (index, word) pair.
// The mixer is the splitmix64 finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom number
// generators", 2014).
__device__ __forceinline__ unsigned long long mix64(unsigned long long x)
{
    x ^= x >> 30;
    x *= 0xbf58476d1ce4e5b9ull;
    x ^= x >> 27;
    x *= 0x94d049bb133111ebull;
    x ^= x >> 31;
    return x;
}

__device__ __forceinline__ unsigned long long word_hash(int w, uint32_t v)
{
    return mix64(((unsigned long long)(unsigned)w << 32) | v);
}

__global__ void __launch_bounds__(256) hash_insert_kernel(const uint32_t *__restrict__ intents, unsigned long long count,
                                                          int wm, int m, uint32_t *slots, unsigned long long mask,
                                                          LatticeCounters *lc)
{
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    for (unsigned long long r = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; r < count; r += stride) {
        unsigned long long h = 0;
        for (int w = 0; w < wm; ++w) h += word_hash(w, __ldg(intents + r * wm + w) & valid_bits(w, wm, m));
        unsigned long long s = h & mask;
        bool done = false;
        for (unsigned long long probe = 0; probe <= mask; ++probe) {
            const uint32_t held = atomicCAS(slots + s, EMPTY_SLOT, (uint32_t)r);
            if (held == EMPTY_SLOT) {
                done = true;
                break;
            }
            // an occupant with the same intent: the set holds a duplicate (each intent must be given
            // once, or a cover would resolve to either copy)
            bool same = true;
            for (int w = 0; w < wm && same; ++w) {
                const uint32_t vm = valid_bits(w, wm, m);
                same = (__ldg(intents + r * wm + w) & vm) == (__ldg(intents + (unsigned long long)held * wm + w) & vm);
            }
            if (same) {
                atomicAdd(&lc->duplicates, 1ull);
                done = true;
                break;
            }
            s = (s + 1) & mask;
        }
        if (!done) atomicAdd(&lc->insert_failed, 1ull);
    }
}

// Per-warp shared memory of covers_kernel, in 32-bit words: R (2M: 64-bit restricted sets by
// attribute), s (M supports), eb (M: rows of the covers found for the current concept), ids (64 object
// ids), scratch (32: B by position), rows of A's objects (64 x W_M, when A has at most 64), the
// attribute list of B (M 16-bit positions); rounded up to an even count. Each warp also has 4 W_N words
// of global workspace: A's non-zero words and their indices, C_k's non-zero words and their indices.
__host__ __device__ inline long long covers_words_per_warp(const Dims &d)
{
    return (4ll * d.m + 64 + 32 + 64ll * d.wm + (d.m + 1) / 2 + 1) & ~1ll;   // even: R 8-byte aligned
}

// Extents of more than 64 objects: attributes whose supports one pass counts, words of A whose
// restriction to a column one compaction step forms (per lane), compacted words of a C_k of more
// than 64 objects one containment step tests (per lane).
constexpr int SUP_BATCH = 4;
constexpr int COMPACT_U = 4;
constexpr int SCAN_BATCH = 8;

struct CoversArgs {
    Dims d;
    const uint32_t *intents;   // count x wm, attribute order
    unsigned long long count;
    const uint32_t *rows;      // n x wm, processing order
    const int32_t *inv;        // processing position -> attribute (null: the identity)
    const int32_t *perm;       // attribute -> processing position (null: the identity)
    const uint32_t *cols_p;    // m x wnp, processing order
    const uint32_t *cols;      // m x wnp, attribute order
    const uint32_t *slots;     // hash table of intents
    unsigned long long mask;   // slots - 1
    uint32_t *edges;           // capacity x 2
    unsigned long long capacity;
    LatticeCounters *lc;
    uint32_t *ws;              // 4 x wn words per warp of the grid
};

// The row of intent D (lane w holds word w) in the intent set, through the hash table; -1 when it is
// not there (warp-wide).
__device__ __forceinline__ long long find_intent(const CoversArgs &a, uint32_t Dw, unsigned lane)
{
    const Dims &d = a.d;
    unsigned long long h = (int)lane < d.wm ? word_hash((int)lane, Dw) : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) h += __shfl_xor_sync(FULL, h, o);
    unsigned long long slot = h & a.mask;
    for (unsigned long long probe = 0; probe <= a.mask; ++probe) {
        const uint32_t idx = a.slots[slot];
        if (idx == EMPTY_SLOT) return -1;
        const bool eq = (int)lane >= d.wm ||
                        (a.intents[(size_t)idx * d.wm + lane] & valid_bits(lane, d.wm, d.m)) == Dw;
        if (__all_sync(FULL, eq)) return idx;
        slot = (slot + 1) & a.mask;
    }
    return -1;
}

// The objects of a set kept as its non-zero words (value v[j] of word index wi[j], j < nw) into
// ids[], ascending; the caller knows there are at most as many as ids[] holds.
__device__ __forceinline__ void list_objects(const uint32_t *v, const uint32_t *wi, int nw, uint32_t *ids,
                                             unsigned lane)
{
    unsigned off = 0;
    for (int j0 = 0; j0 < nw; j0 += 32) {
        const int j = j0 + (int)lane;
        const uint32_t x0 = j < nw ? v[j] : 0u;
        const unsigned c = __popc(x0);
        unsigned pre = c;   // inclusive prefix sum of the popcounts
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(FULL, pre, o);
            if ((int)lane >= o) pre += y;
        }
        unsigned p = off + pre - c;
        uint32_t x = x0;
        while (x) {
            const int b = __ffs(x) - 1;
            x &= x - 1u;
            ids[p++] = (uint32_t)(32 * wi[j] + b);
        }
        off += __shfl_sync(FULL, pre, 31);
    }
    __syncwarp();
}

// Candidates with an empty C_k: such a C_k is maximal only when every C_k outside B is empty, and the
// cover is then the bottom concept (extent empty, intent M), emitted by the smallest such k. One vote
// over the supports (s_k, -1 for k in B) gives both facts to every lane.
__device__ __forceinline__ void empty_vote(const int *s, int m, unsigned lane, bool *nz_any, int *kmin0)
{
    bool nz = false;
    int kmin = 0x7fffffff;
    for (int k = (int)lane; k < m; k += 32) {
        const int sv = s[k];
        nz |= sv > 0;
        if (sv == 0 && k < kmin) kmin = k;
    }
    *nz_any = __any_sync(FULL, nz);
    *kmin0 = __reduce_min_sync(FULL, kmin);
}

__global__ void __launch_bounds__(256, 5) covers_kernel(const __grid_constant__ CoversArgs a)
{
    extern __shared__ __align__(16) uint32_t lat_smem[];
    const Dims d = a.d;
    const unsigned lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint32_t *base = lat_smem + (size_t)warp * covers_words_per_warp(d);
    unsigned long long *R = reinterpret_cast<unsigned long long *>(base);
    int *s = reinterpret_cast<int *>(base + 2 * d.m);
    uint32_t *eb = base + 3 * d.m;
    uint32_t *ids = base + 4 * d.m;
    uint32_t *Aw = a.ws + ((size_t)blockIdx.x * (blockDim.x >> 5) + warp) * 4 * (size_t)d.wn;
    uint32_t *Ai = Aw + d.wn;
    uint32_t *Cv = Ai + d.wn;
    uint32_t *Ci = Cv + d.wn;
    uint32_t *scratch = ids + 64;
    uint32_t *rowsm = scratch + 32;
    uint16_t *list = reinterpret_cast<uint16_t *>(rowsm + 64 * d.wm);
    const int chunks = (d.m + 31) >> 5;   // = wm

    // One concept per claim, the next one claimed while this one runs: the concepts with large
    // extents sit next to each other in the enumeration's output, and claims of several at a time
    // gave some warps a run of them.
    unsigned long long inext = 0;
    if (lane == 0) inext = atomicAdd(&a.lc->next, 1ull);
    for (;;) {
        const unsigned long long i = __shfl_sync(FULL, inext, 0);
        if (i >= a.count) break;
        if (lane == 0) inext = atomicAdd(&a.lc->next, 1ull);
        {
            // B: lane w holds word w
            const uint32_t Bw = (int)lane < d.wm ? a.intents[i * d.wm + lane] & valid_bits(lane, d.wm, d.m) : 0u;

            // A = B': AND of the columns of B's attributes (rarest first), kept as its non-zero words
            const int nb = attr_list(Bw, a.perm, list, scratch, d.wm, lane);
            int nnz = 0, objs = 0;
            for (long long w0 = 0; w0 < d.wn; w0 += 32 * EXT_U) {
                uint32_t acc[EXT_U];
#pragma unroll
                for (int u = 0; u < EXT_U; ++u) {
                    const long long w = w0 + 32 * u + lane;
                    acc[u] = w < d.wn ? valid_bits(w, d.wn, d.n) : 0u;
                }
                extent_words<EXT_U>(acc, list, nb, a.cols_p, d.wnp, w0, lane);
#pragma unroll
                for (int u = 0; u < EXT_U; ++u) {
                    const unsigned nzb = __ballot_sync(FULL, acc[u] != 0u);
                    if (acc[u]) {
                        const int p = nnz + __popc(nzb & ((1u << lane) - 1u));
                        Aw[p] = acc[u];
                        Ai[p] = (uint32_t)(w0 + 32 * u + lane);
                    }
                    nnz += __popc(nzb);
                    objs += __reduce_add_sync(FULL, (unsigned)__popc(acc[u]));
                }
            }
            __syncwarp();

            int ne = 0;   // covers found for concept i (rows in eb)
            bool nz_any = false;   // some C_k outside B is not empty
            int kmin0 = 0;         // the smallest k outside B with C_k empty
            const bool small = objs <= 64;
            if (small) {
                list_objects(Aw, Ai, nnz, ids, lane);   // object ids of A (at most 64)
                // the rows of A's objects (processing order), then the restricted sets by attribute:
                // R[k] bit o = object ids[o] has attribute k (inv maps a position back to its attribute)
                for (int x = (int)lane; x < objs * d.wm; x += 32) {
                    const int o = x / d.wm;
                    rowsm[x] = __ldg(a.rows + (size_t)ids[o] * d.wm + (x - o * d.wm));
                }
                __syncwarp();
                for (int t = 0; t < d.wm; ++t) {
                    const uint32_t lo = warp_transpose32((int)lane < objs ? rowsm[lane * d.wm + t] : 0u);
                    const uint32_t hi =
                        objs > 32 ? warp_transpose32((int)lane + 32 < objs ? rowsm[(lane + 32) * d.wm + t] : 0u) : 0u;
                    const int p = 32 * t + (int)lane;
                    if (p < d.m) R[a.inv ? a.inv[p] : p] = ((unsigned long long)hi << 32) | lo;
                }
                __syncwarp();
                // supports s_k = |C_k| for k not in B (-1 for k in B)
                for (int c = 0; c < chunks; ++c) {
                    const int k = 32 * c + (int)lane;
                    const bool inB = (__shfl_sync(FULL, Bw, c) >> lane) & 1u;
                    if (k < d.m) s[k] = inB ? -1 : __popcll(R[k]);
                }
                __syncwarp();
                empty_vote(s, d.m, lane, &nz_any, &kmin0);
                // the covers: candidates k whose C_k is maximal among the C_k and that are the smallest
                // attribute of their class (no other k2 has C_k inside C_k2 with more objects, or the
                // same set and a smaller index). The k2 with C_k inside C_k2 are the attributes of
                // D_k = C_k', the AND of the rows of C_k's objects (every attribute when C_k is empty),
                // so each lane closes its own candidate and checks the supports of D_k outside B.
                for (int c = 0; c < chunks; ++c) {
                    const int k = 32 * c + (int)lane;
                    const int sk = k < d.m ? s[k] : -1;
                    bool bad = sk < 0;
                    if (sk == 0) {
                        bad = nz_any || k != kmin0;
                    } else if (!bad) {
                        const unsigned long long Rk = R[k];
                        for (int t = 0; t < d.wm && !bad; ++t) {
                            uint32_t dk = valid_bits(t, d.wm, d.m);
                            unsigned long long x = Rk;
                            while (x && dk) {
                                const int o = __ffsll(x) - 1;
                                x &= x - 1ull;
                                dk &= rowsm[o * d.wm + t];
                            }
                            dk &= ~scratch[t];   // D_k outside B, by processing position
                            while (dk) {
                                const int p = 32 * t + __ffs(dk) - 1;
                                dk &= dk - 1u;
                                const int k2 = a.inv ? a.inv[p] : p;
                                if (k2 == k) continue;
                                const int s2 = s[k2];
                                if (s2 > sk || (s2 == sk && k2 < k)) {
                                    bad = true;
                                    break;
                                }
                            }
                        }
                    }
                    unsigned emit = __ballot_sync(FULL, !bad);
                    while (emit) {
                        const int kk = 32 * c + __ffs(emit) - 1;
                        emit &= emit - 1u;
                        const int skk = s[kk];
                        const unsigned long long Rkk = R[kk];
                        // D = B + {k2 : C_k2 = C_kk}
                        uint32_t Dw = Bw;
                        for (int c2 = 0; c2 < chunks; ++c2) {
                            const int k2 = 32 * c2 + (int)lane;
                            const bool in = k2 < d.m && s[k2] == skk && (Rkk & ~R[k2]) == 0ull;
                            const uint32_t word = __ballot_sync(FULL, in);
                            if ((int)lane == c2) Dw |= word;
                        }
                        const long long row = find_intent(a, Dw, lane);
                        if (row < 0) {
                            if (lane == 0) atomicAdd(&a.lc->missing, 1ull);
                        } else {
                            if (lane == 0) eb[ne] = (uint32_t)row;
                            ++ne;
                        }
                    }
                }
            } else {
                // supports, SUP_BATCH attributes per pass: lanes over A's non-zero words, each word of
                // A read once per pass and the batch's column words gathered together
                for (int c = 0; c < chunks; ++c) {
                    const int k = 32 * c + (int)lane;
                    if (k < d.m) s[k] = -1;
                }
                __syncwarp();
                for (int c = 0; c < chunks; ++c) {
                    uint32_t cand = ~__shfl_sync(FULL, Bw, c) & valid_bits(c, d.wm, d.m);
                    while (cand) {
                        int kk[SUP_BATCH];
                        const uint32_t *colb[SUP_BATCH];
#pragma unroll
                        for (int u = 0; u < SUP_BATCH; ++u) {
                            kk[u] = cand ? 32 * c + __ffs(cand) - 1 : -1;
                            cand &= cand - 1u;
                            colb[u] = a.cols + (size_t)(kk[u] < 0 ? kk[0] : kk[u]) * d.wnp;   // kk[0] >= 0
                        }
                        unsigned cnt[SUP_BATCH];
#pragma unroll
                        for (int u = 0; u < SUP_BATCH; ++u) cnt[u] = 0u;
#pragma unroll 2
                        for (int j = (int)lane; j < nnz; j += 32) {
                            const uint32_t aw = Aw[j];
                            const uint32_t ai = Ai[j];
#pragma unroll
                            for (int u = 0; u < SUP_BATCH; ++u) cnt[u] += __popc(aw & __ldg(colb[u] + ai));
                        }
#pragma unroll
                        for (int u = 0; u < SUP_BATCH; ++u) {
                            const unsigned t = __reduce_add_sync(FULL, cnt[u]);
                            if (lane == 0 && kk[u] >= 0) s[kk[u]] = (int)t;
                        }
                    }
                }
                __syncwarp();
                empty_vote(s, d.m, lane, &nz_any, &kmin0);
                // each candidate k in turn. Only attributes k2 outside B with s_k2 >= s_k can hold C_k
                // (C_k inside C_k2 gives |C_k| <= |C_k2|); with none, C_k is maximal, the smallest of
                // its class, and its cover's intent is B + {k}. Otherwise C_k's non-zero words are
                // compacted and lanes take the k2 and test C_k inside column k2 on those words only,
                // the warp reading the compacted words together and gathering SCAN_BATCH of them at a time.
                for (int c = 0; c < chunks; ++c) {
                    uint32_t cand = ~__shfl_sync(FULL, Bw, c) & valid_bits(c, d.wm, d.m);
                    while (cand) {
                        const int k = 32 * c + __ffs(cand) - 1;
                        cand &= cand - 1u;
                        const int sk = s[k];
                        uint32_t Dw = Bw;
                        bool any_holder = false;
                        if (sk == 0) {
                            if (nz_any || k != kmin0) continue;
                            Dw = (int)lane < d.wm ? valid_bits(lane, d.wm, d.m) : 0u;   // the bottom: M
                        } else {
                            for (int c2 = 0; c2 < chunks; ++c2) {
                                const int k2 = 32 * c2 + (int)lane;
                                any_holder |= k2 < d.m && k2 != k && s[k2] >= sk;   // s < 0 for attributes of B
                            }
                        }
                        if (__any_sync(FULL, any_holder)) {
                            const uint32_t *col = a.cols + (size_t)k * d.wnp;
                            int cnz = 0;
                            __syncwarp();
                            for (int j0 = 0; j0 < nnz; j0 += 32 * COMPACT_U) {
                                uint32_t v[COMPACT_U], wi[COMPACT_U];
#pragma unroll
                                for (int u = 0; u < COMPACT_U; ++u) {
                                    const int j = j0 + 32 * u + (int)lane;
                                    v[u] = j < nnz ? Aw[j] : 0u;   // A's listed words are non-zero
                                    wi[u] = j < nnz ? Ai[j] : 0u;
                                }
#pragma unroll
                                for (int u = 0; u < COMPACT_U; ++u) v[u] = v[u] ? v[u] & __ldg(col + wi[u]) : 0u;
#pragma unroll
                                for (int u = 0; u < COMPACT_U; ++u) {
                                    const unsigned nzb = __ballot_sync(FULL, v[u] != 0u);
                                    if (v[u]) {
                                        const int p = cnz + __popc(nzb & ((1u << lane) - 1u));
                                        Cv[p] = v[u];
                                        Ci[p] = wi[u];
                                    }
                                    cnz += __popc(nzb);
                                }
                            }
                            __syncwarp();
                            bool bad = false;
                            if (sk <= 64) {
                                // D_k = C_k' (processing positions, lane t holds word t): the AND of
                                // the rows of C_k's objects, at most two per lane; the k2 holding C_k
                                // are the attributes of D_k outside B
                                list_objects(Cv, Ci, cnz, ids, lane);
                                const uint32_t o0 = (int)lane < sk ? ids[lane] : 0u;
                                const uint32_t o1 = (int)lane + 32 < sk ? ids[lane + 32] : 0u;
                                uint32_t Dp = 0u;
#pragma unroll 4
                                for (int t = 0; t < d.wm; ++t) {
                                    uint32_t v = (int)lane < sk ? __ldg(a.rows + (size_t)o0 * d.wm + t) : FULL;
                                    if ((int)lane + 32 < sk) v &= __ldg(a.rows + (size_t)o1 * d.wm + t);
                                    v = __reduce_and_sync(FULL, v);
                                    if ((int)lane == t) Dp = v;
                                }
                                for (int c2 = 0; c2 < chunks; ++c2) {
                                    const int k2 = 32 * c2 + (int)lane;
                                    const int p = k2 < d.m ? (a.perm ? a.perm[k2] : k2) : 0;
                                    const uint32_t wd = __shfl_sync(FULL, Dp, p >> 5);
                                    const bool held = k2 < d.m && k2 != k && s[k2] >= 0 && ((wd >> (p & 31)) & 1u);
                                    if (held && (s[k2] > sk || k2 < k)) bad = true;
                                    const uint32_t word = __ballot_sync(FULL, held);
                                    if ((int)lane == c2) Dw |= word;
                                }
                                bad = __any_sync(FULL, bad);
                            } else {
                                for (int c2 = 0; c2 < chunks && !bad; ++c2) {
                                    const int k2 = 32 * c2 + (int)lane;
                                    bool held = k2 < d.m && k2 != k && s[k2] >= sk;
                                    const uint32_t *col2 = a.cols + (size_t)(held ? k2 : 0) * d.wnp;
                                    for (int j0 = 0; j0 < cnz && __any_sync(FULL, held); j0 += 32) {
                                        const int jl = j0 + (int)lane;
                                        const uint32_t myv = jl < cnz ? Cv[jl] : 0u;
                                        const uint32_t myi = jl < cnz ? Ci[jl] : 0u;
                                        int u0 = 0;
                                        if (j0 == 0) {
                                            // most k2 miss C_k on its first word: test that word alone
                                            const uint32_t cv = __shfl_sync(FULL, myv, 0);
                                            const uint32_t ci = __shfl_sync(FULL, myi, 0);
                                            if (held && (cv & ~__ldg(col2 + ci))) held = false;
                                            u0 = 1;
                                        }
                                        for (; u0 < 32 && j0 + u0 < cnz && __any_sync(FULL, held); u0 += SCAN_BATCH) {
                                            uint32_t viol = 0u;
#pragma unroll
                                            for (int u = 0; u < SCAN_BATCH; ++u) {
                                                const int src = u0 + u;
                                                const uint32_t cv = __shfl_sync(FULL, myv, src & 31);
                                                const uint32_t ci = __shfl_sync(FULL, myi, src & 31);
                                                if (held && src < 32 && cv) viol |= cv & ~__ldg(col2 + ci);
                                            }
                                            held = held && viol == 0u;
                                        }
                                    }
                                    if (held && (s[k2] > sk || k2 < k)) bad = true;
                                    bad = __any_sync(FULL, bad);
                                    const uint32_t word = __ballot_sync(FULL, held);
                                    if ((int)lane == c2) Dw |= word;
                                }
                            }
                            __syncwarp();
                            if (bad) continue;
                        }
                        if ((int)lane == (k >> 5)) Dw |= 1u << (k & 31);
                        const long long row = find_intent(a, Dw, lane);
                        if (row < 0) {
                            if (lane == 0) atomicAdd(&a.lc->missing, 1ull);
                        } else {
                            if (lane == 0) eb[ne] = (uint32_t)row;
                            ++ne;
                        }
                    }
                }
            }
            // the concept's edges: one slot allocation, then the rows
            __syncwarp();
            if (ne) {
                unsigned long long e0 = 0;
                if (lane == 0) e0 = atomicAdd(&a.lc->edges, (unsigned long long)ne);
                e0 = __shfl_sync(FULL, e0, 0);
                for (int j = (int)lane; j < ne; j += 32) {
                    const unsigned long long e = e0 + j;
                    if (e < a.capacity) {
                        a.edges[2 * e] = (uint32_t)i;
                        a.edges[2 * e + 1] = eb[j];
                    }
                }
            }
            __syncwarp();
        }
    }
}

}  // namespace

int launch_extents(const uint32_t *intents, uint64_t count, const uint32_t *cols, const uint32_t *cols_p,
                   const int32_t *perm, const Dims &d, uint32_t *extents, int sm_count, void *stream)
{
    if (count == 0) return (int)cudaSuccess;
    int g = 1;
    while (g < 32 && g < d.wn) g <<= 1;
    const unsigned long long rows_per_block = 8ull * (32 / g);
    const unsigned blocks = (unsigned)std::min<unsigned long long>((count + rows_per_block - 1) / rows_per_block,
                                                                   8ull * sm_count);
    cudaStream_t st = (cudaStream_t)stream;
    switch (g) {
    case 1: extents_kernel<1><<<blocks, 256, 0, st>>>(intents, count, cols, cols_p, perm, d, extents); break;
    case 2: extents_kernel<2><<<blocks, 256, 0, st>>>(intents, count, cols, cols_p, perm, d, extents); break;
    case 4: extents_kernel<4><<<blocks, 256, 0, st>>>(intents, count, cols, cols_p, perm, d, extents); break;
    case 8: extents_kernel<8><<<blocks, 256, 0, st>>>(intents, count, cols, cols_p, perm, d, extents); break;
    case 16: extents_kernel<16><<<blocks, 256, 0, st>>>(intents, count, cols, cols_p, perm, d, extents); break;
    default: extents_kernel<32><<<blocks, 256, 0, st>>>(intents, count, cols, cols_p, perm, d, extents); break;
    }
    return (int)cudaGetLastError();
}

size_t covers_smem_per_warp(const Dims &d) { return (size_t)covers_words_per_warp(d) * 4; }

int covers_shape(const Dims &d, uint64_t count, int sm_count, int *wpb, unsigned *blocks, size_t *smem)
{
    // Each warp holds its own shared memory, so the block size only decides how much of an SM's
    // shared memory blocks can fill: take the size (at most 8 warps) with the most warps resident.
    const size_t per_warp = covers_smem_per_warp(d);
    const size_t limit = 227 * 1024;
    if (per_warp > limit) return (int)cudaErrorInvalidValue;
    const int wmax = (int)std::min<size_t>(8, limit / per_warp);
    cudaError_t e =
        cudaFuncSetAttribute(covers_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(per_warp * wmax));
    if (e != cudaSuccess) return (int)e;
    int per_sm = 0, best = -1;
    for (int w = wmax; w >= 1; --w) {
        int b = 0;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, covers_kernel, w * 32, per_warp * w)) != cudaSuccess)
            return (int)e;
        if (b * w > best) {
            best = b * w;
            *wpb = w;
            per_sm = b;
        }
    }
    *smem = per_warp * *wpb;
    per_sm = std::max(1, per_sm);
    *blocks = (unsigned)std::max<unsigned long long>(
        1, std::min<unsigned long long>((std::max<uint64_t>(count, 1) + *wpb - 1) / *wpb,
                                        (unsigned long long)per_sm * sm_count));
    return (int)cudaSuccess;
}

int launch_covers(const uint32_t *intents, uint64_t count, const uint32_t *rows, const int32_t *inv,
                  const int32_t *perm, const uint32_t *cols, const uint32_t *cols_p, const Dims &d, uint32_t *slots,
                  uint64_t nslots, uint32_t *edges, uint64_t capacity, LatticeCounters *lc, uint32_t *ws, int wpb,
                  unsigned blocks, size_t smem, int sm_count, void *stream)
{
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(slots, 0xff, (size_t)nslots * 4, st);
    if (e != cudaSuccess) return (int)e;
    if (count == 0) return (int)cudaSuccess;
    const unsigned ib = (unsigned)std::min<unsigned long long>((count + 255) / 256, 16ull * sm_count);
    hash_insert_kernel<<<ib, 256, 0, st>>>(intents, count, d.wm, d.m, slots, nslots - 1, lc);
    if ((e = cudaGetLastError()) != cudaSuccess) return (int)e;
    CoversArgs a;
    a.d = d;
    a.intents = intents;
    a.count = count;
    a.rows = rows;
    a.inv = inv;
    a.perm = perm;
    a.cols_p = cols_p;
    a.cols = cols;
    a.slots = slots;
    a.mask = nslots - 1;
    a.edges = edges;
    a.capacity = capacity;
    a.lc = lc;
    a.ws = ws;
    covers_kernel<<<blocks, wpb * 32, smem, st>>>(a);
    return (int)cudaGetLastError();
}

}  // namespace fca
