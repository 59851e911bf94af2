// Concept-lattice kernels of libfca (sm_103a): the extent of each intent and the cover relation of
// the lattice (FCbO-to-CUDA article, section 4.4: the concept pool keeps extents beside intents, and
// the lattice's edges are rebuilt afterwards by extent inclusion; Parallel FCBO article, section 3.4).
//
//  extents_kernel      A = B' for each given attribute set B: the AND of the columns of B's
//                      attributes (every object for the empty set). One thread per output word.
//  hash_insert_kernel  an open-addressing table from intent to row index (linear probing).
//  covers_kernel       the lower covers of each concept (A, B), one warp per concept. For k not in
//                      B let C_k = A & column k. The extents of the lower covers are exactly the
//                      maximal sets among the distinct C_k (a concept below (A, B) has an extent
//                      inside some C_k; a maximal C_k is closed, since C_k'' = A & (B + k)' = C_k), and
//                      the cover with extent C has intent D = B + {k : C_k = C}. Each cover is
//                      emitted once, by the smallest k with C_k = C, and its row index is looked up.
//                      With at most 64 objects in A, the sets C_k are 64-bit masks over A's objects
//                      (built from the rows by 32 x 32 bit transposes); above that they are words of
//                      the object bitmap, restricted to the words where A is not zero.
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

__global__ void __launch_bounds__(256) extents_kernel(const uint32_t *__restrict__ intents, unsigned long long count,
                                                      const uint32_t *__restrict__ cols, Dims d,
                                                      uint32_t *__restrict__ extents)
{
    const unsigned long long total = count * (unsigned long long)d.wn;
    const unsigned long long stride = (unsigned long long)gridDim.x * blockDim.x;
    for (unsigned long long t = (unsigned long long)blockIdx.x * blockDim.x + threadIdx.x; t < total; t += stride) {
        const unsigned long long r = t / (unsigned long long)d.wn;
        const long long w = (long long)(t - r * (unsigned long long)d.wn);
        uint32_t acc = valid_bits(w, d.wn, d.n);
        const uint32_t *b = intents + r * (unsigned long long)d.wm;
        for (int iw = 0; iw < d.wm && acc; ++iw) {
            uint32_t bits = __ldg(b + iw) & valid_bits(iw, d.wm, d.m);
            while (bits && acc) {
                const int a = 32 * iw + __ffs(bits) - 1;
                bits &= bits - 1u;
                acc &= __ldg(cols + (size_t)a * d.wnp + w);
            }
        }
        extents[t] = acc;
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
            if (atomicCAS(slots + s, EMPTY_SLOT, (uint32_t)r) == EMPTY_SLOT) {
                done = true;
                break;
            }
            s = (s + 1) & mask;
        }
        if (!done) atomicAdd(&lc->insert_failed, 1ull);
    }
}

// Per-warp shared memory of covers_kernel, in 32-bit words: R (2M: 64-bit restricted columns by
// processing position), s (M supports), Aw / Ai / Cw (wn each: A's non-zero words, their indices, C_k
// on them), ids (64 object ids); rounded up to an even count.
__host__ __device__ inline long long covers_words_per_warp(const Dims &d)
{
    return (3ll * d.m + 3ll * d.wn + 64 + 1) & ~1ll;   // even: R stays 8-byte aligned
}

struct CoversArgs {
    Dims d;
    const uint32_t *intents;   // count x wm, attribute order
    unsigned long long count;
    const uint32_t *rows;      // n x wm, processing order
    const int32_t *perm;       // attribute -> processing position (null: the identity)
    const uint32_t *cols;      // m x wnp, attribute order
    const uint32_t *slots;     // hash table of intents
    unsigned long long mask;   // slots - 1
    uint32_t *edges;           // capacity x 2
    unsigned long long capacity;
    LatticeCounters *lc;
};

__global__ void __launch_bounds__(256) covers_kernel(const __grid_constant__ CoversArgs a)
{
    extern __shared__ __align__(16) uint32_t lat_smem[];
    const Dims d = a.d;
    const unsigned lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    uint32_t *base = lat_smem + (size_t)warp * covers_words_per_warp(d);
    unsigned long long *R = reinterpret_cast<unsigned long long *>(base);
    int *s = reinterpret_cast<int *>(base + 2 * d.m);
    uint32_t *Aw = base + 3 * d.m;
    uint32_t *Ai = Aw + d.wn;
    uint32_t *Cw = Ai + d.wn;
    uint32_t *ids = Cw + d.wn;
    const int chunks = (d.m + 31) >> 5;   // = wm

    for (;;) {
        unsigned long long i = 0;
        if (lane == 0) i = atomicAdd(&a.lc->next, 1ull);
        i = __shfl_sync(FULL, i, 0);
        if (i >= a.count) break;

        // B: lane w holds word w
        const uint32_t Bw = (int)lane < d.wm ? a.intents[i * d.wm + lane] & valid_bits(lane, d.wm, d.m) : 0u;

        // A = B': AND of the columns of B's attributes, kept as its non-zero words
        int nnz = 0, objs = 0;
        for (long long w0 = 0; w0 < d.wn; w0 += 32) {
            const long long w = w0 + lane;
            uint32_t acc = w < d.wn ? valid_bits(w, d.wn, d.n) : 0u;
            for (int t = 0; t < d.wm; ++t) {
                uint32_t bits = __shfl_sync(FULL, Bw, t);
                while (bits) {
                    if (!__any_sync(FULL, acc != 0u)) break;
                    const int at = 32 * t + __ffs(bits) - 1;
                    bits &= bits - 1u;
                    if (acc) acc &= __ldg(a.cols + (size_t)at * d.wnp + w);
                }
            }
            const unsigned nzb = __ballot_sync(FULL, acc != 0u);
            if (acc) {
                const int p = nnz + __popc(nzb & ((1u << lane) - 1u));
                Aw[p] = acc;
                Ai[p] = (uint32_t)w;
            }
            nnz += __popc(nzb);
            objs += __reduce_add_sync(FULL, (unsigned)__popc(acc));
        }
        __syncwarp();

        const bool small = objs <= 64;
        if (small) {
            // object ids of A (at most 64; every non-zero word holds at least one object)
            unsigned off = 0;
            for (int j0 = 0; j0 < nnz; j0 += 32) {
                const int j = j0 + (int)lane;
                const uint32_t v = j < nnz ? Aw[j] : 0u;
                const unsigned c = __popc(v);
                unsigned pre = c;   // inclusive prefix sum of the popcounts
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned y = __shfl_up_sync(FULL, pre, o);
                    if ((int)lane >= o) pre += y;
                }
                unsigned p = off + pre - c;
                uint32_t x = v;
                while (x) {
                    const int b = __ffs(x) - 1;
                    x &= x - 1u;
                    ids[p++] = (uint32_t)(32 * Ai[j] + b);
                }
                off += __shfl_sync(FULL, pre, 31);
            }
            __syncwarp();
            // restricted columns by processing position: R[p] bit o = object ids[o] has the
            // attribute at position p (rows are in processing order)
            const uint32_t *r0 = (int)lane < objs ? a.rows + (size_t)ids[lane] * d.wm : nullptr;
            const uint32_t *r1 = (int)lane + 32 < objs ? a.rows + (size_t)ids[lane + 32] * d.wm : nullptr;
            for (int t = 0; t < d.wm; ++t) {
                const uint32_t lo = warp_transpose32(r0 ? __ldg(r0 + t) : 0u);
                const uint32_t hi = objs > 32 ? warp_transpose32(r1 ? __ldg(r1 + t) : 0u) : 0u;
                const int p = 32 * t + (int)lane;
                if (p < d.m) R[p] = ((unsigned long long)hi << 32) | lo;
            }
            __syncwarp();
        }

        // supports s_k = |C_k| for k not in B (-1 for k in B)
        for (int c = 0; c < chunks; ++c) {
            const int k = 32 * c + (int)lane;
            const uint32_t bword = __shfl_sync(FULL, Bw, c);
            const bool inB = (bword >> lane) & 1u;
            int sk = -1;
            if (k < d.m && !inB) {
                if (small) {
                    const int p = a.perm ? a.perm[k] : k;
                    sk = __popcll(R[p]);
                } else {
                    sk = 0;
                    const uint32_t *col = a.cols + (size_t)k * d.wnp;
                    for (int j = 0; j < nnz; ++j) sk += __popc(Aw[j] & __ldg(col + Ai[j]));
                }
            }
            if (k < d.m) s[k] = sk;
        }
        __syncwarp();

        // each candidate k: maximal among the C_k and the smallest attribute of its class
        for (int c = 0; c < chunks; ++c) {
            uint32_t cand = ~__shfl_sync(FULL, Bw, c) & valid_bits(c, d.wm, d.m);
            while (cand) {
                const int k = 32 * c + __ffs(cand) - 1;
                cand &= cand - 1u;
                const int sk = s[k];
                unsigned long long Rk = 0;
                if (small) {
                    Rk = R[a.perm ? a.perm[k] : k];
                } else {
                    const uint32_t *col = a.cols + (size_t)k * d.wnp;
                    for (int j = (int)lane; j < nnz; j += 32) Cw[j] = Aw[j] & __ldg(col + Ai[j]);
                    __syncwarp();
                }
                bool bad = false;
                uint32_t Dw = Bw;
                for (int c2 = 0; c2 < chunks && !bad; ++c2) {
                    const int k2 = 32 * c2 + (int)lane;
                    bool in = false;
                    if (k2 < d.m && k2 != k) {
                        const int s2 = s[k2];
                        if (s2 >= sk) {   // s2 < 0 for attributes of B
                            if (small) {
                                in = (Rk & ~R[a.perm ? a.perm[k2] : k2]) == 0ull;
                            } else {
                                const uint32_t *col2 = a.cols + (size_t)k2 * d.wnp;
                                in = true;
                                for (int j = 0; j < nnz; ++j) {
                                    if (Cw[j] & ~__ldg(col2 + Ai[j])) {
                                        in = false;
                                        break;
                                    }
                                }
                            }
                            if (in && (s2 > sk || k2 < k)) bad = true;
                        }
                    }
                    bad = __any_sync(FULL, bad);
                    const uint32_t word = __ballot_sync(FULL, in);
                    if ((int)lane == c2) Dw |= word;
                }
                if (!small) __syncwarp();
                if (bad) continue;
                if ((int)lane == (k >> 5)) Dw |= 1u << (k & 31);

                // row index of D
                unsigned long long h = (int)lane < d.wm ? word_hash(lane, Dw) : 0ull;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) h += __shfl_xor_sync(FULL, h, o);
                unsigned long long slot = h & a.mask;
                long long found = -1;
                for (unsigned long long probe = 0; probe <= a.mask; ++probe) {
                    const uint32_t idx = a.slots[slot];
                    if (idx == EMPTY_SLOT) break;
                    const bool eq = (int)lane >= d.wm ||
                                    (a.intents[(size_t)idx * d.wm + lane] & valid_bits(lane, d.wm, d.m)) == Dw;
                    if (__all_sync(FULL, eq)) {
                        found = idx;
                        break;
                    }
                    slot = (slot + 1) & a.mask;
                }
                if (lane == 0) {
                    if (found < 0) {
                        atomicAdd(&a.lc->missing, 1ull);
                    } else {
                        const unsigned long long e = atomicAdd(&a.lc->edges, 1ull);
                        if (e < a.capacity) {
                            a.edges[2 * e] = (uint32_t)i;
                            a.edges[2 * e + 1] = (uint32_t)found;
                        }
                    }
                }
            }
        }
        __syncwarp();
    }
}

}  // namespace

int launch_extents(const uint32_t *intents, uint64_t count, const uint32_t *cols, const Dims &d, uint32_t *extents,
                   int sm_count, void *stream)
{
    if (count == 0) return (int)cudaSuccess;
    const unsigned long long total = count * (unsigned long long)d.wn;
    const unsigned long long want = (total + 255) / 256;
    const unsigned blocks = (unsigned)std::min<unsigned long long>(want, 16ull * sm_count);
    extents_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(intents, count, cols, d, extents);
    return (int)cudaGetLastError();
}

size_t covers_smem_per_warp(const Dims &d) { return (size_t)covers_words_per_warp(d) * 4; }

int launch_covers(const uint32_t *intents, uint64_t count, const uint32_t *rows, const int32_t *perm,
                  const uint32_t *cols, const Dims &d, uint32_t *slots, uint64_t nslots, uint32_t *edges,
                  uint64_t capacity, LatticeCounters *lc, int sm_count, void *stream)
{
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaMemsetAsync(slots, 0xff, (size_t)nslots * 4, st);
    if (e != cudaSuccess) return (int)e;
    if (count == 0) return (int)cudaSuccess;
    const unsigned ib = (unsigned)std::min<unsigned long long>((count + 255) / 256, 16ull * sm_count);
    hash_insert_kernel<<<ib, 256, 0, st>>>(intents, count, d.wm, d.m, slots, nslots - 1, lc);
    if ((e = cudaGetLastError()) != cudaSuccess) return (int)e;

    const size_t per_warp = covers_smem_per_warp(d);
    const size_t limit = 200 * 1024;
    const int wpb = (int)std::max<size_t>(1, std::min<size_t>(8, limit / per_warp));
    const size_t smem = per_warp * wpb;
    if (smem > 227 * 1024) return (int)cudaErrorInvalidValue;
    if ((e = cudaFuncSetAttribute(covers_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
        return (int)e;
    int per_sm = 1;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, covers_kernel, wpb * 32, smem)) != cudaSuccess)
        return (int)e;
    per_sm = std::max(1, per_sm);
    const unsigned long long warps_needed = count;
    const unsigned blocks = (unsigned)std::max<unsigned long long>(
        1, std::min<unsigned long long>((warps_needed + wpb - 1) / wpb, (unsigned long long)per_sm * sm_count));
    CoversArgs a;
    a.d = d;
    a.intents = intents;
    a.count = count;
    a.rows = rows;
    a.perm = perm;
    a.cols = cols;
    a.slots = slots;
    a.mask = nslots - 1;
    a.edges = edges;
    a.capacity = capacity;
    a.lc = lc;
    covers_kernel<<<blocks, wpb * 32, smem, st>>>(a);
    return (int)cudaGetLastError();
}

}  // namespace fca
