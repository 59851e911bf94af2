// Mid tier of libfca (sm_103a): expand_mid_kernel expands the entries of a level's mid pool, whose
// extents hold more than SMALL_MAX and at most mid_max objects, one entry per warp, on columns
// restricted to the entry's objects (FCbO-to-CUDA article, sections 2.1-2.3, 3.4 and 5.3; Parallel FCBO article,
// sections 2.1 and 3.2). Bitwise set algebra only: no tensor cores.
//
// Such an entry stores its extent A as the ascending list of its object ids. The warp loads the rows
// of those objects and transposes them, 32 objects and 32 attributes at a time, into the restricted
// columns R[k] = A & {k}' as G = ceil(|A| / 32) words per attribute, kept in the warp's shared memory.
// Then for each candidate j >= y outside B:
//   C = R[j] (no intersection left to do: the restriction is the intersection with A);
//   the closure D = C' = B + j + {k : C inside R[k]} over the attributes held by some but not all of
//   A, tested by the lanes 32 attributes at a time in ascending order, so that an attribute below j
//   found in D ends the candidate (the canonical test) after the fewest rounds;
//   a canonical child writes its intent and goes to an object-list queue (at most SMALL_MAX objects)
//   or to the mid pool of the next level as an id list, compacted from the bits of C.
// No block barrier: the warps of a block take entries on their own from a launch-wide cursor.
#include <cuda_runtime.h>

#include <algorithm>

#include "fca_device.cuh"

namespace fca {
namespace {

// Mid-pool children of one entry whose inherited failures are written when the entry is done.
constexpr int WIT_SLOTS = 32;

// Per-warp shared memory in 32-bit words: R (M attributes, stride G | 1, at most GMAX + 1: an odd
// stride keeps the per-attribute reads of one word by 32 lanes and the lane-wise stores of the
// transposes free of bank conflicts), then the object ids (32 GMAX), then the entry's failure
// witnesses (ww words, one byte per attribute) and the slots of its mid-pool children.
template <int GMAX>
struct MidLayout {
    static constexpr int GS = GMAX + 1;
    __host__ __device__ static size_t words(int m, int ww)
    {
        return (size_t)m * GS + 32u * GMAX + (ww > 0 ? (size_t)ww + WIT_SLOTS : 0u);
    }
};

// The ids of the objects of C (bits of word `cw` of lane g < G: object 32 g + b of the list `ids`)
// written in ascending order to dst[0 .. |C|) and, when `fill` > |C|, zeros up to dst[fill).
__device__ __forceinline__ void write_ids(uint32_t cw, const uint32_t *ids, uint32_t *dst, unsigned cnt, int fill,
                                          unsigned lane)
{
    const unsigned pc = __popc(cw);
    unsigned incl = pc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const unsigned t = __shfl_up_sync(FULL, incl, off);
        if (lane >= (unsigned)off) incl += t;
    }
    unsigned pos = incl - pc;
    while (cw) {
        const int b = __ffs(cw) - 1;
        cw &= cw - 1u;
        dst[pos++] = ids[32 * lane + b];
    }
    for (int i = (int)cnt + (int)lane; i < fill; i += 32) dst[i] = 0u;
}

template <bool COUNT, int GMAX, bool INHERIT>
__global__ void __launch_bounds__(256) expand_mid_kernel(const __grid_constant__ ExpandArgs a)
{
    extern __shared__ __align__(16) uint32_t mid_smem[];
    const Dims d = a.d;
    const int wm = d.wm;
    const unsigned lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    uint32_t *R = mid_smem + (size_t)wib * MidLayout<GMAX>::words(d.m, a.wit_words);
    uint32_t *ids = R + (size_t)d.m * MidLayout<GMAX>::GS;
    // inherited failures (the Fast Close-by-One rule): witness byte per attribute, 0xff for none
    constexpr bool inherit = INHERIT;
    uint32_t *witw = ids + 32 * GMAX;
    uint8_t *wit = reinterpret_cast<uint8_t *>(witw);
    uint32_t *slots = witw + a.wit_words;
    const uint32_t valid_last = (d.m & 31) ? ((1u << (d.m & 31)) - 1u) : FULL;
    const unsigned long long p_count = a.p_count_dev ? *a.p_count_dev : a.p_count;
    const unsigned long long nwarps = (unsigned long long)gridDim.x * (blockDim.x >> 5);

    unsigned long long my_closures = 0, my_bytes = 0;
    unsigned long long next = 0, end = 0, seen = 0;
    for (;;) {
        if (next >= end) {
            // claim a run of entries: a quarter of this warp's share of what it last saw left (at
            // most 8), so that claims shrink to single entries near the end
            unsigned long long base = 0, k = 1;
            if (lane == 0) {
                const unsigned long long left = p_count > seen ? p_count - seen : 0;
                k = min(8ull, max(1ull, left / (4 * nwarps)));
                base = atomicAdd(&a.ctr->mid_head, k);
            }
            base = __shfl_sync(FULL, base, 0);
            k = __shfl_sync(FULL, k, 0);
            if (base >= p_count) break;
            next = base;
            end = min(p_count, base + k);
            seen = base + k;
        }
        const unsigned long long p = a.p_begin + next++;
        const int n = a.in.n[p];
        const int y = a.in.y[p];
        const int G = (n + 31) >> 5;
        const int gs = G | 1;
        const uint32_t *src = a.in.ext + p * (size_t)a.in.stride;
        for (int i = (int)lane; i < n; i += 32) ids[i] = src[i];
        if (inherit)
            for (int i = (int)lane; i < a.wit_words; i += 32) witw[i] = src[a.wit_off + i];
        const uint32_t Bw = (int)lane < wm ? a.in.itt[p * wm + lane] : 0u;
        int nslots = 0;   // mid-pool children recorded in slots[]
        __syncwarp();

        // ---- restricted columns: per group g of 32 objects and row word w, one register transpose
        //      gives lane b the bits of attribute 32 w + b over the group. The rows of the next group
        //      (8 words at a time) are loaded while the current one is transposed.
        uint32_t held = 0;   // bit w: attribute 32 w + lane is held by some object of A
        const int chunks = (wm + 7) >> 3;
        const int steps = G * chunks;
        auto load8 = [&](int step, uint32_t (&v)[8]) {
            const int g = step / chunks, w0 = (step - g * chunks) * 8;
            const int i = 32 * g + (int)lane;
            const uint32_t *row = a.rows + (size_t)(i < n ? ids[i] : 0u) * wm + w0;
            if (wm == 8 && i < n) {   // one 32-byte row: two 16-byte loads
                const uint4 x = __ldg(reinterpret_cast<const uint4 *>(row));
                const uint4 y = __ldg(reinterpret_cast<const uint4 *>(row) + 1);
                v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
                v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
            } else {
#pragma unroll
                for (int t = 0; t < 8; ++t) v[t] = (i < n && w0 + t < wm) ? __ldg(row + t) : 0u;
            }
        };
        uint32_t nxt[8];
        load8(0, nxt);
        for (int step = 0; step < steps; ++step) {
            uint32_t v[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) v[t] = nxt[t];
            if (step + 1 < steps) load8(step + 1, nxt);
            const int g = step / chunks, w0 = (step - g * chunks) * 8;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                if (w0 + t < wm) {
                    const uint32_t col = warp_transpose32(v[t]);
                    const int k = 32 * (w0 + t) + (int)lane;
                    if (k < d.m) R[(size_t)k * gs + g] = col;
                    held |= (col != 0u ? 1u : 0u) << (w0 + t);
                }
            }
        }
        __syncwarp();
        if (COUNT && lane == 0) my_bytes += 4ull * n + 4ull * n * wm;   // the list and the rows of A

        // attributes whose subset test can succeed: held by some object of A and not in B (bit t of
        // `rel` is attribute 32 t + lane); attributes in B are in every child's intent
        uint32_t rel = held;
        for (int t = 0; t < wm; ++t)
            if ((__shfl_sync(FULL, Bw, t) >> lane) & 1u) rel &= ~(1u << t);
        // candidates: j >= y outside B (lane u holds word u)
        uint32_t cand = (int)lane < wm ? ~Bw & ge_mask((int)lane, y) : 0u;
        if ((int)lane == wm - 1) cand &= valid_last;

        for (;;) {
            const unsigned bal = __ballot_sync(FULL, cand != 0u);
            if (!bal) break;
            const int u = __ffs(bal) - 1;
            const uint32_t cw0 = __shfl_sync(FULL, cand, u);
            const int jb = __ffs(cw0) - 1;
            const int j = 32 * u + jb;
            if ((int)lane == u) cand &= cand - 1u;
            ++my_closures;
            // no object of A holds j: C is empty (its closure is the bottom, added by the host)
            if (!((__shfl_sync(FULL, held, jb) >> u) & 1u)) continue;
            // j failed at an ancestor whose extent holds A, its closure there containing the witness
            // k < j: while k stays outside B, j's closure here contains k too and j fails again
            if (inherit) {
                const unsigned w = wit[j];
                if (w != 0xffu && !((__shfl_sync(FULL, Bw, (int)(w >> 5)) >> (w & 31)) & 1u)) continue;
            }

            uint32_t c[GMAX];
            unsigned cnt = 0;
#pragma unroll
            for (int g = 0; g < GMAX; ++g) {
                c[g] = g < G ? R[(size_t)j * gs + g] : 0u;
                cnt += __popc(c[g]);
            }
            // the closure, 32 attributes per round in ascending order; a round at or below j's
            // word that puts an attribute below j into D ends the candidate
            uint32_t Dw = Bw | ((int)lane == u ? 1u << jb : 0u);
            bool canonical = true;
            for (int t = 0; t < wm; ++t) {
                bool in = false;
                const int k = 32 * t + (int)lane;
                if (((rel >> t) & 1u) && k != j) {
                    // every word at once (independent loads): C inside R[k]
                    const uint32_t *Rk = R + (size_t)k * gs;
                    uint32_t bad = 0u;
#pragma unroll
                    for (int g = 0; g < GMAX; ++g)
                        if (g < G) bad |= c[g] & ~Rk[g];
                    in = bad == 0u;
                }
                if (inherit) {
                    // the lowest attribute below j in the closure is the failure's witness
                    const uint32_t dt = __ballot_sync(FULL, in);
                    const uint32_t viol = t < u ? dt : (t == u ? dt & lt_mask(t, j) : 0u);
                    if (viol) {
                        if (lane == 0) wit[j] = (uint8_t)(32 * t + __ffs(viol) - 1);
                        canonical = false;
                        break;
                    }
                    if ((int)lane == t) Dw |= dt;
                    continue;
                }
                if (t < u) {
                    // a word below j's: any attribute of it in the closure (none is in B) ends j
                    if (__any_sync(FULL, in)) {
                        canonical = false;
                        break;
                    }
                    continue;
                }
                const uint32_t dt = __ballot_sync(FULL, in);
                if (t == u && (dt & lt_mask(t, j))) {
                    canonical = false;
                    break;
                }
                if ((int)lane == t) Dw |= dt;
            }
            if (!canonical) continue;
            if (inherit && lane == 0) wit[j] = 0xffu;

            // ---- emit the intent
            unsigned long long slot = 0;
            if (lane == 0) slot = atomicAdd(&a.ctr->out_count, 1ull);
            slot = __shfl_sync(FULL, slot, 0);
            if (slot < a.capacity && (int)lane < wm) a.out[slot * wm + lane] = Dw;
            if (COUNT && lane == 0)
                my_bytes += 4ull * wm + (cnt <= (unsigned)SMALL_MAX ? 4ull * queue_entry_words(cnt, wm)
                                                                    : 4ull * (cnt + wm + 2));

            // ---- the child (C, D, j+1): an object-list root, or an entry of the next level's mid pool.
            // A destination that is full only counts; the driver rolls the launch back and retries.
            const uint32_t cwl = (int)lane < G ? R[(size_t)j * gs + lane] : 0u;
            if (cnt <= (unsigned)SMALL_MAX) {
                const int qi = cnt <= 32u ? 0 : 1;
                const Queue &Q = a.q[qi];
                const int per = 32 << qi;
                unsigned long long s = 0;
                if (lane == 0) s = atomicAdd(&a.ctr->q_count[qi], 1ull);
                s = __shfl_sync(FULL, s, 0);
                if (s >= Q.cap) {
                    if (lane == 0) atomicOr(&a.ctr->error, ERR_QUEUE0 << qi);
                    continue;
                }
                write_ids(cwl, ids, Q.ids + s * per, cnt, per, lane);
                if ((int)lane < wm) Q.itt[s * wm + lane] = Dw;
                if (lane == 0) {
                    Q.y[s] = j + 1;
                    Q.n[s] = (int)cnt;
                }
            } else {
                // |C| <= |A| <= mid_max: the child belongs to the mid pool as well
                const Level &X = a.next_mid;
                unsigned long long s = 0;
                if (lane == 0) s = atomicAdd(&a.ctr->next_mid, 1ull);
                s = __shfl_sync(FULL, s, 0);
                if (s >= X.cap) {
                    if (lane == 0) atomicOr(&a.ctr->error, ERR_NEXT_MID);
                    continue;
                }
                write_ids(cwl, ids, X.ext + s * (size_t)X.stride, cnt, 0, lane);
                if ((int)lane < wm) X.itt[s * wm + lane] = Dw;
                if (lane == 0) {
                    X.y[s] = j + 1;
                    X.n[s] = (int)cnt;
                }
                // its inherited failures are written once every candidate of this entry is done
                // (past WIT_SLOTS children: none)
                if (inherit) {
                    if (nslots < WIT_SLOTS) {
                        if (lane == 0) slots[nslots] = (uint32_t)s;
                        ++nslots;
                    } else {
                        for (int i = (int)lane; i < a.wit_words; i += 32)
                            X.ext[s * (size_t)X.stride + a.wit_off + i] = FULL;
                    }
                }
            }
        }
        __syncwarp();
        if (inherit)
            for (int ci = 0; ci < nslots; ++ci) {
                uint32_t *dst = a.next_mid.ext + (size_t)slots[ci] * a.next_mid.stride + a.wit_off;
                for (int i = (int)lane; i < a.wit_words; i += 32) dst[i] = witw[i];
            }
        __syncwarp();   // ids, R and the witnesses are rewritten by the next entry
    }
    if (lane == 0) {
        if (my_closures) atomicAdd(&a.ctr->closures, my_closures);
        if (COUNT && my_bytes) atomicAdd(&a.ctr->bytes, my_bytes);
    }
}

// Words of restricted column a warp may hold per attribute, by M (the per-warp shared memory is
// M x (GMAX + 1) words plus the object ids).
int mid_gmax(int m) { return m <= 512 ? 8 : 4; }

template <bool COUNT, int GMAX, bool INHERIT>
int launch_mid_t(const ExpandArgs &a, int sm_count, void *stream)
{
    const size_t per_warp = MidLayout<GMAX>::words(a.d.m, a.wit_words) * 4;
    // warps per block: the shape with the most resident warps per SM (ties: the larger block)
    static thread_local ShapeCache cache;
    int dev = 0;
    cudaGetDevice(&dev);
    if (cache.dev != dev || cache.smem != per_warp) {
        int best_w = 0, best_wpb = 1, best_ps = 1;
        for (int wpb = 8; wpb >= 1; wpb >>= 1) {
            const size_t smem = per_warp * wpb;
            if (smem > 200 * 1024) continue;
            cudaError_t e = cudaFuncSetAttribute(expand_mid_kernel<COUNT, GMAX, INHERIT>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return (int)e;
            int ps = 0;
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ps, expand_mid_kernel<COUNT, GMAX, INHERIT>, wpb * 32, smem);
            if (ps * wpb > best_w) {
                best_w = ps * wpb;
                best_wpb = wpb;
                best_ps = ps;
            }
        }
        if (best_w == 0) return (int)cudaErrorInvalidConfiguration;
        cudaError_t e = cudaFuncSetAttribute(expand_mid_kernel<COUNT, GMAX, INHERIT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(per_warp * best_wpb));
        if (e != cudaSuccess) return (int)e;
        cache = ShapeCache{dev, per_warp, best_wpb, best_ps};
    }
    const int wpb = cache.wpb;
    const unsigned long long resident = (unsigned long long)sm_count * cache.per_sm;
    unsigned long long blocks = a.p_count_dev ? resident
                                              : std::min<unsigned long long>(resident, (a.p_count + wpb - 1) / wpb);
    if (blocks < 1) blocks = 1;
    expand_mid_kernel<COUNT, GMAX, INHERIT><<<(unsigned)blocks, wpb * 32, per_warp * wpb, (cudaStream_t)stream>>>(a);
    return (int)cudaGetLastError();
}

}  // namespace

int mid_max_for(const Dims &d)
{
    const int store = list_max_for(d);
    if (store <= SMALL_MAX) return 0;
    return std::min(32 * mid_gmax(d.m), store);
}

int launch_expand_mid(const ExpandArgs &a, int sm_count, void *stream)
{
    // inherited failures are kept only for M <= 256 (one byte per attribute), where GMAX is 8
    if (mid_gmax(a.d.m) == 8) {
        if (a.wit_words > 0)
            return a.count_work ? launch_mid_t<true, 8, true>(a, sm_count, stream)
                                : launch_mid_t<false, 8, true>(a, sm_count, stream);
        return a.count_work ? launch_mid_t<true, 8, false>(a, sm_count, stream)
                            : launch_mid_t<false, 8, false>(a, sm_count, stream);
    }
    return a.count_work ? launch_mid_t<true, 4, false>(a, sm_count, stream)
                        : launch_mid_t<false, 4, false>(a, sm_count, stream);
}

}  // namespace fca
