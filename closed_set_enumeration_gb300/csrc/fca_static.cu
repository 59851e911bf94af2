// An enumerate entry point that allocates nothing, for callers that may not call cudaMalloc.
//
// Some callers cannot allocate device memory while they run: a process whose device memory is
// owned entirely by another allocator (a framework's caching allocator, or a fixed-budget arena
// reserved at start-up), or a latency-critical loop where cudaMalloc and cudaFree, which can
// synchronize the whole device and fail under memory pressure, are not allowed. For small
// contexts (at most STATIC_MAX_OBJECTS objects, so the whole search is one object-list subtree)
// fca_enumerate_small_noalloc runs the object-list kernel with all of its scratch - the work
// counters, a copy of the rows, the single subtree root and the bottom intent - in one
// file-scope device array. The caller passes the rows and the output buffer; nothing is
// allocated or freed.
//
// Every GPU that loads the library holds this array (STATIC_SCRATCH_WORDS words, under 10 KB)
// until the process exits. All calls on a device share it and each call starts by rewriting it,
// so calls whose GPU work overlaps in time (on different streams or host threads) race on it.
// The array's device address is looked up once per device and kept: a cudaDeviceReset unloads the
// module that holds it (and frees every context of the library on that device), so the library is
// not to be used on a device after a reset.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "fca.h"
#include "fca_internal.cuh"

using namespace fca;

namespace {

constexpr int STATIC_MAX_OBJECTS = 64;                 // one subtree root of the 1- or 2-word tier
constexpr int STATIC_MAX_WORDS = MAX_ATTRS / 32;       // intent words
constexpr int MAX_DEVICES = 64;

// Word offsets inside the scratch array.
constexpr int OFF_CTR = 0;                                             // Counters (128 bytes)
constexpr int OFF_FLAG = 32;                                           // some row holds every attribute
constexpr int OFF_ROWS = 64;                                           // rows, padding cleared
constexpr int OFF_IDS = OFF_ROWS + STATIC_MAX_OBJECTS * STATIC_MAX_WORDS;
constexpr int OFF_ITT = OFF_IDS + STATIC_MAX_OBJECTS;                  // root intent = top intent
constexpr int OFF_Y = OFF_ITT + STATIC_MAX_WORDS;                      // root cursor
constexpr int OFF_N = OFF_Y + 1;                                       // root object count
constexpr int OFF_FULL = OFF_N + 1;                                    // every attribute (bottom)
constexpr int STATIC_SCRATCH_WORDS = OFF_FULL + STATIC_MAX_WORDS;

static_assert(sizeof(Counters) <= OFF_FLAG * 4, "counters overlap the flag word");

static __device__ __align__(256) uint32_t fca_static_scratch[STATIC_SCRATCH_WORDS];

std::mutex g_lock;
uint32_t *g_scratch[MAX_DEVICES] = {};

// One block: clear the counters (the top intent holds output row 0), clear the padding bits of
// the copied rows, compute the top intent and the full-row flag, write the single subtree root.
__global__ void static_setup_kernel(uint32_t *s, int n, int m, uint32_t *out, unsigned long long capacity)
{
    const int wm = (m + 31) / 32;
    const int t = threadIdx.x;
    uint32_t *rows = s + OFF_ROWS;
    if (t < OFF_ROWS) s[t] = 0u;
    __syncthreads();
    if (t == 0) reinterpret_cast<Counters *>(s + OFF_CTR)->out_count = 1ull;
    const uint32_t last = (m & 31) ? ((1u << (m & 31)) - 1u) : 0xffffffffu;
    if (t < n) rows[t * wm + wm - 1] &= last;
    __syncthreads();
    if (t < wm) {
        const uint32_t mask = t == wm - 1 ? last : 0xffffffffu;
        uint32_t top = mask;
        for (int o = 0; o < n; ++o) top &= rows[o * wm + t];
        s[OFF_ITT + t] = top;
        s[OFF_FULL + t] = mask;
        if (capacity >= 1ull) out[t] = top;
    }
    if (t < n) {
        bool full = true;
        for (int w = 0; w < wm; ++w) {
            const uint32_t mask = w == wm - 1 ? last : 0xffffffffu;
            full = full && rows[t * wm + w] == mask;
        }
        if (full) atomicOr(s + OFF_FLAG, 1u);
    }
    if (t < STATIC_MAX_OBJECTS) s[OFF_IDS + t] = t < n ? (uint32_t)t : 0u;
    if (t == 0) {
        s[OFF_Y] = 0u;
        s[OFF_N] = (uint32_t)n;
    }
}

}  // namespace

extern "C" fca_status fca_enumerate_small_noalloc(const uint32_t *rows, int64_t n_objects, int32_t n_attrs,
                                                  uint32_t *out, uint64_t capacity, uint64_t *out_count,
                                                  void *stream)
{
    if (!rows || !out_count || (capacity > 0 && !out) || n_objects < 1 ||
        n_objects > STATIC_MAX_OBJECTS || n_attrs < 1 || n_attrs > MAX_ATTRS)
        return FCA_ERR_INVALID;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FCA_ERR_CUDA;
    // set-up, once per device, with that device current: the device address of the scratch array
    // (in host code its name is only a host-side stand-in)
    uint32_t *s = nullptr;
    {
        std::lock_guard<std::mutex> g(g_lock);
        if (!g_scratch[dev]) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, fca_static_scratch) != cudaSuccess) {
                cudaGetLastError();
                return FCA_ERR_CUDA;
            }
            g_scratch[dev] = static_cast<uint32_t *>(p);
        }
        s = g_scratch[dev];
    }
    cudaStream_t st = (cudaStream_t)stream;
    const int n = (int)n_objects, m = n_attrs, wm = (m + 31) / 32;
    if (cudaMemcpyAsync(s + OFF_ROWS, rows, (size_t)n * wm * 4, cudaMemcpyDefault, st) != cudaSuccess)
        return FCA_ERR_CUDA;
    static_setup_kernel<<<1, 256, 0, st>>>(s, n, m, out, capacity);
    if (cudaGetLastError() != cudaSuccess) return FCA_ERR_CUDA;

    SubtreeArgs a{};
    a.d.n = n;
    a.d.m = m;
    a.d.wm = wm;
    a.d.wn = (n + 31) / 32;
    a.d.wnp = (a.d.wn + 3) & ~(int64_t)3;
    a.rows = s + OFF_ROWS;
    a.q.ids = s + OFF_IDS;
    a.q.itt = s + OFF_ITT;
    a.q.y = reinterpret_cast<int32_t *>(s + OFF_Y);
    a.q.n = reinterpret_cast<int32_t *>(s + OFF_N);
    a.q.cap = 1;
    a.q_count = 1;
    a.q_index = 0;
    a.out = out;
    a.capacity = capacity;
    a.ctr = reinterpret_cast<Counters *>(s + OFF_CTR);
    a.count_work = 0;
    if (launch_subtree(a, n <= 32 ? 1 : 2, sms, st) != (int)cudaSuccess) return FCA_ERR_CUDA;

    // counters and the full-row flag back to the host (a local variable: no host allocation)
    uint32_t head[OFF_ROWS];
    if (cudaMemcpyAsync(head, s, sizeof head, cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return FCA_ERR_CUDA;
    Counters ctr;
    memcpy(&ctr, head + OFF_CTR, sizeof ctr);
    if (ctr.fault) return FCA_ERR_CUDA;
    uint64_t total = ctr.out_count;
    // the bottom concept, when no object holds every attribute (its extent is then empty)
    if (head[OFF_FLAG] == 0u) {
        if (total < capacity &&
            cudaMemcpyAsync(out + total * wm, s + OFF_FULL, (size_t)wm * 4, cudaMemcpyDeviceToDevice, st) !=
                cudaSuccess)
            return FCA_ERR_CUDA;
        total += 1;
        if (cudaStreamSynchronize(st) != cudaSuccess) return FCA_ERR_CUDA;
    }
    *out_count = total;
    return total > capacity ? FCA_ERR_CAPACITY : FCA_OK;
}
