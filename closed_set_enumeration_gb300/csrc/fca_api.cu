// C ABI and host driver of libfca.
//
// The driver runs the Close-by-One search level by level (Parallel FCBO
// article, section 2.1: a level is expanded in one launch over all its
// (parent, j) pairs, and the loop ends when no level holds work). A level is
// launched optimistically into the current pools; when a destination turns
// out too small, the launch is rolled back (the device counters are restored
// from the copy taken before it, so everything it appended is dropped) and
// retried after the destination was emptied (queues run, levels drained depth
// first) or grown, up to a memory limit beyond which the level is split into
// smaller chunks. Storage therefore stays bounded (the memory concern of the
// FCbO-to-CUDA article, sections 3.4 and 6.1), and no global dedupe is needed
// because the canonical test is local (section 2.2).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstddef>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <utility>
#include <vector>

#include "fca.h"
#include "fca_internal.cuh"

using namespace fca;

struct fca_ctx {
    int device = 0;
    int sm_count = 0;
    Dims d{};
    uint32_t *rows = nullptr;      // n x wm
    uint32_t *cols = nullptr;      // m x wnp, in processing order (one of cols_buf)
    uint32_t *top = nullptr;       // wm, in processing order (one of top_buf)
    // Processing order of the attributes (fca_set_option FCA_OPT_ATTR_ORDER: 0 attribute order, 1
    // ascending support when the supports vary, 2 ascending support): the table kernels write
    // cols_buf[0] and top_buf[0] in attribute order; in support order the permuted tables are
    // cols_buf[1], top_buf[1] and the rows (overwritten), and every output intent is mapped back at
    // the end of a call.
    uint32_t *cols_buf[2]{};
    uint32_t *top_buf[2]{};
    uint32_t *sup = nullptr;        // m: attribute supports
    int32_t *perm = nullptr;        // m: attribute -> position
    int32_t *inv = nullptr;         // m: position -> attribute
    int attr_order = 1;             // the option
    bool decide = true;             // the next table load chooses the order (from its supports)
    bool use_order = false;         // the choice: support order
    bool ordered = false;           // the tables in use are in support order
    uint32_t *full_mask = nullptr; // wm: every attribute (the bottom intent)
    uint32_t *root_ext = nullptr;  // wnp: every object
    uint32_t *botext = nullptr;    // wn: objects holding every attribute (the bottom extent)

    // work pools, allocated on first use, grown on demand and kept for later calls
    std::vector<Level> levels;        // per level: the big pool (slots of W_Np words)
    std::vector<Level> mids;          // per level: the mid pool (slots of mid_stride words; cap 0 when
                                      // there is no mid tier)
    std::vector<uint64_t> level_count, mid_count;   // entries waiting in each pool
    Queue q[NQ]{};
    // roots spilled by object-list searches that ran past their time budget, per queue width; two
    // sets, used in turn by the rounds that search them (spill_rounds)
    Queue spq[2][NQ]{};
    uint64_t q_count[NQ]{};
    Counters *ctr = nullptr;        // device
    Counters *ctr_snap = nullptr;   // device copy taken before each bitmap-tier launch (rollback)
    Counters *ctr_host = nullptr;   // pinned host copy, read after each bitmap-tier launch
    ChainSlots *chain = nullptr;        // device records of a chain of bitmap-tier launches
    ChainSlots *chain_host = nullptr;   // pinned host copy
    // parents per bitmap level in the last call and its number of levels: they set how many levels
    // are launched as one chain, and the launch shapes of the chained launches
    std::vector<uint64_t> prev_counts, cur_counts;   // big-pool parents per level
    std::vector<uint64_t> prev_mids, cur_mids;       // mid-pool parents per level
    uint64_t prev_levels = 0;
    uint64_t prev_q[NQ]{}, last_q[NQ]{};   // roots of the last object-list launches (last call, this one)

    uint32_t *host_out_dev = nullptr;   // device buffer behind fca_enumerate_host
    uint64_t host_out_rows = 0;

    size_t pool_bytes = 0;          // bytes held by levels and queues
    size_t pool_limit = 0;          // growth stops here; levels are then split into chunks
    uint64_t level_bytes = 0, queue_entries = 0;   // initial pool sizes
    int count_work = 0;
    // growth ahead of a level launch (unchained levels): the destinations are grown to what the
    // previous launch's children per parent predict for this one, so that a first call on a table
    // does not overflow and re-run most of its levels (FCA_PREGROW=0 turns it off)
    int pregrow = 1;
    bool ratio_known = false;
    size_t ratio_lv = 0;            // level whose launch gave the ratios
    double ratio_big = 0, ratio_mid = 0, ratio_q[NQ]{};
    // extents of SMALL_MAX < n <= list_max objects are stored as object-id lists; those of at most
    // mid_max objects are kept in the mid pools (slots of mid_stride words) and expanded one per warp
    // by the mid-tier kernel (0: off)
    int list_max = 0, mid_max = 0;
    int64_t mid_stride = 0;
    // inherited failures (M <= 256: one byte per attribute) kept in every level entry after its
    // extent: at word wit_off of a mid-pool slot, at word wnp of a big-pool slot (big_stride words)
    int wit_off = 0, wit_words = 0;
    int64_t big_stride = 0;
    uint64_t mid_min = 0;           // smallest mid-pool launch given to the mid-tier kernel
    uint64_t wait_ns = 0;           // bound of a work-sharing wait (0: the kernels' default)
    uint64_t table_launches = 0;    // kernels launched by the last table load

    // a second stream for the object-list launch that runs beside the other one
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    cudaEvent_t lat_ev[2]{};        // around the kernels of the last lattice call
    bool lat_timed = false;

    // device timing of kernel launches: event pairs recorded around each launch
    std::vector<cudaEvent_t> events;
    std::vector<int> event_kind;    // per pair: 0 = bitmap-tier expand, 1 = subtree, 2 = mid-tier expand
    size_t pairs_used = 0;

    fca_stats stats{};
    std::string err;
};

namespace {

const char *kStatus[] = {"ok", "invalid argument", "out of memory", "capacity exceeded",
                         "CUDA error"};

fca_status cuda_fail(fca_ctx *c, cudaError_t e, const char *what)
{
    if (c) {
        char buf[256];
        snprintf(buf, sizeof buf, "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
        c->err = buf;
    }
    return e == cudaErrorMemoryAllocation ? FCA_ERR_OOM : FCA_ERR_CUDA;
}

#define CK(call, what)                                        \
    do {                                                      \
        cudaError_t e_ = (call);                              \
        if (e_ != cudaSuccess) return cuda_fail(c, e_, what); \
    } while (0)

// Smallest coefficient of variation of the attribute supports for which option 1 of
// FCA_OPT_ATTR_ORDER takes the support order.
constexpr double ORDER_MIN_CV = 0.25;

// Time budget of one object-list search, in SM clock cycles (about 100 us): a search running
// longer spills its unexplored nodes as new roots, searched in parallel by a following launch.
constexpr long long SEARCH_BUDGET_CYCLES = 200000;
// Roots each spill queue holds.
constexpr uint64_t SPILL_CAP = 1ull << 16;
// Levels of at least this many parents are first launched on an eighth of them when their children
// per parent are not known yet (the first call on a table)
constexpr uint64_t PROBE_MIN_PARENTS = 1ull << 16;

uint64_t env_u64(const char *name, uint64_t dflt)
{
    const char *v = getenv(name);
    if (!v || !*v) return dflt;
    char *end = nullptr;
    unsigned long long x = strtoull(v, &end, 10);
    return (end && *end == 0 && x > 0) ? (uint64_t)x : dflt;
}

fca_status alloc_raw(fca_ctx *c, void **p, size_t bytes, const char *what)
{
    cudaError_t e = cudaMalloc(p, bytes ? bytes : 16);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        c->err = std::string("cudaMalloc failed for ") + what;
        return FCA_ERR_OOM;
    }
    return FCA_OK;
}

uint64_t level_entry_bytes(const fca_ctx *c) { return ((uint64_t)c->big_stride + c->d.wm + 2) * 4; }
uint64_t mid_entry_bytes(const fca_ctx *c) { return ((uint64_t)c->mid_stride + c->d.wm + 2) * 4; }
uint64_t queue_entry_bytes(const Dims &d, int qi) { return ((uint64_t)(32 << qi) + d.wm + 2) * 4; }

uint64_t initial_level_cap(const fca_ctx *c)
{
    return std::max<uint64_t>(4 * (uint64_t)c->d.m, c->level_bytes / level_entry_bytes(c));
}

uint64_t initial_mid_cap(const fca_ctx *c)
{
    return std::max<uint64_t>(4 * (uint64_t)c->d.m, c->level_bytes / mid_entry_bytes(c));
}

uint64_t initial_queue_cap(const fca_ctx *c) { return std::max<uint64_t>(4 * (uint64_t)c->d.m, c->queue_entries); }

void free_level(Level &L)
{
    cudaFree(L.ext);
    cudaFree(L.itt);
    cudaFree(L.y);
    cudaFree(L.n);
    L = Level{};
}

void free_queue(Queue &Q)
{
    cudaFree(Q.ids);
    cudaFree(Q.itt);
    cudaFree(Q.y);
    cudaFree(Q.n);
    Q = Queue{};
}

void free_pools(fca_ctx *c)
{
    for (Level &L : c->levels) free_level(L);
    for (Level &L : c->mids) free_level(L);
    c->levels.clear();
    c->mids.clear();
    c->level_count.clear();
    c->mid_count.clear();
    for (Queue &Q : c->q) free_queue(Q);
    for (int k = 0; k < 2; ++k)
        for (Queue &Q : c->spq[k]) free_queue(Q);
    c->pool_bytes = 0;
}

fca_status make_level(fca_ctx *c, Level *L, uint64_t cap, int64_t stride)
{
    const Dims &d = c->d;
    // the level kernels record child slots in 31 bits (the inherited-failure patch lists)
    if (cap >= (1ull << 31)) {
        c->err = "level pool capacity past 2^31 entries";
        return FCA_ERR_OOM;
    }
    Level n{};
    n.cap = cap;
    n.stride = stride;
    fca_status s;
    if ((s = alloc_raw(c, (void **)&n.ext, cap * stride * 4, "frontier extents")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&n.itt, cap * d.wm * 4, "frontier intents")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&n.y, cap * 4, "frontier cursors")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&n.n, cap * 4, "frontier sizes")) != FCA_OK) {
        free_level(n);
        return s;
    }
    *L = n;
    return FCA_OK;
}

fca_status make_queue(fca_ctx *c, Queue *Q, int qi, uint64_t cap)
{
    const Dims &d = c->d;
    Queue n{};
    n.cap = cap;
    fca_status s;
    if ((s = alloc_raw(c, (void **)&n.ids, cap * (32 << qi) * 4, "queue ids")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&n.itt, cap * d.wm * 4, "queue intents")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&n.y, cap * 4, "queue cursors")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&n.n, cap * 4, "queue sizes")) != FCA_OK) {
        free_queue(n);
        return s;
    }
    *Q = n;
    return FCA_OK;
}

fca_status ensure_level(fca_ctx *c, size_t idx)
{
    while (c->levels.size() <= idx) {
        const uint64_t cap = initial_level_cap(c);
        Level L{}, M{};
        fca_status s = make_level(c, &L, cap, c->big_stride);
        if (s != FCA_OK) return s;
        c->pool_bytes += cap * level_entry_bytes(c);
        if (c->mid_max > SMALL_MAX) {
            const uint64_t mcap = initial_mid_cap(c);
            if ((s = make_level(c, &M, mcap, c->mid_stride)) != FCA_OK) {
                free_level(L);
                return s;
            }
            c->pool_bytes += mcap * mid_entry_bytes(c);
        }
        c->levels.push_back(L);
        c->mids.push_back(M);
        c->level_count.push_back(0);
        c->mid_count.push_back(0);
    }
    return FCA_OK;
}

fca_status ensure_queues(fca_ctx *c)
{
    for (int k = 0; k < 2; ++k)
        for (int qi = 0; qi < NQ; ++qi) {
            if (c->spq[k][qi].ids) continue;
            fca_status s = make_queue(c, &c->spq[k][qi], qi, SPILL_CAP);
            if (s != FCA_OK) return s;
        }
    for (int qi = 0; qi < NQ; ++qi) {
        if (c->q[qi].ids) continue;
        const uint64_t cap = initial_queue_cap(c);
        fca_status s = make_queue(c, &c->q[qi], qi, cap);
        if (s != FCA_OK) return s;
        c->pool_bytes += cap * queue_entry_bytes(c->d, qi);
    }
    return FCA_OK;
}

// Grow a pool of level `idx` (the mid pool when `mid`) to hold at least `need` entries, keeping its
// current entries. Returns FCA_ERR_CAPACITY (nothing changed) when that would pass the pool limit.
fca_status grow_level(fca_ctx *c, size_t idx, bool mid, uint64_t need, cudaStream_t st, size_t limit = 0)
{
    Level &L = mid ? c->mids[idx] : c->levels[idx];
    constexpr uint64_t CAP_MAX = (1ull << 31) - 1;   // see make_level
    if (need > CAP_MAX) return FCA_ERR_CAPACITY;
    // an overflow grows with headroom; a growth ahead of a launch (limit given) to the prediction
    const uint64_t cap = limit ? need : std::min<uint64_t>(CAP_MAX, std::max<uint64_t>(2 * L.cap, need + need / 4));
    const uint64_t eb = mid ? mid_entry_bytes(c) : level_entry_bytes(c);
    if (c->pool_bytes + (cap - L.cap) * eb > (limit ? limit : c->pool_limit)) return FCA_ERR_CAPACITY;
    Level n{};
    fca_status s = make_level(c, &n, cap, L.stride);
    if (s != FCA_OK) return s;
    const uint64_t cnt = mid ? c->mid_count[idx] : c->level_count[idx];
    const Dims &d = c->d;
    CK(cudaMemcpyAsync(n.ext, L.ext, cnt * L.stride * 4, cudaMemcpyDeviceToDevice, st), "level grow");
    CK(cudaMemcpyAsync(n.itt, L.itt, cnt * d.wm * 4, cudaMemcpyDeviceToDevice, st), "level grow");
    CK(cudaMemcpyAsync(n.y, L.y, cnt * 4, cudaMemcpyDeviceToDevice, st), "level grow");
    CK(cudaMemcpyAsync(n.n, L.n, cnt * 4, cudaMemcpyDeviceToDevice, st), "level grow");
    CK(cudaStreamSynchronize(st), "stream synchronize");
    c->pool_bytes += (cap - L.cap) * eb;
    free_level(L);
    L = n;
    return FCA_OK;
}

// Grow (empty) queue qi to hold at least `need` entries.
fca_status grow_queue(fca_ctx *c, int qi, uint64_t need, cudaStream_t st, size_t limit = 0)
{
    Queue &Q = c->q[qi];
    const uint64_t cap = limit ? need : std::max<uint64_t>(2 * Q.cap, need + need / 4);
    const uint64_t eb = queue_entry_bytes(c->d, qi);
    if (c->pool_bytes + (cap - Q.cap) * eb > (limit ? limit : c->pool_limit)) return FCA_ERR_CAPACITY;
    Queue n{};
    fca_status s = make_queue(c, &n, qi, cap);
    if (s != FCA_OK) return s;
    // keep the roots waiting in the queue
    const uint64_t cnt = c->q_count[qi];
    if (cnt) {
        const Dims &d = c->d;
        CK(cudaMemcpyAsync(n.ids, Q.ids, cnt * (32u << qi) * 4, cudaMemcpyDeviceToDevice, st), "queue grow");
        CK(cudaMemcpyAsync(n.itt, Q.itt, cnt * d.wm * 4, cudaMemcpyDeviceToDevice, st), "queue grow");
        CK(cudaMemcpyAsync(n.y, Q.y, cnt * 4, cudaMemcpyDeviceToDevice, st), "queue grow");
        CK(cudaMemcpyAsync(n.n, Q.n, cnt * 4, cudaMemcpyDeviceToDevice, st), "queue grow");
        CK(cudaStreamSynchronize(st), "stream synchronize");
    }
    c->pool_bytes += (cap - Q.cap) * eb;
    free_queue(Q);
    Q = n;
    return FCA_OK;
}

struct Run {
    fca_ctx *c;
    uint32_t *out;
    uint64_t capacity;
    cudaStream_t st;
};

// Record the start event of a timed launch; returns the pair index.
fca_status time_begin(Run &r, int kind, size_t *pair, cudaStream_t st)
{
    fca_ctx *c = r.c;
    if (c->pairs_used == c->event_kind.size()) {
        cudaEvent_t e0, e1;
        CK(cudaEventCreate(&e0), "cudaEventCreate");
        CK(cudaEventCreate(&e1), "cudaEventCreate");
        c->events.push_back(e0);
        c->events.push_back(e1);
        c->event_kind.push_back(0);
    }
    *pair = c->pairs_used++;
    c->event_kind[*pair] = kind;
    CK(cudaEventRecord(c->events[2 * *pair], st), "cudaEventRecord");
    return FCA_OK;
}

fca_status time_end(Run &r, size_t pair, cudaStream_t st)
{
    fca_ctx *c = r.c;
    CK(cudaEventRecord(c->events[2 * pair + 1], st), "cudaEventRecord");
    return FCA_OK;
}

// The device times of the launches recorded by the last call (read when statistics are asked for,
// so that a call does not wait on them), per kind of kernel in ms: the length of the union of the
// launches' intervals, so that launches that run side by side on two streams count once.
void launch_times(const fca_ctx *c, double *expand_ms, double *subtree_ms, double *mid_ms)
{
    *expand_ms = *subtree_ms = *mid_ms = 0.0;
    if (c->pairs_used == 0) return;
    std::vector<std::pair<float, float>> iv[3];
    for (size_t i = 0; i < c->pairs_used; ++i) {
        float t0 = 0.f, t1 = 0.f;
        if (cudaEventElapsedTime(&t0, c->events[0], c->events[2 * i]) != cudaSuccess ||
            cudaEventElapsedTime(&t1, c->events[0], c->events[2 * i + 1]) != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        const int k = c->event_kind[i];
        if (k >= 0 && k < 3) iv[k].emplace_back(t0, t1);
    }
    double *dst[3] = {expand_ms, subtree_ms, mid_ms};
    for (int k = 0; k < 3; ++k) {
        std::sort(iv[k].begin(), iv[k].end());
        double total = 0.0;
        float lo = 0.f, hi = 0.f;
        bool open = false;
        for (const auto &v : iv[k]) {
            if (open && v.first <= hi) {
                hi = std::max(hi, v.second);
                continue;
            }
            if (open) total += hi - lo;
            lo = v.first;
            hi = v.second;
            open = true;
        }
        if (open) total += hi - lo;
        *dst[k] = total;
    }
}

fca_status read_counters(Run &r)
{
    fca_ctx *c = r.c;
    CK(cudaMemcpyAsync(c->ctr_host, c->ctr, sizeof(Counters), cudaMemcpyDeviceToHost, r.st),
       "counter readback");
    CK(cudaStreamSynchronize(r.st), "stream synchronize");
    return FCA_OK;
}

// Process every root waiting in object-list queue qi, then empty it; all on stream `st`. `share`
// allows the launch to hand work between the warps of a block (see subtree_kernel).
// With `guarded`, the root count is read on the device and the launch does nothing unless the
// bitmap search ended cleanly (a launch queued before the host knew; see SubtreeArgs::guard).
fca_status run_subtree(Run &r, int qi, cudaStream_t st, bool share = true, bool reset = true, bool guarded = false)
{
    fca_ctx *c = r.c;
    if (!guarded && c->q_count[qi] == 0) return FCA_OK;
    const int nw = 1 << qi;
    fca_status s;
    SubtreeArgs a{};
    a.d = c->d;
    a.rows = c->rows;
    a.q = c->q[qi];
    a.q_count = guarded ? std::max<uint64_t>(1, c->prev_q[qi]) : c->q_count[qi];
    a.q_count_dev = guarded ? &c->ctr->q_count[qi] : nullptr;
    a.guard = guarded ? 1 : 0;
    a.q_index = qi;
    a.out = r.out;
    a.capacity = r.capacity;
    a.ctr = c->ctr;
    a.count_work = c->count_work;
    a.share = share ? 1 : 0;
    a.budget = SEARCH_BUDGET_CYCLES;
    a.wait_ns = c->wait_ns;
    a.spill = c->spq[0][qi];
    size_t pair = 0;
    if ((s = time_begin(r, 1, &pair, st)) != FCA_OK) return s;
    CK((cudaError_t)launch_subtree(a, nw, c->sm_count, st), "subtree kernel launch");
    if ((s = time_end(r, pair, st)) != FCA_OK) return s;
    c->stats.launches++;
    c->stats.subtree_launches++;
    if (!guarded) {
        c->stats.small_roots += c->q_count[qi];
        c->last_q[qi] = c->q_count[qi];
    }
    // empty the queue: its append counter and its work cursor (not needed after the last launches
    // of a call: the next call starts from zeroed counters)
    if (reset) {
        CK(cudaMemsetAsync(&c->ctr->q_count[qi], 0, sizeof(unsigned long long), st), "queue reset");
        CK(cudaMemsetAsync(&c->ctr->q_head[qi], 0, sizeof(unsigned long long), st), "queue reset");
    }
    c->q_count[qi] = 0;
    return FCA_OK;
}

void count_level(fca_ctx *c, size_t lv, uint64_t kb, uint64_t km)
{
    if (c->cur_counts.size() <= lv) c->cur_counts.resize(lv + 1, 0);
    if (c->cur_mids.size() <= lv) c->cur_mids.resize(lv + 1, 0);
    c->cur_counts[lv] += kb;
    c->cur_mids[lv] += km;
    c->stats.large_parents += kb + km;
    c->stats.levels = std::max<uint64_t>(c->stats.levels, lv + 2);
}

fca_status drain(Run &r, size_t lv, bool chain = true);

// Mid-pool parents per SM below which a level's mid pool is expanded by the block-wide kernel
// instead (it reads id lists as well): with fewer parents than about twice the warps the mid-tier
// kernel keeps resident, a launch lasts as long as its slowest parent searched by a single warp,
// while a block of 8 to 16 warps takes one parent's candidates together. Measured on zipf, whose mid
// levels hold at most 3 769 parents: 0.90 ms of mid-tier launches per enumeration against ... with
// blocks. FCA_MID_MIN (parents) in the environment replaces the bound (1: every mid level).
constexpr uint64_t MID_MIN_PARENTS_PER_SM = 32;

// Launch one level (or a chunk of it): mid-pool parents [bm, bm + km) and big-pool parents
// [bb, bb + kb), both writing into level lv + 1 and the object-list queues. The mid pool goes to the
// mid-tier kernel (one parent per warp) when it holds enough parents to fill the GPU, else to the
// block-wide kernel like the big pool. With `chain_i` >= 1 the parent counts are read on the device
// (the launch is queued behind the one that produces its level: km and kb are then the last call's
// counts, used for the launch shapes; a kernel without parents returns at once). Each kernel is
// timed by its own pair of events.
fca_status launch_level(Run &r, size_t lv, uint64_t bb, uint64_t kb, uint64_t bm, uint64_t km, int chain_i)
{
    fca_ctx *c = r.c;
    fca_status s;
    size_t pair = 0;
    ExpandArgs a{};
    a.d = c->d;
    a.rows = c->rows;
    a.cols = c->cols;
    a.next = c->levels[lv + 1];
    a.next_mid = c->mids[lv + 1];
    for (int qi = 0; qi < NQ; ++qi) a.q[qi] = c->q[qi];
    a.out = r.out;
    a.capacity = r.capacity;
    a.ctr = c->ctr;
    a.count_work = c->count_work;
    a.list_max = c->list_max;
    a.mid_max = c->mid_max;
    a.wit_off = c->wit_off;
    a.wit_words = c->wit_words;
    a.wit_off_big = (int)c->d.wnp;
    const bool on_device = chain_i >= 1;
    const bool has_mid = c->mid_max > SMALL_MAX && (km > 0 || on_device);
    const bool warps = has_mid && km >= c->mid_min;
    if (warps) {
        ExpandArgs m = a;
        m.in = c->mids[lv];
        m.p_begin = bm;
        m.p_count = std::max<uint64_t>(1, km);
        m.p_count_dev = on_device ? &c->chain->pcount_mid : nullptr;
        if ((s = time_begin(r, 2, &pair, r.st)) != FCA_OK) return s;
        CK((cudaError_t)launch_expand_mid(m, c->sm_count, r.st), "mid kernel launch");
        if ((s = time_end(r, pair, r.st)) != FCA_OK) return s;
        c->stats.launches++;
        c->stats.mid_launches++;
    } else if (has_mid) {
        // a small mid pool goes to the block-wide kernel, in the big pool's launch
        a.in2 = c->mids[lv];
        a.p_begin2 = bm;
        a.p_count2 = km;
        a.p_count2_dev = on_device ? &c->chain->pcount_mid : nullptr;
    }
    if (kb > 0 || on_device || (has_mid && !warps)) {
        a.in = c->levels[lv];
        a.p_begin = bb;
        a.p_count = kb;
        a.p_count_dev = on_device ? &c->chain->pcount : nullptr;
        if ((s = time_begin(r, 0, &pair, r.st)) != FCA_OK) return s;
        CK((cudaError_t)launch_expand(a, c->sm_count, r.st), "expand kernel launch");
        if ((s = time_end(r, pair, r.st)) != FCA_OK) return s;
        c->stats.launches++;
        c->stats.expand_launches++;
    }
    return FCA_OK;
}

bool level_empty(const fca_ctx *c, size_t lv)
{
    return lv >= c->levels.size() || (c->level_count[lv] == 0 && c->mid_count[lv] == 0);
}

// Launch levels lv .. lv+K-1 (level lv whole, the next level empty) back to back, each reading its
// parent counts on the device, and read the counters once at the end. Launches up to the first that
// overflowed are committed; that one's counters as they were before it are restored and *failed
// is set. *next_lv is the first level still holding parents.
fca_status enqueue_chain(Run &r, size_t lv, int K)
{
    fca_ctx *c = r.c;
    fca_status s;
    for (int i = 0; i < K; ++i)
        if ((s = ensure_level(c, lv + i + 1)) != FCA_OK) return s;
    const uint64_t n0 = c->level_count[lv], m0 = c->mid_count[lv];
    for (int i = 0; i < K; ++i) {
        const size_t L = lv + i;
        CK((cudaError_t)launch_prepare_chain(c->ctr, c->chain, i, n0, m0, r.st), "chain set-up kernel");
        c->stats.launches++;
        // launch shapes of the device-counted launches: the last call's counts of the level
        const uint64_t eb = i == 0 ? n0 : (L < c->prev_counts.size() ? c->prev_counts[L] : n0);
        const uint64_t em = i == 0 ? m0 : (L < c->prev_mids.size() ? c->prev_mids[L] : m0);
        if ((s = launch_level(r, L, 0, eb, 0, em, i)) != FCA_OK) return s;
    }
    return FCA_OK;
}

// Read back the records of a chain queued by enqueue_chain (and the counters, after whatever was
// queued behind it), commit it up to the first launch that overflowed, and restore that one.
fca_status collect_chain(Run &r, size_t lv, int K, size_t *next_lv, bool *failed)
{
    fca_ctx *c = r.c;
    CK(cudaMemcpyAsync(c->chain_host, c->chain, sizeof(ChainSlots), cudaMemcpyDeviceToHost, r.st), "chain read-back");
    CK(cudaMemcpyAsync(c->ctr_host, c->ctr, sizeof(Counters), cudaMemcpyDeviceToHost, r.st), "counter readback");
    CK(cudaStreamSynchronize(r.st), "stream synchronize");
    const ChainSlots &cs = *c->chain_host;
    const Counters &fin = *c->ctr_host;
    int f = -1;   // the first launch after which the error word was set
    for (int i = 0; i < K && f < 0; ++i)
        if ((i + 1 < K ? cs.snaps[i + 1].error : fin.error) != 0u) f = i;
    const int ok = f < 0 ? K : f;
    for (int i = 0; i < ok; ++i) {
        count_level(c, lv + i, cs.counts[i], cs.mcounts[i]);
        const uint64_t produced = i + 1 < K ? cs.counts[i + 1] + cs.mcounts[i + 1] : fin.next_count + fin.next_mid;
        c->stats.max_frontier = std::max<uint64_t>(c->stats.max_frontier, produced);
        c->level_count[lv + i] = 0;
        c->mid_count[lv + i] = 0;
    }
    if (f < 0) {
        c->level_count[lv + K] = fin.next_count;
        c->mid_count[lv + K] = fin.next_mid;
        for (int qi = 0; qi < NQ; ++qi) c->q_count[qi] = fin.q_count[qi];
        *next_lv = lv + K;
        *failed = false;
        return FCA_OK;
    }
    // launch f overflowed a destination: the counters come back as they were before it, its parents
    // wait again in level lv+f, and the caller continues there launch by launch
    CK(cudaMemcpyAsync(c->ctr, &c->chain->snaps[f], sizeof(Counters), cudaMemcpyDeviceToDevice, r.st),
       "counter restore");
    c->level_count[lv + f] = cs.counts[f];
    c->mid_count[lv + f] = cs.mcounts[f];
    c->level_count[lv + f + 1] = 0;
    c->mid_count[lv + f + 1] = 0;
    for (int qi = 0; qi < NQ; ++qi) c->q_count[qi] = cs.snaps[f].q_count[qi];
    c->stats.retries++;
    *next_lv = lv + f;
    *failed = true;
    return FCA_OK;
}

fca_status drain_chain(Run &r, size_t lv, int K, size_t *next_lv, bool *failed)
{
    fca_status s = enqueue_chain(r, lv, K);
    if (s != FCA_OK) return s;
    return collect_chain(r, lv, K, next_lv, failed);
}

// Make room in pool `mid` of level lv + 1 for what a rolled-back launch wanted to append (`after`
// its counters): grow it, or past the pool limit empty the level (drain it depth first) and grow it
// only if the launch alone needs more. Sets *limited when even that is not possible (the caller
// then expands smaller chunks).
fca_status make_room(Run &r, size_t lv, bool mid, const Counters &after, bool *limited)
{
    fca_ctx *c = r.c;
    const uint64_t wanted = mid ? after.next_mid : after.next_count;
    const uint64_t need = wanted - (mid ? c->mid_count[lv + 1] : c->level_count[lv + 1]);
    fca_status s = grow_level(c, lv + 1, mid, wanted, r.st);
    if (s == FCA_OK) return FCA_OK;
    if (s != FCA_ERR_CAPACITY) return s;
    if ((s = drain(r, lv + 1)) != FCA_OK) return s;
    if (need > (mid ? c->mids[lv + 1].cap : c->levels[lv + 1].cap)) {
        s = grow_level(c, lv + 1, mid, need, r.st);
        if (s == FCA_ERR_CAPACITY) *limited = true;
        else if (s != FCA_OK) return s;
    }
    return FCA_OK;
}

// Expand every entry of level `lv` (both pools), depth first. With `chain`, a whole level whose next
// level is empty starts a chain of launches as deep as the last call's search (drain_chain).
fca_status drain(Run &r, size_t lv, bool chain)
{
    fca_ctx *c = r.c;
    fca_status s;
    if (chain && !level_empty(c, lv) && level_empty(c, lv + 1) && c->prev_levels > lv + 2) {
        const int K = (int)std::min<uint64_t>(CHAIN_MAX, c->prev_levels - 1 - lv);
        size_t next = lv;
        bool failed = false;
        if ((s = drain_chain(r, lv, K, &next, &failed)) != FCA_OK) return s;
        if (failed) return drain(r, next, false);
        if (!level_empty(c, next)) return drain(r, next, true);
        return FCA_OK;
    }
    uint64_t kmax = ~(uint64_t)0;    // chunk limit per pool, lowered only when the pools may not grow
    while (!level_empty(c, lv)) {
        if ((s = ensure_level(c, lv + 1)) != FCA_OK) return s;
        const uint64_t hb = c->level_count[lv], hm = c->mid_count[lv];
        uint64_t kb = std::min(hb, kmax), km = std::min(hm, kmax);
        const bool same_level = c->ratio_known && c->ratio_lv == lv;
        // Growth ahead of the launch: what the last launch's children per parent predict for `par`
        // parents, with a margin, allocated exactly. A prediction from an earlier part of the same
        // level may use the whole pool limit; one from the previous level only half of it (a wrong
        // prediction must not take the memory that the overflow path below may need). Returns
        // whether some destination could not be grown that far.
        auto grow_ahead = [&](double par, size_t lim, double margin, bool *refused) -> fca_status {
            auto want = [&](uint64_t have, double ratio) { return have + (uint64_t)(margin * ratio * par) + 16; };
            auto note = [&](fca_status g) {
                if (g == FCA_ERR_CAPACITY) *refused = true;
                return g == FCA_ERR_CAPACITY ? FCA_OK : g;
            };
            fca_status g;
            uint64_t need = want(c->level_count[lv + 1], c->ratio_big);
            if (need > c->levels[lv + 1].cap && (g = note(grow_level(c, lv + 1, false, need, r.st, lim))) != FCA_OK)
                return g;
            if (c->mid_max > SMALL_MAX) {
                need = want(c->mid_count[lv + 1], c->ratio_mid);
                if (need > c->mids[lv + 1].cap && (g = note(grow_level(c, lv + 1, true, need, r.st, lim))) != FCA_OK)
                    return g;
            }
            for (int qi = 0; qi < NQ; ++qi) {
                need = want(c->q_count[qi], c->ratio_q[qi]);
                if (need > c->q[qi].cap && (g = note(grow_queue(c, qi, need, r.st, lim))) != FCA_OK) return g;
            }
            return FCA_OK;
        };
        bool refused = false;
        if (c->pregrow && c->ratio_known &&
            (s = grow_ahead((double)(kb + km), same_level ? c->pool_limit : c->pool_limit / 2,
                            same_level ? 1.5 : 1.25, &refused)) != FCA_OK)
            return s;
        // a large level whose growth could not be predicted (the first level of a call, or a
        // prediction past the bound) is first launched on an eighth of its parents, which measures
        // its children per parent for the rest
        if (c->pregrow && !same_level && (refused || !c->ratio_known) && hb + hm >= PROBE_MIN_PARENTS) {
            kb = std::min(kb, std::max<uint64_t>(1, hb / 8));
            km = std::min(km, std::max<uint64_t>(1, hm / 8));
            // the eighth itself: the previous level's prediction, within the whole limit (an eighth
            // of a wrong prediction costs little)
            bool r2 = false;
            if (c->ratio_known && (s = grow_ahead((double)(kb + km), c->pool_limit, 1.25, &r2)) != FCA_OK) return s;
        }
        const uint64_t bb = hb - kb, bm = hm - km;

        // the next level appends after its current fills; the counters as they are then are kept on
        // the device, to be restored if the launch has to be rolled back (one small kernel)
        CK((cudaError_t)launch_prepare_expand(c->ctr, c->ctr_snap, c->level_count[lv + 1], c->mid_count[lv + 1],
                                              r.st),
           "counter set-up kernel");
        c->stats.launches++;
        if ((s = launch_level(r, lv, bb, kb, bm, km, 0)) != FCA_OK) return s;
        if ((s = read_counters(r)) != FCA_OK) return s;
        const Counters after = *c->ctr_host;

        if (after.error) {
            // roll back: drop everything the launch appended, then make room and retry
            c->stats.retries++;
            CK(cudaMemcpyAsync(c->ctr, c->ctr_snap, sizeof(Counters), cudaMemcpyDeviceToDevice, r.st),
               "counter restore");
            // A full destination is first grown to hold what the launch wanted, keeping what waits
            // in it (the pools are kept for later calls, so a workload stops overflowing once they
            // have grown); past the pool limit it is emptied instead (its subtrees searched, or the
            // next level drained) and grown only if one launch alone needs more.
            bool limited = false;
            for (int qi = 0; qi < NQ; ++qi) {
                if (!(after.error & (ERR_QUEUE0 << qi))) continue;
                const uint64_t need = after.q_count[qi] - c->q_count[qi];
                s = grow_queue(c, qi, after.q_count[qi], r.st);
                if (s == FCA_OK) continue;
                if (s != FCA_ERR_CAPACITY) return s;
                if ((s = run_subtree(r, qi, r.st)) != FCA_OK) return s;
                if (need > c->q[qi].cap) {
                    s = grow_queue(c, qi, need, r.st);
                    if (s == FCA_ERR_CAPACITY) limited = true;
                    else if (s != FCA_OK) return s;
                }
            }
            if ((after.error & ERR_NEXT) && (s = make_room(r, lv, false, after, &limited)) != FCA_OK) return s;
            if ((after.error & ERR_NEXT_MID) && (s = make_room(r, lv, true, after, &limited)) != FCA_OK) return s;
            if (limited) {
                if (kb + km <= 1) {
                    c->err = "work pools too small for one search node (raise FCA_POOL_LIMIT_BYTES)";
                    return FCA_ERR_OOM;
                }
                kmax = std::max<uint64_t>(1, std::max(kb, km) / 2);
            }
            continue;
        }
        if (kb + km > 0) {
            const double parents = (double)(kb + km);
            c->ratio_big = (double)(after.next_count - c->level_count[lv + 1]) / parents;
            c->ratio_mid = (double)(after.next_mid - c->mid_count[lv + 1]) / parents;
            for (int qi = 0; qi < NQ; ++qi) c->ratio_q[qi] = (double)(after.q_count[qi] - c->q_count[qi]) / parents;
            c->ratio_known = true;
            c->ratio_lv = lv;
        }
        c->level_count[lv] = bb;
        c->mid_count[lv] = bm;
        c->level_count[lv + 1] = after.next_count;
        c->mid_count[lv + 1] = after.next_mid;
        for (int qi = 0; qi < NQ; ++qi) c->q_count[qi] = after.q_count[qi];
        count_level(c, lv, kb, km);
        c->stats.max_frontier = std::max<uint64_t>(c->stats.max_frontier, after.next_count + after.next_mid);
    }
    if (!level_empty(c, lv + 1)) return drain(r, lv + 1, true);
    return FCA_OK;
}

// Copy the rows in (host or device source), clear padding bits, rebuild the columns (transpose),
// the top intent and the full-row flag. Everything on stream `st`; returns after it completes.
fca_status load_table(fca_ctx *c, const uint32_t *rows, cudaStream_t st)
{
    const Dims &d = c->d;
    CK(cudaSetDevice(c->device), "cudaSetDevice");
    // device rows are read in place by the table kernel; other memory is copied in first
    cudaPointerAttributes pa{};
    const bool on_device = cudaPointerGetAttributes(&pa, rows) == cudaSuccess && pa.type == cudaMemoryTypeDevice &&
                           pa.device == c->device;
    cudaGetLastError();
    const uint32_t *src = rows;
    if (!on_device) {
        CK(cudaMemcpyAsync(c->rows, rows, (size_t)d.n * d.wm * 4, cudaMemcpyDefault, st), "row copy");
        src = c->rows;
    }
    const bool need_sup = c->decide ? c->attr_order != 0 : c->use_order;
    CK((cudaError_t)launch_table(src, c->rows, c->cols_buf[0], c->top_buf[0], c->full_mask, c->botext,
                                 need_sup ? c->sup : nullptr, d, st),
       "table kernels");
    c->table_launches = 2;
    if (c->decide) {
        // the order is chosen once (at creation, or after the option changed): with option 1 the
        // support order is taken when the supports vary (coefficient of variation above 0.25):
        // then rare attributes come first and far fewer candidates fail the canonical test,
        // while on evenly dense tables a reordering saves little and its kernels cost more
        c->use_order = c->attr_order == 2;
        if (c->attr_order == 1) {
            std::vector<uint32_t> h(d.m);
            CK(cudaMemcpyAsync(h.data(), c->sup, (size_t)d.m * 4, cudaMemcpyDeviceToHost, st), "support read-back");
            CK(cudaStreamSynchronize(st), "stream synchronize");
            double sum = 0.0, sq = 0.0;
            for (uint32_t v : h) {
                sum += v;
                sq += (double)v * v;
            }
            const double mean = sum / d.m, var = std::max(0.0, sq / d.m - mean * mean);
            c->use_order = mean > 0.0 && std::sqrt(var) > ORDER_MIN_CV * mean;
        }
        c->decide = false;
    }
    c->ordered = c->use_order;
    if (c->ordered) {
        CK((cudaError_t)launch_order(c->sup, c->perm, c->inv, c->cols_buf[0], c->cols_buf[1], c->rows, c->top_buf[0],
                                     c->top_buf[1], d, st),
           "order kernels");
        c->table_launches += 2;
    }
    c->cols = c->cols_buf[c->ordered ? 1 : 0];
    c->top = c->top_buf[c->ordered ? 1 : 0];
    return FCA_OK;
}

// Search the roots that object-list searches spilled (the counters in ctr_host are current): one
// launch per queue width and round, the next round taking what this one spilled, until none is
// left; then the intents they output are mapped back to attribute order.
fca_status spill_rounds(Run &r)
{
    fca_ctx *c = r.c;
    fca_status s;
    uint64_t cnt[NQ];
    for (int qi = 0; qi < NQ; ++qi) cnt[qi] = std::min<uint64_t>(c->ctr_host->spill[qi], SPILL_CAP);
    if (cnt[0] == 0 && cnt[1] == 0) return FCA_OK;
    const uint64_t start = c->ctr_host->out_count;
    int cur = 0;
    while (cnt[0] || cnt[1]) {
        c->stats.spill_rounds++;
        CK(cudaMemsetAsync(c->ctr->spill, 0, sizeof(c->ctr->spill), r.st), "spill reset");
        for (int qi = NQ - 1; qi >= 0; --qi) {
            if (!cnt[qi]) continue;
            SubtreeArgs a{};
            a.d = c->d;
            a.rows = c->rows;
            a.q = c->spq[cur][qi];
            a.q_count = cnt[qi];
            a.q_index = qi;
            a.out = r.out;
            a.capacity = r.capacity;
            a.ctr = c->ctr;
            a.count_work = c->count_work;
            a.share = 1;
            a.budget = SEARCH_BUDGET_CYCLES;
            a.wait_ns = c->wait_ns;
            a.spill = c->spq[1 - cur][qi];
            CK(cudaMemsetAsync(&c->ctr->q_head[qi], 0, sizeof(unsigned long long), r.st), "cursor reset");
            size_t pair = 0;
            if ((s = time_begin(r, 1, &pair, r.st)) != FCA_OK) return s;
            CK((cudaError_t)launch_subtree(a, 1 << qi, c->sm_count, r.st), "subtree kernel launch");
            if ((s = time_end(r, pair, r.st)) != FCA_OK) return s;
            c->stats.launches++;
            c->stats.subtree_launches++;
            c->stats.small_roots += cnt[qi];
        }
        if ((s = read_counters(r)) != FCA_OK) return s;
        for (int qi = 0; qi < NQ; ++qi) cnt[qi] = std::min<uint64_t>(c->ctr_host->spill[qi], SPILL_CAP);
        cur = 1 - cur;
    }
    if (c->ordered) {
        CK((cudaError_t)launch_unpermute(r.out, r.capacity, c->ctr, c->perm, c->d, c->sm_count, r.st, 0, start),
           "unpermute kernel");
        c->stats.launches++;
        if ((s = read_counters(r)) != FCA_OK) return s;
    }
    return FCA_OK;
}

// The roots left in the two queues: one launch each. The larger extents run first on the caller's
// stream; the smaller ones on a side stream, so their blocks take the SMs that the last long
// subtrees of the first launch leave idle. The caller's stream waits for both. Only the heavier
// launch (a root of the wider queue counted as four) may hand work between warps: helpers kept busy
// in the lighter one would take issue slots from the heavier one, which ends the call. `guarded`:
// counts read on the device, estimates from the last call (see run_subtree).
fca_status final_launches(Run &r, bool guarded)
{
    fca_ctx *c = r.c;
    fca_status s;
    const uint64_t q0 = guarded ? c->prev_q[0] : c->q_count[0];
    const uint64_t q1 = guarded ? c->prev_q[1] : c->q_count[1];
    if (guarded || (q0 > 0 && q1 > 0)) {
        const bool wide_heavier = 4 * q1 >= q0;
        CK(cudaEventRecord(c->fork, r.st), "cudaEventRecord");
        if ((s = run_subtree(r, 1, r.st, wide_heavier, false, guarded)) != FCA_OK) return s;
        CK(cudaStreamWaitEvent(c->side, c->fork, 0), "cudaStreamWaitEvent");
        if ((s = run_subtree(r, 0, c->side, !wide_heavier, false, guarded)) != FCA_OK) return s;
        CK(cudaEventRecord(c->join, c->side), "cudaEventRecord");
        CK(cudaStreamWaitEvent(r.st, c->join, 0), "cudaStreamWaitEvent");
        return FCA_OK;
    }
    for (int qi = NQ - 1; qi >= 0; --qi)
        if ((s = run_subtree(r, qi, r.st, true, false)) != FCA_OK) return s;
    return FCA_OK;
}

fca_status enumerate_impl(fca_ctx *c, uint32_t *out, uint64_t capacity, uint64_t *out_count,
                          cudaStream_t st)
{
    CK(cudaSetDevice(c->device), "cudaSetDevice");
    fca_status s;
    c->stats = fca_stats{};
    std::fill(c->cur_counts.begin(), c->cur_counts.end(), 0);
    std::fill(c->cur_mids.begin(), c->cur_mids.end(), 0);
    c->pairs_used = 0;
    if ((s = ensure_queues(c)) != FCA_OK) return s;
    if ((s = ensure_level(c, 0)) != FCA_OK) return s;
    for (size_t i = 0; i < c->levels.size(); ++i) c->level_count[i] = c->mid_count[i] = 0;
    for (int qi = 0; qi < NQ; ++qi) c->q_count[qi] = c->last_q[qi] = 0;
    c->ratio_known = false;

    Run r{c, out, capacity, st};
    const Dims &d = c->d;
    // counters (the top intent occupies output row 0) and the root node (G, G', 0): an object-list
    // root when it has at most SMALL_MAX objects, else entry 0 of bitmap level 0 (one small kernel)
    const int root_q = d.n <= SMALL_MAX ? (d.n <= 32 ? 0 : 1) : -1;
    CK((cudaError_t)launch_start(c->ctr, c->top, c->root_ext, d, out, capacity, c->levels[0],
                                 c->q[root_q < 0 ? 0 : root_q], root_q, st),
       "start kernel");
    c->stats.launches++;
    if (root_q >= 0) c->q_count[root_q] = 1;
    else c->level_count[0] = 1;

    // When the last call's bitmap search fit in one chain, queue it and, behind it, the last
    // object-list launches and the bottom concept, guarded on the device: they run only if the
    // chain ends the bitmap search cleanly (no overflow, no deeper level). One read-back then ends
    // the call; otherwise they did nothing and the search goes on as below.
    bool finished = false;
    if (root_q < 0 && c->prev_levels > 2) {
        const int K = (int)std::min<uint64_t>(CHAIN_MAX, c->prev_levels - 1);
        size_t next = 0;
        bool failed = false;
        if ((s = enqueue_chain(r, 0, K)) != FCA_OK) return s;
        if ((s = final_launches(r, true)) != FCA_OK) return s;
        CK((cudaError_t)launch_append_bottom(c->botext, c->full_mask, out, capacity, c->ctr, d, st, 1),
           "bottom kernel");
        c->stats.launches++;
        if (c->ordered) {
            CK((cudaError_t)launch_unpermute(out, capacity, c->ctr, c->perm, d, c->sm_count, st, 1),
               "unpermute kernel");
            c->stats.launches++;
        }
        if ((s = collect_chain(r, 0, K, &next, &failed)) != FCA_OK) return s;
        if (!failed && level_empty(c, next)) {
            finished = true;
            for (int qi = 0; qi < NQ; ++qi) {
                c->stats.small_roots += c->ctr_host->q_count[qi];
                c->last_q[qi] = c->ctr_host->q_count[qi];
            }
        } else if ((s = drain(r, next, !failed)) != FCA_OK) {
            return s;
        }
    } else if ((s = drain(r, 0)) != FCA_OK) {
        return s;
    }
    if (!finished) {
        if ((s = final_launches(r, false)) != FCA_OK) return s;
        // The bottom concept (M', M). When some object holds every attribute its extent is not
        // empty and the search reaches it. Otherwise only empty candidate extents close to it; the
        // search skips those, and it is appended here (a concept is output exactly once either way).
        CK((cudaError_t)launch_append_bottom(c->botext, c->full_mask, out, capacity, c->ctr, d, st),
           "bottom kernel");
        c->stats.launches++;
        // intents back from processing order to attribute order
        if (c->ordered) {
            CK((cudaError_t)launch_unpermute(out, capacity, c->ctr, c->perm, d, c->sm_count, st, 0),
               "unpermute kernel");
            c->stats.launches++;
        }
        if ((s = read_counters(r)) != FCA_OK) return s;
    }
    if ((s = spill_rounds(r)) != FCA_OK) return s;
    if (c->ctr_host->fault & FAULT_WAIT) {
        c->err = "object-list kernel: a warp waited past its limit for work from its block";
        return FCA_ERR_CUDA;
    }
    const uint64_t total = c->ctr_host->out_count;
    c->stats.concepts = total;
    c->stats.closures = c->ctr_host->closures;
    c->stats.frontier_bytes = c->pool_bytes;
    c->stats.subtree_word_ops = c->ctr_host->word_ops;
    c->stats.expand_bytes = c->ctr_host->bytes;
    *out_count = total;
    c->prev_counts = c->cur_counts;
    c->prev_mids = c->cur_mids;
    c->prev_levels = c->stats.levels;
    for (int qi = 0; qi < NQ; ++qi) c->prev_q[qi] = c->last_q[qi];
    return total > capacity ? FCA_ERR_CAPACITY : FCA_OK;
}

}  // namespace

extern "C" {

const char *fca_status_string(fca_status s)
{
    int i = (int)s;
    return (i >= 0 && i < 5) ? kStatus[i] : "unknown status";
}

const char *fca_last_error(const fca_ctx *ctx) { return ctx ? ctx->err.c_str() : ""; }

void fca_free(fca_ctx *ctx)
{
    if (!ctx) return;
    cudaSetDevice(ctx->device);
    cudaFree(ctx->rows);
    for (int i = 0; i < 2; ++i) {
        cudaFree(ctx->cols_buf[i]);
        cudaFree(ctx->top_buf[i]);
    }
    cudaFree(ctx->sup);
    cudaFree(ctx->perm);
    cudaFree(ctx->inv);
    cudaFree(ctx->full_mask);
    cudaFree(ctx->root_ext);
    free_pools(ctx);
    for (cudaEvent_t e : ctx->events) cudaEventDestroy(e);
    if (ctx->fork) cudaEventDestroy(ctx->fork);
    for (cudaEvent_t e : ctx->lat_ev)
        if (e) cudaEventDestroy(e);
    if (ctx->join) cudaEventDestroy(ctx->join);
    if (ctx->side) cudaStreamDestroy(ctx->side);
    cudaFree(ctx->ctr);
    cudaFree(ctx->ctr_snap);
    cudaFree(ctx->chain);
    cudaFreeHost(ctx->chain_host);
    cudaFree(ctx->host_out_dev);
    cudaFreeHost(ctx->ctr_host);
    cudaFree(ctx->botext);
    delete ctx;
}

fca_status fca_context_create(const uint32_t *rows, int64_t n_objects, int32_t n_attrs,
                              fca_ctx **out_ctx)
{
    if (out_ctx) *out_ctx = nullptr;
    if (!rows || !out_ctx || n_objects < 1 || n_attrs < 1 || n_attrs > MAX_ATTRS ||
        n_objects > ((int64_t)1 << 31) - 64)
        return FCA_ERR_INVALID;
    fca_ctx *c = new fca_ctx();
    auto fail = [&](fca_status s) {
        *out_ctx = nullptr;
        fca_free(c);
        return s;
    };
    cudaError_t e = cudaGetDevice(&c->device);
    if (e != cudaSuccess) { cuda_fail(c, e, "cudaGetDevice"); return fail(FCA_ERR_CUDA); }
    e = cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, c->device);
    if (e != cudaSuccess) { cuda_fail(c, e, "device query"); return fail(FCA_ERR_CUDA); }
    Dims &d = c->d;
    d.n = n_objects;
    d.m = n_attrs;
    d.wm = (n_attrs + 31) / 32;
    d.wn = (n_objects + 31) / 32;
    d.wnp = (d.wn + 3) & ~(int64_t)3;
    // the expand kernel stages an extent's chunks and one intersection per warp in shared memory
    if (expand_smem_per_warp(d) > 200 * 1024) return fail(FCA_ERR_INVALID);

    fca_status s;
    if ((s = alloc_raw(c, (void **)&c->rows, (size_t)d.n * d.wm * 4, "rows")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&c->cols_buf[0], (size_t)d.m * d.wnp * 4, "columns")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&c->cols_buf[1], (size_t)d.m * d.wnp * 4, "columns")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&c->top_buf[0], (size_t)d.wm * 4, "top")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&c->top_buf[1], (size_t)d.wm * 4, "top")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&c->sup, (size_t)d.m * 4, "supports")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&c->perm, (size_t)d.m * 4, "order")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&c->inv, (size_t)d.m * 4, "order")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&c->full_mask, (size_t)d.wm * 4, "mask")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&c->root_ext, (size_t)d.wnp * 4, "root extent")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&c->ctr, sizeof(Counters), "counters")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&c->ctr_snap, sizeof(Counters), "counter snapshot")) != FCA_OK ||
        (s = alloc_raw(c, (void **)&c->chain, sizeof(ChainSlots), "chain records")) != FCA_OK)
        return fail(s);
    if ((s = alloc_raw(c, (void **)&c->botext, (size_t)d.wn * 4, "bottom extent")) != FCA_OK) return fail(s);
    // the padding words of the columns (past wn) stay zero; the table kernel writes only the others
    if ((e = cudaMemset(c->cols_buf[0], 0, (size_t)d.m * d.wnp * 4)) != cudaSuccess ||
        (e = cudaMemset(c->cols_buf[1], 0, (size_t)d.m * d.wnp * 4)) != cudaSuccess) {
        cuda_fail(c, e, "column clear");
        return fail(FCA_ERR_CUDA);
    }
    if (cudaMallocHost((void **)&c->ctr_host, sizeof(Counters)) != cudaSuccess ||
        cudaMallocHost((void **)&c->chain_host, sizeof(ChainSlots)) != cudaSuccess) {
        cudaGetLastError();
        c->err = "pinned host allocation failed";
        return fail(FCA_ERR_OOM);
    }
    if ((e = cudaStreamCreateWithFlags(&c->side, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&c->fork, cudaEventDisableTiming)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&c->join, cudaEventDisableTiming)) != cudaSuccess) {
        cuda_fail(c, e, "stream set-up");
        return fail(FCA_ERR_CUDA);
    }

    // host-side constants: the all-attribute intent and the all-object extent
    std::vector<uint32_t> mask(d.wm, 0xffffffffu), ext(d.wnp, 0u);
    if (d.m & 31) mask[d.wm - 1] = (1u << (d.m & 31)) - 1u;
    for (int64_t w = 0; w < d.wn; ++w) ext[w] = 0xffffffffu;
    if (d.n & 31) ext[d.wn - 1] = (1u << (d.n & 31)) - 1u;
    if ((e = cudaMemcpy(c->full_mask, mask.data(), d.wm * 4, cudaMemcpyHostToDevice)) != cudaSuccess ||
        (e = cudaMemcpy(c->root_ext, ext.data(), d.wnp * 4, cudaMemcpyHostToDevice)) != cudaSuccess) {
        cuda_fail(c, e, "context set-up");
        return fail(FCA_ERR_CUDA);
    }
    {
        // processing order of the attributes (FCA_OPT_ATTR_ORDER), 1 unless FCA_ATTR_ORDER says 0 or 2
        const char *v = getenv("FCA_ATTR_ORDER");
        c->attr_order = (v && (v[0] == '0' || v[0] == '2') && v[1] == 0) ? v[0] - '0' : 1;
    }
    if ((s = load_table(c, rows, 0)) != FCA_OK) return fail(s);
    if ((e = cudaStreamSynchronize(0)) != cudaSuccess) {
        cuda_fail(c, e, "context set-up");
        return fail(FCA_ERR_CUDA);
    }

    // work pools: initial sizes and the growth limit (half of the free device memory by default)
    size_t free_b = 0, total_b = 0;
    if (cudaMemGetInfo(&free_b, &total_b) != cudaSuccess) {
        cudaGetLastError();
        free_b = (size_t)8 << 30;
    }
    c->level_bytes = env_u64("FCA_LEVEL_BYTES", 64ull << 20);
    {
        const char *v = getenv("FCA_PREGROW");
        c->pregrow = !(v && v[0] == '0' && v[1] == 0);
    }
    c->queue_entries = env_u64("FCA_QUEUE_ENTRIES", 1ull << 18);
    c->pool_limit = (size_t)env_u64("FCA_POOL_LIMIT_BYTES", free_b / 2);
    c->wait_ns = env_u64("FCA_WAIT_LIMIT_NS", 0);
    // id lists and the mid tier (FCA_LIST_MAX=0 stores every level entry as a bitmap; FCA_MID_MAX=0
    // leaves the id-list entries to the bitmap-tier kernel)
    c->list_max = list_max_for(c->d);
    c->mid_max = mid_max_for(c->d);
    {
        const char *v = getenv("FCA_LIST_MAX");
        if (v && v[0] == '0' && v[1] == 0) c->list_max = c->mid_max = 0;
        v = getenv("FCA_MID_MAX");
        if (v && v[0] == '0' && v[1] == 0) c->mid_max = 0;
    }
    c->mid_stride = c->mid_max > SMALL_MAX ? ((int64_t)c->mid_max + 3) & ~(int64_t)3 : 0;
    c->big_stride = c->d.wnp;
    if (c->d.m <= 256 && !(getenv("FCA_NO_INHERIT") && getenv("FCA_NO_INHERIT")[0] == '1')) {
        c->wit_words = ((c->d.m + 3) / 4 + 3) & ~3;
        c->big_stride += c->wit_words;
        if (c->mid_stride > 0) {
            c->wit_off = (int)c->mid_stride;
            c->mid_stride += c->wit_words;
        }
    }
    c->mid_min = env_u64("FCA_MID_MIN", MID_MIN_PARENTS_PER_SM * (uint64_t)c->sm_count);
    *out_ctx = c;
    return FCA_OK;
}

fca_status fca_context_load(fca_ctx *ctx, const uint32_t *rows, void *stream)
{
    if (!ctx || !rows) return FCA_ERR_INVALID;
    ctx->err.clear();
    return load_table(ctx, rows, (cudaStream_t)stream);
}

fca_status fca_enumerate(fca_ctx *ctx, uint32_t *out, uint64_t capacity, uint64_t *out_count, void *stream)
{
    if (!ctx || !out_count || (capacity > 0 && !out)) return FCA_ERR_INVALID;
    ctx->err.clear();
    return enumerate_impl(ctx, out, capacity, out_count, (cudaStream_t)stream);
}

fca_status fca_enumerate_host(fca_ctx *ctx, uint32_t *out_host, uint64_t capacity, uint64_t *out_count,
                              void *stream)
{
    if (!ctx || !out_count || (capacity > 0 && !out_host)) return FCA_ERR_INVALID;
    fca_ctx *c = ctx;
    c->err.clear();
    CK(cudaSetDevice(c->device), "cudaSetDevice");
    if (capacity > c->host_out_rows) {
        cudaFree(c->host_out_dev);
        c->host_out_dev = nullptr;
        c->host_out_rows = 0;
        void *p = nullptr;
        if (cudaMalloc(&p, capacity * c->d.wm * 4) != cudaSuccess) {
            cudaGetLastError();
            c->err = "cudaMalloc failed for the output buffer";
            return FCA_ERR_OOM;
        }
        c->host_out_dev = (uint32_t *)p;
        c->host_out_rows = capacity;
    }
    cudaStream_t st = (cudaStream_t)stream;
    fca_status s = enumerate_impl(c, c->host_out_dev, capacity, out_count, st);
    if (s != FCA_OK && s != FCA_ERR_CAPACITY) return s;
    const uint64_t rows = std::min<uint64_t>(*out_count, capacity);
    if (rows) {
        CK(cudaMemcpyAsync(out_host, c->host_out_dev, rows * c->d.wm * 4, cudaMemcpyDeviceToHost, st),
           "output copy");
        CK(cudaStreamSynchronize(st), "stream synchronize");
    }
    return s;
}

fca_status fca_set_option(fca_ctx *ctx, int option, int64_t value)
{
    if (!ctx || value < 0) return FCA_ERR_INVALID;
    fca_ctx *c = ctx;
    switch (option) {
    case FCA_OPT_COUNT_WORK:
        c->count_work = value != 0;
        return FCA_OK;
    case FCA_OPT_WAIT_LIMIT_NS:
        c->wait_ns = (uint64_t)value;
        return FCA_OK;
    case FCA_OPT_ATTR_ORDER:
        if (value > 2) return FCA_ERR_INVALID;
        c->attr_order = (int)value;
        c->decide = true;
        return FCA_OK;
    case FCA_OPT_LEVEL_BYTES:
    case FCA_OPT_QUEUE_ENTRIES:
    case FCA_OPT_POOL_LIMIT_BYTES:
        CK(cudaSetDevice(c->device), "cudaSetDevice");
        CK(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
        free_pools(c);
        if (option == FCA_OPT_LEVEL_BYTES) c->level_bytes = (uint64_t)value;
        else if (option == FCA_OPT_QUEUE_ENTRIES) c->queue_entries = (uint64_t)value;
        else c->pool_limit = (size_t)value;
        return FCA_OK;
    default:
        return FCA_ERR_INVALID;
    }
}

fca_status fca_get_stats(const fca_ctx *ctx, fca_stats *out)
{
    if (!ctx || !out) return FCA_ERR_INVALID;
    *out = ctx->stats;
    cudaSetDevice(ctx->device);
    launch_times(ctx, &out->expand_ms, &out->subtree_ms, &out->mid_ms);
    out->list_max = ctx->list_max > SMALL_MAX ? (uint64_t)ctx->list_max : 0;
    out->mid_max = ctx->mid_max > SMALL_MAX ? (uint64_t)ctx->mid_max : 0;
    out->lattice_ms = 0.0;
    float ms = 0.f;
    if (ctx->lat_timed) {
        if (cudaEventElapsedTime(&ms, ctx->lat_ev[0], ctx->lat_ev[1]) == cudaSuccess) out->lattice_ms = ms;
        else cudaGetLastError();
    }
    return FCA_OK;
}

fca_status fca_context_dims(const fca_ctx *ctx, int64_t *n_objects, int32_t *n_attrs)
{
    if (!ctx || !n_objects || !n_attrs) return FCA_ERR_INVALID;
    *n_objects = ctx->d.n;
    *n_attrs = ctx->d.m;
    return FCA_OK;
}

fca_status fca_context_copy(const fca_ctx *ctx, int which, uint32_t *dst, uint64_t dst_words)
{
    if (!ctx || !dst) return FCA_ERR_INVALID;
    const uint32_t *src = nullptr;
    uint64_t words = 0;
    switch (which) {
    case 0: src = ctx->rows; words = (uint64_t)ctx->d.n * ctx->d.wm; break;
    case 1: src = ctx->cols; words = (uint64_t)ctx->d.m * ctx->d.wnp; break;
    case 2: src = ctx->top; words = (uint64_t)ctx->d.wm; break;
    case 3:
        if (!ctx->ordered) {   // attribute order: the identity
            if (dst_words < (uint64_t)ctx->d.m) return FCA_ERR_INVALID;
            for (int32_t a = 0; a < ctx->d.m; ++a) dst[a] = (uint32_t)a;
            return FCA_OK;
        }
        src = reinterpret_cast<const uint32_t *>(ctx->perm);
        words = (uint64_t)ctx->d.m;
        break;
    default: return FCA_ERR_INVALID;
    }
    if (dst_words < words) return FCA_ERR_INVALID;
    fca_ctx *c = const_cast<fca_ctx *>(ctx);
    CK(cudaSetDevice(c->device), "cudaSetDevice");
    CK(cudaMemcpy(dst, src, words * 4, cudaMemcpyDefault), "context copy");
    return FCA_OK;
}

// Create the lattice-call event pair on first use and record its start on `st`.
static fca_status lattice_time_begin(fca_ctx *c, cudaStream_t st)
{
    for (cudaEvent_t &e : c->lat_ev)
        if (!e) CK(cudaEventCreate(&e), "cudaEventCreate");
    c->lat_timed = false;
    CK(cudaEventRecord(c->lat_ev[0], st), "cudaEventRecord");
    return FCA_OK;
}

static fca_status lattice_time_end(fca_ctx *c, cudaStream_t st)
{
    CK(cudaEventRecord(c->lat_ev[1], st), "cudaEventRecord");
    c->lat_timed = true;
    return FCA_OK;
}

fca_status fca_extents(fca_ctx *ctx, const uint32_t *intents, uint64_t count, uint32_t *extents, void *stream)
{
    if (!ctx || (count > 0 && (!intents || !extents))) return FCA_ERR_INVALID;
    fca_ctx *c = ctx;
    c->err.clear();
    if (count > (uint64_t)INT64_MAX / (uint64_t)c->d.wn) {
        c->err = "count x W_N words exceeds 64 bits";
        return FCA_ERR_INVALID;
    }
    if (count == 0) return FCA_OK;
    CK(cudaSetDevice(c->device), "cudaSetDevice");
    cudaStream_t st = (cudaStream_t)stream;
    fca_status s = lattice_time_begin(c, st);
    if (s != FCA_OK) return s;
    CK((cudaError_t)launch_extents(intents, count, c->cols_buf[0], c->cols, c->ordered ? c->perm : nullptr, c->d,
                                   extents, c->sm_count, st),
       "extents kernel");
    return lattice_time_end(c, st);
}

fca_status fca_cover_edges(fca_ctx *ctx, const uint32_t *intents, uint64_t count, uint32_t *edges,
                           uint64_t capacity, uint64_t *out_edges, void *stream)
{
    if (!ctx || !out_edges || (count > 0 && !intents) || (capacity > 0 && !edges)) return FCA_ERR_INVALID;
    fca_ctx *c = ctx;
    c->err.clear();
    *out_edges = 0;
    if (count >= 0xffffffffull) {
        c->err = "cover edges take fewer than 2^32 - 1 intents";
        return FCA_ERR_INVALID;
    }
    if (count == 0) return FCA_OK;
    CK(cudaSetDevice(c->device), "cudaSetDevice");
    cudaStream_t st = (cudaStream_t)stream;
    uint64_t nslots = 64;
    while (nslots < 2 * count) nslots <<= 1;
    int wpb = 0;
    unsigned blocks = 0;
    size_t smem = 0;
    CK((cudaError_t)covers_shape(c->d, count, c->sm_count, &wpb, &blocks, &smem), "cover kernel shape");
    const size_t ws_bytes = (size_t)blocks * wpb * 4 * (size_t)c->d.wn * 4;
    LatticeCounters *lc = nullptr;
    uint32_t *slots = nullptr, *ws = nullptr;
    CK(cudaMallocAsync((void **)&lc, sizeof(LatticeCounters), st), "cudaMallocAsync");
    cudaError_t e = cudaMallocAsync((void **)&slots, nslots * 4, st);
    if (e == cudaSuccess) e = cudaMallocAsync((void **)&ws, ws_bytes, st);
    LatticeCounters h{};
    if (e == cudaSuccess) e = cudaMemsetAsync(lc, 0, sizeof(LatticeCounters), st);
    if (e == cudaSuccess && lattice_time_begin(c, st) != FCA_OK) e = cudaErrorUnknown;
    if (e == cudaSuccess)
        e = (cudaError_t)launch_covers(intents, count, c->rows, c->ordered ? c->inv : nullptr,
                                       c->ordered ? c->perm : nullptr, c->cols_buf[0], c->cols, c->d, slots, nslots,
                                       edges, capacity, lc, ws, wpb, blocks, smem, c->sm_count, st);
    if (e == cudaSuccess && lattice_time_end(c, st) != FCA_OK) e = cudaErrorUnknown;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&h, lc, sizeof h, cudaMemcpyDeviceToHost, st);
    if (ws) cudaFreeAsync(ws, st);
    if (slots) cudaFreeAsync(slots, st);
    cudaFreeAsync(lc, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(c, e, "cover edges");
    *out_edges = h.edges;
    if (h.duplicates) {
        char buf[120];
        snprintf(buf, sizeof buf, "cover edges: %llu given intents repeat an earlier one (each must be given once)",
                 (unsigned long long)h.duplicates);
        c->err = buf;
        return FCA_ERR_INVALID;
    }
    if (h.insert_failed || h.missing) {
        char buf[160];
        snprintf(buf, sizeof buf, "cover edges: %llu cover intents missing from the given set (%llu not stored)",
                 (unsigned long long)h.missing, (unsigned long long)h.insert_failed);
        c->err = buf;
        return FCA_ERR_INVALID;
    }
    return h.edges > capacity ? FCA_ERR_CAPACITY : FCA_OK;
}

}  // extern "C"
