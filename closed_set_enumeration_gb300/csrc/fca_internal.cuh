// Internal declarations shared by the host driver and the kernels of libfca.
//
// Search model (FCbO-to-CUDA article, sections 2.1-2.4 and 5.3; Parallel FCBO
// article, sections 1.3 and 2.1): a search node is (A, B, y) with extent A,
// intent B = A' and cursor y. Its candidates are the attributes j >= y that
// are not in B (the saturation skip: j in B <=> A is inside column j). For a
// candidate, C = A & column j and D = C'; the child (C, D, j+1) exists iff D
// adds no attribute below j to B (the canonical prefix test, bit j itself
// excluded). Every intent is produced by exactly one node.
//
// Tiers, chosen by extent size:
//  * frontier levels: nodes whose extent has more than SMALL_MAX objects are
//    held in level-synchronous frontiers, each level in two pools. The mid
//    pool holds the nodes of at most mid_max objects, each as the ascending
//    list of its object ids in a slot of mid_max words; they are expanded one
//    per warp on columns restricted to their objects (expand_mid_kernel). The
//    big pool holds the larger ones in slots of W_Np words: an extent of at
//    most list_max objects as its id list, a larger one as an N-bit bitmap;
//    they are expanded one per thread block (expand_bitmap_kernel);
//  * object-list tier: a node with at most 32*NW objects (NW = 1, 2) is
//    handed over as a list of object ids, and one warp runs its whole subtree
//    on the columns restricted to those objects (subtree_kernel<NW>). Every
//    descendant of such a node has a subset of its objects, so the subtree
//    never needs the bitmaps again; this is the FCbO-to-CUDA article's
//    section 5.3 rule of finishing small extents in-block instead of
//    re-enqueueing them.
#pragma once
#include <cstdint>

namespace fca {

constexpr int SMALL_MAX = 64;      // largest extent handed to the object-list tier
constexpr int NQ = 2;              // object-list queues: queue q holds extents of <= 32 << q objects
constexpr int MAX_ATTRS = 1024;    // M limit (intent words fit one per lane)

// Overflow bits of Counters::error (a destination was too small; the driver rolls back and retries).
constexpr unsigned ERR_NEXT = 1u << 4;     // big pool of the next level
constexpr unsigned ERR_NEXT_MID = 1u << 5; // mid pool of the next level
constexpr unsigned ERR_QUEUE0 = 1u;        // queue q sets ERR_QUEUE0 << q
// Bits of Counters::fault (the call fails with FCA_ERR_CUDA).
constexpr unsigned FAULT_WAIT = 1u;        // an object-list warp waited too long for its block

// Device-side counters of one enumerate call.
struct Counters {
    unsigned long long out_count;      // intents emitted so far (row index allocator)
    unsigned long long closures;       // candidates evaluated
    unsigned long long next_count;     // entries appended to the next bitmap level
    unsigned long long work_head;      // work-distribution cursor of the bitmap-tier launch
    unsigned long long q_count[NQ];    // entries appended to the object-list queues
    unsigned long long q_head[NQ];     // work-distribution cursors of the subtree kernels
    unsigned long long word_ops;       // counted object-mid-tier word operations (when counting)
    unsigned long long bytes;          // counted bitmap-tier bytes (when counting)
    unsigned int error;                // overflow bits (ERR_*)
    unsigned int fault;                // FAULT_* bits: a bounded wait inside a kernel ran out
    unsigned int pad[2];
    unsigned long long spill[NQ];      // roots written to the spill queues (object-list searches
                                       // that ran past their time budget)
    unsigned long long mid_head;       // work-distribution cursor of the mid-tier launch
    unsigned long long next_mid;       // entries appended to the mid pool of the next level
};

// Device records of a chain of level launches queued without host synchronisation between them:
// the parent counts of each launch (big and mid pools) and the counters as they were before it.
constexpr int CHAIN_MAX = 32;
struct ChainSlots {
    unsigned long long pcount;               // big-pool parents of the launch being run
    unsigned long long pcount_mid;           // mid-pool parents of the launch being run
    unsigned long long counts[CHAIN_MAX];    // big-pool parents of launch i (0 after a failed launch)
    unsigned long long mcounts[CHAIN_MAX];   // mid-pool parents of launch i (0 after a failed launch)
    Counters snaps[CHAIN_MAX];               // counters before launch i
};

// Device counters of one cover-edge call (fca_cover_edges).
struct LatticeCounters {
    unsigned long long next;            // work cursor: next concept to take
    unsigned long long edges;           // cover edges found (row index allocator)
    unsigned long long missing;         // cover intents not found in the given set
    unsigned long long insert_failed;   // intents the hash table had no room for
    unsigned long long duplicates;      // given intents equal to an earlier-stored one
};

// One pool of a frontier level (structure of arrays).
struct Level {
    uint32_t *ext;   // cap x stride words, 16-byte aligned rows: the extent as a bitmap, or (n <=
                     // list_max; always in a mid pool) its n object ids in ascending order
    uint32_t *itt;   // cap x wm words (intents)
    int32_t *y;      // cap cursors
    int32_t *n;      // cap extent sizes (objects)
    uint64_t cap;
    int64_t stride;  // words per extent slot: W_Np (big pool) or mid_max rounded up to 4 (mid pool)
};

// A queue of subtree roots for the NW-word object-list tier.
struct Queue {
    uint32_t *ids;   // cap x (32*NW) object ids, ascending
    uint32_t *itt;   // cap x wm words (intents)
    int32_t *y;      // cap cursors
    int32_t *n;      // cap object counts (1..32*NW)
    uint64_t cap;
};

struct Dims {
    int64_t n;       // objects
    int32_t m;       // attributes
    int32_t wm;      // words per intent / row
    int64_t wn;      // words per extent
    int64_t wnp;     // wn rounded up to a multiple of 4 (uint4 rows)
};

struct ExpandArgs {
    Dims d;
    const uint32_t *rows;   // n x wm
    const uint32_t *cols;   // m x wnp
    Level in;               // parents (a big pool for expand_bitmap_kernel, a mid pool for expand_mid_kernel)
    uint64_t p_begin, p_count;
    // expand_bitmap_kernel only: a second pool expanded in the same launch after `in` (a small mid
    // pool), parents [p_begin2, p_begin2 + p_count2) or, with p_count2_dev, that many read there
    Level in2;
    uint64_t p_begin2, p_count2;
    const unsigned long long *p_count2_dev;
    // when not null, the parent count is read here on the device (a launch queued behind the one
    // that produces its level); p_count is then only the launcher's estimate for the grid size
    const unsigned long long *p_count_dev;
    int parts;              // work items per parent: parts of the attribute range (set by the launcher;
                            // 0: chosen by the kernel from the device count)
    unsigned long long resident;   // resident blocks of the launch (set by the launcher)
    int restrict_max;       // largest extent rebuilt as restricted columns (set by the launcher)
    int list_max;           // extents of SMALL_MAX < n <= list_max objects are object-id lists (list_max
                            // <= SMALL_MAX: every level entry is a bitmap)
    int mid_max;            // children of SMALL_MAX < n <= mid_max objects go to the mid pool of the next
                            // level (mid_max <= SMALL_MAX: no mid tier)
    Level next;             // children with more than max(SMALL_MAX, mid_max) objects (big pool)
    Level next_mid;         // children with SMALL_MAX < n <= mid_max objects (mid pool)
    int wit_off;            // mid-pool entries: word offset, inside the entry's slot, of its inherited
                            // failures (one byte per attribute: the witness of a candidate that failed
                            // at an ancestor, 0xff for none); 0 when they are not kept
    int wit_words;          // words of those bytes (0: failures are not inherited)
    int wit_off_big;        // the same offset in a big-pool entry (after its W_Np extent words)
    Queue q[NQ];            // children with <= 32 << q objects
    uint32_t *out;          // capacity x wm
    uint64_t capacity;
    Counters *ctr;
    int count_work;         // 1: accumulate Counters::bytes
};

struct SubtreeArgs {
    Dims d;
    const uint32_t *rows;
    Queue q;
    uint64_t q_count;       // roots (the launcher's estimate when q_count_dev is set)
    const unsigned long long *q_count_dev;   // when not null, the root count is read here
    int guard;              // 1: do nothing unless the bitmap search ended cleanly (Counters::error
                            // and next_count both zero): a launch queued before the host knew
    int q_index;            // which q_head counter this queue uses
    int slices;             // work items per root (set by the launcher)
    int share;              // 1: warps may hand work to idle warps of their block (the launcher
                            // keeps it only for launches with few items per warp)
    uint32_t *out;
    uint64_t capacity;
    Counters *ctr;
    int count_work;         // 1: accumulate Counters::word_ops
    // Time budget of one search (clock cycles; 0: none). A search still running past it writes what
    // it has not explored to `spill` as new roots (Counters::spill[q_index] counts them; when the
    // spill queue is full the search goes on instead).
    long long budget;
    Queue spill;
    // Longest a warp of a work-sharing launch waits for a hand-over or for its block to finish
    // (nanoseconds; 0: DEFAULT_WAIT_NS). Past it the kernel records FAULT_WAIT and the warp stops
    // waiting.
    unsigned long long wait_ns;
};
constexpr unsigned long long DEFAULT_WAIT_NS = 1000000000ull;   // 1 s: far above any one search

// Launch wrappers (defined in fca_context.cu, fca_expand.cu and fca_subtree.cu). Each returns a
// cudaError_t value.
// The context's tables from the rows at `src` (device memory; copied into `rows` when it is
// another buffer): padding bits cleared, columns (m x wnp, padding words left as they are), the top
// intent, the bottom extent botext (wn words) and, when sup is not null, the attribute supports
// (m words). Two launches.
int launch_table(const uint32_t *src, uint32_t *rows, uint32_t *cols, uint32_t *top, const uint32_t *full_mask,
                 uint32_t *botext, uint32_t *sup, const Dims &d, void *stream);
// Processing order by ascending support (perm: attribute -> position, inv: position -> attribute),
// then the tables in that order: cols2 from cols, rows (overwritten), top2 from top. Two launches.
int launch_order(const uint32_t *sup, int32_t *perm, int32_t *inv, const uint32_t *cols, uint32_t *cols2,
                 uint32_t *rows, const uint32_t *top, uint32_t *top2, const Dims &d, void *stream);
// Output rows [start, min(out_count, capacity)) mapped back to attribute order (guard as for the
// guarded launches).
int launch_unpermute(uint32_t *out, uint64_t capacity, const Counters *ctr, const int32_t *perm, const Dims &d,
                     int sm_count, void *stream, int guard, uint64_t start = 0);
int launch_expand(const ExpandArgs &a, int sm_count, void *stream);
// The mid pool of a level (a.mid_max > SMALL_MAX): entries of at most a.mid_max objects, one per warp.
int launch_expand_mid(const ExpandArgs &a, int sm_count, void *stream);
// Largest extent expand_mid_kernel takes for these dimensions (<= SMALL_MAX: none), and the largest
// extent stored as an object-id list (<= SMALL_MAX: none; at least the former when that is on).
int mid_max_for(const Dims &d);
int list_max_for(const Dims &d);
// Before a level launch: Counters::next_count = next_fill and next_mid = next_mid_fill (the next
// level's pools), zero work cursors and error, then the counters copied to *snap (for a rollback).
int launch_prepare_expand(Counters *ctr, Counters *snap, uint64_t next_fill, uint64_t next_mid_fill, void *stream);
// Start of an enumeration: zero counters, the top intent in row 0, the root node as entry 0 of
// level L0 (qi < 0) or as the first root of queue Q (queue index qi).
int launch_start(Counters *ctr, const uint32_t *top, const uint32_t *root_ext, const Dims &d, uint32_t *out,
                 uint64_t capacity, const Level &L0, const Queue &Q, int qi, void *stream);
// Before launch i of a chain: its parent counts (n0 / n0_mid for the first, else the previous
// launch's next_count / next_mid; 0 once a launch of the chain has overflowed), zero next level
// fills and cursors, and the counters copied to cs->snaps[i].
int launch_prepare_chain(Counters *ctr, ChainSlots *cs, int i, uint64_t n0, uint64_t n0_mid, void *stream);
// Append the all-attribute intent when the bottom extent botext (wn words) is empty (one slot from
// Counters::out_count). With guard, only when Counters::error and next_count are both zero (see
// SubtreeArgs::guard).
int launch_append_bottom(const uint32_t *botext, const uint32_t *full_mask, uint32_t *out,
                         uint64_t capacity, Counters *ctr, const Dims &d, void *stream, int guard = 0);
int launch_subtree(const SubtreeArgs &a, int nw, int sm_count, void *stream);
// The same with work sharing inside blocks, for a launch whose slices are already set in `b`
// (called by launch_subtree; rw = register words of the search, 2, 4 or 8).
int launch_subtree_shared(const SubtreeArgs &b, int nw, int rw, int sm_count, void *stream);
size_t expand_smem_per_warp(const Dims &d);
// Extent (wn words, padding bits zero) of each of `count` attribute sets (wm words each, attribute
// order) from the columns in attribute order (cols) and in processing order (cols_p; perm: attribute
// -> position, null when the two orders are the same). One launch.
int launch_extents(const uint32_t *intents, uint64_t count, const uint32_t *cols, const uint32_t *cols_p,
                   const int32_t *perm, const Dims &d, uint32_t *extents, int sm_count, void *stream);
// Launch shape of the cover kernel for `count` intents: warps per block, blocks (a persistent grid of
// at most the resident blocks) and dynamic shared memory; the caller allocates 4 x wn words of
// workspace per warp of that grid.
int covers_shape(const Dims &d, uint64_t count, int sm_count, int *wpb, unsigned *blocks, size_t *smem);
// Cover edges of a complete intent set: a hash table of the intents in `slots` (nslots, a power of two
// of at least twice count), then the lower covers of every concept as (row, row of the cover) pairs.
// rows and cols_p are in processing order (inv: position -> attribute, perm: attribute -> position,
// both null for the identity), cols in attribute order; lc zeroed by the caller; ws, wpb, blocks and
// smem from covers_shape. A memset and two launches.
int launch_covers(const uint32_t *intents, uint64_t count, const uint32_t *rows, const int32_t *inv,
                  const int32_t *perm, const uint32_t *cols, const uint32_t *cols_p, const Dims &d, uint32_t *slots,
                  uint64_t nslots, uint32_t *edges, uint64_t capacity, LatticeCounters *lc, uint32_t *ws, int wpb,
                  unsigned blocks, size_t smem, int sm_count, void *stream);
// Shared memory of one covers_kernel warp (bytes).
size_t covers_smem_per_warp(const Dims &d);

}  // namespace fca
