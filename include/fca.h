/*
 * fca.h - formal-concept enumeration (Close-by-One with saturation pruning)
 * on one GB300 GPU (sm_103a). Plain C ABI: no C++ or framework types.
 *
 * A formal context is a binary table of N objects x M attributes. For an
 * object set X, X' is the set of attributes shared by every object of X; for
 * an attribute set Y, Y' is the set of objects having every attribute of Y.
 * A concept is a pair (A, B) with A' = B and B' = A; B is its intent
 * (FCbO-to-CUDA page, sections 1.1-1.2; Parallel FCBO page, section 1.1).
 * fca_enumerate outputs every intent exactly once, found by the Close-by-One
 * search with the canonical prefix test and the saturation skip
 * (FCbO-to-CUDA page, sections 2.1-2.3 and 4.3; Parallel FCBO page,
 * sections 1.2-1.3 and 2.1).
 *
 * Bit layout (FCbO-to-CUDA page, section 4.3; Parallel FCBO page, section
 * 3.1): attribute a of a row is bit (a & 31) of 32-bit word (a >> 5), least
 * significant bit first. A row / intent is W_M = ceil(M/32) words.
 *
 * Error behaviour: every call returns a status; nothing aborts the process.
 * A CUDA error is reported as FCA_ERR_CUDA and its text is kept in the
 * context (fca_last_error). The library never falls back to the CPU.
 */
#ifndef FCA_H
#define FCA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct fca_ctx fca_ctx; /* opaque; owns the device copies and work pools */

typedef enum {
    FCA_OK = 0,
    FCA_ERR_INVALID = 1,  /* bad argument (NULL pointer, N < 1, M < 1, sizes beyond limits) */
    FCA_ERR_OOM = 2,      /* a device or host allocation failed */
    FCA_ERR_CAPACITY = 3, /* more concepts than `capacity`; *out_count holds the true total */
    FCA_ERR_CUDA = 4      /* a CUDA runtime call or kernel failed; see fca_last_error */
} fca_status;

/* Statistics of the last fca_enumerate call on a context. Device times are
 * the union of the launches' intervals per kind of kernel (launches that run
 * side by side count once). */
typedef struct {
    uint64_t concepts;         /* intents found (= *out_count) */
    uint64_t closures;         /* candidates (A, B, j) considered: j >= cursor, j not in B (with
                                  M <= 256 the bitmap and mid tiers skip the closure of a candidate
                                  whose failure a search-tree ancestor recorded with a witness still
                                  outside B, the Fast Close-by-One rule; such candidates are counted
                                  here too; FCA_NO_INHERIT=1 in the environment turns the rule off) */
    uint64_t large_parents;    /* search nodes of more than 64 objects (list- and bitmap-tier kernels) */
    uint64_t small_roots;      /* subtrees handed to the object-list kernels (extent <= 64) */
    uint64_t launches;         /* kernels launched by the call */
    uint64_t levels;           /* deepest bitmap-frontier level used, plus one */
    uint64_t max_frontier;     /* largest number of bitmap entries held by one level */
    uint64_t frontier_bytes;   /* device bytes held by frontier and queue buffers */
    uint64_t expand_launches;  /* launches of the bitmap-tier kernel */
    uint64_t subtree_launches; /* launches of the object-list kernels */
    uint64_t subtree_word_ops; /* counted work of the object-list tier (FCA_OPT_COUNT_WORK) */
    uint64_t expand_bytes;     /* counted bytes moved by the list and bitmap tiers (FCA_OPT_COUNT_WORK) */
    uint64_t retries;          /* level launches rolled back because a work pool was full (before
                                  each unchained level launch the pools are grown to what the last
                                  launch predicts; FCA_PREGROW=0 in the environment turns that off) */
    uint64_t spill_rounds;     /* launch rounds over subtrees spilled by searches past their time
                                  budget (their roots are counted in small_roots) */
    double expand_ms;          /* device time of the bitmap-tier kernel launches */
    double subtree_ms;         /* device time of the object-list kernel launches */
    double lattice_ms;         /* device time of the kernels of the last fca_extents or
                                  fca_cover_edges call on the context (0 before the first) */
    uint64_t mid_launches;     /* launches of the mid-tier kernel (search nodes of 65 to a few
                                  hundred objects, held as object-id lists, one per warp) */
    double mid_ms;             /* device time of the mid-tier kernel launches */
    uint64_t list_max;         /* largest search-node extent kept as an object-id list (0: none;
                                  fixed by N and M, or FCA_LIST_MAX=0 in the environment) */
    uint64_t mid_max;          /* largest search-node extent expanded by the mid-tier kernel (0:
                                  no mid tier; FCA_MID_MAX=0 turns it off) */
} fca_stats;

/* Options for fca_set_option. */
typedef enum {
    FCA_OPT_COUNT_WORK = 1,       /* 0/1: count the algorithmic work of each kernel (slower) */
    FCA_OPT_LEVEL_BYTES = 2,      /* initial bytes of one bitmap-frontier level (default 64 MiB) */
    FCA_OPT_QUEUE_ENTRIES = 3,    /* initial entries of each object-list queue (default 2^18) */
    FCA_OPT_POOL_LIMIT_BYTES = 4, /* growth limit of all work pools (default: half the free memory) */
    FCA_OPT_ATTR_ORDER = 5,       /* processing order of the attributes: 0 attribute order,
                                     1 (default) ascending support when the supports vary,
                                     2 ascending support; chosen by the next table load */
    FCA_OPT_WAIT_LIMIT_NS = 6     /* bound, in ns, of a device-side wait of the object-list
                                     kernel (0: the default, 1 s); see fca_set_option */
} fca_option;

/*
 * Build a context: device copies of the object rows (ctxRows, N x W_M words)
 * and of their transpose, the attribute columns (ctxCols, M x W_N words with
 * W_N = ceil(N/32), each column padded to a 16-byte multiple), plus the top
 * intent G' (AND of all rows). This is the dual row/column layout of the
 * FCbO-to-CUDA page, section 3.1, and the Parallel FCBO page, section 2.3;
 * the transpose is built on the GPU (Parallel FCBO page, section 3.1).
 *
 *   rows       N x W_M uint32 words, row-major, LSB-first. Host or device
 *              pointer (copied with cudaMemcpyDefault, read once, not kept).
 *              Padding bits past M are ignored.
 *   n_objects  1 <= N <= about 720 000 (a thread block of the bitmap-extent
 *              kernel stages one extent and one intersection in shared memory;
 *              larger N returns FCA_ERR_INVALID).
 *   n_attrs    1 <= M <= 1024.
 *   out_ctx    receives the new context (NULL on failure).
 * Runs on the legacy default stream and returns after it completes.
 * Uses the current CUDA device; the context must be used on that device.
 */
fca_status fca_context_create(const uint32_t *rows, int64_t n_objects, int32_t n_attrs,
                              fca_ctx **out_ctx);

/*
 * Replace the context's table with new rows of the same N x M and rebuild
 * its columns and top intent, reusing every allocation (a new batch of the
 * same shape). `rows` as for fca_context_create (host or device pointer).
 * The work is enqueued on `stream` (cudaStream_t, NULL = legacy default
 * stream) and the call returns without waiting for it: `rows` must stay
 * valid until it has run, and a later fca_enumerate must be ordered after it
 * (the same stream does that).
 */
fca_status fca_context_load(fca_ctx *ctx, const uint32_t *rows, void *stream);

/*
 * Enumerate every intent of the context.
 *
 *   out        device pointer, capacity x W_M uint32 words, caller-owned.
 *              Row r receives one intent. Output order is unspecified; the
 *              top intent G' is row 0 when capacity >= 1. Padding bits are 0.
 *   capacity   rows available in `out` (0 allowed: count only).
 *   out_count  host pointer; receives the total number of intents, also when
 *              it exceeds `capacity`.
 *   stream     cudaStream_t to run on (NULL = legacy default stream).
 * Returns FCA_OK, or FCA_ERR_CAPACITY when the total exceeds `capacity`
 * (the first `capacity` rows are written, the count is exact: retry with a
 * larger buffer). The call returns after the work on `stream` completes.
 * One context serves one caller at a time.
 */
fca_status fca_enumerate(fca_ctx *ctx, uint32_t *out, uint64_t capacity, uint64_t *out_count,
                         void *stream);

/*
 * Like fca_enumerate, but `out_host` is a host pointer (pinned or pageable,
 * capacity x W_M words). The intents are produced in a device buffer held
 * by the context and copied back before return.
 */
fca_status fca_enumerate_host(fca_ctx *ctx, uint32_t *out_host, uint64_t capacity,
                              uint64_t *out_count, void *stream);

/*
 * The extent of each given attribute set: Y' = the objects having every
 * attribute of Y (FCbO-to-CUDA page, sections 1.1 and 4.4: the concept pool
 * holds each concept's extent beside its intent; Parallel FCBO page,
 * section 1.1). For the intents written by fca_enumerate this yields the
 * concepts (B', B).
 *
 *   intents    device pointer, count x W_M words in attribute order (as
 *              fca_enumerate writes them); padding bits past M are ignored.
 *   count      rows of `intents` (0: nothing to do).
 *   extents    device pointer, count x W_N words (W_N = ceil(N/32)),
 *              caller-owned: row r receives the extent of row r, object o
 *              being bit (o & 31) of word (o >> 5); padding bits are 0.
 *   stream     cudaStream_t (NULL = legacy default stream).
 * The work is enqueued on `stream` and the call returns without waiting;
 * it reads the context's table, so it must be ordered after any
 * fca_context_load that precedes it (the same stream does that).
 * FCA_ERR_INVALID for NULL pointers with count > 0.
 */
fca_status fca_extents(fca_ctx *ctx, const uint32_t *intents, uint64_t count, uint32_t *extents, void *stream);

/*
 * The cover relation of the concept lattice (its Hasse diagram): the
 * edges (i, j) such that concept j lies directly below concept i, i.e.
 * intent i is a proper subset of intent j and no intent lies strictly
 * between them (FCbO-to-CUDA page, section 4.4, and Parallel FCBO page,
 * section 3.4: the lattice's edges are rebuilt from the concepts after the
 * search, because the search tree's links are not them).
 *
 *   intents    device pointer, count x W_M words in attribute order: every
 *              intent of the context, each once, in any order (the output
 *              of fca_enumerate). 1 <= count < 2^32 - 1.
 *   edges      device pointer, capacity x 2 uint32, caller-owned: edge e is
 *              (edges[2e], edges[2e+1]) = (row of the upper concept, row of
 *              the lower concept) in `intents`. Edge order is unspecified.
 *   capacity   edges available (0 allowed: count only).
 *   out_edges  host pointer; receives the number of edges, also when it
 *              exceeds `capacity` (then FCA_ERR_CAPACITY, the first
 *              `capacity` edges written).
 *   stream     cudaStream_t (NULL = legacy default stream).
 * Uses stream-ordered device scratch (about 8 bytes per intent, plus
 * 16 W_N bytes for each warp of the kernel's grid, which is sized to the
 * warps resident on the GPU) and returns after the work on `stream`
 * completes. It reads the context's table, so it must be ordered after
 * any fca_context_load that precedes it (the same stream does that).
 * FCA_ERR_INVALID when a cover's intent is not in the given set (the set
 * was not complete) or when an intent is given more than once (the edges
 * are then not computed; *out_edges is not meaningful).
 */
fca_status fca_cover_edges(fca_ctx *ctx, const uint32_t *intents, uint64_t count, uint32_t *edges,
                           uint64_t capacity, uint64_t *out_edges, void *stream);

/*
 * Set an option of a context (fca_option).
 *
 * FCA_OPT_WAIT_LIMIT_NS: in launches that hand work between the warps of a
 * thread block, a warp with nothing left to do waits for a hand-over or for
 * the block's busy warps to finish. The wait is bounded: past the limit the
 * warp stops waiting and the call returns FCA_ERR_CUDA with a message in
 * fca_last_error (the kernel records the fault instead of hanging; the
 * context stays usable). The default, 1 s, is far above the time of any one
 * subtree search; the environment variable FCA_WAIT_LIMIT_NS sets it before
 * creation.
 *
 * FCA_OPT_ATTR_ORDER: the search runs over the attributes in a processing
 * order: attribute order (0), or ascending support (number of objects holding
 * the attribute; ties by index), computed on the device (2). Every output
 * intent is mapped back to attribute order, so the output set does not depend
 * on the order, while the number of evaluated candidates (closures) does: a
 * search that meets rare attributes first fails far fewer canonical tests
 * (the usual ordering heuristic of Close-by-One implementations). With 1, the
 * default, the support order is taken when the supports vary (coefficient of
 * variation above 0.25); on evenly dense tables the reordering saves little
 * and costs three kernels per call. The choice is made by the table load at
 * creation, or by the next fca_context_load after the option is set (with 1
 * it reads the supports back, one synchronisation), and kept for later loads.
 * FCA_ATTR_ORDER=0, 1 or 2 in the environment sets the option before creation.
 *
 * Pools start at the initial sizes
 * (rounded up to at least 4*M entries) and grow on demand up to the limit;
 * past the limit a frontier level is expanded in smaller chunks. Changing a
 * pool option frees the pools, which are allocated again by the next
 * enumerate call. The same sizes can be set before creation through the
 * environment variables FCA_LEVEL_BYTES, FCA_QUEUE_ENTRIES and
 * FCA_POOL_LIMIT_BYTES. FCA_ERR_INVALID for an unknown option or a negative
 * value; FCA_ERR_OOM from enumerate when the limit cannot hold the children
 * of a single search node.
 */
fca_status fca_set_option(fca_ctx *ctx, int option, int64_t value);

/*
 * Enumerate every intent of a small context without allocating any memory.
 * The paper has no counterpart: this entry point serves callers that may not
 * call cudaMalloc/cudaFree while they run, because their device memory is
 * owned entirely by another allocator (a framework's caching allocator or a
 * fixed arena reserved at start-up) or because they run on a latency-critical
 * path where an allocation, which can synchronize the device, is not allowed.
 *
 *   rows       N x W_M uint32 words as for fca_context_create (host or device
 *              pointer); padding bits past M are ignored.
 *   n_objects  1 <= N <= 64 (the whole search is one object-list subtree).
 *   n_attrs    1 <= M <= 1024.
 *   out, capacity, out_count, stream: as for fca_enumerate (out on the device).
 * Larger sizes return FCA_ERR_INVALID. Its scratch (under 10 KB) is one
 * file-scope device array, held by every GPU that loads the library until the
 * process exits; the first call on a device looks up that array's device
 * address, so make that first call before any stream capture. The address is
 * kept for the life of the process: after a cudaDeviceReset (which also ends
 * every context of this library on that device) do not call the library on
 * that device again. All calls on a device share the array and rewrite it:
 * calls whose GPU work overlaps in time race. The call returns after the work
 * on `stream` completes.
 */
fca_status fca_enumerate_small_noalloc(const uint32_t *rows, int64_t n_objects, int32_t n_attrs,
                                       uint32_t *out, uint64_t capacity, uint64_t *out_count,
                                       void *stream);

/* Statistics of the last enumerate call (zeros before the first). */
fca_status fca_get_stats(const fca_ctx *ctx, fca_stats *out);

/* N and M of the context. */
fca_status fca_context_dims(const fca_ctx *ctx, int64_t *n_objects, int32_t *n_attrs);

/*
 * Copy the context's device tables into `dst` (host or device pointer), in
 * processing order (FCA_OPT_ATTR_ORDER): which = 0 -> rows (N x W_M words),
 * 1 -> columns (M x W_Np words, W_Np = W_N rounded up to a multiple of 4),
 * 2 -> top intent (W_M words), 3 -> the processing order (M words: the
 * position of each attribute). `dst_words` is the room in `dst`;
 * FCA_ERR_INVALID if too small.
 */
fca_status fca_context_copy(const fca_ctx *ctx, int which, uint32_t *dst, uint64_t dst_words);

/* Text of the last error on this context ("" when none). Valid until the next call. */
const char *fca_last_error(const fca_ctx *ctx);

/* Release the context and everything it holds. NULL is ignored. */
void fca_free(fca_ctx *ctx);

/* Static description of a status code. */
const char *fca_status_string(fca_status s);

#ifdef __cplusplus
}
#endif

#endif /* FCA_H */
