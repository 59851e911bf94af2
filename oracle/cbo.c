/*
 * CPU oracle: plain recursive Close-by-One over a formal context.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously correct
 * definition that the CUDA library is checked against. Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg load it. It shares no
 * code, header or table with the library.
 *
 * What it computes (FCbO-to-CUDA page, sections 1.1-1.2; Parallel FCBO page,
 * section 1.1): every intent B of the context, i.e. every attribute set with
 * B'' = B, where Y' is the set of objects having all attributes of Y and X'
 * is the set of attributes common to all objects of X.
 *
 * How (FCbO-to-CUDA page, sections 2.1-2.3 and 4.3; Parallel FCBO page,
 * section 1.2):
 *   top concept: A = all objects, B = A' ; visit(A, B, 0)
 *   visit(A, B, y):
 *     output B
 *     for j = y .. M-1:
 *       if j in B: skip             -- A is already inside column j, so
 *                                      adding j cannot shrink the extent
 *                                      (the saturation pruning, section 2.3)
 *       C = A & column j            -- extent intersection
 *       D = C'                      -- AND of the rows of the objects of C;
 *                                      the empty extent gives all M attributes
 *       if D and B agree on attributes 0..j-1 (bit j itself excluded,
 *          section 4.3): visit(C, D, j+1)
 *
 * Readings of points the pages leave open:
 *   - bit order: attribute a is bit (a & 31) of 32-bit word (a >> 5), LSB
 *     first; objects likewise (section 4.3 mask, Parallel FCBO section 3.1);
 *   - the child's cursor is j+1 (the child extends attributes after j);
 *   - the top concept is output first, and the bottom concept (all M
 *     attributes, possibly with an empty extent) is output whenever the
 *     recursion reaches it;
 *   - padding bits past M in the input rows are ignored; output padding is 0;
 *   - word counts are ceil(N/32) / ceil(M/32) (never floor).
 *
 * Internally the sets are 64-bit words (its own bitset code). Multi-thread
 * mode splits the top level loop over j between threads: subtrees below
 * distinct top-level candidates are independent because the canonical test
 * uses only the local state (A, B, j) (FCbO-to-CUDA page, section 2.2).
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t n;       /* objects */
    int32_t m;       /* attributes */
    int64_t wn;      /* 64-bit words of an extent */
    int32_t wm;      /* 64-bit words of an intent */
    uint64_t *rows;  /* n x wm : row o = attribute set of object o */
    uint64_t *cols;  /* m x wn : column j = object set of attribute j */
    uint64_t last_attr_mask; /* valid bits of the last intent word */
} octx;

typedef struct {
    uint64_t *intents;   /* count x wm */
    uint64_t *extents;   /* count x wn, only when wanted */
    uint64_t count, cap;
    uint64_t closures;   /* candidates (A, B, j) with j >= y, j not in B */
    uint64_t *depth_counts; /* m + 2 entries */
    int want_extents;
    int oom;
    uint64_t limit;      /* stop descending once this many intents are output (0 = no limit) */
    int digest_only;     /* keep no intents; accumulate an order-independent digest instead */
    int32_t words32;     /* 32-bit words of an intent (for the digest) */
    uint64_t hsum, hxor; /* sum and xor of the per-intent hashes */
    const int32_t *label; /* digest only, optional: attribute at position r is label[r] */
    uint64_t *relabeled; /* scratch for the renumbered intent (wm words) */
} osink;

/* splitmix64 finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom number generators"). */
static uint64_t mix64(uint64_t z)
{
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    z ^= z >> 31;
    return z;
}

/* Hash of one intent: its 32-bit words folded in order, then the word count. */
static uint64_t intent_hash(const uint64_t *intent, int32_t words32)
{
    uint64_t h = 0x9E3779B97F4A7C15ull;
    for (int32_t i = 0; i < words32; ++i) {
        uint64_t w = (intent[i >> 1] >> (32 * (i & 1))) & 0xFFFFFFFFull;
        h = mix64(h ^ w);
    }
    return mix64(h + (uint64_t)words32);
}

static int bit_of(const uint64_t *set, int64_t i) { return (int)((set[i >> 6] >> (i & 63)) & 1u); }

/* Y' for one attribute: the stored column. X' : AND of the rows of X. */
static void intent_of(const octx *c, const uint64_t *extent, uint64_t *out)
{
    for (int32_t w = 0; w < c->wm; ++w) out[w] = ~(uint64_t)0;
    out[c->wm - 1] = c->last_attr_mask;          /* empty extent -> all M */
    for (int64_t ew = 0; ew < c->wn; ++ew) {      /* every set bit o of the extent */
        uint64_t x = extent[ew];
        while (x) {
            int64_t o = ew * 64 + __builtin_ctzll(x);
            x &= x - 1u;
            const uint64_t *row = c->rows + (size_t)o * (size_t)c->wm;
            for (int32_t w = 0; w < c->wm; ++w) out[w] &= row[w];
        }
    }
}

/* D and B agree on attributes 0 .. j-1 (attribute j itself not compared). */
static int same_prefix(const uint64_t *d, const uint64_t *b, int32_t j)
{
    int32_t full = j >> 6;
    for (int32_t w = 0; w < full; ++w)
        if (d[w] != b[w]) return 0;
    uint64_t mask = (j & 63) ? ((((uint64_t)1) << (j & 63)) - 1u) : 0u;
    return (d[full] & mask) == (b[full] & mask);
}

static void sink_emit(const octx *c, osink *s, const uint64_t *extent, const uint64_t *intent,
                      int depth)
{
    if (s->oom) return;
    if (s->digest_only) {
        if (s->label) {   /* hash the intent with its attributes renumbered */
            memset(s->relabeled, 0, (size_t)c->wm * sizeof(uint64_t));
            for (int32_t r = 0; r < c->m; ++r)
                if (bit_of(intent, r)) {
                    int32_t a = s->label[r];
                    s->relabeled[a >> 6] |= ((uint64_t)1) << (a & 63);
                }
            intent = s->relabeled;
        }
        uint64_t h = intent_hash(intent, s->words32);
        s->hsum += h;
        s->hxor ^= h;
        s->count += 1;
        s->depth_counts[depth] += 1;
        return;
    }
    if (s->count == s->cap) {
        uint64_t ncap = s->cap ? s->cap * 2 : 1024;
        uint64_t *ni = (uint64_t *)realloc(s->intents, ncap * (size_t)c->wm * sizeof(uint64_t));
        if (!ni) { s->oom = 1; return; }
        s->intents = ni;
        if (s->want_extents) {
            uint64_t *ne = (uint64_t *)realloc(s->extents, ncap * (size_t)c->wn * sizeof(uint64_t));
            if (!ne) { s->oom = 1; return; }
            s->extents = ne;
        }
        s->cap = ncap;
    }
    memcpy(s->intents + s->count * (size_t)c->wm, intent, (size_t)c->wm * sizeof(uint64_t));
    if (s->want_extents)
        memcpy(s->extents + s->count * (size_t)c->wn, extent, (size_t)c->wn * sizeof(uint64_t));
    s->count += 1;
    s->depth_counts[depth] += 1;
}

/* Scratch: one (C, D) pair per recursion depth, depth <= m + 1. */
typedef struct { uint64_t *ext; uint64_t *itt; } oframe;

static void visit(const octx *c, osink *s, oframe *stack, const uint64_t *a, const uint64_t *b,
                  int32_t y, int depth)
{
    sink_emit(c, s, a, b, depth);
    if (s->limit && s->count >= s->limit) return;   /* bounded sample (timing only) */
    uint64_t *cc = stack[depth + 1].ext;
    uint64_t *dd = stack[depth + 1].itt;
    for (int32_t j = y; j < c->m; ++j) {
        if (bit_of(b, j)) continue;
        s->closures += 1;
        const uint64_t *col = c->cols + (size_t)j * (size_t)c->wn;
        for (int64_t w = 0; w < c->wn; ++w) cc[w] = a[w] & col[w];
        intent_of(c, cc, dd);
        if (same_prefix(dd, b, j)) visit(c, s, stack, cc, dd, j + 1, depth + 1);
    }
}

static int build_ctx(octx *c, const uint32_t *rows32, int64_t n, int32_t m)
{
    c->n = n;
    c->m = m;
    c->wn = (n + 63) / 64;
    c->wm = (m + 63) / 64;
    c->last_attr_mask = (m % 64) ? ((((uint64_t)1) << (m % 64)) - 1u) : ~(uint64_t)0;
    c->rows = (uint64_t *)calloc((size_t)n * (size_t)c->wm, sizeof(uint64_t));
    c->cols = (uint64_t *)calloc((size_t)m * (size_t)c->wn, sizeof(uint64_t));
    if (!c->rows || !c->cols) return -1;
    int64_t w32 = (m + 31) / 32;
    for (int64_t o = 0; o < n; ++o) {
        for (int32_t a = 0; a < m; ++a) {
            uint32_t word = rows32[(size_t)o * (size_t)w32 + (size_t)(a >> 5)];
            if ((word >> (a & 31)) & 1u) {
                c->rows[(size_t)o * (size_t)c->wm + (size_t)(a >> 6)] |= ((uint64_t)1) << (a & 63);
                c->cols[(size_t)a * (size_t)c->wn + (size_t)(o >> 6)] |= ((uint64_t)1) << (o & 63);
            }
        }
    }
    return 0;
}

static void free_ctx(octx *c) { free(c->rows); free(c->cols); }

static oframe *alloc_stack(const octx *c)
{
    int frames = c->m + 2;
    oframe *st = (oframe *)calloc((size_t)frames, sizeof(oframe));
    if (!st) return NULL;
    for (int i = 0; i < frames; ++i) {
        st[i].ext = (uint64_t *)calloc((size_t)c->wn, sizeof(uint64_t));
        st[i].itt = (uint64_t *)calloc((size_t)c->wm, sizeof(uint64_t));
        if (!st[i].ext || !st[i].itt) return NULL;
    }
    return st;
}

static void free_stack(const octx *c, oframe *st)
{
    if (!st) return;
    for (int i = 0; i < c->m + 2; ++i) { free(st[i].ext); free(st[i].itt); }
    free(st);
}

/* Thread mode: the top concept is output once; threads share the top-level j loop. */
typedef struct {
    const octx *c;
    const uint64_t *top_ext, *top_int;
    osink sink;
    pthread_mutex_t *lock;
    int32_t *next_j;
    int fail;
} oworker;

static void *worker_main(void *arg)
{
    oworker *wk = (oworker *)arg;
    const octx *c = wk->c;
    oframe *stack = alloc_stack(c);
    if (!stack) { wk->fail = 1; return NULL; }
    for (;;) {
        pthread_mutex_lock(wk->lock);
        int32_t j = (*wk->next_j)++;
        pthread_mutex_unlock(wk->lock);
        if (j >= c->m) break;
        if (wk->sink.limit && wk->sink.count >= wk->sink.limit) break;
        if (bit_of(wk->top_int, j)) continue;
        wk->sink.closures += 1;
        uint64_t *cc = stack[1].ext, *dd = stack[1].itt;
        const uint64_t *col = c->cols + (size_t)j * (size_t)c->wn;
        for (int64_t w = 0; w < c->wn; ++w) cc[w] = wk->top_ext[w] & col[w];
        intent_of(c, cc, dd);
        if (same_prefix(dd, wk->top_int, j)) visit(c, &wk->sink, stack, cc, dd, j + 1, 1);
    }
    free_stack(c, stack);
    return NULL;
}

static void to_words32(const uint64_t *src, uint64_t count, int32_t wm64, int64_t w32,
                       uint32_t *dst)
{
    for (uint64_t i = 0; i < count; ++i)
        for (int64_t w = 0; w < w32; ++w) {
            uint64_t x = src[i * (size_t)wm64 + (size_t)(w >> 1)];
            dst[i * (size_t)w32 + (size_t)w] = (uint32_t)((w & 1) ? (x >> 32) : x);
        }
}

/*
 * Enumerate all intents.
 *   rows32        n x ceil(m/32) uint32 words, LSB-first, padding ignored.
 *   threads       1 = single recursive pass; >1 = top-level split.
 *   want_extents  also return each intent's extent (ceil(n/32) words).
 * Outputs (malloc'd, free with oracle_free): intents count x ceil(m/32),
 * extents count x ceil(n/32) or NULL; closures; depth_counts[m+2] (caller array).
 * Returns 0, or -1 on bad arguments / allocation failure.
 * `limit` > 0 stops each thread once it has output `limit` intents: a bounded
 * sample of the search for timing; the result is then incomplete.
 */
int oracle_cbo_limited(const uint32_t *rows32, int64_t n, int32_t m, int threads, int want_extents,
                       uint64_t limit, uint32_t **out_intents, uint32_t **out_extents,
                       uint64_t *out_count, uint64_t *out_closures, uint64_t *depth_counts);

static int run_cbo(const uint32_t *rows32, int64_t n, int32_t m, int threads, int want_extents,
                   uint64_t limit, int digest_only, const int32_t *label, uint32_t **out_intents,
                   uint32_t **out_extents, uint64_t *out_count, uint64_t *out_closures,
                   uint64_t *depth_counts, uint64_t *hsum, uint64_t *hxor);

int oracle_cbo(const uint32_t *rows32, int64_t n, int32_t m, int threads, int want_extents,
               uint32_t **out_intents, uint32_t **out_extents, uint64_t *out_count,
               uint64_t *out_closures, uint64_t *depth_counts)
{
    return oracle_cbo_limited(rows32, n, m, threads, want_extents, 0, out_intents, out_extents,
                              out_count, out_closures, depth_counts);
}

int oracle_cbo_limited(const uint32_t *rows32, int64_t n, int32_t m, int threads, int want_extents,
                       uint64_t limit, uint32_t **out_intents, uint32_t **out_extents,
                       uint64_t *out_count, uint64_t *out_closures, uint64_t *depth_counts)
{
    return run_cbo(rows32, n, m, threads, want_extents, limit, 0, NULL, out_intents, out_extents,
                   out_count, out_closures, depth_counts, NULL, NULL);
}

/*
 * Same search, keeping no intents: returns their number, the closures, the depth
 * counts and an order-independent digest of the intent set (the sum and the xor,
 * modulo 2^64, of one 64-bit hash per intent), for workloads whose intents do not
 * fit in host memory.
 */
int oracle_cbo_digest(const uint32_t *rows32, int64_t n, int32_t m, int threads, uint64_t *out_count,
                      uint64_t *out_closures, uint64_t *depth_counts, uint64_t *hsum, uint64_t *hxor)
{
    if (!hsum || !hxor) return -1;
    return run_cbo(rows32, n, m, threads, 0, 0, 1, NULL, NULL, NULL, out_count, out_closures,
                   depth_counts, hsum, hxor);
}

/*
 * The digest of a table whose attributes were renumbered (columns listed in another order), taken
 * over the intents in the original numbering: label[r] is the original number of the attribute at
 * position r (a permutation of 0 .. m-1). The set of intents does not depend on the order in which
 * the search takes the attributes, so the digest equals that of the original table, while the
 * closures counted are those of the search in the given order.
 */
int oracle_cbo_digest_relabel(const uint32_t *rows32, int64_t n, int32_t m, int threads,
                              const int32_t *label, uint64_t *out_count, uint64_t *out_closures,
                              uint64_t *depth_counts, uint64_t *hsum, uint64_t *hxor)
{
    if (!hsum || !hxor || !label || m < 1) return -1;
    char *seen = (char *)calloc((size_t)m, 1);
    if (!seen) return -1;
    int ok = 1;
    for (int32_t r = 0; r < m; ++r) {
        if (label[r] < 0 || label[r] >= m || seen[label[r]]) ok = 0;
        else seen[label[r]] = 1;
    }
    free(seen);
    if (!ok) return -1;
    return run_cbo(rows32, n, m, threads, 0, 0, 1, label, NULL, NULL, out_count, out_closures,
                   depth_counts, hsum, hxor);
}

static int run_cbo(const uint32_t *rows32, int64_t n, int32_t m, int threads, int want_extents,
                   uint64_t limit, int digest_only, const int32_t *label, uint32_t **out_intents,
                   uint32_t **out_extents, uint64_t *out_count, uint64_t *out_closures,
                   uint64_t *depth_counts, uint64_t *hsum, uint64_t *hxor)
{
    if (!rows32 || n < 1 || m < 1 || (!digest_only && !out_intents) || !out_count || !out_closures ||
        !depth_counts)
        return -1;
    octx c;
    if (build_ctx(&c, rows32, n, m) != 0) { free_ctx(&c); return -1; }
    memset(depth_counts, 0, (size_t)(m + 2) * sizeof(uint64_t));

    uint64_t *top_ext = (uint64_t *)calloc((size_t)c.wn, sizeof(uint64_t));
    uint64_t *top_int = (uint64_t *)calloc((size_t)c.wm, sizeof(uint64_t));
    if (!top_ext || !top_int) { free(top_ext); free(top_int); free_ctx(&c); return -1; }
    for (int64_t o = 0; o < n; ++o) top_ext[o >> 6] |= ((uint64_t)1) << (o & 63);
    intent_of(&c, top_ext, top_int);

    int nthr = threads < 1 ? 1 : threads;
    oworker *wks = (oworker *)calloc((size_t)nthr, sizeof(oworker));
    if (!wks) { free(top_ext); free(top_int); free_ctx(&c); return -1; }
    for (int t = 0; t < nthr; ++t) {
        wks[t].sink.want_extents = want_extents;
        wks[t].sink.limit = limit;
        wks[t].sink.digest_only = digest_only;
        wks[t].sink.words32 = (m + 31) / 32;
        wks[t].sink.depth_counts = (uint64_t *)calloc((size_t)(m + 2), sizeof(uint64_t));
        wks[t].sink.label = label;
        wks[t].sink.relabeled = (uint64_t *)calloc((size_t)c.wm, sizeof(uint64_t));
        if (!wks[t].sink.depth_counts || !wks[t].sink.relabeled) wks[t].sink.oom = 1;
    }
    int rc = 0;
    if (nthr == 1) {
        oframe *stack = alloc_stack(&c);
        if (!stack) rc = -1;
        else visit(&c, &wks[0].sink, stack, top_ext, top_int, 0, 0);
        free_stack(&c, stack);
    } else {
        /* the top concept itself, then the shared top-level loop */
        sink_emit(&c, &wks[0].sink, top_ext, top_int, 0);
        pthread_mutex_t lock = PTHREAD_MUTEX_INITIALIZER;
        int32_t next_j = 0;
        pthread_t *tid = (pthread_t *)calloc((size_t)nthr, sizeof(pthread_t));
        for (int t = 0; t < nthr; ++t) {
            wks[t].c = &c;
            wks[t].top_ext = top_ext;
            wks[t].top_int = top_int;
            wks[t].lock = &lock;
            wks[t].next_j = &next_j;
            pthread_create(&tid[t], NULL, worker_main, &wks[t]);
        }
        for (int t = 0; t < nthr; ++t) pthread_join(tid[t], NULL);
        free(tid);
    }

    uint64_t total = 0, closures = 0, hs = 0, hx = 0;
    for (int t = 0; t < nthr; ++t) {
        if (wks[t].fail || wks[t].sink.oom) rc = -1;
        total += wks[t].sink.count;
        hs += wks[t].sink.hsum;
        hx ^= wks[t].sink.hxor;
        closures += wks[t].sink.closures;
        for (int d = 0; d < m + 2; ++d) depth_counts[d] += wks[t].sink.depth_counts[d];
    }
    int64_t w32m = (m + 31) / 32, w32n = (n + 31) / 32;
    uint32_t *oi = NULL, *oe = NULL;
    for (int t = 0; t < nthr; ++t) free(wks[t].sink.relabeled);
    if (digest_only) {
        for (int t = 0; t < nthr; ++t) free(wks[t].sink.depth_counts);
        free(wks);
        free(top_ext);
        free(top_int);
        free_ctx(&c);
        if (rc != 0) return -1;
        *out_count = total;
        *out_closures = closures;
        *hsum = hs;
        *hxor = hx;
        return 0;
    }
    if (rc == 0) {
        oi = (uint32_t *)malloc((size_t)(total ? total : 1) * (size_t)w32m * sizeof(uint32_t));
        if (want_extents)
            oe = (uint32_t *)malloc((size_t)(total ? total : 1) * (size_t)w32n * sizeof(uint32_t));
        if (!oi || (want_extents && !oe)) rc = -1;
    }
    uint64_t at = 0;
    for (int t = 0; t < nthr; ++t) {
        if (rc == 0) {
            to_words32(wks[t].sink.intents, wks[t].sink.count, c.wm, w32m, oi + at * (size_t)w32m);
            if (want_extents)
                to_words32(wks[t].sink.extents, wks[t].sink.count, (int32_t)c.wn, w32n,
                           oe + at * (size_t)w32n);
        }
        at += wks[t].sink.count;
        free(wks[t].sink.intents);
        free(wks[t].sink.extents);
        free(wks[t].sink.depth_counts);
    }
    free(wks);
    free(top_ext);
    free(top_int);
    free_ctx(&c);
    if (rc != 0) { free(oi); free(oe); return -1; }
    *out_intents = oi;
    if (out_extents) *out_extents = oe; else free(oe);
    *out_count = total;
    *out_closures = closures;
    return 0;
}

void oracle_free(void *p) { free(p); }
