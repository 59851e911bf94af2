/*
 * Counting pass: the algorithmic work of Close-by-One enumeration, counted exactly in 32-bit
 * words. TEST AND MEASUREMENT INFRASTRUCTURE ONLY: it gives the roofline its numerator (the words
 * the method must touch) and is pinned by the test suite. It shares no code with the library, nor
 * with the oracle in cbo.c (it runs its own search).
 *
 * The search is plain Close-by-One (FCbO-to-CUDA page, sections 2.1-2.3): node (A, B, y); for each
 * j >= y with j not in B: C = A & column j, D = C', and the child (C, D, j+1) exists iff D adds no
 * attribute below j to B. What is counted, per unit:
 *
 *   parent (every node, when its candidates are evaluated):
 *     hbm   += W_N                    its extent read once, shared by its candidates
 *   candidate (a closure):
 *     isect += nnzw(A)                C = A & column j over the non-zero words of A: one column
 *                                     word read and one AND per word (section 3.1, 4.2)
 *     close += min(|C| * W_M, sum_k s_k)
 *                                     the closure, by rows (AND of |C| rows of W_M words) or by
 *                                     columns, whichever touches fewer words. By columns, k runs
 *                                     over the attributes not in B and not j in ascending order;
 *                                     s_k is the number of non-zero words of C probed for
 *                                     C & ~column k up to and including the first non-zero
 *                                     result, or nnzw(C) when C is inside column k. The sum stops
 *                                     after the first k < j with C inside column k (the canonical
 *                                     test has failed there).
 *     canon += W_M                    the prefix comparison of D and B
 *   canonical child:
 *     hbm   += W_N + W_M + W_M        its frontier entry (extent and intent) and its output row
 *
 * W_N = ceil(N/32), W_M = ceil(M/32), nnzw() = number of non-zero 32-bit words. Every count is
 * split by the tier of the parent: extents of at most 64 objects (object-list tier), of at most
 * mid_max objects (mid tier; none when mid_max <= 64), or larger (bitmap tier).
 *
 * A second model counts what the tiered representation moves instead of an N-bit bitmap per node
 * (the memory-lean frontier: extents of at most list_max objects stored as object-id lists,
 * subtrees of at most 64 objects searched inside one warp):
 *   parent:  hbm_lean += |A| ids (id list: object-list root, mid tier, bitmap tier up to list_max)
 *                        or W_N (bitmap tier above list_max); a node of the object-list tier that
 *                        is not a root (its parent is in that tier too) reads nothing: it lives in
 *                        the searching warp's registers and shared memory;
 *            l2_lean  += |A| * W_M for an object-list root or a parent kept as an id list (the
 *                        rows of its objects, gathered once to build its columns restricted to
 *                        A); for a parent kept as a bitmap, its candidates' intersection and
 *                        closure words as above;
 *   canonical child: hbm_lean += W_M (output row), plus its entry when it leaves the parent's warp
 *                        or block (every child but one of an object-list-tier parent): |C| ids or
 *                        W_N words as above, and W_M intent words.
 *
 * The search keeps each extent as its non-zero words and their indices, so that a candidate costs
 * the host time of its own counts, not a scan of W_N words.
 *
 * Multi-thread mode splits the top-level j loop between threads, as the oracle does; the totals do
 * not depend on the split.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SMALL_EXTENT 64

typedef struct {
    int64_t n, wn;        /* objects, 32-bit words of an extent */
    int32_t m, wm;        /* attributes, 32-bit words of an intent */
    uint32_t *rows;       /* n x wm */
    uint32_t *cols;       /* m x wn */
    uint32_t last_mask;   /* valid bits of the last intent word */
    int64_t mid_max;      /* largest extent of the mid tier */
    int64_t list_max;     /* largest extent stored as an object-id list */
} wctx;

/* Per tier: 0 = object-list tier (|A| <= 64), 1 = mid tier (|A| <= mid_max), 2 = bitmap tier. */
typedef struct {
    uint64_t parents, closures, children;
    uint64_t isect, close, canon, hbm;
    uint64_t hbm_lean, l2_lean;
} wtier;

typedef struct {
    uint32_t *aw;         /* this node's extent: its non-zero words (values) ... */
    int64_t *ai;          /* ... and their word indices, ascending */
    int64_t nza;          /* their number */
    uint32_t *itt;        /* this node's intent (wm words) */
} wframe;

static int popc32(uint32_t x) { return __builtin_popcount(x); }

static int has_attr(const uint32_t *set, int32_t a) { return (int)((set[a >> 5] >> (a & 31)) & 1u); }

/* The tier of a parent with `na` objects: 0 = at most 64, 1 = at most mid_max, 2 = larger. */
static int tier_of(const wctx *c, int64_t na)
{
    if (na <= SMALL_EXTENT) return 0;
    return na <= c->mid_max ? 1 : 2;
}

/* D = AND of the rows of the objects of C (all M attributes when C is empty); C given by its
   non-zero words (values cw, indices ci, nz of them). */
static void closure_rows(const wctx *c, const uint32_t *cw, const int64_t *ci, int64_t nz, uint32_t *d)
{
    for (int32_t w = 0; w < c->wm; ++w) d[w] = 0xffffffffu;
    d[c->wm - 1] = c->last_mask;
    for (int64_t t = 0; t < nz; ++t) {
        uint32_t bits = cw[t];
        while (bits) {
            const int b = __builtin_ctz(bits);
            bits &= bits - 1u;
            const uint32_t *row = c->rows + (size_t)(ci[t] * 32 + b) * c->wm;
            for (int32_t v = 0; v < c->wm; ++v) d[v] &= row[v];
        }
    }
}

/* The column-route word count of one candidate, stopped once it reaches `cap` (the row route). */
static uint64_t column_route(const wctx *c, const uint32_t *b, int32_t j, const uint32_t *cw,
                             const int64_t *ci, int64_t nz, uint64_t cap)
{
    uint64_t sum = 0;
    for (int32_t k = 0; k < c->m && sum < cap; ++k) {
        if (k == j || has_attr(b, k)) continue;
        const uint32_t *col = c->cols + (size_t)k * c->wn;
        int64_t t = 0;
        int inside = 1;
        for (; t < nz; ++t) {
            if (cw[t] & ~col[ci[t]]) { inside = 0; ++t; break; }
        }
        sum += (uint64_t)t;
        if (inside && k < j) break;   /* C inside column k, k < j: not canonical */
    }
    return sum < cap ? sum : cap;
}

/* Words of an extent of `na` objects kept in a frontier entry or queue: its ids, or the bitmap. */
static uint64_t entry_words(const wctx *c, int64_t na)
{
    return (na <= SMALL_EXTENT || na <= c->list_max) ? (uint64_t)na : (uint64_t)c->wn;
}

/* The lean-model reads of a parent of `na` objects in tier `tier` whose parent was in `up`
   (-1 for the top node). */
static void lean_parent(const wctx *c, wtier *t, int tier, int up, int64_t na)
{
    if (tier == 0 && up == 0) return;           /* inside an object-list subtree */
    t->hbm_lean += entry_words(c, na);
    if (tier <= 1 || na <= c->list_max) t->l2_lean += (uint64_t)na * (uint64_t)c->wm;
}

/* The candidates j in [j_begin, m) with step `stride` of the node at `depth` (its extent and intent
   in st[depth]); each candidate's C is built in st[depth + 1], which is the child's frame. */
static void expand(const wctx *c, wtier *tiers, wframe *st, int depth, int32_t j_begin, int32_t stride)
{
    const wframe *f = &st[depth];
    wframe *g = &st[depth + 1];
    int64_t na = 0;
    for (int64_t i = 0; i < f->nza; ++i) na += popc32(f->aw[i]);
    const int tier = tier_of(c, na);
    wtier *t = &tiers[tier];
    for (int32_t j = j_begin; j < c->m; j += stride) {
        if (has_attr(f->itt, j)) continue;
        t->closures++;
        t->isect += (uint64_t)f->nza;
        const uint32_t *col = c->cols + (size_t)j * c->wn;
        int64_t nzc = 0, cnt = 0;
        for (int64_t i = 0; i < f->nza; ++i) {
            const uint32_t v = f->aw[i] & col[f->ai[i]];
            if (v) { g->aw[nzc] = v; g->ai[nzc] = f->ai[i]; ++nzc; cnt += popc32(v); }
        }
        g->nza = nzc;
        const uint64_t rows_words = (uint64_t)cnt * (uint64_t)c->wm;
        const uint64_t close = column_route(c, f->itt, j, g->aw, g->ai, nzc, rows_words);
        t->close += close;
        t->canon += (uint64_t)c->wm;
        if (tier == 2 && na > c->list_max) t->l2_lean += (uint64_t)f->nza + close;
        closure_rows(c, g->aw, g->ai, nzc, g->itt);
        /* canonical iff D and B agree below j (D contains B) */
        int canonical = 1;
        for (int32_t w = 0; w <= (j >> 5) && canonical; ++w) {
            uint32_t below = w < (j >> 5) ? 0xffffffffu : ((1u << (j & 31)) - 1u);
            if ((g->itt[w] ^ f->itt[w]) & below) canonical = 0;
        }
        if (!canonical) continue;
        t->children++;
        t->hbm += (uint64_t)c->wn + 2u * (uint64_t)c->wm;
        const int ctier = tier_of(c, cnt);
        t->hbm_lean += (uint64_t)c->wm;
        if (!(tier == 0 && ctier == 0)) t->hbm_lean += entry_words(c, cnt) + (uint64_t)c->wm;
        /* the child: a parent of its own */
        wtier *tc = &tiers[ctier];
        tc->parents++;
        tc->hbm += (uint64_t)c->wn;
        lean_parent(c, tc, ctier, tier, cnt);
        expand(c, tiers, st, depth + 1, j + 1, 1);
    }
}

typedef struct {
    const wctx *c;
    int32_t j0, stride;
    wtier tiers[3];
    int err;
} wjob;

static wframe *alloc_frames(const wctx *c)
{
    const int depth = c->m + 2;
    wframe *st = (wframe *)calloc((size_t)depth, sizeof(wframe));
    if (!st) return NULL;
    for (int i = 0; i < depth; ++i) {
        st[i].aw = (uint32_t *)calloc((size_t)c->wn, sizeof(uint32_t));
        st[i].ai = (int64_t *)calloc((size_t)c->wn, sizeof(int64_t));
        st[i].itt = (uint32_t *)calloc((size_t)c->wm, sizeof(uint32_t));
        if (!st[i].aw || !st[i].ai || !st[i].itt) return NULL;
    }
    return st;
}

static void free_frames(const wctx *c, wframe *st)
{
    if (!st) return;
    for (int i = 0; i < c->m + 2; ++i) {
        free(st[i].aw);
        free(st[i].ai);
        free(st[i].itt);
    }
    free(st);
}

/* Thread `j0` of `stride`: the top node's candidates j = j0, j0 + stride, ... and their subtrees.
   Thread 0 also counts the top node as a parent. */
static void *worker(void *arg)
{
    wjob *job = (wjob *)arg;
    const wctx *c = job->c;
    wframe *st = alloc_frames(c);
    if (!st) { job->err = 1; free_frames(c, st); return NULL; }
    wframe *f = &st[0];
    for (int64_t w = 0; w < c->wn; ++w) {
        f->aw[w] = 0xffffffffu;
        f->ai[w] = w;
    }
    if (c->n & 31) f->aw[c->wn - 1] = (1u << (c->n & 31)) - 1u;
    f->nza = c->wn;
    closure_rows(c, f->aw, f->ai, f->nza, f->itt);
    if (job->j0 == 0) {
        const int tier = tier_of(c, c->n);
        wtier *t = &job->tiers[tier];
        t->parents++;
        t->hbm += (uint64_t)c->wn;
        lean_parent(c, t, tier, -1, c->n);
    }
    expand(c, job->tiers, st, 0, job->j0, job->stride);
    free_frames(c, st);
    return NULL;
}

/* Count the work of enumerating the context `rows32` (n x ceil(m/32) words, LSB-first; padding
   bits ignored). out[3][7] receives, per tier (0: extents <= 64 objects, 1: <= mid_max objects,
   2: larger), parents, closures, canonical children, intersection words, closure words, canonical-
   test words, HBM words, and the lean model's HBM and L2 words, in that order (out[3][9]). Returns
   0, or -1 on bad arguments or memory exhaustion. The top concept is a parent; its own output row
   is not counted (it is not a child). */
int workcount(const uint32_t *rows32, int64_t n, int32_t m, int threads, int64_t mid_max, int64_t list_max,
              uint64_t *out)
{
    if (!rows32 || n < 1 || m < 1 || !out) return -1;
    if (threads < 1) threads = 1;
    wctx c;
    c.n = n;
    c.m = m;
    c.wn = (n + 31) / 32;
    c.wm = (m + 31) / 32;
    c.last_mask = (m & 31) ? ((1u << (m & 31)) - 1u) : 0xffffffffu;
    c.mid_max = mid_max;
    c.list_max = list_max;
    c.rows = (uint32_t *)calloc((size_t)n * (size_t)c.wm, sizeof(uint32_t));
    c.cols = (uint32_t *)calloc((size_t)m * (size_t)c.wn, sizeof(uint32_t));
    if (!c.rows || !c.cols) { free(c.rows); free(c.cols); return -1; }
    for (int64_t o = 0; o < n; ++o) {
        for (int32_t w = 0; w < c.wm; ++w) {
            uint32_t v = rows32[(size_t)o * c.wm + w];
            if (w == c.wm - 1) v &= c.last_mask;
            c.rows[(size_t)o * c.wm + w] = v;
            while (v) {
                const int b = __builtin_ctz(v);
                v &= v - 1u;
                const int32_t a = w * 32 + b;
                c.cols[(size_t)a * c.wn + (o >> 5)] |= 1u << (o & 31);
            }
        }
    }
    wjob *jobs = (wjob *)calloc((size_t)threads, sizeof(wjob));
    pthread_t *tid = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    int err = (!jobs || !tid);
    for (int i = 0; i < threads && !err; ++i) {
        jobs[i].c = &c;
        jobs[i].j0 = i;
        jobs[i].stride = threads;
    }
    int started = 0;
    for (int i = 1; i < threads && !err; ++i, ++started)
        if (pthread_create(&tid[i], NULL, worker, &jobs[i]) != 0) { err = 1; break; }
    if (!err) worker(&jobs[0]);
    for (int i = 1; i <= started; ++i) pthread_join(tid[i], NULL);
    if (!err) {
        memset(out, 0, sizeof(uint64_t) * 27);
        for (int i = 0; i < threads; ++i) {
            err |= jobs[i].err;
            for (int k = 0; k < 3; ++k) {
                const wtier *t = &jobs[i].tiers[k];
                uint64_t *o = out + 9 * k;
                o[0] += t->parents;
                o[1] += t->closures;
                o[2] += t->children;
                o[3] += t->isect;
                o[4] += t->close;
                o[5] += t->canon;
                o[6] += t->hbm;
                o[7] += t->hbm_lean;
                o[8] += t->l2_lean;
            }
        }
    }
    free(jobs);
    free(tid);
    free(c.rows);
    free(c.cols);
    return err ? -1 : 0;
}
