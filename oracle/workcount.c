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
 * split by the tier of the parent: extents of more than 64 objects (bitmap tier) or at most 64
 * (object-list tier).
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
} wctx;

/* Per tier: 0 = object-list tier (|A| <= 64), 1 = bitmap tier. */
typedef struct {
    uint64_t parents, closures, children;
    uint64_t isect, close, canon, hbm;
} wtier;

typedef struct {
    uint32_t *ext, *itt;  /* extent (wn) and intent (wm) of the node at this depth */
    uint32_t *cw;         /* non-zero words of C (values) */
    int64_t *ci;          /* their word indices */
    int64_t *ai;          /* non-zero word indices of this node's extent */
} wframe;

static int popc32(uint32_t x) { return __builtin_popcount(x); }

static int has_attr(const uint32_t *set, int32_t a) { return (int)((set[a >> 5] >> (a & 31)) & 1u); }

/* D = AND of the rows of the objects of C (all M attributes when C is empty). */
static void closure_rows(const wctx *c, const uint32_t *ext, uint32_t *d)
{
    for (int32_t w = 0; w < c->wm; ++w) d[w] = 0xffffffffu;
    d[c->wm - 1] = c->last_mask;
    for (int64_t w = 0; w < c->wn; ++w) {
        uint32_t bits = ext[w];
        while (bits) {
            const int b = __builtin_ctz(bits);
            bits &= bits - 1u;
            const uint32_t *row = c->rows + (size_t)(w * 32 + b) * c->wm;
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

static void visit(const wctx *c, wtier *tiers, wframe *st, int depth, int32_t y)
{
    wframe *f = &st[depth];
    const uint32_t *a = f->ext, *b = f->itt;
    int64_t na = 0, nza = 0;
    for (int64_t w = 0; w < c->wn; ++w) {
        if (a[w]) { f->ai[nza++] = w; na += popc32(a[w]); }
    }
    wtier *t = &tiers[na > SMALL_EXTENT ? 1 : 0];
    t->parents++;
    t->hbm += (uint64_t)c->wn;
    wframe *g = &st[depth + 1];
    for (int32_t j = y; j < c->m; ++j) {
        if (has_attr(b, j)) continue;
        t->closures++;
        t->isect += (uint64_t)nza;
        const uint32_t *col = c->cols + (size_t)j * c->wn;
        memset(g->ext, 0, sizeof(uint32_t) * (size_t)c->wn);
        int64_t nzc = 0, cnt = 0;
        for (int64_t i = 0; i < nza; ++i) {
            const int64_t w = f->ai[i];
            const uint32_t v = a[w] & col[w];
            g->ext[w] = v;
            if (v) { f->cw[nzc] = v; f->ci[nzc] = w; ++nzc; cnt += popc32(v); }
        }
        const uint64_t rows_words = (uint64_t)cnt * (uint64_t)c->wm;
        t->close += column_route(c, b, j, f->cw, f->ci, nzc, rows_words);
        t->canon += (uint64_t)c->wm;
        closure_rows(c, g->ext, g->itt);
        /* canonical iff D and B agree below j (D contains B) */
        int canonical = 1;
        for (int32_t w = 0; w <= (j >> 5) && canonical; ++w) {
            uint32_t below = w < (j >> 5) ? 0xffffffffu : ((1u << (j & 31)) - 1u);
            if ((g->itt[w] ^ b[w]) & below) canonical = 0;
        }
        if (!canonical) continue;
        t->children++;
        t->hbm += (uint64_t)c->wn + 2u * (uint64_t)c->wm;
        visit(c, tiers, st, depth + 1, j + 1);
    }
}

typedef struct {
    const wctx *c;
    int32_t j0, stride;
    wtier tiers[2];
    int err;
} wjob;

static wframe *alloc_frames(const wctx *c)
{
    const int depth = c->m + 2;
    wframe *st = (wframe *)calloc((size_t)depth, sizeof(wframe));
    if (!st) return NULL;
    for (int i = 0; i < depth; ++i) {
        st[i].ext = (uint32_t *)calloc((size_t)c->wn, sizeof(uint32_t));
        st[i].itt = (uint32_t *)calloc((size_t)c->wm, sizeof(uint32_t));
        st[i].cw = (uint32_t *)calloc((size_t)c->wn, sizeof(uint32_t));
        st[i].ci = (int64_t *)calloc((size_t)c->wn, sizeof(int64_t));
        st[i].ai = (int64_t *)calloc((size_t)c->wn, sizeof(int64_t));
        if (!st[i].ext || !st[i].itt || !st[i].cw || !st[i].ci || !st[i].ai) return NULL;
    }
    return st;
}

static void free_frames(const wctx *c, wframe *st)
{
    if (!st) return;
    for (int i = 0; i < c->m + 2; ++i) {
        free(st[i].ext);
        free(st[i].itt);
        free(st[i].cw);
        free(st[i].ci);
        free(st[i].ai);
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
    for (int64_t w = 0; w < c->wn; ++w) f->ext[w] = 0xffffffffu;
    if (c->n & 31) f->ext[c->wn - 1] = (1u << (c->n & 31)) - 1u;
    closure_rows(c, f->ext, f->itt);
    /* the top node: its own accounting, then only this thread's share of its candidates */
    int64_t na = c->n, nza = 0;
    for (int64_t w = 0; w < c->wn; ++w)
        if (f->ext[w]) f->ai[nza++] = w;
    wtier *t = &job->tiers[na > SMALL_EXTENT ? 1 : 0];
    if (job->j0 == 0) {
        t->parents++;
        t->hbm += (uint64_t)c->wn;
    }
    wframe *g = &st[1];
    for (int32_t j = job->j0; j < c->m; j += job->stride) {
        if (has_attr(f->itt, j)) continue;
        t->closures++;
        t->isect += (uint64_t)nza;
        const uint32_t *col = c->cols + (size_t)j * c->wn;
        int64_t nzc = 0, cnt = 0;
        for (int64_t i = 0; i < nza; ++i) {
            const int64_t w = f->ai[i];
            const uint32_t v = f->ext[w] & col[w];
            g->ext[w] = v;
            if (v) { f->cw[nzc] = v; f->ci[nzc] = w; ++nzc; cnt += popc32(v); }
        }
        const uint64_t rows_words = (uint64_t)cnt * (uint64_t)c->wm;
        t->close += column_route(c, f->itt, j, f->cw, f->ci, nzc, rows_words);
        t->canon += (uint64_t)c->wm;
        closure_rows(c, g->ext, g->itt);
        int canonical = 1;
        for (int32_t w = 0; w <= (j >> 5) && canonical; ++w) {
            uint32_t below = w < (j >> 5) ? 0xffffffffu : ((1u << (j & 31)) - 1u);
            if ((g->itt[w] ^ f->itt[w]) & below) canonical = 0;
        }
        if (!canonical) continue;
        t->children++;
        t->hbm += (uint64_t)c->wn + 2u * (uint64_t)c->wm;
        visit(c, job->tiers, st, 1, j + 1);
    }
    free_frames(c, st);
    return NULL;
}

/* Count the work of enumerating the context `rows32` (n x ceil(m/32) words, LSB-first; padding
   bits ignored). out[2][7] receives, per tier (0: extents <= 64 objects, 1: larger), parents,
   closures, canonical children, intersection words, closure words, canonical-test words and HBM
   words, in that order. Returns 0, or -1 on bad arguments or memory exhaustion. The top concept
   is a parent; its own output row is not counted (it is not a child). */
int workcount(const uint32_t *rows32, int64_t n, int32_t m, int threads, uint64_t *out)
{
    if (!rows32 || n < 1 || m < 1 || !out) return -1;
    if (threads < 1) threads = 1;
    wctx c;
    c.n = n;
    c.m = m;
    c.wn = (n + 31) / 32;
    c.wm = (m + 31) / 32;
    c.last_mask = (m & 31) ? ((1u << (m & 31)) - 1u) : 0xffffffffu;
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
        memset(out, 0, sizeof(uint64_t) * 14);
        for (int i = 0; i < threads; ++i) {
            err |= jobs[i].err;
            for (int k = 0; k < 2; ++k) {
                const wtier *t = &jobs[i].tiers[k];
                uint64_t *o = out + 7 * k;
                o[0] += t->parents;
                o[1] += t->closures;
                o[2] += t->children;
                o[3] += t->isect;
                o[4] += t->close;
                o[5] += t->canon;
                o[6] += t->hbm;
            }
        }
    }
    free(jobs);
    free(tid);
    free(c.rows);
    free(c.cols);
    return err ? -1 : 0;
}
