/*
 * Counting pass for the lower-cover search of the concept lattice: the algorithmic work, in 32-bit
 * words, of finding every concept's lower covers from the intent set. TEST AND MEASUREMENT
 * INFRASTRUCTURE ONLY: it gives the cover-edge roofline its numerator. It shares no code with the
 * library, nor with cbo.c, workcount.c or lattice.py.
 *
 * The method (the lattice rebuild of the FCbO-to-CUDA page, section 4.4, and of the Parallel FCBO
 * page, section 3.4, read as in the cover relation): for a concept (A, B), every attribute k outside
 * B gives the sub-extent C_k = A & column k; the lower covers are the distinct maximal non-empty
 * C_k, and the closure D_k of C_k (the AND of the rows of its objects) tells which attributes k2
 * have C_k inside C_k2 (exactly those of D_k), hence whether C_k is maximal. What is counted, per
 * concept (A, B):
 *
 *   extent   += W_N                       A = B' formed once (W_N words written or read)
 *   isect    += (M - |B|) * nnzw(A)       every C_k over the non-zero words of A
 *   closure  += sum over k not in B with C_k non-empty of |C_k| * W_M
 *                                         each D_k as the AND of |C_k| rows of W_M words
 *
 * W_N = ceil(N/32), W_M = ceil(M/32), nnzw() = number of non-zero 32-bit words. The counts do not
 * depend on the order of the intents. Multi-thread mode splits the intents between threads.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t n, wn;
    int32_t m, wm;
    const uint32_t *rows;    /* n x wm, padding bits cleared */
    uint32_t *cols;          /* m x wn */
    const uint32_t *intents; /* k x wm */
    int64_t k;
    uint32_t last_mask;
} cctx;

typedef struct {
    const cctx *c;
    int64_t i0, stride;
    uint64_t extent, isect, closure;
    int err;
} cjob;

static void *cover_worker(void *arg)
{
    cjob *jb = (cjob *)arg;
    const cctx *c = jb->c;
    uint32_t *a = (uint32_t *)malloc(sizeof(uint32_t) * (size_t)c->wn);
    if (!a) { jb->err = 1; return NULL; }
    for (int64_t i = jb->i0; i < c->k; i += jb->stride) {
        const uint32_t *b = c->intents + (size_t)i * c->wm;
        /* A = B': every object when B is empty, else the AND of the columns of B */
        for (int64_t q = 0; q < c->wn; ++q) a[q] = 0xffffffffu;
        if (c->n & 31) a[c->wn - 1] = (1u << (c->n & 31)) - 1u;
        int32_t nb = 0;
        for (int32_t att = 0; att < c->m; ++att) {
            if (!((b[att >> 5] >> (att & 31)) & 1u)) continue;
            ++nb;
            const uint32_t *col = c->cols + (size_t)att * c->wn;
            for (int64_t q = 0; q < c->wn; ++q) a[q] &= col[q];
        }
        int64_t nnz = 0;
        for (int64_t q = 0; q < c->wn; ++q) nnz += a[q] != 0u;
        jb->extent += (uint64_t)c->wn;
        jb->isect += (uint64_t)(c->m - nb) * (uint64_t)nnz;
        for (int32_t att = 0; att < c->m; ++att) {
            if ((b[att >> 5] >> (att & 31)) & 1u) continue;
            const uint32_t *col = c->cols + (size_t)att * c->wn;
            uint64_t s = 0;
            for (int64_t q = 0; q < c->wn; ++q) s += (uint64_t)__builtin_popcount(a[q] & col[q]);
            jb->closure += s * (uint64_t)c->wm;
        }
    }
    free(a);
    return NULL;
}

/* Count the work of the lower-cover search over `k` intents (k x ceil(m/32) words, LSB-first) of
   the context `rows32` (n x ceil(m/32) words; padding bits ignored). out[0..3] receives the
   concepts, extent words, intersection words and closure words. Returns 0, or -1 on bad arguments
   or memory exhaustion. */
int coverwork(const uint32_t *rows32, int64_t n, int32_t m, const uint32_t *intents, int64_t k, int threads,
              uint64_t *out)
{
    if (!rows32 || n < 1 || m < 1 || k < 0 || (k > 0 && !intents) || !out) return -1;
    if (threads < 1) threads = 1;
    cctx c;
    c.n = n;
    c.m = m;
    c.wn = (n + 31) / 32;
    c.wm = (m + 31) / 32;
    c.last_mask = (m & 31) ? ((1u << (m & 31)) - 1u) : 0xffffffffu;
    c.intents = intents;
    c.k = k;
    c.rows = rows32;
    c.cols = (uint32_t *)calloc((size_t)m * (size_t)c.wn, sizeof(uint32_t));
    if (!c.cols) return -1;
    for (int64_t o = 0; o < n; ++o)
        for (int32_t w = 0; w < c.wm; ++w) {
            uint32_t v = rows32[(size_t)o * c.wm + w];
            if (w == c.wm - 1) v &= c.last_mask;
            while (v) {
                const int bit = __builtin_ctz(v);
                v &= v - 1u;
                const int32_t att = w * 32 + bit;
                c.cols[(size_t)att * c.wn + (o >> 5)] |= 1u << (o & 31);
            }
        }
    cjob *jobs = (cjob *)calloc((size_t)threads, sizeof(cjob));
    pthread_t *tid = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    int err = (!jobs || !tid);
    for (int i = 0; i < threads && !err; ++i) {
        jobs[i].c = &c;
        jobs[i].i0 = i;
        jobs[i].stride = threads;
    }
    int started = 0;
    for (int i = 1; i < threads && !err; ++i, ++started)
        if (pthread_create(&tid[i], NULL, cover_worker, &jobs[i]) != 0) { err = 1; break; }
    if (!err) cover_worker(&jobs[0]);
    for (int i = 1; i <= started; ++i) pthread_join(tid[i], NULL);
    if (!err) {
        memset(out, 0, sizeof(uint64_t) * 4);
        out[0] = (uint64_t)k;
        for (int i = 0; i < threads; ++i) {
            err |= jobs[i].err;
            out[1] += jobs[i].extent;
            out[2] += jobs[i].isect;
            out[3] += jobs[i].closure;
        }
    }
    free(jobs);
    free(tid);
    free(c.cols);
    return err ? -1 : 0;
}
