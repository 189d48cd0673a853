/*
 * k2t_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU restatement of what a k^2-tree
 * sparse matrix-vector product computes, written from the text of
 * "A GPU Engine for Sparse Matrix-Vector Products on k^2-Tree-Compressed
 * Graphs" (Tosoni & Mencagli).  Only the test suite, the smoke check and
 * the CPU-baseline leg of the benchmark may load this file.  It shares no
 * code, header, table or helper with the library under test.
 *
 * Contents
 *   orc_build      the k^2-tree of a Boolean matrix by recursive
 *                  subdivision (section 2.1 "The k^2-tree": one bit per
 *                  quadrant, set iff the quadrant holds a non-zero; level
 *                  order; rectangular matrices padded with empty rows and
 *                  columns).  Duplicated coordinates need no special care:
 *                  a quadrant is non-empty whatever the multiplicity.
 *   orc_rank1      rank1(T, p) = set bits of T[0..p], inclusive (section 2.1).
 *   orc_spmv       the product by a recursive top-down descent in which
 *                  every step down is a rank query (section 2.1: children of
 *                  the bit at offset p start at k^2 * rank1(T, p)), applying
 *                  the contribution w (x) x_j of Table 1 at every cell.
 *                  Right: y_r (+)= w (x) x_c.  Left (section 3.6): y_c (+)=
 *                  w (x) x_r.
 *   orc_spmv_bands the same descent shared among POSIX threads: the subtrees
 *                  of one level are grouped into row bands (right products)
 *                  or column bands (left products), and the threads take
 *                  whole bands, so no two threads write one output.  Every
 *                  output receives its contributions in the order orc_spmv
 *                  gives them, so the results are identical.  This is the
 *                  multicore CPU descent the pages measure against (section
 *                  4, "Baselines"), kept here as a timed baseline.
 *   orc_rows_product  the plain definition y_i = (+)_{j: A_ij = 1} w (x) x_j
 *                  (section 2.2) evaluated from the edge list, for a sample
 *                  of outputs only, in one pass over the edges.
 *
 * Semirings (Table 1, section 2.2):
 *   0  plus-times  contribution w*x_j, accumulated in fp64 (the GPU path
 *                  accumulates in fp32; tests allow the stated tolerance).
 *                  The oracle also returns sum_j |w*x_j| per output, the
 *                  scale of that tolerance.
 *   1  Boolean     x, y are bit-packed: one uint32 word per vertex holding up
 *                  to 32 vectors; the contribution is x_j's word masked to
 *                  the batch's bits, accumulated by OR.  w is not used.
 *   2  tropical    contribution w + x_j rounded to fp32, accumulated by min
 *                  in the total order of IEEE floats without NaN, in which
 *                  -0 < +0; the empty min is +inf.
 *
 * Hybrid trees: the first n_k4 levels may use k = 4 (16-bit signatures,
 * quadrant b = 4*br + bc in row-major order, which reduces to b = 2*b1 + b0
 * for k = 2).  The pages describe k = 2 only; this is the plainest extension.
 * The leaf level may use k = 4 as well (leaf_k4 = 1): leaves are then 4x4
 * bitmaps, cell (dr, dc) at bit 4*dr + dc, the "leaves larger than 2x2" the
 * pages name as the next lever (section 5.6).  Every other level keeps k = 2.
 */
#define _POSIX_C_SOURCE 200809L
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORC_MAX_LEVELS 64

typedef struct {
    int32_t levels;                     /* number of levels; root = 0, leaves = levels-1 */
    int32_t n_k4;                       /* leading levels with k = 4 */
    int32_t dim_bits;                   /* padded side = 2^dim_bits */
    int32_t leaf_k4;                    /* 1: the leaf level has k = 4 */
    uint64_t nodes[ORC_MAX_LEVELS];     /* nodes per level */
    uint64_t start[ORC_MAX_LEVELS + 1]; /* bit offset of each level; start[levels] = total bits */
    uint64_t t_bits;                    /* bits in T (levels 0..levels-2) */
    uint64_t nwords;                    /* 64-bit words of the bitstring T followed by L */
    uint64_t *bits;                     /* bit p lives at bits[p/64] >> (p%64) */
    uint64_t *cum;                      /* cum[w] = set bits in words [0, w) */
} orc_tree;

static int level_k(const orc_tree *t, int d)
{
    if (d < t->n_k4) return 4;
    if (t->leaf_k4 && d == t->levels - 1) return 4;
    return 2;
}

/* side of the square block covered by a node of level d */
static uint64_t level_side(const orc_tree *t, int d)
{
    int used = 0;
    for (int e = 0; e < d; ++e) used += level_k(t, e) == 4 ? 2 : 1;
    return (uint64_t)1 << (t->dim_bits - used);
}

static int get_bit(const orc_tree *t, uint64_t p) { return (int)((t->bits[p >> 6] >> (p & 63)) & 1u); }

static int popcount64(uint64_t v)
{
    int c = 0;
    while (v) { v &= v - 1; ++c; }
    return c;
}

void orc_free(orc_tree *t)
{
    if (!t) return;
    free(t->bits);
    free(t->cum);
    t->bits = NULL;
    t->cum = NULL;
}

typedef struct { uint64_t r0, c0; uint64_t lo, hi; } orc_node; /* block origin, edge range */

/* Returns 0 on success, -1 on bad arguments, -2 on allocation failure.
 * The side is padded to 2^bits with at least one k = 2 level below the k = 4
 * top (so a last internal level with k = 2 exists): bits >= 2*n_k4 + 2, and
 * with 4x4 leaves bits >= 2*n_k4 + 3. */
int orc_build(const uint32_t *rows, const uint32_t *cols, uint64_t nnz,
              uint64_t n_rows, uint64_t n_cols, int32_t n_k4, int32_t leaf_k4, orc_tree *out)
{
    memset(out, 0, sizeof(*out));
    if (n_rows == 0 || n_cols == 0 || n_k4 < 0 || leaf_k4 < 0 || leaf_k4 > 1) return -1;
    uint64_t n = n_rows > n_cols ? n_rows : n_cols;
    int bits = 0;
    while (((uint64_t)1 << bits) < n) ++bits;
    if (bits < 2) bits = 2;
    if (bits < 2 * n_k4 + 2 + leaf_k4) bits = 2 * n_k4 + 2 + leaf_k4;
    if (bits > 32) return -1;
    for (uint64_t i = 0; i < nnz; ++i)
        if (rows[i] >= n_rows || cols[i] >= n_cols) return -1;
    out->dim_bits = bits;
    out->n_k4 = n_k4;
    out->leaf_k4 = leaf_k4;
    out->levels = bits - n_k4 - leaf_k4;

    /* Edge indices, partitioned per node; two arrays alternate per level. */
    uint64_t *idx = (uint64_t *)malloc((nnz ? nnz : 1) * sizeof(uint64_t));
    uint64_t *nidx = (uint64_t *)malloc((nnz ? nnz : 1) * sizeof(uint64_t));
    orc_node *cur = (orc_node *)malloc(sizeof(orc_node));
    /* signatures are collected per level in a growing byte array of bits */
    uint64_t cap_bits = 1024, nbits = 0;
    uint64_t *bitbuf = (uint64_t *)calloc(cap_bits / 64, sizeof(uint64_t));
    if (!idx || !nidx || !cur || !bitbuf) { free(idx); free(nidx); free(cur); free(bitbuf); return -2; }
    for (uint64_t i = 0; i < nnz; ++i) idx[i] = i;
    cur[0].r0 = 0; cur[0].c0 = 0; cur[0].lo = 0; cur[0].hi = nnz;
    uint64_t ncur = 1;

    for (int d = 0; d < out->levels; ++d) {
        int k = level_k(out, d);
        int kk = k * k;
        uint64_t sub = level_side(out, d) / (uint64_t)k;
        out->nodes[d] = ncur;
        out->start[d] = nbits;
        /* the next level has at most min(kk * ncur, nnz) nodes */
        uint64_t maxnext = ncur * (uint64_t)kk;
        if (maxnext > nnz) maxnext = nnz;
        orc_node *next = (orc_node *)malloc((maxnext ? maxnext : 1) * sizeof(orc_node));
        if (!next) { free(idx); free(nidx); free(cur); free(bitbuf); return -2; }
        uint64_t nnext = 0;
        uint64_t wpos = 0; /* write position in nidx */
        while (nbits + ncur * (uint64_t)kk > cap_bits) {
            uint64_t ncap = cap_bits * 2;
            uint64_t *nb = (uint64_t *)realloc(bitbuf, (ncap / 64) * sizeof(uint64_t));
            if (!nb) { free(next); free(idx); free(nidx); free(cur); free(bitbuf); return -2; }
            memset(nb + cap_bits / 64, 0, (ncap - cap_bits) / 64 * sizeof(uint64_t));
            bitbuf = nb;
            cap_bits = ncap;
        }
        for (uint64_t u = 0; u < ncur; ++u) {
            orc_node nd = cur[u];
            /* stable partition of the node's edges into its kk quadrants:
             * count per quadrant, then place in quadrant order */
            uint64_t cnt[16], at[16];
            for (int b = 0; b < kk; ++b) cnt[b] = 0;
            for (uint64_t e = nd.lo; e < nd.hi; ++e) {
                uint64_t ei = idx[e];
                uint64_t br = (rows[ei] - nd.r0) / sub;
                uint64_t bc = (cols[ei] - nd.c0) / sub;
                cnt[br * (uint64_t)k + bc]++;
            }
            at[0] = wpos;
            for (int b = 1; b < kk; ++b) at[b] = at[b - 1] + cnt[b - 1];
            for (uint64_t e = nd.lo; e < nd.hi; ++e) {
                uint64_t ei = idx[e];
                uint64_t br = (rows[ei] - nd.r0) / sub;
                uint64_t bc = (cols[ei] - nd.c0) / sub;
                nidx[at[br * (uint64_t)k + bc]++] = ei;
            }
            for (int b = 0; b < kk; ++b) {
                if (cnt[b] == 0) continue;
                uint64_t p = nbits + (uint64_t)b;
                bitbuf[p >> 6] |= (uint64_t)1 << (p & 63);
                if (d + 1 < out->levels) {
                    next[nnext].r0 = nd.r0 + (uint64_t)(b / k) * sub;
                    next[nnext].c0 = nd.c0 + (uint64_t)(b % k) * sub;
                    next[nnext].lo = at[b] - cnt[b];
                    next[nnext].hi = at[b];
                    ++nnext;
                }
            }
            wpos = at[kk - 1];
            nbits += (uint64_t)kk;
        }
        uint64_t *tmp = idx; idx = nidx; nidx = tmp;
        free(cur);
        cur = next;
        ncur = nnext;
    }
    out->start[out->levels] = nbits;
    out->t_bits = out->start[out->levels - 1];
    out->nwords = (nbits + 63) / 64;
    out->bits = bitbuf;
    out->cum = (uint64_t *)malloc((out->nwords + 1) * sizeof(uint64_t));
    free(idx); free(nidx); free(cur);
    if (!out->cum) { free(out->bits); out->bits = NULL; return -2; }
    out->cum[0] = 0;
    for (uint64_t w = 0; w < out->nwords; ++w) out->cum[w + 1] = out->cum[w] + (uint64_t)popcount64(out->bits[w]);
    return 0;
}

/* Set bits of the bitstring in positions [0..p], inclusive. */
uint64_t orc_rank1(const orc_tree *t, uint64_t p)
{
    uint64_t w = p >> 6;
    uint64_t b = p & 63;
    uint64_t mask = (b == 63) ? ~(uint64_t)0 : (((uint64_t)1 << (b + 1)) - 1);
    return t->cum[w] + (uint64_t)popcount64(t->bits[w] & mask);
}

/* Position of the first bit of the child node reached through the set bit at
 * position p, which lies in level d.  For k = 2 throughout this equals the
 * pages' 4 * rank1(T, p); with per-level k the set bits before level d are
 * discounted and the child's level start added back. */
uint64_t orc_child_pos(const orc_tree *t, int d, uint64_t p)
{
    uint64_t before = (t->start[d] == 0) ? 0 : orc_rank1(t, t->start[d] - 1);
    uint64_t child_index = orc_rank1(t, p) - before - 1;
    uint64_t kk = (uint64_t)level_k(t, d + 1) * (uint64_t)level_k(t, d + 1);
    return t->start[d + 1] + kk * child_index;
}

/* --- semiring helpers (fp32 total order for tropical) ------------------- */
typedef union { float f; uint32_t u; } orc_fu;

static int32_t order_key(float v)
{
    orc_fu a; a.f = v;
    uint32_t k = (a.u & 0x80000000u) ? (a.u ^ 0x7fffffffu) : a.u;
    return (int32_t)k;
}

typedef struct {
    int32_t dir;        /* 0 right, 1 left */
    int32_t semiring;   /* 0 plus-times, 1 Boolean, 2 tropical */
    float w;
    uint32_t B;
    uint32_t mask;      /* Boolean: bits of the batch */
    const void *x;
    void *y;            /* plus-times: double[n_out*B]; Boolean: uint32[n_out]; tropical: float[n_out*B] */
    double *scale;      /* plus-times: sum |w*x| per output (may be NULL) */
    uint64_t cells;     /* cells visited */
} orc_ctx;

static void apply_cell(orc_ctx *c, uint64_t r, uint64_t col)
{
    uint64_t in = c->dir == 0 ? col : r;
    uint64_t o = c->dir == 0 ? r : col;
    c->cells++;
    if (c->semiring == 0) {
        const float *x = (const float *)c->x;
        double *y = (double *)c->y;
        for (uint32_t k = 0; k < c->B; ++k) {
            double v = (double)c->w * (double)x[in * c->B + k];
            y[o * c->B + k] += v;
            if (c->scale) c->scale[o * c->B + k] += v < 0 ? -v : v;
        }
    } else if (c->semiring == 1) {
        const uint32_t *x = (const uint32_t *)c->x;
        uint32_t *y = (uint32_t *)c->y;
        y[o] |= x[in] & c->mask;
    } else {
        const float *x = (const float *)c->x;
        float *y = (float *)c->y;
        for (uint32_t k = 0; k < c->B; ++k) {
            volatile float s = c->w + x[in * c->B + k]; /* one fp32 rounding, no contraction */
            float v = s;
            if (order_key(v) < order_key(y[o * c->B + k])) y[o * c->B + k] = v;
        }
    }
}

static void visit(const orc_tree *t, orc_ctx *c, int d, uint64_t pos, uint64_t r0, uint64_t c0)
{
    int k = level_k(t, d);
    uint64_t sub = level_side(t, d) / (uint64_t)k;
    for (int b = 0; b < k * k; ++b) {
        if (!get_bit(t, pos + (uint64_t)b)) continue;
        uint64_t r = r0 + (uint64_t)(b / k) * sub;
        uint64_t col = c0 + (uint64_t)(b % k) * sub;
        if (d == t->levels - 1) {
            apply_cell(c, r, col);
        } else {
            visit(t, c, d + 1, orc_child_pos(t, d, pos + (uint64_t)b), r, col);
        }
    }
}

/*
 * y = A x (dir 0) or y^T = x^T A (dir 1) over the semiring, from the tree alone.
 * y must be sized n_out*B (Boolean: n_out words) and is overwritten with the
 * semiring zero first (Algorithm 1, line 1).  Returns the number of cells
 * visited (= nnz of the deduplicated matrix).
 */
uint64_t orc_spmv(const orc_tree *t, uint64_t n_rows, uint64_t n_cols,
                  int32_t dir, int32_t semiring, float w, uint32_t B,
                  const void *x, void *y, double *scale)
{
    uint64_t n_out = dir == 0 ? n_rows : n_cols;
    orc_ctx c;
    c.dir = dir; c.semiring = semiring; c.w = w; c.B = B;
    c.mask = (B >= 32) ? 0xffffffffu : ((1u << B) - 1u);
    c.x = x; c.y = y; c.scale = scale; c.cells = 0;
    if (semiring == 0) {
        double *yy = (double *)y;
        for (uint64_t i = 0; i < n_out * B; ++i) yy[i] = 0.0;
        if (scale) for (uint64_t i = 0; i < n_out * B; ++i) scale[i] = 0.0;
    } else if (semiring == 1) {
        memset(y, 0, n_out * sizeof(uint32_t));
    } else {
        orc_fu inf; inf.u = 0x7f800000u;
        float *yy = (float *)y;
        for (uint64_t i = 0; i < n_out * B; ++i) yy[i] = inf.f;
    }
    visit(t, &c, 0, 0, 0, 0);
    return c.cells;
}

/* --- the descent shared among threads by bands ------------------------- */
typedef struct { uint64_t pos, r0, c0, band, seq; } orc_sub;  /* a level-bd node */
typedef struct { orc_sub *v; uint64_t n, cap; int bd; int dir; } orc_subs;

static int collect_visit(const orc_tree *t, orc_subs *s, int d, uint64_t pos, uint64_t r0, uint64_t c0)
{
    if (d == s->bd) {
        if (s->n == s->cap) {
            uint64_t ncap = s->cap ? 2 * s->cap : 1024;
            orc_sub *nv = (orc_sub *)realloc(s->v, ncap * sizeof(orc_sub));
            if (!nv) return -2;
            s->v = nv;
            s->cap = ncap;
        }
        orc_sub *e = &s->v[s->n];
        e->pos = pos; e->r0 = r0; e->c0 = c0; e->seq = s->n;
        e->band = (s->dir == 0 ? r0 : c0) / level_side(t, d);
        s->n++;
        return 0;
    }
    int k = level_k(t, d);
    uint64_t sub = level_side(t, d) / (uint64_t)k;
    for (int b = 0; b < k * k; ++b) {
        if (!get_bit(t, pos + (uint64_t)b)) continue;
        uint64_t r = r0 + (uint64_t)(b / k) * sub;
        uint64_t col = c0 + (uint64_t)(b % k) * sub;
        int rc = collect_visit(t, s, d + 1, orc_child_pos(t, d, pos + (uint64_t)b), r, col);
        if (rc) return rc;
    }
    return 0;
}

static int sub_cmp(const void *a, const void *b)
{
    const orc_sub *x = (const orc_sub *)a, *y = (const orc_sub *)b;
    if (x->band != y->band) return x->band < y->band ? -1 : 1;
    return x->seq < y->seq ? -1 : (x->seq > y->seq ? 1 : 0);
}

typedef struct {
    const orc_tree *t;
    const orc_subs *subs;
    const uint64_t *group;   /* group g = subs [group[g], group[g+1]) */
    uint64_t ngroups;
    uint64_t next;           /* next group to take (atomic) */
    orc_ctx proto;
} orc_shared;

typedef struct { orc_shared *sh; uint64_t cells; } orc_worker;

static void *band_worker(void *arg)
{
    orc_worker *w = (orc_worker *)arg;
    orc_shared *sh = w->sh;
    orc_ctx c = sh->proto;
    c.cells = 0;
    for (;;) {
        uint64_t g = __atomic_fetch_add(&sh->next, 1, __ATOMIC_RELAXED);
        if (g >= sh->ngroups) break;
        for (uint64_t i = sh->group[g]; i < sh->group[g + 1]; ++i) {
            const orc_sub *e = &sh->subs->v[i];
            visit(sh->t, &c, sh->subs->bd, e->pos, e->r0, e->c0);
        }
    }
    w->cells = c.cells;
    return NULL;
}

/*
 * orc_spmv with the level-bd subtrees grouped into bands of their node row
 * (dir 0) or column (dir 1) and the bands shared among `threads` threads
 * (0: one per online core).  bd < 0 picks the shallowest level with at least
 * 8192 nodes per thread (at most the last internal level): enough bands to
 * balance power-law rows, few enough that collecting them stays cheap.  *used receives the
 * thread count.  Returns the cells visited, or (uint64_t)-1 if memory ran out.
 */
uint64_t orc_spmv_bands(const orc_tree *t, uint64_t n_rows, uint64_t n_cols,
                        int32_t dir, int32_t semiring, float w, uint32_t B,
                        const void *x, void *y, double *scale, int32_t bd, int32_t threads, int32_t *used)
{
    int nt = threads > 0 ? threads : (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nt < 1) nt = 1;
    if (bd < 0) {
        bd = 0;
        while (bd < t->levels - 2 && t->nodes[bd] < (uint64_t)8192 * (uint64_t)nt) ++bd;
    }
    if (bd > t->levels - 1) bd = t->levels - 1;
    /* fill y and scale with the semiring zero, as orc_spmv does */
    uint64_t n_out = dir == 0 ? n_rows : n_cols;
    if (semiring == 0) {
        double *yy = (double *)y;
        for (uint64_t i = 0; i < n_out * B; ++i) yy[i] = 0.0;
        if (scale) for (uint64_t i = 0; i < n_out * B; ++i) scale[i] = 0.0;
    } else if (semiring == 1) {
        memset(y, 0, n_out * sizeof(uint32_t));
    } else {
        orc_fu inf; inf.u = 0x7f800000u;
        float *yy = (float *)y;
        for (uint64_t i = 0; i < n_out * B; ++i) yy[i] = inf.f;
    }
    orc_subs subs;
    memset(&subs, 0, sizeof(subs));
    subs.bd = bd;
    subs.dir = dir;
    if (collect_visit(t, &subs, 0, 0, 0, 0)) { free(subs.v); return (uint64_t)-1; }
    qsort(subs.v, subs.n, sizeof(orc_sub), sub_cmp);
    uint64_t *group = (uint64_t *)malloc((subs.n + 1) * sizeof(uint64_t));
    orc_worker *wk = (orc_worker *)calloc((size_t)nt, sizeof(orc_worker));
    pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    if (!group || !wk || !th) { free(group); free(wk); free(th); free(subs.v); return (uint64_t)-1; }
    uint64_t ng = 0;
    for (uint64_t i = 0; i < subs.n; ++i)
        if (i == 0 || subs.v[i].band != subs.v[i - 1].band) group[ng++] = i;
    group[ng] = subs.n;
    orc_shared sh;
    sh.t = t; sh.subs = &subs; sh.group = group; sh.ngroups = ng; sh.next = 0;
    sh.proto.dir = dir; sh.proto.semiring = semiring; sh.proto.w = w; sh.proto.B = B;
    sh.proto.mask = (B >= 32) ? 0xffffffffu : ((1u << B) - 1u);
    sh.proto.x = x; sh.proto.y = y; sh.proto.scale = scale; sh.proto.cells = 0;
    int started = 0;
    for (int i = 0; i < nt; ++i) {
        wk[i].sh = &sh;
        if (i > 0 && pthread_create(&th[i], NULL, band_worker, &wk[i]) == 0) ++started;
        else if (i > 0) break;
    }
    band_worker(&wk[0]);
    uint64_t cells = wk[0].cells;
    for (int i = 1; i <= started; ++i) {
        pthread_join(th[i], NULL);
        cells += wk[i].cells;
    }
    if (used) *used = started + 1;
    free(group); free(wk); free(th); free(subs.v);
    return cells;
}

/* Decode the tree into its cells, in descent order.  Returns the number of
 * cells; writes at most cap of them. */
typedef struct { uint32_t *rows, *cols; uint64_t cap, n; } orc_dec;

static void decode_visit(const orc_tree *t, orc_dec *o, int d, uint64_t pos, uint64_t r0, uint64_t c0)
{
    int k = level_k(t, d);
    uint64_t sub = level_side(t, d) / (uint64_t)k;
    for (int b = 0; b < k * k; ++b) {
        if (!get_bit(t, pos + (uint64_t)b)) continue;
        uint64_t r = r0 + (uint64_t)(b / k) * sub;
        uint64_t col = c0 + (uint64_t)(b % k) * sub;
        if (d == t->levels - 1) {
            if (o->n < o->cap) { o->rows[o->n] = (uint32_t)r; o->cols[o->n] = (uint32_t)col; }
            o->n++;
        } else {
            decode_visit(t, o, d + 1, orc_child_pos(t, d, pos + (uint64_t)b), r, col);
        }
    }
}

uint64_t orc_decode(const orc_tree *t, uint32_t *rows, uint32_t *cols, uint64_t cap)
{
    orc_dec o;
    o.rows = rows; o.cols = cols; o.cap = cap; o.n = 0;
    decode_visit(t, &o, 0, 0, 0, 0);
    return o.n;
}

/* Copy the bitstring words out (T followed by L). */
void orc_copy_bits(const orc_tree *t, uint64_t *dst) { memcpy(dst, t->bits, t->nwords * sizeof(uint64_t)); }

/*
 * Definition from the edge list, for sampled outputs only: for each output
 * index listed in `sample` (sorted or not, no duplicates), compute
 * y = (+)_{edges into it} w (x) x.  `slot` maps an output index to its
 * position in the sample (-1 elsewhere) and has n_out entries.  Edges are
 * deduplicated by the caller or counted once per distinct (row, col) by
 * passing unique edges.  Result layout as orc_spmv, one row per sample.
 */
void orc_rows_product(const uint32_t *rows, const uint32_t *cols, uint64_t nnz,
                      int32_t dir, int32_t semiring, float w, uint32_t B,
                      const void *x, const int64_t *slot,
                      uint64_t n_sample, void *y, double *scale)
{
    orc_ctx c;
    c.dir = 0; c.semiring = semiring; c.w = w; c.B = B;
    c.mask = (B >= 32) ? 0xffffffffu : ((1u << B) - 1u);
    c.x = x; c.y = y; c.scale = scale; c.cells = 0;
    if (semiring == 0) {
        double *yy = (double *)y;
        for (uint64_t i = 0; i < n_sample * B; ++i) yy[i] = 0.0;
        if (scale) for (uint64_t i = 0; i < n_sample * B; ++i) scale[i] = 0.0;
    } else if (semiring == 1) {
        memset(y, 0, n_sample * sizeof(uint32_t));
    } else {
        orc_fu inf; inf.u = 0x7f800000u;
        float *yy = (float *)y;
        for (uint64_t i = 0; i < n_sample * B; ++i) yy[i] = inf.f;
    }
    for (uint64_t e = 0; e < nnz; ++e) {
        uint64_t o = dir == 0 ? rows[e] : cols[e];
        uint64_t in = dir == 0 ? cols[e] : rows[e];
        int64_t s = slot[o];
        if (s < 0) continue;
        /* apply with output index = slot, input index = in (dir 0 layout) */
        apply_cell(&c, (uint64_t)s, in);
    }
}
