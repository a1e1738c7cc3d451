/*
 * orc.c -- plain, slow fp64 CPU oracle for tensor-relational join-agg.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the CPU-baseline
 * leg of the benchmark call it; the product never does.  It shares no code,
 * header or table with the CUDA path.
 *
 * Semantics ("Every Kernel Is a Join", Section 1 and Definition 3.7): in the
 * degenerate relational form every key is one cell and every sub-tensor is
 * a scalar.  A join-agg over input relations R_0..R_{n-1} is
 *   (1) Join:      every combination of one tuple per relation that agrees
 *                  on each shared index letter (an optional cell predicate
 *                  "a <= b" on two letters filters the joined tuples);
 *   (2) Map:       f applied to the joined values;
 *   (3) Aggregate: group the mapped tuples by the output letters and
 *                  combine each group with an associative, commutative op
 *                  (SUM or MAX), or keep the single tuple (NONE);
 *   (4) Recompose: write each group at its output cell.
 *
 * Dense arrays carry relations: a cell holding NaN is ABSENT (no tuple).
 * Generated inputs are NaN-free, so NaN only ever marks absence (produced
 * by a filtered join, e.g. the causal predicate).
 *
 * Two tiers compute the same thing:
 *   orc_joinagg_lit -- literal: hash join + hash group-by over tuple lists.
 *   orc_joinagg_idx -- index nested loop over dense keys, threaded.
 * And the re-blocking exchange is written from its definition
 * ("Every Kernel Is a Join", Section 5.3: overlay of two tilings; every
 * element keeps its global coordinates).
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define MAXR 8
#define MAXIN 4
#define NLET 26

enum { M_PRODUCT = 0, M_IDENTITY, M_SILU_MUL, M_ADD, M_EXP_SUB, M_DIV, M_SQUARE, M_RMS_APPLY };
enum { A_NONE = 0, A_SUM, A_MAX };

static __thread char g_err[512];

const char *orc_last_error(void) { return g_err; }

static int fail(const char *msg) {
    snprintf(g_err, sizeof g_err, "%s", msg);
    return -1;
}

/* ------------------------------------------------------------------ spec */

typedef struct {
    int n_in;
    int rank[MAXIN];
    int let[MAXIN][MAXR];
    int out_rank;
    int out_let[MAXR];
    int64_t ext[NLET];
    int in_out[NLET];     /* letter appears in the output */
    int used[NLET];
    int pred_a, pred_b;   /* keep joined tuple iff val[a] <= val[b]; -1 = none */
    int64_t lo[NLET];     /* global offset of each letter (the predicate compares global values) */
} spec_t;

static int parse_term(const char **p, int *let, int *rank) {
    int r = 0;
    while (**p >= 'a' && **p <= 'z') {
        if (r == MAXR) return fail("spec: a term has too many letters");
        int l = **p - 'a';
        for (int i = 0; i < r; i++)
            if (let[i] == l) return fail("spec: repeated letter inside one term");
        let[r++] = l;
        (*p)++;
    }
    *rank = r;
    return 0;
}

static int parse_spec(const char *s, const int64_t *shapes, const char *pred, const int64_t *lo, spec_t *sp) {
    memset(sp, 0, sizeof *sp);
    if (lo) memcpy(sp->lo, lo, sizeof sp->lo);
    const char *p = s;
    sp->n_in = 0;
    for (;;) {
        if (sp->n_in == MAXIN) return fail("spec: too many inputs");
        if (parse_term(&p, sp->let[sp->n_in], &sp->rank[sp->n_in])) return -1;
        sp->n_in++;
        if (*p == ',') { p++; continue; }
        break;
    }
    if (p[0] != '-' || p[1] != '>') return fail("spec: expected '->'");
    p += 2;
    if (parse_term(&p, sp->out_let, &sp->out_rank)) return -1;
    if (*p != 0) return fail("spec: trailing characters");
    for (int l = 0; l < NLET; l++) sp->ext[l] = -1;
    int si = 0;
    for (int k = 0; k < sp->n_in; k++)
        for (int d = 0; d < sp->rank[k]; d++) {
            int l = sp->let[k][d];
            int64_t e = shapes[si++];
            if (e < 0) return fail("shape: negative extent");
            if (sp->ext[l] >= 0 && sp->ext[l] != e) return fail("shape: a letter has two extents");
            sp->ext[l] = e;
            sp->used[l] = 1;
        }
    for (int d = 0; d < sp->out_rank; d++) {
        int l = sp->out_let[d];
        if (!sp->used[l]) return fail("spec: output letter missing from the inputs");
        sp->in_out[l] = 1;
    }
    sp->pred_a = sp->pred_b = -1;
    if (pred && pred[0]) {
        if (!(pred[0] >= 'a' && pred[0] <= 'z' && pred[1] >= 'a' && pred[1] <= 'z' && pred[2] == 0))
            return fail("predicate: expected two letters");
        sp->pred_a = pred[0] - 'a';
        sp->pred_b = pred[1] - 'a';
        if (!sp->used[sp->pred_a] || !sp->used[sp->pred_b]) return fail("predicate: unknown letter");
    }
    return 0;
}

static int map_arity_ok(int map, int n) {
    switch (map) {
    case M_PRODUCT: return n >= 1;
    case M_IDENTITY: case M_SQUARE: return n == 1;
    case M_SILU_MUL: case M_ADD: case M_EXP_SUB: case M_DIV: return n == 2;
    case M_RMS_APPLY: return n == 3;
    }
    return 0;
}

static double apply_map(int map, const double *v, int n, double scale, double eps) {
    switch (map) {
    case M_PRODUCT: {
        double r = scale;
        for (int k = 0; k < n; k++) r *= v[k];
        return r;
    }
    case M_IDENTITY: return scale * v[0];
    case M_SILU_MUL: return v[0] / (1.0 + exp(-v[0])) * v[1];
    case M_ADD: return v[0] + v[1];
    case M_EXP_SUB: return exp(v[0] - v[1]);
    case M_DIV: return v[0] / v[1];
    case M_SQUARE: return scale * v[0] * v[0];
    case M_RMS_APPLY: return v[0] / sqrt(v[1] + eps) * v[2];
    }
    return NAN;
}

static int64_t out_cells(const spec_t *sp) {
    int64_t n = 1;
    for (int d = 0; d < sp->out_rank; d++) n *= sp->ext[sp->out_let[d]];
    return n;
}

/* ------------------------------------------------- literal tier: relations */

typedef struct {
    int r;
    int let[MAXR];
    int64_t n;
    int64_t *key; /* n * r letter values */
    double *val;
} rel_t;

static int rel_from_dense(const spec_t *sp, int k, const double *a, rel_t *R) {
    R->r = sp->rank[k];
    memcpy(R->let, sp->let[k], sizeof R->let);
    int64_t cells = 1;
    for (int d = 0; d < R->r; d++) cells *= sp->ext[R->let[d]];
    R->key = (int64_t *)malloc(sizeof(int64_t) * (size_t)(cells * (R->r ? R->r : 1) + 1));
    R->val = (double *)malloc(sizeof(double) * (size_t)(cells + 1));
    if (!R->key || !R->val) return fail("oracle: out of host memory");
    int64_t idx[MAXR] = {0};
    R->n = 0;
    for (int64_t c = 0; c < cells; c++) {
        if (!isnan(a[c])) {
            for (int d = 0; d < R->r; d++) R->key[R->n * R->r + d] = idx[d];
            R->val[R->n] = a[c];
            R->n++;
        }
        for (int d = R->r - 1; d >= 0; d--) {
            if (++idx[d] < sp->ext[R->let[d]]) break;
            idx[d] = 0;
        }
    }
    return 0;
}

static uint64_t hash_keys(const int64_t *v, int n) {
    uint64_t h = 0xcbf29ce484222325ULL;
    for (int i = 0; i < n; i++) {
        h ^= (uint64_t)v[i] + 0x9e3779b97f4a7c15ULL + (h << 6) + (h >> 2);
        h *= 0x100000001b3ULL;
    }
    h ^= h >> 31;
    return h;
}

/* Hash index of one relation on the positions of its already-bound letters. */
typedef struct {
    int nsub;
    int pos[MAXR];  /* positions in the relation's key */
    int lets[MAXR]; /* their letters */
    uint64_t *h;    /* sorted hashes */
    int64_t *ix;    /* tuple indices in hash order */
} jidx_t;

static const uint64_t *g_sort_h;
static int cmp_ix(const void *x, const void *y) {
    uint64_t a = g_sort_h[*(const int64_t *)x], b = g_sort_h[*(const int64_t *)y];
    return a < b ? -1 : a > b ? 1 : 0;
}

static int build_index(const rel_t *R, const int *bound, jidx_t *I) {
    I->nsub = 0;
    for (int d = 0; d < R->r; d++)
        if (bound[R->let[d]]) {
            I->pos[I->nsub] = d;
            I->lets[I->nsub] = R->let[d];
            I->nsub++;
        }
    I->h = NULL;
    I->ix = NULL;
    if (I->nsub == 0) return 0;
    uint64_t *hh = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(R->n + 1));
    I->ix = (int64_t *)malloc(sizeof(int64_t) * (size_t)(R->n + 1));
    I->h = (uint64_t *)malloc(sizeof(uint64_t) * (size_t)(R->n + 1));
    if (!hh || !I->ix || !I->h) return fail("oracle: out of host memory");
    int64_t sub[MAXR];
    for (int64_t t = 0; t < R->n; t++) {
        for (int j = 0; j < I->nsub; j++) sub[j] = R->key[t * R->r + I->pos[j]];
        hh[t] = hash_keys(sub, I->nsub);
        I->ix[t] = t;
    }
    g_sort_h = hh;
    qsort(I->ix, (size_t)R->n, sizeof(int64_t), cmp_ix);
    for (int64_t t = 0; t < R->n; t++) I->h[t] = hh[I->ix[t]];
    free(hh);
    return 0;
}

/* Group-by table: open addressing on the output key. */
typedef struct {
    int64_t cap;
    int r;
    int64_t *key;
    double *acc;
    int64_t *cnt;
} gtab_t;

typedef struct {
    const spec_t *sp;
    rel_t *rel;
    jidx_t *idx;
    int map, agg;
    double scale, eps;
    int64_t val[NLET];
    double v[MAXIN];
    gtab_t g;
    int err;
    int64_t joined;
} jctx_t;

static void emit(jctx_t *c) {
    const spec_t *sp = c->sp;
    if (sp->pred_a >= 0 && !(c->val[sp->pred_a] + sp->lo[sp->pred_a] <= c->val[sp->pred_b] + sp->lo[sp->pred_b])) return;
    c->joined++;
    double f = apply_map(c->map, c->v, sp->n_in, c->scale, c->eps);
    int64_t key[MAXR];
    for (int d = 0; d < sp->out_rank; d++) key[d] = c->val[sp->out_let[d]];
    uint64_t h = hash_keys(key, sp->out_rank);
    int64_t s = (int64_t)(h & (uint64_t)(c->g.cap - 1));
    for (;;) {
        if (c->g.cnt[s] == 0) {
            memcpy(&c->g.key[s * c->g.r], key, sizeof(int64_t) * (size_t)c->g.r);
            c->g.acc[s] = f;
            c->g.cnt[s] = 1;
            return;
        }
        if (memcmp(&c->g.key[s * c->g.r], key, sizeof(int64_t) * (size_t)c->g.r) == 0) {
            if (c->agg == A_SUM) c->g.acc[s] += f;
            else if (c->agg == A_MAX) c->g.acc[s] = fmax(c->g.acc[s], f);
            else c->err = 1; /* NONE with two tuples in one group */
            c->g.cnt[s]++;
            return;
        }
        s = (s + 1) & (c->g.cap - 1);
    }
}

static void join_rec(jctx_t *c, int k) {
    if (k == c->sp->n_in) {
        emit(c);
        return;
    }
    const rel_t *R = &c->rel[k];
    const jidx_t *I = &c->idx[k];
    if (I->nsub == 0) {
        for (int64_t t = 0; t < R->n; t++) {
            for (int d = 0; d < R->r; d++) c->val[R->let[d]] = R->key[t * R->r + d];
            c->v[k] = R->val[t];
            join_rec(c, k + 1);
        }
        return;
    }
    int64_t sub[MAXR];
    for (int j = 0; j < I->nsub; j++) sub[j] = c->val[I->lets[j]];
    uint64_t h = hash_keys(sub, I->nsub);
    int64_t lo = 0, hi = R->n;
    while (lo < hi) {
        int64_t mid = (lo + hi) / 2;
        if (I->h[mid] < h) lo = mid + 1;
        else hi = mid;
    }
    for (int64_t j = lo; j < R->n && I->h[j] == h; j++) {
        int64_t t = I->ix[j];
        int ok = 1;
        for (int q = 0; q < I->nsub; q++)
            if (R->key[t * R->r + I->pos[q]] != sub[q]) { ok = 0; break; }
        if (!ok) continue;
        for (int d = 0; d < R->r; d++) c->val[R->let[d]] = R->key[t * R->r + d];
        c->v[k] = R->val[t];
        join_rec(c, k + 1);
    }
}

int orc_joinagg_lit(const char *spec, const int64_t *shapes, const double *const *ins, int map, int agg,
                    double scale, double eps, const char *pred, const int64_t *lo, double *out, int64_t *n_joined) {
    spec_t sp;
    if (parse_spec(spec, shapes, pred, lo, &sp)) return -1;
    if (!map_arity_ok(map, sp.n_in)) return fail("map: wrong number of inputs");
    if (agg < A_NONE || agg > A_MAX) return fail("agg: unknown");
    int rc = -1;
    rel_t rel[MAXIN];
    jidx_t idx[MAXIN];
    memset(rel, 0, sizeof rel);
    memset(idx, 0, sizeof idx);
    jctx_t c;
    memset(&c, 0, sizeof c);
    int bound[NLET] = {0};
    for (int k = 0; k < sp.n_in; k++) {
        if (rel_from_dense(&sp, k, ins[k], &rel[k])) goto done;
        if (build_index(&rel[k], bound, &idx[k])) goto done;
        for (int d = 0; d < rel[k].r; d++) bound[rel[k].let[d]] = 1;
    }
    int64_t cells = out_cells(&sp);
    int64_t cap = 16;
    while (cap < 2 * cells + 2) cap <<= 1;
    c.g.cap = cap;
    c.g.r = sp.out_rank ? sp.out_rank : 1;
    c.g.key = (int64_t *)calloc((size_t)(cap * c.g.r), sizeof(int64_t));
    c.g.acc = (double *)calloc((size_t)cap, sizeof(double));
    c.g.cnt = (int64_t *)calloc((size_t)cap, sizeof(int64_t));
    if (!c.g.key || !c.g.acc || !c.g.cnt) { fail("oracle: out of host memory"); goto done; }
    if (sp.out_rank == 0) c.g.r = 0;
    c.sp = &sp;
    c.rel = rel;
    c.idx = idx;
    c.map = map;
    c.agg = agg;
    c.scale = scale;
    c.eps = eps;
    join_rec(&c, 0);
    if (c.err) { fail("agg NONE: a group holds more than one joined tuple"); goto done; }
    /* Recompose: absent cells stay NaN. */
    for (int64_t i = 0; i < cells; i++) out[i] = NAN;
    for (int64_t s = 0; s < cap; s++) {
        if (!c.g.cnt[s]) continue;
        int64_t off = 0;
        for (int d = 0; d < sp.out_rank; d++) off = off * sp.ext[sp.out_let[d]] + c.g.key[s * sp.out_rank + d];
        out[off] = c.g.acc[s];
    }
    if (n_joined) *n_joined = c.joined;
    rc = 0;
done:
    for (int k = 0; k < MAXIN; k++) {
        free(rel[k].key);
        free(rel[k].val);
        free(idx[k].h);
        free(idx[k].ix);
    }
    free(c.g.key);
    free(c.g.acc);
    free(c.g.cnt);
    return rc;
}

/* ----------------------------------------- index tier: dense nested loops */

typedef struct {
    const spec_t *sp;
    const double *const *ins;
    double *out;
    int map, agg;
    double scale, eps;
    int n_inner;
    int inner[NLET];
    int64_t stride[MAXIN][NLET]; /* 0 when the letter is not in the input */
    int64_t cells;
    int64_t chunk;
    _Atomic int64_t next;
    _Atomic int err;
} ictx_t;

static void *idx_worker(void *arg) {
    ictx_t *c = (ictx_t *)arg;
    const spec_t *sp = c->sp;
    int n = sp->n_in;
    int64_t val[NLET];
    double v[MAXIN];
    int64_t off[MAXIN];
    for (;;) {
        int64_t start = atomic_fetch_add(&c->next, c->chunk);
        if (start >= c->cells) break;
        int64_t end = start + c->chunk < c->cells ? start + c->chunk : c->cells;
        for (int64_t o = start; o < end; o++) {
            int64_t rem = o;
            for (int d = sp->out_rank - 1; d >= 0; d--) {
                int l = sp->out_let[d];
                val[l] = rem % sp->ext[l];
                rem /= sp->ext[l];
            }
            int64_t base[MAXIN];
            for (int k = 0; k < n; k++) {
                base[k] = 0;
                for (int d = 0; d < sp->out_rank; d++) base[k] += val[sp->out_let[d]] * c->stride[k][sp->out_let[d]];
            }
            int64_t inner_count = 1;
            for (int j = 0; j < c->n_inner; j++) inner_count *= sp->ext[c->inner[j]];
            double acc = 0.0;
            int64_t cnt = 0;
            if (c->n_inner == 1) {
                /* one aggregated letter: walk it directly (same order as below) */
                int l = c->inner[0];
                for (int64_t x = 0; x < inner_count; x++) {
                    int absent = 0;
                    for (int k = 0; k < n; k++) {
                        v[k] = c->ins[k][base[k] + x * c->stride[k][l]];
                        if (isnan(v[k])) absent = 1;
                    }
                    if (absent) continue;
                    val[l] = x;
                    if (sp->pred_a >= 0 && !(val[sp->pred_a] + sp->lo[sp->pred_a] <= val[sp->pred_b] + sp->lo[sp->pred_b]))
                        continue;
                    double f = apply_map(c->map, v, n, c->scale, c->eps);
                    if (cnt == 0) acc = f;
                    else if (c->agg == A_SUM) acc += f;
                    else if (c->agg == A_MAX) acc = fmax(acc, f);
                    else atomic_store(&c->err, 1);
                    cnt++;
                }
                c->out[o] = cnt ? acc : NAN;
                continue;
            }
            for (int j = 0; j < c->n_inner; j++) val[c->inner[j]] = 0;
            for (int64_t it = 0; it < inner_count; it++) {
                if (it > 0) {
                    for (int j = c->n_inner - 1; j >= 0; j--) {
                        int l = c->inner[j];
                        if (++val[l] < sp->ext[l]) break;
                        val[l] = 0;
                    }
                }
                int absent = 0;
                for (int k = 0; k < n; k++) {
                    off[k] = base[k];
                    for (int j = 0; j < c->n_inner; j++) off[k] += val[c->inner[j]] * c->stride[k][c->inner[j]];
                    v[k] = c->ins[k][off[k]];
                    if (isnan(v[k])) absent = 1;
                }
                if (absent) continue;
                if (sp->pred_a >= 0 && !(val[sp->pred_a] + sp->lo[sp->pred_a] <= val[sp->pred_b] + sp->lo[sp->pred_b])) continue;
                double f = apply_map(c->map, v, n, c->scale, c->eps);
                if (cnt == 0) acc = f;
                else if (c->agg == A_SUM) acc += f;
                else if (c->agg == A_MAX) acc = fmax(acc, f);
                else atomic_store(&c->err, 1);
                cnt++;
            }
            c->out[o] = cnt ? acc : NAN;
        }
    }
    return NULL;
}

static int hw_threads(int want) {
    if (want > 0) return want;
    /* ORC_THREADS caps the default (the benchmark's one-core baseline) */
    const char *env = getenv("ORC_THREADS");
    if (env && atoi(env) > 0) return atoi(env);
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

int orc_joinagg_idx(const char *spec, const int64_t *shapes, const double *const *ins, int map, int agg,
                    double scale, double eps, const char *pred, const int64_t *lo, double *out, int nthreads) {
    spec_t sp;
    if (parse_spec(spec, shapes, pred, lo, &sp)) return -1;
    if (!map_arity_ok(map, sp.n_in)) return fail("map: wrong number of inputs");
    if (agg < A_NONE || agg > A_MAX) return fail("agg: unknown");
    ictx_t *c = (ictx_t *)calloc(1, sizeof(ictx_t));
    if (!c) return fail("oracle: out of host memory");
    c->sp = &sp;
    c->ins = ins;
    c->out = out;
    c->map = map;
    c->agg = agg;
    c->scale = scale;
    c->eps = eps;
    /* Inner letters: in the inputs but not in the output, in order of first appearance. */
    int seen[NLET] = {0};
    for (int k = 0; k < sp.n_in; k++)
        for (int d = 0; d < sp.rank[k]; d++) {
            int l = sp.let[k][d];
            if (!sp.in_out[l] && !seen[l]) {
                seen[l] = 1;
                c->inner[c->n_inner++] = l;
            }
        }
    for (int k = 0; k < sp.n_in; k++) {
        int64_t s = 1;
        for (int d = sp.rank[k] - 1; d >= 0; d--) {
            c->stride[k][sp.let[k][d]] = s;
            s *= sp.ext[sp.let[k][d]];
        }
    }
    c->cells = out_cells(&sp);
    int nt = hw_threads(nthreads);
    c->chunk = c->cells / ((int64_t)nt * 16) + 1;
    atomic_store(&c->next, 0);
    atomic_store(&c->err, 0);
    pthread_t th[256];
    if (nt > 256) nt = 256;
    int started = 0;
    for (int t = 1; t < nt; t++)
        if (pthread_create(&th[started], NULL, idx_worker, c) == 0) started++;
    idx_worker(c);
    for (int t = 0; t < started; t++) pthread_join(th[t], NULL);
    int rc = 0;
    if (atomic_load(&c->err)) rc = fail("agg NONE: a group holds more than one joined tuple");
    free(c);
    return rc;
}

/* ------------------------------------------------------------ exchange */

/* Tilings are given per dimension as nb[d] intervals with bounds
 * b[d][0] = 0 < ... < b[d][nb[d]] = dims[d] (flattened, dimension after
 * dimension).  Blocks are numbered row-major over the block grid; each
 * block is stored row-major and blocks follow one another in id order.  */
typedef struct {
    int rank;
    int64_t dims[MAXR];
    int nb[MAXR];
    const int64_t *b[MAXR];
    int64_t nblocks;
    int64_t *off; /* element offset of each block in the arena */
} tiling_t;

static int tiling_make(int rank, const int64_t *dims, const int32_t *nb, const int64_t *bounds, tiling_t *t) {
    memset(t, 0, sizeof *t);
    t->rank = rank;
    const int64_t *p = bounds;
    t->nblocks = 1;
    for (int d = 0; d < rank; d++) {
        t->dims[d] = dims[d];
        t->nb[d] = nb[d];
        t->b[d] = p;
        if (nb[d] < 1 || p[0] != 0 || p[nb[d]] != dims[d]) return fail("tiling: bounds must run from 0 to the extent");
        for (int i = 0; i < nb[d]; i++)
            if (p[i + 1] < p[i]) return fail("tiling: bounds must not decrease");
        p += nb[d] + 1;
        t->nblocks *= nb[d];
    }
    t->off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(t->nblocks + 1));
    if (!t->off) return fail("oracle: out of host memory");
    int64_t bi[MAXR] = {0};
    int64_t acc = 0;
    for (int64_t id = 0; id < t->nblocks; id++) {
        t->off[id] = acc;
        int64_t sz = 1;
        for (int d = 0; d < rank; d++) sz *= t->b[d][bi[d] + 1] - t->b[d][bi[d]];
        acc += sz;
        for (int d = rank - 1; d >= 0; d--) {
            if (++bi[d] < nb[d]) break;
            bi[d] = 0;
        }
    }
    t->off[t->nblocks] = acc;
    return 0;
}

/* Arena position of the element at global coordinates g. */
static int64_t tiling_locate(const tiling_t *t, const int64_t *g) {
    int64_t id = 0, inner = 0;
    int64_t bi[MAXR];
    for (int d = 0; d < t->rank; d++) {
        int lo = 0, hi = t->nb[d] - 1;
        while (lo < hi) { /* last block whose lower bound is <= g */
            int mid = (lo + hi + 1) / 2;
            if (t->b[d][mid] <= g[d]) lo = mid;
            else hi = mid - 1;
        }
        while (t->b[d][lo + 1] <= g[d]) lo++; /* skip empty blocks */
        bi[d] = lo;
        id = id * t->nb[d] + lo;
    }
    for (int d = 0; d < t->rank; d++) {
        int64_t ext = t->b[d][bi[d] + 1] - t->b[d][bi[d]];
        inner = inner * ext + (g[d] - t->b[d][bi[d]]);
    }
    return t->off[id] + inner;
}

typedef struct {
    const tiling_t *src, *dst;
    int esize;
    const unsigned char *sa;
    unsigned char *da;
    int64_t *perm;
    _Atomic int64_t next;
} xctx_t;

static void *x_worker(void *arg) {
    xctx_t *c = (xctx_t *)arg;
    const tiling_t *D = c->dst;
    for (;;) {
        int64_t id = atomic_fetch_add(&c->next, 1);
        if (id >= D->nblocks) break;
        int64_t rem = id, bi[MAXR], lo[MAXR], ext[MAXR];
        for (int d = D->rank - 1; d >= 0; d--) {
            bi[d] = rem % D->nb[d];
            rem /= D->nb[d];
        }
        int64_t n = 1;
        for (int d = 0; d < D->rank; d++) {
            lo[d] = D->b[d][bi[d]];
            ext[d] = D->b[d][bi[d] + 1] - lo[d];
            n *= ext[d];
        }
        int64_t loc[MAXR] = {0}, g[MAXR];
        for (int64_t e = 0; e < n; e++) {
            for (int d = 0; d < D->rank; d++) g[d] = lo[d] + loc[d];
            int64_t s = tiling_locate(c->src, g);
            int64_t dpos = D->off[id] + e;
            if (c->perm) c->perm[dpos] = s;
            if (c->da) memcpy(c->da + dpos * c->esize, c->sa + s * c->esize, (size_t)c->esize);
            for (int d = D->rank - 1; d >= 0; d--) {
                if (++loc[d] < ext[d]) break;
                loc[d] = 0;
            }
        }
    }
    return NULL;
}

static int exchange_impl(int rank, const int64_t *dims, int esize, const int32_t *src_nb, const int64_t *src_b,
                         const int32_t *dst_nb, const int64_t *dst_b, const void *src, void *dst, int64_t *perm,
                         int nthreads) {
    if (rank < 1 || rank > MAXR) return fail("exchange: rank out of range");
    tiling_t S, D;
    memset(&S, 0, sizeof S);
    memset(&D, 0, sizeof D);
    int rc = -1;
    if (tiling_make(rank, dims, src_nb, src_b, &S)) goto done;
    if (tiling_make(rank, dims, dst_nb, dst_b, &D)) goto done;
    xctx_t c;
    c.src = &S;
    c.dst = &D;
    c.esize = esize;
    c.sa = (const unsigned char *)src;
    c.da = (unsigned char *)dst;
    c.perm = perm;
    atomic_store(&c.next, 0);
    int nt = hw_threads(nthreads);
    if (nt > 256) nt = 256;
    pthread_t th[256];
    int started = 0;
    for (int t = 1; t < nt; t++)
        if (pthread_create(&th[started], NULL, x_worker, &c) == 0) started++;
    x_worker(&c);
    for (int t = 0; t < started; t++) pthread_join(th[t], NULL);
    rc = 0;
done:
    free(S.off);
    free(D.off);
    return rc;
}

int orc_exchange(int rank, const int64_t *dims, int esize, const int32_t *src_nb, const int64_t *src_b,
                 const int32_t *dst_nb, const int64_t *dst_b, const void *src, void *dst, int nthreads) {
    return exchange_impl(rank, dims, esize, src_nb, src_b, dst_nb, dst_b, src, dst, NULL, nthreads);
}

int orc_exchange_perm(int rank, const int64_t *dims, const int32_t *src_nb, const int64_t *src_b,
                      const int32_t *dst_nb, const int64_t *dst_b, int64_t *perm, int nthreads) {
    return exchange_impl(rank, dims, 1, src_nb, src_b, dst_nb, dst_b, NULL, NULL, perm, nthreads);
}

int orc_threads(void) { return hw_threads(0); }
