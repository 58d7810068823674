/* oracle.c -- plain CPU oracle for continuity-aware draft-tree construction.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, by the package smoke check and
 * by the benchmark's CPU-baseline leg; never by the product path.  No code is
 * shared with the CUDA implementation.
 *
 * The method is a heuristic (per-depth beam pruning), so this file follows its
 * steps in the pages' order rather than a closed form:
 *   1. per position j: p_j = log_softmax(z_j / T) and C_j, the k best tokens
 *      of that position's own logit vector (DART, Figure 3 caption);
 *   2. per depth: every frontier node is expanded by every candidate and each
 *      child scored as parent score + p_j[c] + lambda * ngram(context, c), with
 *      beta standing in for an n-gram the model lacks (DART, Figure 3 caption,
 *      the N-gram continuity step; DARTree, Tree Construction: all nodes of a
 *      depth are expanded and scored together);
 *   3. the W best children over the whole frontier survive, the rest are
 *      dropped (DARTree, Tree Construction, best-first pruning per depth);
 *   4. token ids, parent indices, depths and ancestor masks are emitted for
 *      tree-attention verification (DART, Figure 3 caption; DARTree,
 *      Verification).
 * Readings where the pages are silent: the root is the last committed token
 * and is not a node; T = 0 (greedy decoding, DART Figure 2 caption) names
 * the target's sampling, not a log-softmax: candidates come from the raw
 * logits whatever T is, and the tree is scored with the draft's own
 * log-probabilities, log_softmax(z), exactly as at T = 1, so that the first
 * child of each depth extends the argmax chain when lambda = 0; the n-gram context is the last n-1 tokens of (committed
 * context ++ path); candidates are ranked on the raw logits, lower id first on
 * equal values; children are ranked by score, then lower parent index, then
 * lower token id, and nodes of a depth are numbered in that order.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- decoding */

static double f16_to_double(uint16_t h) {
    /* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits */
    int s = h >> 15, e = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v;
    if (e == 0) v = ldexp((double)m, -24);
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp((double)(m + 1024), e - 25);
    return s ? -v : v;
}

static double bf16_to_double(uint16_t b) {
    /* bfloat16 is the upper half of an IEEE 754 binary32 */
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_decode(const void* logits, int dtype, int64_t i) {
    if (dtype == 0) return (double)((const float*)logits)[i];
    if (dtype == 1) return f16_to_double(((const uint16_t*)logits)[i]);
    return bf16_to_double(((const uint16_t*)logits)[i]);
}

/* ------------------------------------------------- step 1: rows (a1 + a2) */

typedef struct { double z; int32_t id; } zid_t;

static int cmp_zid(const void* pa, const void* pb) {
    const zid_t* a = (const zid_t*)pa;
    const zid_t* b = (const zid_t*)pb;
    if (a->z > b->z) return -1;
    if (a->z < b->z) return 1;
    return (a->id > b->id) - (a->id < b->id);
}

static void one_row(const void* logits, int dtype, int64_t r, int V, double T, int k,
                    int32_t* ids, double* logp, double* lse, zid_t* work) {
    int64_t off = r * (int64_t)V;
    double m = -INFINITY, S = 0.0;
    for (int v = 0; v < V; ++v) {
        double z = oracle_decode(logits, dtype, off + v);
        work[v].z = z;
        work[v].id = v;
        double x = z / T;
        if (x > m) m = x;
    }
    for (int v = 0; v < V; ++v) S += exp(work[v].z / T - m);
    double l = m + log(S);
    if (lse) lse[r] = l;
    qsort(work, (size_t)V, sizeof(zid_t), cmp_zid);
    for (int c = 0; c < k; ++c) {
        ids[r * k + c] = work[c].id;
        logp[r * k + c] = work[c].z / T - l;
    }
}

/* The temperature the scores use: T itself, or 1 for greedy T = 0. */
static double score_temperature(double T) { return T == 0.0 ? 1.0 : T; }

int oracle_rows(const void* logits, int dtype, int64_t rows, int V, double T, int k,
                int32_t* ids, double* logp, double* lse, int threads) {
    if (!logits || rows < 0 || V < 1 || k < 1 || k > V || !(T >= 0.0) || !ids || !logp) return 1;
    T = score_temperature(T);
    int fail = 0;
#ifdef _OPENMP
    if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel num_threads(threads) reduction(| : fail)
#endif
    {
        zid_t* work = (zid_t*)malloc(sizeof(zid_t) * (size_t)V);
        if (!work) fail = 1;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t r = 0; r < rows; ++r)
            if (work) one_row(logits, dtype, r, V, T, k, ids, logp, lse, work);
        free(work);
    }
    return fail;
}

/* -------------------------------------------------------- n-gram model */

typedef struct { int32_t t[4]; float v; int64_t order; } ngram_t;

struct oracle_ngram { int n; int64_t M; ngram_t* e; };

static int cmp_tokens(const int32_t* a, const int32_t* b, int n) {
    for (int i = 0; i < n; ++i) {
        if (a[i] < b[i]) return -1;
        if (a[i] > b[i]) return 1;
    }
    return 0;
}

static int cmp_ngram(const void* pa, const void* pb) {
    const ngram_t* a = (const ngram_t*)pa;
    const ngram_t* b = (const ngram_t*)pb;
    int c = cmp_tokens(a->t, b->t, 4);
    if (c) return c;
    return (a->order > b->order) - (a->order < b->order);
}

oracle_ngram* oracle_ngram_new(int n, const int32_t* keys, const float* vals, int64_t M) {
    if (n < 1 || n > 4 || M < 0 || (M > 0 && (!keys || !vals))) return NULL;
    oracle_ngram* t = (oracle_ngram*)calloc(1, sizeof *t);
    if (!t) return NULL;
    t->n = n;
    t->M = M;
    t->e = (ngram_t*)malloc(sizeof(ngram_t) * (size_t)(M > 0 ? M : 1));
    if (!t->e) { free(t); return NULL; }
    for (int64_t i = 0; i < M; ++i) {
        for (int f = 0; f < 4; ++f) t->e[i].t[f] = f < n ? keys[i * n + f] : 0;
        t->e[i].v = vals[i];
        t->e[i].order = i;
    }
    qsort(t->e, (size_t)M, sizeof(ngram_t), cmp_ngram);
    return t;
}

void oracle_ngram_free(oracle_ngram* t) {
    if (t) { free(t->e); free(t); }
}

/* the first entry (lowest insertion order) holding exactly key[0..3] */
static const ngram_t* ngram_find(const oracle_ngram* t, const int32_t key4[4]) {
    int64_t lo = 0, hi = t->M; /* first index whose tokens are >= key */
    while (lo < hi) {
        int64_t mid = lo + (hi - lo) / 2;
        if (cmp_tokens(t->e[mid].t, key4, 4) < 0) lo = mid + 1;
        else hi = mid;
    }
    if (lo < t->M && cmp_tokens(t->e[lo].t, key4, 4) == 0) return &t->e[lo];
    return NULL;
}

static int ngram_get(const oracle_ngram* t, const int32_t* key, float* val) {
    int32_t k4[4] = {0, 0, 0, 0};
    for (int f = 0; f < t->n; ++f) k4[f] = key[f];
    const ngram_t* e = ngram_find(t, k4);
    if (!e) return 0;
    *val = e->v;
    return 1;
}

void oracle_ngram_lookup(const oracle_ngram* t, const int32_t* keys, int64_t Q,
                         float* vals, int32_t* found) {
    for (int64_t q = 0; q < Q; ++q) {
        float v = 0.0f;
        found[q] = ngram_get(t, keys + q * t->n, &v);
        vals[q] = v;
    }
}

/* ------------------------------------------- steps 2-4: the tree (a3-a6) */

int oracle_num_nodes(int d, int k, int W) {
    if (d < 1 || k < 1 || W < 1) return -1;
    long long total = 0, width = 1;
    for (int j = 1; j <= d; ++j) {
        width *= k;
        if (width > W) width = W;
        total += width;
        if (total > (1LL << 30)) return -1;
    }
    return (int)total;
}

typedef struct { double key, Z, G, g; int32_t i; int32_t tok; int32_t col; int32_t found; } cand_t;

static int cmp_cand(const void* pa, const void* pb) {
    const cand_t* a = (const cand_t*)pa;
    const cand_t* b = (const cand_t*)pb;
    if (a->key > b->key) return -1;       /* higher score first */
    if (a->key < b->key) return 1;
    if (a->i != b->i) return a->i < b->i ? -1 : 1;       /* then lower parent */
    return (a->tok > b->tok) - (a->tok < b->tok);        /* then lower token id */
}

int oracle_mask_from_parents(int B, int N, const int32_t* parents, uint32_t* mask) {
    if (B < 0 || N < 0 || (N > 0 && (!parents || !mask))) return 1;
    int MW = (N + 31) / 32;
    memset(mask, 0, sizeof(uint32_t) * (size_t)B * (size_t)N * (size_t)MW);
    for (int b = 0; b < B; ++b) {
        for (int x = 0; x < N; ++x) {
            uint32_t* row = mask + ((size_t)b * N + x) * MW;
            int a = x, steps = 0;
            while (a >= 0) {
                if (a >= N || steps > N) return 2;
                row[a >> 5] |= 1u << (a & 31);
                int p = parents[(size_t)b * N + a];
                if (p >= a) return 2;
                a = p;
                ++steps;
            }
        }
    }
    return 0;
}

/* One tree.  A node's path score is sum_j p_j[c_j] + lam * sum_j g_j with
 * p_j[c] = base_j[c] * invT - off_j.  Every node of one depth carries the same
 * sum of off_j, so children are ranked by key = Z * invT + lam * G, where Z is
 * the sum of the base values along the path and G the sum of n-gram terms,
 * each accumulated in double from the root in path order; the reported score
 * is key minus that common sum.  Ranking on the key keeps every tie that the
 * inputs hold exactly (equal sums of logits along two paths) an exact tie,
 * whatever the rounding of the log-partition terms. */
static int one_tree(int b, int d, int k, int W, int N,
                    const int32_t* ids, const double* base, double invT, const double* off,
                    double lam, double beta, const oracle_ngram* tab, int n,
                    const float* pair, const int32_t* ctx,
                    int32_t* tokens, int32_t* parents, int32_t* pos, double* scores,
                    double* min_pos_gap, oracle_trace_entry* trace) {
    int L = (n > 1 ? n - 1 : 0) + d;             /* longest sequence */
    int Wmax = W;
    double* fZ = (double*)malloc(sizeof(double) * Wmax);
    double* fG = (double*)malloc(sizeof(double) * Wmax);
    int* fnode = (int*)malloc(sizeof(int) * Wmax);
    int* fcol = (int*)malloc(sizeof(int) * Wmax);     /* each frontier node's column in its row */
    int* ncol = (int*)malloc(sizeof(int) * Wmax);
    int32_t* fseq = (int32_t*)malloc(sizeof(int32_t) * (size_t)Wmax * (L > 0 ? L : 1));
    double* nZ = (double*)malloc(sizeof(double) * Wmax);
    double* nG = (double*)malloc(sizeof(double) * Wmax);
    int* nnode = (int*)malloc(sizeof(int) * Wmax);
    int32_t* nseq = (int32_t*)malloc(sizeof(int32_t) * (size_t)Wmax * (L > 0 ? L : 1));
    cand_t* cand = (cand_t*)malloc(sizeof(cand_t) * (size_t)Wmax * k);
    int rc = 0;
    if (!fZ || !fG || !fnode || !fcol || !ncol || !fseq || !nZ || !nG || !nnode || !nseq || !cand) rc = 1;
    int nc = n > 1 ? n - 1 : 0;                  /* committed context length */
    int F = 1, len = nc, next = 0;
    double Lsum = 0.0;
    if (!rc) {
        fZ[0] = 0.0;
        fG[0] = 0.0;
        fnode[0] = -1;
        fcol[0] = 0;                             /* the root counts as column 0 */
        for (int c = 0; c < nc; ++c) fseq[c] = ctx[(size_t)b * nc + c];
    }
    for (int j = 0; j < d && !rc; ++j) {
        const int32_t* C = ids + ((size_t)b * d + j) * k;
        const double* P = base + ((size_t)b * d + j) * k;
        if (off) Lsum = Lsum + off[(size_t)b * d + j];
        int m = 0;
        for (int i = 0; i < F; ++i) {
            const int32_t* seq = fseq + (size_t)i * L;
            for (int c = 0; c < k; ++c) {
                double Z = fZ[i] + P[c];
                double G = fG[i];
                double term = 0.0;
                int found = 0;
                if (tab) {
                    int32_t key[4];
                    for (int q = 0; q < n - 1; ++q) key[q] = seq[len - (n - 1) + q];
                    key[n - 1] = C[c];
                    float g = 0.0f;
                    found = ngram_get(tab, key, &g);
                    double gg = found ? (double)g : beta;
                    G = G + gg;
                    term = gg;
                } else if (pair) {
                    /* caller-supplied continuity score of (parent's column, c) */
                    term = (double)pair[(((size_t)b * d + j) * k + fcol[i]) * k + c];
                    G = G + term;
                    found = 1;
                }
                cand[m].Z = Z;
                cand[m].G = G;
                cand[m].key = Z * invT + lam * G;
                cand[m].i = i;
                cand[m].tok = C[c];
                cand[m].col = c;
                cand[m].g = term;
                cand[m].found = found;
                ++m;
            }
        }
        qsort(cand, (size_t)m, sizeof(cand_t), cmp_cand);
        int keep = m < W ? m : W;
        if (trace) {
            for (int r = 0; r < m; ++r, ++trace) {
                trace->depth = j + 1;
                trace->parent = fnode[cand[r].i];
                trace->parent_rank = cand[r].i;
                trace->token = cand[r].tok;
                trace->column = cand[r].col;
                trace->found = cand[r].found;
                trace->node = r < keep ? next + r : -1;
                trace->pad = 0;
                trace->g = cand[r].g;
                trace->Z = cand[r].Z;
                trace->G = cand[r].G;
                trace->key = cand[r].key;
            }
        }
        if (min_pos_gap) {
            double g = 1e300;
            for (int r = 0; r < keep && r + 1 < m; ++r) {
                double gap = cand[r].key - cand[r + 1].key;
                if (gap > 0.0 && gap < g) g = gap;
            }
            min_pos_gap[(size_t)b * d + j] = g;
        }
        for (int r = 0; r < keep; ++r) {
            int node = next + r;
            if (node >= N) { rc = 2; break; }
            const cand_t* e = &cand[r];
            tokens[(size_t)b * N + node] = e->tok;
            parents[(size_t)b * N + node] = fnode[e->i];
            pos[(size_t)b * N + node] = j + 1;
            if (scores) scores[(size_t)b * N + node] = e->key - Lsum;
            nZ[r] = e->Z;
            nG[r] = e->G;
            nnode[r] = node;
            ncol[r] = e->col;
            memcpy(nseq + (size_t)r * L, fseq + (size_t)e->i * L, sizeof(int32_t) * (size_t)len);
            nseq[(size_t)r * L + len] = e->tok;
        }
        next += keep;
        F = keep;
        len += 1;
        if (!rc) {
            memcpy(fZ, nZ, sizeof(double) * F);
            memcpy(fG, nG, sizeof(double) * F);
            memcpy(fnode, nnode, sizeof(int) * F);
            memcpy(fcol, ncol, sizeof(int) * F);
            memcpy(fseq, nseq, sizeof(int32_t) * (size_t)F * L);
        }
    }
    free(fZ); free(fG); free(fnode); free(fcol); free(ncol); free(fseq); free(nZ); free(nG); free(nnode); free(nseq); free(cand);
    if (rc) return rc;
    return next == N ? 0 : 3;
}

int oracle_tree_from_lists(int B, int d, int k, int W,
                           const int32_t* ids, const double* base, double invT, const double* off,
                           double lam, double beta, const oracle_ngram* tab, int n,
                           const int32_t* ctx,
                           int32_t* tokens, int32_t* parents, int32_t* pos,
                           uint32_t* mask, double* scores, double* min_pos_gap,
                           int threads) {
    int N = oracle_num_nodes(d, k, W);
    if (B < 0 || N < 0 || !ids || !base || !tokens || !parents || !pos) return 1;
    if (tab && (n != tab->n || n < 2 || (!ctx && B > 0))) return 1;
    int fail = 0;
#ifdef _OPENMP
    if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel for num_threads(threads) schedule(dynamic, 1) reduction(| : fail)
#endif
    for (int b = 0; b < B; ++b)
        fail |= one_tree(b, d, k, W, N, ids, base, invT, off, lam, beta, tab, tab ? n : 0, NULL, ctx,
                         tokens, parents, pos, scores, min_pos_gap, NULL);
    if (fail) return fail;
    if (mask) return oracle_mask_from_parents(B, N, parents, mask);
    return 0;
}

/* The tree with a caller-supplied continuity scorer in place of the n-gram
 * model (DARTree, Method / Tree Construction: the children of a depth are
 * scored by the head H in one batch; an order-2 head restricted to the
 * candidate sets is a table of candidate-pair scores).  The term a child with
 * column c of row j adds to G is pair[b][j][c'][c], c' the parent's column in
 * row j-1, and c' = 0 (the root) at j = 0. */
int oracle_tree_from_pairs(int B, int d, int k, int W,
                           const int32_t* ids, const double* base, double invT, const double* off,
                           double lam, const float* pair,
                           int32_t* tokens, int32_t* parents, int32_t* pos,
                           uint32_t* mask, double* scores, double* min_pos_gap,
                           int threads) {
    int N = oracle_num_nodes(d, k, W);
    if (B < 0 || N < 0 || !ids || !base || !pair || !tokens || !parents || !pos) return 1;
    int fail = 0;
#ifdef _OPENMP
    if (threads <= 0) threads = omp_get_max_threads();
#pragma omp parallel for num_threads(threads) schedule(dynamic, 1) reduction(| : fail)
#endif
    for (int b = 0; b < B; ++b)
        fail |= one_tree(b, d, k, W, N, ids, base, invT, off, lam, 0.0, NULL, 0, pair, NULL,
                         tokens, parents, pos, scores, min_pos_gap, NULL);
    if (fail) return fail;
    if (mask) return oracle_mask_from_parents(B, N, parents, mask);
    return 0;
}

/* One tree with every expanded child recorded (see oracle.h). */
int oracle_tree_trace(int d, int k, int W, const int32_t* ids, const double* base, double invT,
                      const double* off, double lam, double beta, const oracle_ngram* tab, int n,
                      const int32_t* ctx, oracle_trace_entry* trace, int64_t trace_cap,
                      int64_t* trace_len) {
    int N = oracle_num_nodes(d, k, W);
    if (N < 0 || !ids || !base || !trace || !trace_len) return 1;
    if (tab && (n != tab->n || n < 2 || !ctx)) return 1;
    int64_t need = 0, width = 1;
    for (int j = 0; j < d; ++j) {
        need += width * k;
        width = width * k < W ? width * k : W;
    }
    if (need > trace_cap) return 1;
    int32_t* tok = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
    int32_t* par = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
    int32_t* pos = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
    int rc = (!tok || !par || !pos) ? 1 : one_tree(0, d, k, W, N, ids, base, invT, off, lam, beta, tab,
                                                   tab ? n : 0, NULL, ctx, tok, par, pos, NULL, NULL, trace);
    free(tok); free(par); free(pos);
    *trace_len = rc ? 0 : need;
    return rc;
}

int oracle_tree_build(const void* logits, int dtype, int B, int d, int V, double T,
                      int k, int W, double lam, double beta,
                      const oracle_ngram* tab, int n, const int32_t* ctx,
                      int32_t* tokens, int32_t* parents, int32_t* pos, uint32_t* mask,
                      double* scores, double* min_pos_gap,
                      int32_t* row_ids, double* row_logp, double* row_lse, int threads) {
    if (B < 0 || d < 1 || k < 1 || k > V || !(T >= 0.0)) return 1;
    T = score_temperature(T);
    size_t R = (size_t)B * d;
    int32_t* ids = row_ids ? row_ids : (int32_t*)malloc(sizeof(int32_t) * (R * k + 1));
    double* lp = row_logp ? row_logp : (double*)malloc(sizeof(double) * (R * k + 1));
    double* lse = row_lse ? row_lse : (double*)malloc(sizeof(double) * (R + 1));
    double* zc = (double*)malloc(sizeof(double) * (R * k + 1));
    int rc = (!ids || !lp || !lse || !zc) ? 1 : 0;
    if (!rc) rc = oracle_rows(logits, dtype, (int64_t)R, V, T, k, ids, lp, lse, threads);
    if (!rc) {
        /* the candidates' own logits are the base values of the ranking key */
        for (size_t r = 0; r < R; ++r)
            for (int c = 0; c < k; ++c)
                zc[r * k + c] = oracle_decode(logits, dtype, (int64_t)r * V + ids[r * k + c]);
        rc = oracle_tree_from_lists(B, d, k, W, ids, zc, 1.0 / T, lse, lam, beta, tab, n, ctx,
                                    tokens, parents, pos, mask, scores, min_pos_gap, threads);
    }
    if (!row_ids) free(ids);
    if (!row_logp) free(lp);
    if (!row_lse) free(lse);
    free(zc);
    return rc;
}

/* ------------------------------------------------- verification tree selection */

/* Node a beats node b: larger score, then lower index. */
static int sel_better(const double* s, int a, int b) {
    if (s[a] != s[b]) return s[a] > s[b];
    return a < b;
}

int oracle_select_tree(int B, int N, int M, const int32_t* parents, const double* scores,
                       int32_t* index, int32_t* new_parents) {
    if (B < 0 || N < 0 || M < 0) return 1;
    int Mp = M < N ? M : N;
    if (B == 0 || Mp == 0) return 0;
    if (!parents || !scores || !index || !new_parents) return 1;
    int* avail = (int*)malloc(sizeof(int) * (size_t)N);   /* the available nodes, unordered */
    char* taken = (char*)malloc((size_t)N);
    int* newpos = (int*)malloc(sizeof(int) * (size_t)N);
    if (!avail || !taken || !newpos) {
        free(avail); free(taken); free(newpos);
        return 1;
    }
    int rc = 0;
    for (int b = 0; b < B && rc == 0; ++b) {
        const int32_t* par = parents + (size_t)b * N;
        const double* s = scores + (size_t)b * N;
        for (int i = 0; i < N; ++i)
            if (par[i] >= i) rc = 2;
        if (rc) break;
        int na = 0;
        for (int i = 0; i < N; ++i) {
            taken[i] = 0;
            if (par[i] < 0) avail[na++] = i;
        }
        /* best-first: M' times pick the best available node (a plain scan of the
         * available set stands in for the priority queue) */
        for (int t = 0; t < Mp; ++t) {
            if (na == 0) { rc = 2; break; }
            int best = 0;
            for (int a = 1; a < na; ++a)
                if (sel_better(s, avail[a], avail[best])) best = a;
            int x = avail[best];
            avail[best] = avail[--na];
            taken[x] = 1;
            for (int c = x + 1; c < N; ++c)
                if (par[c] == x) avail[na++] = c;
        }
        if (rc) break;
        int m = 0;
        for (int i = 0; i < N; ++i) {
            newpos[i] = -1;
            if (taken[i]) newpos[i] = m, index[(size_t)b * Mp + m++] = i;
        }
        for (int j = 0; j < Mp; ++j) {
            int i = index[(size_t)b * Mp + j];
            new_parents[(size_t)b * Mp + j] = par[i] < 0 ? -1 : newpos[par[i]];
        }
    }
    free(avail); free(taken); free(newpos);
    return rc;
}
