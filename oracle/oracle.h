/* oracle.h -- plain CPU oracle for continuity-aware draft-tree construction.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code with
 * the CUDA path.  Everything is double precision, every ordering is a full
 * sort, the n-gram model is a sorted array searched with bsearch.
 *
 * Sources (page titles and sections):
 *  - "DART: Diffusion-Inspired Speculative Decoding for Fast LLM Inference",
 *    Figure 3 caption: d logits from one forward pass, the first from the last
 *    prefix position; candidates per position taken from that position's
 *    logits; an N-gram model keeps expanded tokens continuous; the pruned tree
 *    is verified with tree attention.
 *  - "DARTree: Speculative Diffusion Decoding with Autoregressive Draft Trees",
 *    Method / Tree Construction: a tree of fixed width; all nodes of the
 *    previous depth are expanded and scored together, and after each depth
 *    only the W best-scoring nodes of the full frontier survive.
 *  - The two pages made precise (the readings are listed in oracle.c):
 *    p_j = log_softmax(z_j / T), C_j = top-k of p_j, child score = parent
 *    score + p_j[c] + lambda * ngram(last n-1 path tokens, c), a missing
 *    n-gram costing beta, ties broken by lower parent index then lower token
 *    id; outputs are tokens, parents, depths and a bit-packed ancestor mask.
 */
#ifndef DART_ORACLE_H
#define DART_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dtype codes of the stored logits: 0 = f32, 1 = f16, 2 = bf16 (bit patterns). */

/* Per row r < rows of logits[rows][V]: lse[r], the k best token ids (value
 * descending, lower id first on equal values) and their log-probabilities
 * log_softmax(z / T).  T >= 0; T = 0 (greedy) scores as T = 1. */
int oracle_rows(const void* logits, int dtype, int64_t rows, int V, double T, int k,
                int32_t* ids, double* logp, double* lse, int threads);

/* Decode one stored logit to double (exact for all three dtypes). */
double oracle_decode(const void* logits, int dtype, int64_t index);

typedef struct oracle_ngram oracle_ngram;
/* keys[M][n] (oldest context token first, predicted token last), vals[M].
 * A repeated key keeps its first value. */
oracle_ngram* oracle_ngram_new(int n, const int32_t* keys, const float* vals, int64_t M);
void oracle_ngram_free(oracle_ngram* t);
/* found[q] = 1 and vals[q] = value when keys[q][0..n) is in the model, else 0. */
void oracle_ngram_lookup(const oracle_ngram* t, const int32_t* keys, int64_t Q,
                         float* vals, int32_t* found);

/* Tree construction from per-depth candidate lists, ids/base [B][d][k].
 * A candidate's log-probability is base * invT - off[b][j] (off may be NULL
 * for 0); with invT = 1 and off = NULL, base holds log-probabilities.
 * Children are ranked by key = Z * invT + lam * G (Z: sum of base values along
 * the path, G: sum of n-gram values or beta), then lower parent index, then
 * lower token id; scores[] = key - sum of off over the node's depths.
 * tab == NULL means no continuity term.  Outputs [B][N] (mask [B][N][MW]);
 * min_pos_gap[B][d] (may be NULL) is, per depth, the smallest positive key
 * gap between neighbours in the sorted candidate list among the pairs that
 * decide a kept node's rank or the cut (1e300 when there is none). */
int oracle_tree_from_lists(int B, int d, int k, int W,
                           const int32_t* ids, const double* base, double invT, const double* off,
                           double lam, double beta, const oracle_ngram* tab, int n,
                           const int32_t* ctx,
                           int32_t* tokens, int32_t* parents, int32_t* pos,
                           uint32_t* mask, double* scores, double* min_pos_gap,
                           int threads);

/* oracle_tree_from_lists with caller-supplied pair scores pair[B][d][k][k]
 * in place of the n-gram model: a child with column c of row j adds
 * pair[b][j][c'][c] to G, c' its parent's column in row j-1 (0 at j = 0, the
 * root).  Ranking, tie rule and outputs as in oracle_tree_from_lists. */
int oracle_tree_from_pairs(int B, int d, int k, int W,
                           const int32_t* ids, const double* base, double invT, const double* off,
                           double lam, const float* pair,
                           int32_t* tokens, int32_t* parents, int32_t* pos,
                           uint32_t* mask, double* scores, double* min_pos_gap,
                           int threads);

/* One expanded child of a traced tree: its depth, parent node (-1 = root) and
 * the parent's rank in the frontier, token and column in its row, whether
 * the n-gram was found, the node index it became (-1 if cut), the continuity
 * term g it added (the n-gram value, or beta when absent), and its Z, G and
 * ranking key. */
typedef struct {
    int32_t depth, parent, parent_rank, token, column, found, node, pad;
    double g, Z, G, key;
} oracle_trace_entry;

/* One tree (ids/base [d][k], ctx [n-1]) with every expanded child recorded:
 * per depth, the whole sorted candidate table (kept children first, in node
 * order).  At most trace_cap entries; *trace_len receives the count. */
int oracle_tree_trace(int d, int k, int W, const int32_t* ids, const double* base, double invT,
                      const double* off, double lam, double beta, const oracle_ngram* tab, int n,
                      const int32_t* ctx, oracle_trace_entry* trace, int64_t trace_cap,
                      int64_t* trace_len);

/* Rows, then the tree, as one call (base = the candidates' logits, invT =
 * 1 / T, off = each row's log-sum-exp; T = 0 scores as T = 1).  row_ids/row_logp/row_lse may be NULL. */
int oracle_tree_build(const void* logits, int dtype, int B, int d, int V, double T,
                      int k, int W, double lam, double beta,
                      const oracle_ngram* tab, int n, const int32_t* ctx,
                      int32_t* tokens, int32_t* parents, int32_t* pos, uint32_t* mask,
                      double* scores, double* min_pos_gap,
                      int32_t* row_ids, double* row_logp, double* row_lse, int threads);

/* N = sum over depths j = 1..d of min(W, k^j); -1 when the arguments are invalid. */
int oracle_num_nodes(int d, int k, int W);

/* Ancestor-or-self mask rows from a parent array (parents[i] < i, -1 for depth 1). */
int oracle_mask_from_parents(int B, int N, const int32_t* parents, uint32_t* mask);

/* Verification tree by best-first selection from a candidate tree (DARTree,
 * abstract and Verification: the candidate tree is built first, then only
 * best-first pruning selects the tree sent to verification; PCTree, abstract:
 * a fixed verification budget goes to the most probable paths).  Per tree b,
 * with nodes 0..N-1 (parents[i] < i, -1 at depth 1) and path scores
 * scores[i]: start with the depth-1 nodes available; M times take the
 * available node of largest score (lower node index on equal scores) and make
 * its children available.  index[b][0..M'-1] receives the taken nodes in
 * increasing node index, M' = min(M, N); new_parents[b][m] is the position in
 * that list of node index[m]'s parent (-1 at depth 1).  Returns 0, 1 on bad
 * arguments, 2 on a parent array that does not point backwards. */
int oracle_select_tree(int B, int N, int M, const int32_t* parents, const double* scores,
                       int32_t* index, int32_t* new_parents);

#ifdef __cplusplus
}
#endif
#endif
