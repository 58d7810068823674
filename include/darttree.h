/* darttree.h -- continuity-aware draft-tree construction on one GPU (C ABI).
 *
 * What the library computes (page titles and sections):
 *  - "DART: Diffusion-Inspired Speculative Decoding for Fast LLM Inference",
 *    Figure 3 caption: a draft model emits d logit vectors per sequence in one
 *    forward pass (vector 0 from the last prefix position, so vector j
 *    predicts depth j+1); candidates at each position come from that
 *    position's own logits; an N-gram model keeps expanded tokens continuous;
 *    the pruned tree goes to tree-attention verification.
 *  - "DARTree: Speculative Diffusion Decoding with Autoregressive Draft
 *    Trees", Method / Tree Construction: every node of the previous depth is
 *    expanded and scored together, then only the W best-scoring children of
 *    the whole frontier survive (best-first pruning per depth, no heap).
 *
 * Made precise (the readings where the pages are silent):
 *   p_j   = log_softmax(z_j / T)                           for j = 0..d-1
 *   C_j   = the k tokens with the largest z_j, lower id first on equal values
 *   child = parent score + p_j[c] + lambda * g,  g = ngram(last n-1 tokens of
 *           (committed context ++ path), c), or beta when the model lacks it
 *   keep  = the min(W, |frontier| * k) best children, ordered by score
 *           (descending), then lower parent index, then lower token id
 *   The root (last committed token) is not a node.  Nodes are numbered depth
 *   by depth in that order; a depth-1 node has parent -1.
 *   T = 0 is greedy decoding (DART, Figure 2 caption, reports results at T = 0
 *   and T = 1): it says how the target samples, and log_softmax(z / 0) is
 *   undefined, so p_j is then log_softmax(z_j), the draft's own
 *   log-probabilities (the T = 1 values).  C_j does not depend on T; with
 *   lambda = 0 node 0 of every depth lies on the argmax chain.
 * All children of one depth share the sum of their rows' log-sum-exp terms,
 * so the ranking uses key = (sum of the path's logits) * (1/T) + lambda *
 * (sum of its g terms), both sums accumulated in double along the path; a
 * node's reported score is key minus that shared sum.  Ties that the inputs
 * hold exactly therefore stay exact ties and fall to the tie rule.
 *
 * Conventions for every entry point:
 *  - All buffers belong to the caller.  The library allocates no memory and
 *    keeps no state between calls; calls on different streams with different
 *    workspaces may run concurrently.  (dart_tree_build_noalloc is the one
 *    exception: it uses a buffer inside the library, described there.)
 *  - Pointers documented as "device" must point to memory of the current CUDA
 *    device; "host" pointers to ordinary host memory.  `stream` is a
 *    cudaStream_t (NULL = the legacy default stream).
 *  - Argument errors are detected on the host and returned before anything is
 *    launched.  Launch errors return DART_ERR_CUDA.  Kernels never trap: a
 *    problem they detect (a wait that ran out, an inconsistency) sets a bit in
 *    the workspace's device error word, read with dart_device_error().
 *  - Every call that launches work is asynchronous with respect to the host.
 */
#ifndef DARTTREE_H
#define DARTTREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Logit element types. */
enum { DART_F32 = 0, DART_F16 = 1, DART_BF16 = 2 };

/* Status codes returned by every entry point (0 = success). */
enum {
  DART_OK = 0,
  DART_ERR_INVALID_ARG = 1,   /* an argument is out of range, NULL or misaligned */
  DART_ERR_UNSUPPORTED = 2,   /* a valid request the library does not handle */
  DART_ERR_WORKSPACE = 3,     /* workspace NULL, misaligned or too small */
  DART_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
  DART_ERR_INTERNAL = 5,      /* a kernel reported an inconsistency */
  DART_ERR_TIMEOUT = 6,       /* a bounded device wait ran out */
  DART_ERR_TABLE_FULL = 7     /* n-gram packing: load over 1/2, or no slot after displacements */
};

/* Bits of the device error word (see dart_device_error). */
enum {
  DART_DEVERR_WAIT_TIMEOUT = 1u << 0,  /* a bulk-copy wait ran out; the call's output is invalid */
  DART_DEVERR_ROW_MAX = 1u << 1,       /* a row's maximum and its best candidate disagreed */
  DART_DEVERR_SELECT = 1u << 2,        /* the tree selection produced an invalid candidate */
  DART_DEVERR_PARENT = 1u << 3,        /* dart_mask_pack / dart_tree_select: a parent index was not below its child */
  DART_DEVERR_SCORE_RISES = 1u << 4    /* dart_tree_select: a node outscored its parent (the result is the M best,
                                          which best-first need not take) */
};

/* An n-gram model in device memory: a two-choice bucketed hash table.
 * Each slot is 16 bytes {uint32 key[3]; float logprob}; two consecutive slots
 * form a 32-byte bucket, and the table holds capacity / 2 buckets.  A key packs
 * the n tokens (t_0 = oldest context token ... t_{n-1} = the predicted token)
 * as 24-bit fields, t_f at bits [24f, 24f+24) of the 96-bit value key[0] |
 * key[1] << 32 | key[2] << 64, unused fields zero.  An empty slot holds
 * 0xFFFFFFFF in all three key words.  With h =
 * splitmix64-finalizer((key[0] | key[1] << 32) ^ (key[2] * 0x9E3779B97F4A7C15))
 * and nb = capacity / 2, a key lives in bucket b1 = h & (nb - 1) or bucket
 * b2 = (h >> 32) & (nb - 1), where b2 = b1 ^ 1 when the two coincide; a lookup
 * reads both buckets (64 bytes) at once, so it always takes one memory round
 * trip.  Build the slots with dart_ngram_table_pack_host. */
typedef struct {
  int32_t n;            /* order, 2..4 */
  int32_t reserved;     /* must be 0 */
  uint64_t capacity;    /* number of slots, a power of two >= 8 */
  const void* slots;    /* device, capacity * 16 bytes, 64-byte aligned */
} dart_ngram_table_t;

/* N = sum over j = 1..d of min(W, k^j): nodes per tree (the root excluded).
 * Returns -1 when d, k or W is below 1 or N would exceed 2^30. */
int dart_tree_num_nodes(int d, int k, int W);

/* MW = ceil(N / 32): 32-bit words per ancestor-mask row; -1 if N < 0. */
int dart_tree_mask_words(int num_nodes);

/* Device workspace bytes that dart_tree_build / dart_row_topk need for these
 * sizes (rows = B * d).  The result does not depend on the device.  0 when
 * the arguments are invalid. */
size_t dart_tree_workspace_bytes(int B, int d, int V, int dtype, int k);

/* The whole hot path in one call: per-row temperature log-softmax and top-k
 * (one streaming pass over the logits), then per-depth expansion, n-gram
 * scoring and top-W pruning for every sequence, then token ids, parents,
 * depths and ancestor masks.
 *
 *  logits      device [B][d][V], element type `dtype`, row-major, base
 *              16-byte aligned.  Row j of sequence b predicts depth j+1.
 *              Every row needs at least one finite value; NaN and +inf are
 *              not supported (results unspecified).
 *  B           sequences, >= 0 (0 = nothing to do, returns DART_OK)
 *  d           depths, 1..32          V  vocabulary, 2..2^24-1
 *  T           temperature, finite and >= 0; T = 0 (greedy) scores with
 *              log_softmax(z), as T = 1 does (see the readings above)
 *  k           candidates per position, 1..min(32, V)
 *  W           frontier width, 1..64; N = dart_tree_num_nodes(d,k,W) <= 1024
 *  lambda,beta finite; lambda scales the n-gram log-probability, beta is the
 *              value used when the model lacks the n-gram (so a miss adds
 *              lambda * beta)
 *  ngram_table host pointer to a table descriptor, or NULL for no
 *              continuity term (then child = parent + p_j[c])
 *  ctx_tokens  device int32 [B][n-1]: the committed context, oldest first,
 *              the root last; may be NULL only when ngram_table is NULL
 *  out_tokens, out_parents, out_pos   device int32 [B][N]
 *  out_mask    device uint32 [B][N][MW]; bit (i & 31) of word (i >> 5) in
 *              row x is set iff node i is x or an ancestor of x
 *  out_scores  device float [B][N] or NULL: each node's path score
 *  workspace   device, >= dart_tree_workspace_bytes(B,d,V,dtype,k) bytes,
 *              256-byte aligned, zero-filled before its first use (the
 *              library keeps no state in it between calls beyond the
 *              device error word, so no per-call clearing is launched)
 * Returns DART_OK or an error code; see the conventions above. */
int dart_tree_build(const void* logits, int B, int d, int V, int dtype,
                    float T, int k, int W, float lambda, float beta,
                    const dart_ngram_table_t* ngram_table, const int32_t* ctx_tokens,
                    int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                    uint32_t* out_mask, float* out_scores,
                    void* workspace, size_t workspace_bytes, void* stream);

/* dart_tree_build for logits whose rows are row_stride >= V elements apart
 * (a vocabulary padded for the projection that produced them): row r of
 * [B][d] holds its V valid logits at logits + r * row_stride elements, and
 * the elements from V up to the stride are never read (they may hold
 * anything).  The buffer must reach (B*d - 1) * row_stride + V elements;
 * its base is 16-byte aligned, rows need not be.  row_stride = V is
 * dart_tree_build itself; row_stride < V or above 2^30 is
 * DART_ERR_INVALID_ARG.  Every other argument as for dart_tree_build. */
int dart_tree_build_strided(const void* logits, int B, int d, int V, int64_t row_stride, int dtype,
                            float T, int k, int W, float lambda, float beta,
                            const dart_ngram_table_t* ngram_table, const int32_t* ctx_tokens,
                            int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                            uint32_t* out_mask, float* out_scores,
                            void* workspace, size_t workspace_bytes, void* stream);

/* A dart_tree_build_strided call captured once as a CUDA graph and replayed,
 * for decode loops that build trees of the same sizes into the same buffers
 * every step (no counterpart in the pages: it changes how the kernels are
 * launched, not what they compute).  dart_tree_plan_create takes
 * dart_tree_build_strided's arguments without the stream, checks them as that
 * call does (returning its error codes, nothing captured), records its
 * launches on a stream of its own (nothing runs) and returns a host handle in
 * *out_plan (NULL on error).  The device buffers must stay allocated at the
 * same addresses while the plan lives; their contents may change between
 * launches; the table descriptor and the scalars are read at creation.
 * dart_tree_plan_launch(plan, stream) replays the captured kernels on `stream`
 * (NULL = the default stream) on the device that was current at creation
 * (another current device: DART_ERR_INVALID_ARG): results and device error
 * bits are exactly those of dart_tree_build_strided with the same arguments.
 * Into a stream that is itself being captured, it launches the kernels
 * directly, so that the caller's graph records them.
 * dart_tree_plan_destroy releases a plan (NULL: nothing to do); launches
 * already queued must be complete or ordered before it (it does not wait).
 * Returns DART_OK or an error code (DART_ERR_CUDA when graph capture or
 * instantiation fails, DART_ERR_INTERNAL when the host is out of memory). */
typedef struct dart_tree_plan_s* dart_tree_plan_t;
int dart_tree_plan_create(dart_tree_plan_t* out_plan, const void* logits, int B, int d, int V, int64_t row_stride,
                          int dtype, float T, int k, int W, float lambda, float beta,
                          const dart_ngram_table_t* ngram_table, const int32_t* ctx_tokens,
                          int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                          uint32_t* out_mask, float* out_scores, void* workspace, size_t workspace_bytes);
int dart_tree_plan_launch(dart_tree_plan_t plan, void* stream);
int dart_tree_plan_destroy(dart_tree_plan_t plan);

/* dart_tree_build_strided that also emits the best-first verification tree
 * of budget M >= 1 (dart_tree_select's result on the candidate trees, with
 * the same reading and outputs), chosen by each tree's CTA right after it has
 * built the tree, so no second launch reads the candidate trees back:
 *  out_vindex, out_vtokens, out_vparents, out_vpos  device int32 [B][M'],
 *  out_vmask device uint32 [B][M'][ceil(M'/32)], out_vscores device float
 *  [B][M'] or NULL; M' = min(M, N).
 * A node that outscores its parent sets DART_DEVERR_SCORE_RISES in the
 * workspace's error word (as dart_tree_select does in its device_err).
 * Every other argument as for dart_tree_build_strided. */
int dart_tree_build_verify(const void* logits, int B, int d, int V, int64_t row_stride, int dtype,
                           float T, int k, int W, float lambda, float beta,
                           const dart_ngram_table_t* ngram_table, const int32_t* ctx_tokens,
                           int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                           uint32_t* out_mask, float* out_scores, int M, int32_t* out_vindex,
                           int32_t* out_vtokens, int32_t* out_vparents, int32_t* out_vpos,
                           uint32_t* out_vmask, float* out_vscores,
                           void* workspace, size_t workspace_bytes, void* stream);

/* dart_tree_build without a workspace argument, for callers that cannot
 * allocate device memory: an engine whose own pool allocator has reserved
 * the device's memory (a side cudaMalloc would fail or fragment it), a
 * plugin or language binding with no handle on the application's
 * allocator, or a latency-critical decode loop where cudaMalloc / cudaFree
 * would synchronise the device.  The pages have no counterpart; this is a
 * deployment variant of the same computation.
 * Arguments and outputs are those of dart_tree_build; the workspace is a
 * fixed 16 MiB buffer inside the library that every device loading the
 * library holds until the process exits.  Sizes whose
 * dart_tree_workspace_bytes(B, d, V, dtype, k) exceeds 16 MiB are rejected
 * with DART_ERR_WORKSPACE before anything is launched.  The call allocates
 * nothing and launches no clearing: no byte of the buffer has to start at
 * zero except its device error word, which is zero when the library loads
 * and is read (and cleared) with dart_noalloc_device_error.
 * The first call in each CUDA context (the current device's primary context,
 * bound if none is current) looks up the buffer's device address and caches
 * it under the context's unique id, so a context that cudaDeviceReset
 * replaced gets a fresh lookup; make that first call before any stream
 * capture.  All calls in a context share the one buffer, which keeps the last
 * call's contents: calls that overlap on the GPU (other streams, other host
 * threads) race and must be serialised by the caller. */
int dart_tree_build_noalloc(const void* logits, int B, int d, int V, int dtype,
                            float T, int k, int W, float lambda, float beta,
                            const dart_ngram_table_t* ngram_table, const int32_t* ctx_tokens,
                            int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                            uint32_t* out_mask, float* out_scores, void* stream);

/* The tree stage alone, from candidate lists a caller already has (for
 * example a drafter that emits its own top-k):
 *  cand_ids   device int32 [B][d][k], token ids in [0, 2^24-1), distinct
 *             within a row (any order; a row with a repeated id still
 *             gives a well-formed tree, its tie order unspecified)
 *  cand_logp  device double [B][d][k], the candidates' log-probabilities
 * Children are ranked by (sum of logp along the path) + lambda * (sum of g),
 * both sums in double, and that value is the reported score.  Other
 * arguments and outputs as in dart_tree_build; no workspace. */
int dart_tree_from_topk(const int32_t* cand_ids, const double* cand_logp,
                        int B, int d, int k, int W, float lambda, float beta,
                        const dart_ngram_table_t* ngram_table, const int32_t* ctx_tokens,
                        int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                        uint32_t* out_mask, float* out_scores, void* stream);

/* The tree stage with a caller-supplied continuity scorer in place of the
 * n-gram table (DARTree, Method / Tree Construction: the children of a depth
 * are scored by a head in one batch; an order-2 head, restricted to the
 * candidate sets, is a table of candidate-pair scores):
 *  pair_scores device float [B][d][k][k]: a child with list position c in
 *              row j adds pair_scores[b][j][c'][c] to its continuity sum,
 *              c' the list position of its parent's token in row j-1; for
 *              row 0 the parent is the root and c' = 0 (the rest of row 0's
 *              k x k block is not read).  Values finite.
 * Children are ranked by (path's log-probability sum) + lambda * (sum of its
 * pair scores), ties as in dart_tree_build.  Other arguments and outputs as
 * in dart_tree_from_topk (no table, no context, no beta). */
int dart_tree_from_topk_pairs(const int32_t* cand_ids, const double* cand_logp, const float* pair_scores,
                              int B, int d, int k, int W, float lambda,
                              int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                              uint32_t* out_mask, float* out_scores, void* stream);

/* The same tree stage on the candidate lists that dart_row_topk (or
 * dart_row_pass followed by dart_row_finish) left in `workspace` for rows =
 * B * d rows of [B][d][V] logits: call it with the same V, dtype, T and k, on
 * the same stream, after the caller has scored the pairs of those candidates
 * (their ids are dart_row_topk's out_ids).  The ranking key is that of
 * dart_tree_build with the pair scores as the continuity term, so the scores
 * are log-probabilities at temperature T plus lambda times the pair sum.  The
 * workspace is only read, apart from its device error word. */
int dart_tree_from_rows_pairs(int B, int d, int V, int dtype, float T, int k, int W, float lambda,
                              const float* pair_scores, int32_t* out_tokens, int32_t* out_parents,
                              int32_t* out_pos, uint32_t* out_mask, float* out_scores,
                              const void* workspace, size_t workspace_bytes, void* stream);

/* The row stage alone: for each of `rows` rows of logits[rows][V] (device,
 * 16-byte aligned): the k best ids (value descending, lower id first),
 * their log-probabilities log_softmax(z / T)[id] and the row's
 * log-sum-exp of z / T (T = 0: of z, as for dart_tree_build).  out_ids device int32 [rows][k], out_logp device
 * float [rows][k], out_lse device float [rows] (each may be NULL).
 * workspace as for dart_tree_build with B = rows, d = 1. */
int dart_row_topk(const void* logits, int rows, int V, int dtype, float T, int k,
                  int32_t* out_ids, float* out_logp, float* out_lse,
                  void* workspace, size_t workspace_bytes, void* stream);

/* dart_row_topk for rows row_stride >= V elements apart (see
 * dart_tree_build_strided; the padding is never read). */
int dart_row_topk_strided(const void* logits, int rows, int V, int64_t row_stride, int dtype, float T, int k,
                          int32_t* out_ids, float* out_logp, float* out_lse,
                          void* workspace, size_t workspace_bytes, void* stream);

/* The row stage in two launches, for callers that overlap other work with
 * the streaming pass or time it alone.  dart_row_pass reads the logits once
 * and leaves each row's per-piece maxima, sums, bounds and candidates in the
 * workspace; dart_row_finish merges them into the results dart_row_topk
 * writes (out_ids, out_logp, out_lse: as there, each may be NULL; the rows'
 * candidate ids, logits and log-sum-exp also stay in the workspace).
 * Arguments as for dart_row_topk_strided (dart_row_finish takes no logits);
 * pass the same sizes and workspace to both, in order on one stream.
 * dart_row_topk_strided is dart_row_pass followed by dart_row_finish. */
int dart_row_pass(const void* logits, int rows, int V, int64_t row_stride, int dtype, float T, int k,
                  void* workspace, size_t workspace_bytes, void* stream);
int dart_row_finish(int rows, int V, int64_t row_stride, int dtype, float T, int k, int32_t* out_ids,
                    float* out_logp, float* out_lse, void* workspace, size_t workspace_bytes, void* stream);

/* Ancestor-or-self masks from a parent array (DART, Figure 3 caption: the
 * tree-attention input).  parents device int32 [B][N], each entry -1 or a
 * smaller node index; out_mask device uint32 [B][N][ceil(N/32)].  An entry
 * that is not below its node stops that walk and sets DART_DEVERR_PARENT in
 * *device_err (device uint32, may be NULL). */
int dart_mask_pack(const int32_t* parents, int B, int N, uint32_t* out_mask,
                   uint32_t* device_err, void* stream);

/* Verification tree chosen best-first with a budget (DARTree, abstract and
 * Verification: the candidate tree is built first, then best-first pruning
 * alone picks the tree that is verified; PCTree, abstract: a fixed
 * verification budget goes to the most probable paths).  Per tree b, M' =
 * min(M, N) times, the node of largest score (lower index on equal scores)
 * among those whose parent is already taken (depth-1 nodes need none) is
 * taken.  When scores never rise from a parent to its children (true for
 * dart_tree_build's scores whenever lambda >= 0, beta <= 0 and the table's
 * values are <= 0) these are the M' best nodes by (score, lower index).
 *  tokens, parents, pos  device int32 [B][N] (parents[i] < i, -1 at depth 1),
 *                        and scores device float [B][N]: candidate trees as
 *                        written by dart_tree_build (N <= 1024)
 *  out_index             device int32 [B][M']: the taken nodes' indices,
 *                        increasing (parents before children)
 *  out_tokens, out_pos   device int32 [B][M']: their tokens and depths
 *  out_parents           device int32 [B][M']: position of the parent within
 *                        the chosen tree, -1 at depth 1
 *  out_mask              device uint32 [B][M'][ceil(M'/32)]: ancestor-or-self
 *                        rows of the chosen tree, LSB first
 *  out_scores            device float [B][M'] or NULL
 *  device_err            device uint32 or NULL: receives DART_DEVERR_PARENT
 *                        for a parent index not below its node and
 *                        DART_DEVERR_SCORE_RISES for a node scoring above its
 *                        parent (its kept children may then lack a parent:
 *                        out_parents -2)
 * Nothing is launched when B or M is 0.  Returns DART_OK or an error code. */
int dart_tree_select(const int32_t* tokens, const int32_t* parents, const int32_t* pos,
                     const float* scores, int B, int N, int M, int32_t* out_index,
                     int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                     uint32_t* out_mask, float* out_scores, uint32_t* device_err, void* stream);

/* Smallest power of two >= max(2 * M, 8) (load factor at most 1/2); 0 on
 * overflow. */
uint64_t dart_ngram_capacity_for(uint64_t M);

/* Build the slots of an n-gram table on the host.
 *  keys host int32 [M][n] (t_0 oldest ... t_{n-1} predicted), each in
 *  [0, 2^24-1); vals host float [M]; host_slots host, capacity * 16 bytes;
 *  capacity a power of two >= 8.
 * A repeated key keeps its first value; *out_distinct (may be NULL)
 * receives the number of distinct keys stored.  Keys whose two buckets are
 * full move earlier keys to their other bucket (cuckoo displacement, a fixed
 * deterministic order).  Returns DART_ERR_TABLE_FULL if more than
 * capacity / 2 distinct keys arrive, or if 500 displacements do not free a
 * slot (the slots are then unusable). */
int dart_ngram_table_pack_host(int n, const int32_t* keys, const float* vals, uint64_t M,
                               uint64_t capacity, void* host_slots, uint64_t* out_distinct);

/* Batch lookup in a device table: keys device int32 [Q][n]; vals device
 * float [Q] (0 when absent); found device int32 [Q] (1 / 0). */
int dart_ngram_lookup(const dart_ngram_table_t* table, const int32_t* keys, int64_t Q,
                      float* vals, int32_t* found, void* stream);

/* Waits for `stream`, then copies the workspace's device error word to
 * *out_flags (host).  The word collects the DART_DEVERR_* bits of every call
 * since the last nonzero read; a nonzero read clears it.  Returns DART_OK, or
 * DART_ERR_CUDA. */
int dart_device_error(const void* workspace, uint32_t* out_flags, void* stream);

/* dart_device_error for dart_tree_build_noalloc's internal buffer in the
 * current context: waits for `stream`, copies the buffer's error word to
 * *out_flags (host) and clears it when nonzero.  The word collects the bits
 * of every dart_tree_build_noalloc call in this context since the last
 * nonzero read.  Returns DART_OK, DART_ERR_INVALID_ARG (out_flags NULL) or
 * DART_ERR_CUDA.  The pages have no counterpart. */
int dart_noalloc_device_error(uint32_t* out_flags, void* stream);

/* Sets the number of SM clock cycles any one wait of the row pass (a bulk
 * copy landing, a slot freeing, a barrier of the CTA) may take before the pass
 * gives up: the CTA then ends every other wait, lets its copies in flight
 * land, sets DART_DEVERR_WAIT_TIMEOUT and returns, and its outputs are
 * invalid.  cycles <= 0 restores the default (4e9, about two seconds).  For
 * tests of the timeout path; applies to later calls from every host thread. */
void dart_set_wait_limit(int64_t cycles);

/* Throughput probe of the exponential unit: blocks x threads threads (threads
 * a multiple of 32, at most 1024) each run 8 independent chains of `iters`
 * steps x <- 2^x - 1.5 (one ex2.approx and one add per step) and write one
 * float to out (device, blocks * threads floats).  Time it on `stream` to get
 * exponentials per second = blocks * threads * iters * 8 / time.  Returns
 * DART_OK or an error code. */
int dart_probe_ex2(int blocks, int threads, int iters, float* out, void* stream);

/* Streaming-read probe: reads `bytes` (rounded down to a multiple of 16) of
 * device memory at `src` (16-byte aligned) once, split into equal contiguous
 * spans, one per warp, over `ctas` CTAs of `warps_per_cta` warps, and writes
 * one float per lane to out (device, ctas * warps_per_cta * 32 floats) so
 * that nothing is optimised away.  mode bit 0: 0 = 16-byte loads straight
 * into registers (eight per lane in flight; warps_per_cta <= 16), 1 = each
 * warp's own ring of `stages` (2..16) 4 KiB shared-memory stages filled by
 * bulk copies (warps_per_cta * stages * 4 KiB must fit in shared memory).
 * mode bit 1: reduce the data as bf16 logits (running maximum, one
 * exponential per element) instead of xor-folding it. mode bit 2 (bulk ring
 * only): the warps of a CTA share one contiguous span of warps_per_cta
 * spans, warp w reading its 4 KiB steps w, w + warps_per_cta, ...  A bulk wait that runs
 * out (about two seconds) sets bit 0 of *device_err (device uint32).  Time it
 * on `stream` to get the bandwidth a row pass of that shape can reach.
 * Returns DART_OK or an error code. */
int dart_probe_stream(const void* src, uint64_t bytes, int mode, int ctas, int warps_per_cta,
                      int stages, float* out, uint32_t* device_err, void* stream);

/* Static text for a status code. */
const char* dart_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* DARTTREE_H */
