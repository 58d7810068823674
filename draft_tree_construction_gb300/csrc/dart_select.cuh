// dart_select.cuh -- the best-first verification tree of one candidate tree,
// chosen by one CTA (included inside namespace dart by dart_select.cu, for the
// standalone kernel, and by dart_tree.cu, whose tree kernel can emit it right
// after building the tree).
//
// DARTree, abstract and Verification: the fixed-width candidate tree is built
// first, and only then does best-first pruning pick the tree that the target
// model verifies; PCTree, abstract: a fixed verification budget goes to the
// most probable paths.  Best-first with budget M takes, M times, the best
// node (largest path score, lower node index on equal scores) among those
// whose parent is already taken.  A node's score is its parent's plus a
// log-probability plus lambda times an n-gram log-probability (or beta), so
// with lambda >= 0 and beta <= 0 scores never rise from a parent to its
// children; then the nodes taken are exactly the M best by (score, lower
// index), and that set holds the parent of each of its nodes.  So each node
// counts the nodes whose 64-bit key (ordered score, then inverted index)
// beats its own (a broadcast read of shared memory per node, no sorting
// network) and is kept when fewer than M beat it.  The kept nodes are
// renumbered in node order and their ancestor masks rebuilt.  A node that
// outscores its parent sets DART_DEVERR_SCORE_RISES: the M best need not be
// the best-first choice then.

// Larger key: larger score, then lower node index.
__device__ __forceinline__ uint64_t sel_key(float s, int i) {
  return (uint64_t(ord_f32(s)) << 32) | uint64_t(0xFFFFFFFFu - uint32_t(i));
}

// Shared-memory arrays of the selection: scores and parents of the N nodes
// (filled by the caller), the nodes' keys and new indices, the renumbered
// parents of the Mp kept nodes, and one count per 32 nodes.
struct SelectShared {
  const float* score;
  const int32_t* parent;
  uint64_t* key;
  int32_t* fresh;
  int32_t* npar;
  uint32_t* chunk;
};
__host__ __device__ inline size_t select_shared_bytes(int N) {
  return size_t(N) * (4 + 4 + 8 + 4 + 4) + 4 * (size_t(kMaxN) / 32) + 64;
}

// The verification tree of one candidate tree of N <= kMaxN nodes, budget
// Mp = min(M, N) >= 1.  tokens / pos: the tree's nodes (global memory);
// out_*: the tree's rows of the outputs (Mp entries, masks Mp x ceil(Mp/32)).
// Every thread of the CTA takes part; the caller has filled S.score and
// S.parent and passed a barrier.
static __device__ void select_best_first(int N, int Mp, const SelectShared& S, const int32_t* tokens,
                                         const int32_t* pos, int32_t* out_index, int32_t* out_tokens,
                                         int32_t* out_parents, int32_t* out_pos, uint32_t* out_mask,
                                         float* out_scores, uint32_t* err) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nwarps = nthreads >> 5;
  for (int i = tid; i < N; i += nthreads) {
    const float si = S.score[i];
    S.key[i] = sel_key(si, i);
    // parents point backwards; scores never rise along a path
    const int p = S.parent[i];
    if (p >= i || p < -1) set_dev_error(err, DART_DEVERR_PARENT);
    else if (p >= 0 && si > S.score[p]) set_dev_error(err, DART_DEVERR_SCORE_RISES);
  }
  __syncthreads();
  // kept: fewer than Mp keys beat the node's (counting stops at Mp; with a
  // small budget most nodes leave early)
  for (int i = tid; i < N; i += nthreads) {
    const uint64_t ki = S.key[i];
    int beat = 0;
    for (int j0 = 0; j0 < N && beat < Mp; j0 += 8) {
#pragma unroll
      for (int j = j0; j < j0 + 8; ++j) beat += (j < N && S.key[j] > ki) ? 1 : 0;
    }
    S.fresh[i] = beat < Mp ? 1 : 0;
  }
  __syncthreads();
  // new indices in node order: a count per 32 nodes, then one prefix
  const int nchunks = (N + 31) / 32;
  for (int c = warp; c < nchunks; c += nwarps) {
    const int i = c * 32 + lane;
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, i < N && S.fresh[i] != 0);
    if (lane == 0) S.chunk[c] = uint32_t(__popc(bal));
  }
  __syncthreads();
  if (warp == 0) {
    const uint32_t v = lane < nchunks ? S.chunk[lane] : 0u;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane < nchunks) S.chunk[lane] = incl - v;
  }
  __syncthreads();
  for (int c = warp; c < nchunks; c += nwarps) {
    const int i = c * 32 + lane;
    const bool keep = i < N && S.fresh[i] != 0;
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, keep);
    __syncwarp();
    if (i < N) S.fresh[i] = keep ? int(S.chunk[c] + uint32_t(__popc(bal & ((1u << lane) - 1u)))) : -1;
  }
  __syncthreads();
  // gather the kept nodes; renumber their parents
  for (int i = tid; i < N; i += nthreads) {
    const int m = S.fresh[i];
    if (m < 0) continue;
    const int p = S.parent[i];
    int q = -1;
    if (p >= 0 && p < i) {
      q = S.fresh[p];
      if (q < 0) {
        set_dev_error(err, DART_DEVERR_SCORE_RISES);   // a kept node without its parent
        q = -2;
      }
    }
    S.npar[m] = q;
    out_index[m] = i;
    out_tokens[m] = tokens[i];
    out_pos[m] = pos[i];
    out_parents[m] = q;
    if (out_scores) out_scores[m] = S.score[i];
  }
  __syncthreads();
  // ancestor-or-self masks of the kept tree
  const int MWp = (Mp + 31) / 32;
  for (int idx = tid; idx < Mp * MWp; idx += nthreads) {
    const int x = idx / MWp;
    const int w = idx - x * MWp;
    uint32_t val = 0;
    int a = x;
    for (int steps = 0; a >= 0 && steps <= Mp; ++steps) {
      if ((a >> 5) == w) val |= 1u << (a & 31);
      const int q = S.npar[a];
      if (q >= a) break;
      a = q;
    }
    out_mask[size_t(x) * MWp + w] = val;
  }
}
