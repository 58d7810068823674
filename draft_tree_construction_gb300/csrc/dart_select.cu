// dart_select.cu -- K4: the verification tree, chosen best-first with a budget
// from candidate trees.
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
// index), and that set holds the parent of each of its nodes.  So one CTA per
// tree gives each of its N <= 1024 nodes a thread, which counts the nodes
// whose 64-bit key (ordered score, then inverted index) beats its own (a
// broadcast read of shared memory per node: no sorting network, no barrier
// inside the count); a node is kept when fewer than M beat it.  The kept
// nodes are renumbered in node order and their ancestor masks rebuilt.  A
// node that outscores its parent sets DART_DEVERR_SCORE_RISES: the M best
// need not be the best-first choice then.
#include "dart_common.cuh"

namespace dart {
namespace {

// Larger key: larger score, then lower node index.
__device__ __forceinline__ uint64_t sel_key(float s, int i) {
  return (uint64_t(ord_f32(s)) << 32) | uint64_t(0xFFFFFFFFu - uint32_t(i));
}

// One CTA per tree, blockDim = N rounded up to a multiple of 32 (<= 1024).
__global__ void __launch_bounds__(kMaxN)
select_kernel(const int32_t* __restrict__ tokens, const int32_t* __restrict__ parents,
              const int32_t* __restrict__ pos, const float* __restrict__ scores, int N, int Mp,
              int32_t* __restrict__ out_index, int32_t* __restrict__ out_tokens,
              int32_t* __restrict__ out_parents, int32_t* __restrict__ out_pos,
              uint32_t* __restrict__ out_mask, float* __restrict__ out_scores, uint32_t* err) {
  __shared__ uint64_t skey[kMaxN];
  __shared__ int32_t spar[kMaxN];
  __shared__ float sscore[kMaxN];
  __shared__ int32_t snew[kMaxN];     // a kept node's new index, else -1
  __shared__ int32_t npar[kMaxN];     // the renumbered parent of new index m
  __shared__ uint32_t chunk[kMaxN / 32];
  const int b = blockIdx.x;
  const int i = threadIdx.x;          // this thread's node
  const int lane = i & 31;
  const int c = i >> 5;
  const size_t tb = (size_t)b * N;

  // every global read of the node up front: one memory round trip
  const float si = i < N ? scores[tb + i] : 0.f;
  const int32_t ti = i < N ? tokens[tb + i] : 0;
  const int32_t di = i < N ? pos[tb + i] : 0;
  const uint64_t ki = i < N ? sel_key(si, i) : 0ull;
  if (i < N) {
    skey[i] = ki;
    spar[i] = parents[tb + i];
    sscore[i] = si;
  }
  __syncthreads();
  bool keep = false;
  if (i < N) {
    // parents point backwards; scores never rise along a path
    const int p = spar[i];
    if (p >= i || p < -1) set_dev_error(err, DART_DEVERR_PARENT);
    else if (p >= 0 && si > sscore[p]) set_dev_error(err, DART_DEVERR_SCORE_RISES);
    // stop once Mp keys beat this one: the node is out (with a small budget
    // most nodes leave early; the best ones, shallow and at low indices, sit
    // together in the first warps)
    int beat = 0;
    for (int j0 = 0; j0 < N && beat < Mp; j0 += 8) {
#pragma unroll
      for (int j = j0; j < j0 + 8; ++j) beat += (j < N && skey[j] > ki) ? 1 : 0;
    }
    keep = beat < Mp;
  }
  // new indices in node order: ballot counts per 32 nodes, then a prefix
  const uint32_t bal = __ballot_sync(0xFFFFFFFFu, keep);
  if (lane == 0) chunk[c] = uint32_t(__popc(bal));
  __syncthreads();
  const int nchunks = (N + 31) / 32;
  if (c == 0) {
    const uint32_t v = lane < nchunks ? chunk[lane] : 0u;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane < nchunks) chunk[lane] = incl - v;
  }
  __syncthreads();
  const int m = keep ? int(chunk[c] + uint32_t(__popc(bal & ((1u << lane) - 1u)))) : -1;
  if (i < N) snew[i] = m;
  __syncthreads();
  // gather the kept nodes; renumber their parents
  const size_t ob = (size_t)b * Mp;
  if (m >= 0) {
    const int p = spar[i];
    int q = -1;
    if (p >= 0 && p < i) {
      q = snew[p];
      if (q < 0) {
        set_dev_error(err, DART_DEVERR_SCORE_RISES);   // a kept node without its parent
        q = -2;
      }
    }
    npar[m] = q;
    out_index[ob + m] = i;
    out_tokens[ob + m] = ti;
    out_pos[ob + m] = di;
    out_parents[ob + m] = q;
    if (out_scores) out_scores[ob + m] = si;
  }
  __syncthreads();
  // ancestor-or-self masks of the kept tree
  const int MWp = (Mp + 31) / 32;
  for (int idx = i; idx < Mp * MWp; idx += blockDim.x) {
    const int x = idx / MWp;
    const int w = idx - x * MWp;
    uint32_t val = 0;
    int a = x;
    for (int steps = 0; a >= 0 && steps <= Mp; ++steps) {
      if ((a >> 5) == w) val |= 1u << (a & 31);
      const int q = npar[a];
      if (q >= a) break;
      a = q;
    }
    out_mask[(ob + x) * MWp + w] = val;
  }
}

}  // namespace
}  // namespace dart

extern "C" int dart_tree_select(const int32_t* tokens, const int32_t* parents, const int32_t* pos,
                                const float* scores, int B, int N, int M, int32_t* out_index,
                                int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                                uint32_t* out_mask, float* out_scores, uint32_t* device_err, void* stream) {
  using namespace dart;
  if (B < 0 || N < 1 || N > kMaxN || M < 0) return DART_ERR_INVALID_ARG;
  const int Mp = M < N ? M : N;
  if (B == 0 || Mp == 0) return DART_OK;
  if (!tokens || !parents || !pos || !scores || !out_index || !out_tokens || !out_parents || !out_pos ||
      !out_mask)
    return DART_ERR_INVALID_ARG;
  const int threads = (N + 31) / 32 * 32;
  select_kernel<<<B, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      tokens, parents, pos, scores, N, Mp, out_index, out_tokens, out_parents, out_pos, out_mask,
      out_scores, device_err);
  return cudaGetLastError() == cudaSuccess ? DART_OK : DART_ERR_CUDA;
}
