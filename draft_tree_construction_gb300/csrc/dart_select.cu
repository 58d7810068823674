// dart_select.cu -- K4: the verification tree, chosen best-first with a budget
// from candidate trees (DARTree, abstract and Verification; PCTree,
// abstract).  The selection itself is in dart_select.cuh, shared with the
// tree kernel, which can emit the verification tree of the tree it has just
// built; this kernel serves candidate trees that are already in memory.
#include "dart_common.cuh"

namespace dart {
namespace {

#include "dart_select.cuh"

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
  const size_t tb = (size_t)b * N;
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    sscore[i] = scores[tb + i];
    spar[i] = parents[tb + i];
  }
  __syncthreads();
  const SelectShared S{sscore, spar, skey, snew, npar, chunk};
  const size_t ob = (size_t)b * Mp;
  const int MWp = (Mp + 31) / 32;
  select_best_first(N, Mp, S, tokens + tb, pos + tb, out_index + ob, out_tokens + ob, out_parents + ob,
                    out_pos + ob, out_mask + ob * MWp, out_scores ? out_scores + ob : nullptr, err);
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
