// dart_probe.cu -- throughput probe of the exponential unit.
//
// The row pass evaluates one base-2 exponential per logit (ex2.approx, the
// special-function unit's exp2); this kernel measures how many of them the GPU
// sustains, so that the exponential is checked, not assumed, as a bound of the
// row pass.  Each thread runs eight independent chains x <- 2^x - 1.5 (one
// exponential and one add per step), enough chains per SM to keep the unit
// busy; the sums are written out so that nothing is optimised away.
#include "dart_common.cuh"

namespace dart {
namespace {

__global__ void ex2_probe_kernel(int iters, float seed, float* __restrict__ out) {
  float a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = seed + 1e-6f * float(threadIdx.x) + 0.1f * float(i);
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = ex2_approx(a[i]) - 1.5f;
  }
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s += a[i];
  out[(size_t)blockIdx.x * blockDim.x + threadIdx.x] = s;
}

}  // namespace
}  // namespace dart

extern "C" int dart_probe_ex2(int blocks, int threads, int iters, float* out, void* stream) {
  if (blocks < 1 || threads < 32 || threads > 1024 || threads % 32 != 0 || iters < 1 || !out)
    return DART_ERR_INVALID_ARG;
  dart::ex2_probe_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(iters, 0.25f, out);
  return cudaGetLastError() == cudaSuccess ? DART_OK : DART_ERR_CUDA;
}
