// dart_probe.cu -- throughput probes: the exponential unit and the streaming
// read ceiling.
//
// The row pass evaluates one base-2 exponential per logit (ex2.approx, the
// special-function unit's exp2); ex2_probe_kernel measures how many of them
// the GPU sustains, so that the exponential is checked, not assumed, as a
// bound of the row pass.  Each thread runs eight independent chains
// x <- 2^x - 1.5 (one exponential and one add per step), enough chains per SM
// to keep the unit busy; the sums are written out so that nothing is
// optimised away.
//
// stream_probe_kernel reads a buffer once, the way a row pass can read its
// logits, and measures what bandwidth that access pattern reaches with and
// without the per-element work of a log-sum-exp (a running maximum and one
// exponential per bf16 element).  Each warp reads one contiguous span, either
// with 16-byte loads straight into registers (eight per lane in flight while
// the previous eight are reduced) or through its own ring of 4 KiB
// shared-memory stages filled by bulk copies (cp.async.bulk) that the warp
// itself issues.  The results are the ceilings a row pass of either kind can
// reach on this GPU.  The bulk ring can also interleave its warps: the CTA
// reads one contiguous span, warp w taking its 4 KiB steps w, w + warps,
// w + 2 warps, ... (fewer, longer sequential streams for the memory system).
#include "dart_common.cuh"

#include <cfloat>

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

constexpr int kProbeVec = 8;                       // 16-byte vectors per lane and step
constexpr int kProbeStage = kProbeVec * 32 * 16;   // 4 KiB: one step of a warp
constexpr long long kProbeWaitLimit = 4000000000LL;

struct StreamProbe {
  const uint4* src;
  unsigned long long nvec;   // 16-byte vectors in the buffer
  unsigned long long span;   // vectors per warp (a multiple of 256)
  int stages;                // bulk ring: stages per warp
  int interleave;            // bulk ring: the CTA's warps share one span, step by step
  float* out;                // one value per warp
  uint32_t* err;             // a bulk wait ran out (bit 0)
};

__device__ __forceinline__ uint4 ldg_stream(const uint4* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ uint32_t bf_max2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Per-lane state of the reduction: running max m, fl(m c), sum of 2^(z c - mc)
// (MATH), or an xor of every word (no MATH).
struct ProbeAcc {
  float m, mc, s;
  uint32_t x;
};

template <bool MATH>
__device__ __forceinline__ void probe_reduce(ProbeAcc& a, const uint4 (&r)[kProbeVec], int valid) {
  if (!MATH) {
#pragma unroll
    for (int u = 0; u < kProbeVec; ++u)
      if (u < valid) a.x ^= r[u].x ^ r[u].y ^ r[u].z ^ r[u].w;
    return;
  }
  constexpr float c = 1.4426950408889634f;
  uint32_t pm = 0xFF80FF80u;
#pragma unroll
  for (int u = 0; u < kProbeVec; ++u)
    if (u < valid) pm = bf_max2(pm, bf_max2(bf_max2(r[u].x, r[u].y), bf_max2(r[u].z, r[u].w)));
  const float vm = fmaxf(__uint_as_float(pm << 16), __uint_as_float(pm & 0xFFFF0000u));
  if (vm > a.m) {
    const float mcn = fmaxf(vm * c, -FLT_MAX);
    a.s *= ex2_approx(a.mc - mcn);
    a.m = vm;
    a.mc = mcn;
  }
  const float2 nmc2 = make_float2(-a.mc, -a.mc);
  const float2 c2 = make_float2(c, c);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int u = 0; u < kProbeVec; ++u) {
    if (u >= valid) continue;
    const uint32_t w[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 z = make_float2(__uint_as_float(w[p] << 16), __uint_as_float(w[p] & 0xFFFF0000u));
      const float2 t = __ffma2_rn(z, c2, nmc2);
      acc = __fadd2_rn(acc, make_float2(ex2_approx(t.x), ex2_approx(t.y)));
    }
  }
  a.s += acc.x + acc.y;
}

template <bool MATH>
__device__ __forceinline__ float probe_result(const ProbeAcc& a) {
  return MATH ? a.s + a.m : __uint_as_float(a.x & 0x3FFFFFFFu);
}

// Direct loads: eight 16-byte loads per lane in flight while the previous
// eight are reduced.
template <bool MATH>
__global__ void __launch_bounds__(512) stream_probe_direct(const StreamProbe P) {
  const int lane = threadIdx.x & 31;
  const unsigned long long gw = (unsigned long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const unsigned long long v0 = gw * P.span;
  const unsigned long long v1 = min(P.nvec, v0 + P.span);
  const uint64_t pol = policy_evict_first();
  ProbeAcc a{-FLT_MAX, -FLT_MAX, 0.f, 0u};
  uint4 cur[kProbeVec], nxt[kProbeVec];
  auto load = [&](uint4 (&r)[kProbeVec], unsigned long long base) {
#pragma unroll
    for (int u = 0; u < kProbeVec; ++u) {
      const unsigned long long v = base + (unsigned long long)(u * 32 + lane);
      r[u] = v < v1 ? ldg_stream(P.src + v, pol) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    }
  };
  if (v0 < v1) {
    load(cur, v0);
    for (unsigned long long base = v0; base < v1; base += 256) {
      if (base + 256 < v1) load(nxt, base + 256);
      probe_reduce<MATH>(a, cur, kProbeVec);
#pragma unroll
      for (int u = 0; u < kProbeVec; ++u) cur[u] = nxt[u];
    }
  }
  P.out[gw * 32 + lane] = probe_result<MATH>(a);
}

// Per-warp bulk ring: lane 0 keeps `stages` 4 KiB copies of the warp's span
// in flight; the warp reduces each stage from shared memory and refills it.
template <bool MATH>
__global__ void __launch_bounds__(1024) stream_probe_bulk(const StreamProbe P) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int lane = threadIdx.x & 31;
  const int wl = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  const unsigned long long gw = (unsigned long long)blockIdx.x * nw + wl;
  // contiguous: the warp's span [v0, v1), step st at v0 + 256 st; interleaved:
  // the CTA's span [c0, c1), step st of the warp at c0 + 256 (st nw + wl)
  const unsigned long long c0 = (unsigned long long)blockIdx.x * nw * P.span;
  const unsigned long long c1 = min(P.nvec, c0 + nw * P.span);
  const unsigned long long v0 = P.interleave ? c0 + 256ull * wl : gw * P.span;
  const unsigned long long v1 = P.interleave ? c1 : min(P.nvec, v0 + P.span);
  const unsigned long long vstep = P.interleave ? 256ull * nw : 256ull;
  uint8_t* ring = smem_raw + (size_t)wl * P.stages * kProbeStage;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + (size_t)nw * P.stages * kProbeStage) + (size_t)wl * P.stages;
  const uint64_t pol = policy_evict_first();
  if (lane == 0) {
    for (int s = 0; s < P.stages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const unsigned long long nstep = v0 < v1 ? (v1 - v0 + vstep - 1) / vstep : 0;
  auto issue = [&](unsigned long long step) {
    const unsigned long long v = v0 + step * vstep;
    const uint32_t bytes = uint32_t(min(256ull, v1 - v) * 16ull);
    const int s = int(step % (unsigned long long)P.stages);
    mbar_expect_tx(&bars[s], bytes);
    bulk_g2s(ring + (size_t)s * kProbeStage, P.src + v, bytes, &bars[s], pol);
  };
  if (lane == 0)
    for (unsigned long long st = 0; st < nstep && st < (unsigned long long)P.stages; ++st) issue(st);
  ProbeAcc a{-FLT_MAX, -FLT_MAX, 0.f, 0u};
  bool ok = true;
  for (unsigned long long st = 0; st < nstep; ++st) {
    const int s = int(st % (unsigned long long)P.stages);
    const uint32_t parity = uint32_t(st / (unsigned long long)P.stages) & 1u;
    // a wait that runs out still lets the copy land (the drain below waits
    // again), so the warp never leaves with a copy writing its ring
    const bool got = mbar_wait_bounded(&bars[s], parity, ok ? kProbeWaitLimit : 0);
    if (!got) {
      ok = false;
      if (lane == 0) atomicOr(P.err, 1u);
      break;
    }
    const unsigned long long v = v0 + st * vstep;
    const int valid_vecs = int(min(256ull, v1 - v));
    const uint4* src = reinterpret_cast<const uint4*>(ring + (size_t)s * kProbeStage);
    uint4 r[kProbeVec];
    int valid = 0;
#pragma unroll
    for (int u = 0; u < kProbeVec; ++u) {
      const bool in = u * 32 + lane < valid_vecs;
      r[u] = in ? src[u * 32 + lane] : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
      valid += in ? 1 : 0;
    }
    probe_reduce<MATH>(a, r, kProbeVec);
    __syncwarp();
    if (lane == 0 && st + P.stages < nstep) issue(st + P.stages);
  }
  if (!ok && lane == 0) {
    // drain: every issued copy lands before the warp leaves
    for (int s = 0; s < P.stages; ++s) (void)mbar_wait_bounded(&bars[s], 0u, kProbeWaitLimit);
  }
  __syncwarp();
  P.out[gw * 32 + lane] = probe_result<MATH>(a);
}

}  // namespace
}  // namespace dart

extern "C" int dart_probe_ex2(int blocks, int threads, int iters, float* out, void* stream) {
  if (blocks < 1 || threads < 32 || threads > 1024 || threads % 32 != 0 || iters < 1 || !out)
    return DART_ERR_INVALID_ARG;
  dart::ex2_probe_kernel<<<blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(iters, 0.25f, out);
  return cudaGetLastError() == cudaSuccess ? DART_OK : DART_ERR_CUDA;
}

extern "C" int dart_probe_stream(const void* src, uint64_t bytes, int mode, int ctas, int warps_per_cta,
                                 int stages, float* out, uint32_t* device_err, void* stream) {
  using namespace dart;
  if (!src || (reinterpret_cast<uintptr_t>(src) & 15u) || !out || !device_err || ctas < 1 || warps_per_cta < 1 ||
      warps_per_cta > 32 || mode < 0 || mode > 7 || (!(mode & 1) && warps_per_cta > 16) ||
      ((mode & 4) && !(mode & 1)))
    return DART_ERR_INVALID_ARG;
  const bool bulk = (mode & 1) != 0, math = (mode & 2) != 0;
  if (bulk && (stages < 2 || stages > 16)) return DART_ERR_INVALID_ARG;
  const size_t smem = bulk ? size_t(warps_per_cta) * stages * (kProbeStage + 8) : 0;
  if (smem > 232448) return DART_ERR_INVALID_ARG;
  StreamProbe P;
  P.src = static_cast<const uint4*>(src);
  P.nvec = bytes / 16;
  const unsigned long long warps = (unsigned long long)ctas * warps_per_cta;
  P.span = ((P.nvec + warps - 1) / warps + 255) / 256 * 256;
  P.stages = stages;
  P.interleave = (mode & 4) ? 1 : 0;
  P.out = out;
  P.err = device_err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int threads = warps_per_cta * 32;
  cudaError_t e = cudaSuccess;
  auto go = [&](auto kernel) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e == cudaSuccess) kernel<<<ctas, threads, smem, s>>>(P);
  };
  if (bulk) {
    if (math) go(stream_probe_bulk<true>);
    else go(stream_probe_bulk<false>);
  } else {
    if (math) go(stream_probe_direct<true>);
    else go(stream_probe_direct<false>);
  }
  if (e != cudaSuccess) return DART_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? DART_OK : DART_ERR_CUDA;
}
