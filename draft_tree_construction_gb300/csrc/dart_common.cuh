// dart_common.cuh -- shared pieces of the CUDA path (sm_103a).
//
// Ordered keys, the n-gram key packing and hash, PTX wrappers for mbarrier /
// bulk copies / ex2, warp bitonic networks, and the workspace layout that the
// host code and the kernels agree on.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "darttree.h"

namespace dart {

constexpr int kMaxK = 32;          // candidates per position
constexpr int kMaxW = 64;          // frontier width
constexpr int kMaxD = 32;          // depths
constexpr int kMaxN = 1024;        // nodes per tree
constexpr int kMaxMW = kMaxN / 32; // mask words per row
constexpr int kMaxV = (1 << 24) - 1;
constexpr long long kMaxRowStride = 1ll << 30;   // elements from one row's start to the next

// ------------------------------------------------------------ ordered keys
// A float maps to a uint32 whose unsigned order is the float order; -0.0 is
// first turned into +0.0 so that equal values give equal keys.
__host__ __device__ __forceinline__ uint32_t ord_f32(float z) {
  uint32_t u;
#ifdef __CUDA_ARCH__
  u = __float_as_uint(z);
#else
  memcpy(&u, &z, 4);
#endif
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__host__ __device__ __forceinline__ float unord_f32(uint32_t o) {
  uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
#ifdef __CUDA_ARCH__
  return __uint_as_float(u);
#else
  float f;
  memcpy(&f, &u, 4);
  return f;
#endif
}
// Candidate key of a row element: larger key = larger logit, then lower id.
// Key 0 never occurs for a real element (it would be a negative NaN).
__device__ __forceinline__ uint64_t elem_key(float z, uint32_t id) {
  return (uint64_t(ord_f32(z)) << 32) | uint64_t(~id);
}
__device__ __forceinline__ float key_value(uint64_t key) { return unord_f32(uint32_t(key >> 32)); }
__device__ __forceinline__ uint32_t key_id(uint64_t key) { return ~uint32_t(key); }

__device__ __forceinline__ uint64_t ord_f64(double s) {
  uint64_t u = uint64_t(__double_as_longlong(s));
  if (u == 0x8000000000000000ull) u = 0ull;
  return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}
__device__ __forceinline__ double unord_f64(uint64_t o) {
  uint64_t u = (o & 0x8000000000000000ull) ? (o & 0x7FFFFFFFFFFFFFFFull) : ~o;
  return __longlong_as_double((long long)u);
}

// --------------------------------------------------------- n-gram hashing
constexpr uint32_t kEmpty = 0xFFFFFFFFu;

struct Key96 { uint32_t w0, w1, w2; };

// tokens t[0..n) as 24-bit fields, t[0] in the lowest bits
__host__ __device__ __forceinline__ Key96 pack_ngram(const int32_t* t, int n) {
  uint64_t f[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = i < n ? (uint64_t(uint32_t(t[i])) & 0xFFFFFFull) : 0ull;
  uint64_t lo = f[0] | (f[1] << 24) | (f[2] << 48);
  uint32_t hi = uint32_t(f[2] >> 16) | uint32_t(f[3] << 8);
  return Key96{uint32_t(lo), uint32_t(lo >> 32), hi};
}

// splitmix64 output function (Steele, Lea & Flood, "Fast splittable
// pseudorandom number generators", OOPSLA 2014) applied to the folded key.
__host__ __device__ __forceinline__ uint64_t hash_key(Key96 k) {
  uint64_t x = uint64_t(k.w0) | (uint64_t(k.w1) << 32);
  x ^= uint64_t(k.w2) * 0x9E3779B97F4A7C15ull;
  x ^= x >> 30;
  x *= 0xBF58476D1CE4E5B9ull;
  x ^= x >> 27;
  x *= 0x94D049BB133111EBull;
  x ^= x >> 31;
  return x;
}

// The two buckets (kBucketSlots slots, 32 bytes each) a key may live in;
// nb = capacity / kBucketSlots >= 2.
constexpr int kBucketSlots = 2;
struct Buckets { uint64_t b1, b2; };
__host__ __device__ __forceinline__ Buckets key_buckets(Key96 k, uint64_t nb) {
  const uint64_t h = hash_key(k);
  Buckets b;
  b.b1 = h & (nb - 1);
  b.b2 = (h >> 32) & (nb - 1);
  if (b.b2 == b.b1) b.b2 = b.b1 ^ 1ull;
  return b;
}
constexpr uint64_t kMinTableSlots = 8;

// ------------------------------------------------------- workspace layout
// [ctrl 256 B]                    <- ctrl word 0 holds error bits until read,
//                                    words 2..3 the rows of the last call
// [row_off R x f64][row_ids R*k x i32][row_base R*k x f64][piece slots]
// row_off = the row's log-sum-exp of z / T; row_base = the candidates' logits.
// A piece slot holds one warp's share of a row: {f32 max; u32 count; f32 sum
// of 2^((z - max) c); pad; u32 bound (an ordered float: a lower bound of the
// row's k-th value); pad}, then cp candidate vectors of 16 bytes, then cp tags
// ((element mask << 24) | row index of the vector's first element).
//
// The row pass cuts the logits into one contiguous span per warp of a fixed
// nominal grid (152 SMs x 12 warps), so that the layout depends on the sizes
// alone, never on the device.
constexpr int kCtrlBytes = 256;
constexpr size_t kMinSpanBytes = 8192;      // smallest contiguous span of logits per warp of the row pass
constexpr unsigned long long kRowPassWarps = 152ull * 12ull;
constexpr int kSlotHeader = 32;

// Bytes per warp of the row pass for a stream of `total` bytes.
__host__ __device__ inline unsigned long long row_pass_span(unsigned long long total) {
  unsigned long long span = (total + kRowPassWarps - 1) / kRowPassWarps;
  span = (span + 15) & ~15ull;
  return span < kMinSpanBytes ? kMinSpanBytes : span;
}
// Candidate vectors a piece keeps (about 2.5 times what a piece of the
// streamed workloads typically needs; more are compacted to the k best).
__host__ __device__ inline int slot_capacity(int k) {
  const int c = 8 + 12 * k;
  return c < 200 ? c : 200;
}

struct WsLayout {
  size_t ctrl;               // control block: word 0 holds the device error bits
  size_t row_off, row_ids, row_base, slots, total;
  unsigned long long wspan;  // bytes per warp when rows are V apart (the smallest span)
  int pmax;                  // piece slots per row
  int cp;                    // candidate vectors per slot
  size_t slot_bytes;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool ws_layout(long long R, int V, int es, int k, WsLayout* L) {
  if (R < 0 || V < 1 || es < 1 || k < 1 || k > kMaxK) return false;
  const size_t row_bytes = size_t(V) * size_t(es);
  // every warp whose span meets the row owns one slot of it; spans are
  // smallest (so pieces most numerous) when rows are packed V apart
  L->wspan = row_pass_span((unsigned long long)R * row_bytes);
  L->pmax = int((row_bytes + L->wspan - 1) / L->wspan) + 1;
  L->cp = slot_capacity(k);
  L->slot_bytes = align_up(kSlotHeader + 20 * size_t(L->cp), 16);
  size_t o = 0;
  L->ctrl = o;      o += kCtrlBytes;
  L->row_off = o;   o = align_up(o + 8 * size_t(R), 256);
  L->row_ids = o;   o = align_up(o + 4 * size_t(R) * k, 256);
  L->row_base = o;  o = align_up(o + 8 * size_t(R) * k, 256);
  L->slots = o;     o = align_up(o + size_t(R) * L->pmax * L->slot_bytes, 256);
  L->total = o;
  return true;
}

// --------------------------------------------------------------- PTX glue
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Like mbar_try_wait, but the thread may sleep up to `hint_ns` nanoseconds
// waiting for the phase before the probe fails.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns) : "memory");
  return ok != 0;
}
// Non-blocking probe of a phase (try_wait may suspend the thread for a while).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait: gives up after `limit` clock cycles and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// One bulk copy global -> shared (both 16-byte aligned, size a multiple of 16),
// completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol) : "memory");
}

// 32 bytes (32-byte aligned) in one load: two 16-byte vectors.
__device__ __forceinline__ void ldg_nc_v8(const void* p, uint4& a, uint4& b) {
  asm volatile("ld.global.nc.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
               : "l"(p));
}
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ void set_dev_error(uint32_t* ctrl, uint32_t bits) {
  if (ctrl) atomicOr(ctrl, bits);
}

// ------------------------------------------------- warp bitonic networks
// One 64-bit key per lane, 32 keys per warp, sorted descending (lane 0 best).
__device__ __forceinline__ uint64_t warp_sort_desc_u64(uint64_t key) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      uint64_t other = __shfl_xor_sync(0xFFFFFFFFu, key, stride);
      bool desc = (lane & size) == 0;
      bool lower = (lane & stride) == 0;
      bool keep_max = (lower == desc);
      uint64_t mx = key > other ? key : other;
      uint64_t mn = key > other ? other : key;
      key = keep_max ? mx : mn;
    }
  }
  return key;
}
// Finishes a bitonic sequence (one key per lane) into descending order.
__device__ __forceinline__ uint64_t warp_bitonic_merge_desc_u64(uint64_t key) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int stride = 16; stride > 0; stride >>= 1) {
    uint64_t other = __shfl_xor_sync(0xFFFFFFFFu, key, stride);
    bool lower = (lane & stride) == 0;
    uint64_t mx = key > other ? key : other;
    uint64_t mn = key > other ? other : key;
    key = lower ? mx : mn;
  }
  return key;
}
// list (sorted desc, one per lane) <- top 32 of list U chunk (any order).
__device__ __forceinline__ uint64_t warp_merge_top32(uint64_t list, uint64_t chunk) {
  const int lane = threadIdx.x & 31;
  uint64_t s = warp_sort_desc_u64(chunk);
  uint64_t rev = __shfl_sync(0xFFFFFFFFu, s, 31 - lane);
  uint64_t c = list > rev ? list : rev;
  return warp_bitonic_merge_desc_u64(c);
}

}  // namespace dart
