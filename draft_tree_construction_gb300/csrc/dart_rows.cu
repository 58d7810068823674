// dart_rows.cu -- K1: one streaming pass over the logits computing, per row,
// the temperature log-sum-exp and the k best candidates.
//
// DART, Figure 3 caption: each of the d logit vectors of a sequence supplies
// the candidates of one depth.  Here every row z[b][j][:] is read exactly once
// from HBM and reduced to (max, sum of exp((z - max) / T), k best (z, id)).
//
// Work split.  The logits are one flat byte stream cut into equal,
// contiguous, 16-byte-aligned spans, one per CTA (one CTA per SM).  Inside a
// CTA one producer thread streams its span through a 192 KiB shared-memory
// ring of stages with cp.async.bulk (an mbarrier per stage counts the bytes
// in, another counts the 12 consumer warps out); each consumer warp reduces
// its own slice of every stage: 2 KiB of 24 KiB stages for rows under 256 KiB,
// 4 KiB of 48 KiB stages for longer rows.  Stages never straddle a row, so all
// consumer warps of a CTA work on the same row at the same time.
//
// Per slice a lane holds four 16-byte vectors.  One running-max update covers
// all of them (maxima taken on packed bf16x2 / f16x2 words), the exponentials
// use packed f32x2 subtract / multiply / add, and one warp vote decides
// whether any element can enter the top-k.
//
// Top-k.  Candidates are 64-bit keys (ordered value, then inverted id), so a
// larger key is a better candidate and equal values fall back to the lower id.
// An element can only matter if it is >= tau, a lower bound of the row's k-th
// value.  At a row's first stage every consumer lane posts the maximum of its
// elements and tau starts at the k-th largest of the 32 column maxima (twelve
// warps' lane j): disjoint elements, so k of them are at least that large.
// Consumer warps keep no lists: they append the rare 16-byte vectors whose
// maximum reaches tau (straight from registers, with their first element id)
// to a per-row ring in shared memory.  A merger warp expands them into keys,
// keeps the CTA's best 32 of the row and publishes the list's k-th value as
// the row's tau.
//
// Row end.  Each consumer warp leaves its (max, scaled sum) in a shared slot
// and moves on; the merger combines them with the list.  A row inside one
// span is finished there; a row cut by span borders leaves one partial per
// CTA, and the last CTA to arrive (an arrival counter, no waiting) merges them
// and writes the row's results.  All global round trips of a row's end sit on
// the merger warp, off the stream.
//
// Every wait is bounded: on a timeout the kernel raises a flag in shared
// memory that ends all other waits of the CTA, records the error bit and
// returns.  Vectors enter the ring in per-warp blocks reserved (and waited
// for) before any lane writes, so a reserved entry is always written promptly.
#include "dart_common.cuh"

#include <atomic>
#include <cfloat>

namespace dart {

constexpr int kConsumers = 12;                  // reducing warps per CTA (plus a producer and a merger warp)
constexpr int kSlice = 2048;                    // bytes one reduce step covers: 4 vectors per lane
constexpr int kRingBytes = 196608;              // 192 KiB of stages in flight per SM
constexpr int kMaxStages = 8;                   // 8 x 24 KiB (short rows) or 4 x 48 KiB stages
constexpr int kVecPerLane = kSlice / 16 / 32;
constexpr int kRowSlots = 4;                    // rows in flight between the consumers and the merger
constexpr int kRingVecs = 256;                  // candidate-vector ring per row slot (power of two)
constexpr uint32_t kSleepNs = 100000;           // longest sleep of one barrier probe
// Copies in flight always land before their CTA retires: that drain is bounded
// by about two seconds of SM clock whatever limit the other waits have.
constexpr long long kDrainLimit = 4000000000LL;
constexpr long long kDefaultWaitLimit = 4000000000LL;
constexpr int kMergerWarp = kConsumers + 1;
constexpr int kRowThreads = (kConsumers + 2) * 32;
static_assert(kVecPerLane == 4, "reduce_slice reduces exactly four vectors per lane");
static_assert((kRingVecs & (kRingVecs - 1)) == 0, "ring index masking");
// one warp reserves at most 32 lanes x 4 vectors, and the merger takes at most
// 32 entries past its head: both fit, so the oldest reservation always proceeds
static_assert(kRingVecs >= 32 * 4 + 32, "vector ring too small for one warp's reservation");

struct RowsParams {
  const uint8_t* logits;
  long long R;
  int V, k, es;
  unsigned long long stride;  // elements from one row's start to the next (>= V; the rest is padding)
  float c;                    // log2(e) / T
  double T;
  double invT;                // 1 / T
  unsigned long long total;   // R * V * es bytes
  unsigned long long span;    // bytes per CTA, multiple of 16
  int grid;
  int nsub;                   // 2 KiB steps per consumer warp and stage (1 or 2)
  int pmax, pstride;
  uint32_t* ctrl;
  uint32_t* row_cnt;
  uint8_t* partials;
  double* row_off;
  int32_t* row_ids;
  double* row_base;
  int32_t* out_ids;   // optional [R][k]
  float* out_logp;    // optional [R][k]
  float* out_lse;     // optional [R]
  long long wait_limit;
};

struct __align__(128) RowSmem {
  uint8_t ring[kRingBytes];
  uint4 vdata[kRowSlots][kRingVecs];     // candidate vectors of a row (16 bytes of logits each)
  uint32_t vid[kRowSlots][kRingVecs];    // (element mask << 24) | (first id + 1); 0 = not written yet
  float2 part[kRowSlots][kConsumers];    // per consumer warp: (max, sum of 2^((z - max) c))
  uint64_t full[kMaxStages];             // bytes of a stage have landed
  uint64_t empty[kMaxStages];            // every consumer warp is done with a stage
  uint64_t row_full[kRowSlots];          // every consumer lane is done with a row
  uint64_t row_free[kRowSlots];          // the merger is done with a row slot
  uint32_t tail[kRowSlots];              // keys reserved in a row's ring
  uint32_t head[kRowSlots];              // keys the merger has taken
  uint32_t tau[kRowSlots];               // ordered form of the row's best published threshold
  uint64_t mkeys[32 * 8];                // the merger's surviving keys of one batch
  uint32_t seed[2][kConsumers][32];      // lane maxima of a row's first stage (alternating rows)
  uint64_t seed_bar[2];                  // every consumer lane has written its lane maximum
  uint32_t abort;                        // a wait timed out: every wait gives up
};

// ------------------------------------------------------------- element types
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t hmax2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t word(const uint4& r, int i) {
  return i == 0 ? r.x : (i == 1 ? r.y : (i == 2 ? r.z : r.w));
}

template <int DT> struct Elem;
template <> struct Elem<DART_F32> {
  static constexpr int kPerVec = 4;
  static constexpr int kShift = 2;      // log2 of the element size
  __device__ static uint4 neg_inf() { return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u); }
  __device__ static float2 pair(const uint4& r, int p) {
    return make_float2(__uint_as_float(word(r, 2 * p)), __uint_as_float(word(r, 2 * p + 1)));
  }
  __device__ static float vmax(const uint4& r) {
    return fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)),
                 fmaxf(__uint_as_float(r.z), __uint_as_float(r.w)));
  }
  __device__ static float vmax4(const uint4* r) {
    return fmaxf(fmaxf(vmax(r[0]), vmax(r[1])), fmaxf(vmax(r[2]), vmax(r[3])));
  }
  __device__ static float scalar(const uint8_t* p) { return __ldg(reinterpret_cast<const float*>(p)); }
  // a vector holding z as element 0 (the rest -inf)
  __device__ static uint4 single(float z) { return make_uint4(__float_as_uint(z), 0xFF800000u, 0xFF800000u, 0xFF800000u); }
};
template <> struct Elem<DART_BF16> {
  static constexpr int kPerVec = 8;
  static constexpr int kShift = 1;
  __device__ static uint4 neg_inf() { return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u); }
  __device__ static float2 pair(const uint4& r, int p) {
    const uint32_t w = word(r, p);
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  }
  __device__ static float unpack_max(uint32_t m) {
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
  }
  __device__ static uint32_t pmax(const uint4& r) { return bmax2(bmax2(r.x, r.y), bmax2(r.z, r.w)); }
  __device__ static float vmax(const uint4& r) { return unpack_max(pmax(r)); }
  __device__ static float vmax4(const uint4* r) {
    return unpack_max(bmax2(bmax2(pmax(r[0]), pmax(r[1])), bmax2(pmax(r[2]), pmax(r[3]))));
  }
  __device__ static float scalar(const uint8_t* p) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(p));
    return __uint_as_float(uint32_t(h) << 16);
  }
  __device__ static uint4 single(float z) {   // z came from a bf16: its top half is exact
    return make_uint4((__float_as_uint(z) >> 16) | 0xFF800000u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
  }
};
template <> struct Elem<DART_F16> {
  static constexpr int kPerVec = 8;
  static constexpr int kShift = 1;
  __device__ static uint4 neg_inf() { return make_uint4(0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u); }
  __device__ static float2 pair(const uint4& r, int p) {
    const uint32_t w = word(r, p);
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
  __device__ static float unpack_max(uint32_t m) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&m));
    return fmaxf(f.x, f.y);
  }
  __device__ static uint32_t pmax(const uint4& r) { return hmax2(hmax2(r.x, r.y), hmax2(r.z, r.w)); }
  __device__ static float vmax(const uint4& r) { return unpack_max(pmax(r)); }
  __device__ static float vmax4(const uint4* r) {
    return unpack_max(hmax2(hmax2(pmax(r[0]), pmax(r[1])), hmax2(pmax(r[2]), pmax(r[3]))));
  }
  __device__ static float scalar(const uint8_t* p) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(p));
    return __half2float(__ushort_as_half(h));
  }
  __device__ static uint4 single(float z) {   // z came from an f16: exact
    return make_uint4(uint32_t(__half_as_ushort(__float2half_rn(z))) | 0xFC000000u, 0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u);
  }
};

// ------------------------------------------------------------ bounded waits
__device__ __forceinline__ bool aborted(const RowSmem& S) {
  return *reinterpret_cast<const volatile uint32_t*>(&S.abort) != 0u;
}
__device__ __forceinline__ void raise_abort(RowSmem& S, uint32_t* ctrl) {
  *reinterpret_cast<volatile uint32_t*>(&S.abort) = 1u;
  set_dev_error(ctrl, DART_DEVERR_WAIT_TIMEOUT);
}
__device__ __forceinline__ bool wait_phase_spin(RowSmem& S, uint64_t* bar, uint32_t parity, long long limit,
                                             uint32_t* ctrl) {
  const long long t0 = clock64();
  for (uint32_t it = 1; !mbar_try_wait_hint(bar, parity, kSleepNs); ++it) {
    if ((it & 63u) != 0u) continue;   // the clock and the abort flag every 64 probes
    if (aborted(S)) return false;
    if (clock64() - t0 > limit) {
      raise_abort(S, ctrl);
      return false;
    }
  }
  return true;
}
// Waits for the phase of `bar` with the given parity; false on a timeout or
// when another wait of the CTA has timed out.
__device__ __forceinline__ bool wait_phase(RowSmem& S, uint64_t* bar, uint32_t parity, long long limit,
                                           uint32_t* ctrl) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_phase_spin(S, bar, parity, limit, ctrl);
}

// ----------------------------------------------------------------- consumers
// Where a consumer warp appends candidate vectors of the current row.
struct VecRing {
  uint32_t* tail;                  // reservation counter
  const volatile uint32_t* head;   // entries the merger has taken
  uint4* vdata;                    // kRingVecs entries
  volatile uint32_t* vid;          // their (mask << 24) | (id + 1), 0 = not written yet
  RowSmem* S;
  uint32_t* ctrl;
  long long limit;
};

__device__ __forceinline__ void sts_v4(void* p, const uint4& v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
               :: "r"(smem_u32(p)), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ uint4 lds_v4_volatile(const void* p) {
  uint4 v;
  asm volatile("ld.volatile.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_u32(p)) : "memory");
  return v;
}

__device__ __forceinline__ void ring_wait(const VecRing& vr, uint32_t pos) {
  const long long t0 = clock64();
  while (pos - *vr.head >= uint32_t(kRingVecs)) {
    if (aborted(*vr.S)) return;
    if (clock64() - t0 > vr.limit) {
      raise_abort(*vr.S, vr.ctrl);
      return;
    }
  }
}
// Reserves ring entries for `cnt` vectors of each lane (0..4) as one block for
// the whole warp and waits, warp-uniformly and before any lane writes, until
// the ring has room for all of them.  Every reserved entry is then written
// without waiting, so the merger, which takes entries in order, never waits on
// an entry whose writer waits on the merger.  Returns false (nothing
// reserved) when no lane has a vector; *pos is the lane's first entry.
__device__ __forceinline__ bool warp_reserve(const VecRing& vr, uint32_t cnt, uint32_t* pos) {
  const int lane = threadIdx.x & 31;
  const uint32_t b0 = __ballot_sync(0xFFFFFFFFu, cnt & 1u);
  const uint32_t b1 = __ballot_sync(0xFFFFFFFFu, cnt & 2u);
  const uint32_t b2 = __ballot_sync(0xFFFFFFFFu, cnt & 4u);
  const uint32_t total = uint32_t(__popc(b0) + 2 * __popc(b1) + 4 * __popc(b2));
  if (total == 0u) return false;
  const uint32_t below = (1u << lane) - 1u;
  uint32_t base = 0;
  if (lane == 0) {
    base = atomicAdd(vr.tail, total);
    if (base + total - 1u - *vr.head >= uint32_t(kRingVecs)) ring_wait(vr, base + total - 1u);
  }
  base = __shfl_sync(0xFFFFFFFFu, base, 0);
  *pos = base + uint32_t(__popc(b0 & below) + 2 * __popc(b1 & below) + 4 * __popc(b2 & below));
  return true;
}
// One entry: the vector first, then (after a fence) its tag, which the merger polls.
__device__ __forceinline__ void ring_put(const VecRing& vr, uint32_t pos, const uint4& v, uint32_t tag) {
  const uint32_t i = pos & uint32_t(kRingVecs - 1);
  sts_v4(vr.vdata + i, v);
  __threadfence_block();
  vr.vid[i] = tag;
}

// Appends the lane's vectors of a 2 KiB step whose maximum reaches tau
// (vector u*32 + lane holds elements id_base + (u*32 + lane) * EPV ...).
template <int DT, bool FULL>
__device__ __forceinline__ void push_vectors(const uint4 (&raw)[kVecPerLane], int nvec, uint32_t id_base, float tau,
                                             const VecRing& vr) {
  using E = Elem<DT>;
  constexpr int EPV = E::kPerVec;
  constexpr uint32_t kMask = (1u << EPV) - 1u;
  const int lane = threadIdx.x & 31;
  uint32_t hm = 0;
#pragma unroll
  for (int u = 0; u < kVecPerLane; ++u)
    if ((FULL || u * 32 + lane < nvec) && E::vmax(raw[u]) >= tau) hm |= 1u << u;
  uint32_t pos;
  if (!warp_reserve(vr, uint32_t(__popc(hm)), &pos)) return;
#pragma unroll
  for (int u = 0; u < kVecPerLane; ++u)
    if ((hm >> u) & 1u) ring_put(vr, pos++, raw[u], (kMask << 24) | (id_base + uint32_t((u * 32 + lane) * EPV) + 1u));
  __syncwarp();
}

// Bitonic sort of one 32-bit value per lane, descending (lane 0 largest).
__device__ __forceinline__ uint32_t warp_sort_desc_u32(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xFFFFFFFFu, v, stride);
      const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
      v = keep_max ? max(v, o) : min(v, o);
    }
  }
  return v;
}

// CTA-wide seed of a row's threshold from its first stage.  Every consumer
// lane posts the maximum of its elements of the stage; lane j then takes the
// maximum of column j (the twelve warps' lane j), and the k-th largest of
// those 32 column maxima is a lower bound of the row's k-th value: the
// columns cover disjoint elements, so k distinct elements are at least that
// large.  Returns the bound in ordered form (0 = none or a wait gave up).
template <int DT>
__device__ __forceinline__ uint32_t seed_stage(const uint4* src, int nvec, RowSmem* Sp, int nseed, int w, int k,
                                            long long limit, uint32_t* ctrl) {
  using E = Elem<DT>;
  RowSmem& S = *Sp;
  const int lane = threadIdx.x & 31;
  float vm = -INFINITY;
#pragma unroll 2
  for (int v = lane; v < nvec; v += 32) vm = fmaxf(vm, E::vmax(src[v]));
  const int sb = nseed & 1;
  S.seed[sb][w][lane] = lane < nvec ? ord_f32(vm) : 0u;
  mbar_arrive(&S.seed_bar[sb]);
  if (!__all_sync(0xFFFFFFFFu, wait_phase(S, &S.seed_bar[sb], uint32_t(nseed >> 1) & 1u, limit, ctrl))) return 0u;
  uint32_t col = 0;
#pragma unroll
  for (int i = 0; i < kConsumers; ++i) col = max(col, S.seed[sb][i][lane]);
  const uint32_t v = warp_sort_desc_u32(col);
  return __shfl_sync(0xFFFFFFFFu, v, k - 1);
}

// Per-warp state for one row segment.
// A lane's sum s is kept against mc = fl(m c) rather than m c: each term is
// 2^fma(z, c, -mc), one fused multiply-add per element.  Since m c - mc is
// exact in float (fma(m, c, -mc)), the row end turns s back into the sum of
// 2^((z - m) c).
struct RowCtx {
  float m, mc, s;        // per lane: running max of z, fl(m c), sum of 2^(z c - mc)
  uint32_t tau_ord;      // ordered form of the filter threshold (0 = none yet)
  float tau;             // filter threshold value (-inf = none yet)
  uint32_t* tau_slot;    // the row's shared threshold
};

__device__ __forceinline__ void raise_tau(RowCtx& rc, uint32_t o) {
  if (o > rc.tau_ord) {
    rc.tau_ord = o;
    rc.tau = unord_f32(o);
  }
}
// Adopt a larger threshold published for the row.
__device__ __forceinline__ void refresh_tau(RowCtx& rc) {
  raise_tau(rc, *reinterpret_cast<volatile uint32_t*>(rc.tau_slot));
}

// fl(m c), kept finite (-FLT_MAX before the first element) so that
// fma(-inf, c, -mc) stays -inf.
__device__ __forceinline__ float scaled_max(float m, float c) { return fmaxf(m * c, -FLT_MAX); }
// Raises the lane's running max to v (if larger), rescaling its sum.
__device__ __forceinline__ void raise_max(float& m, float& mc, float& s, float v, float c) {
  if (v > m) {
    const float mcn = scaled_max(v, c);
    s *= ex2_approx(mc - mcn);
    m = v;
    mc = mcn;
  }
}
// s against exact m c: s * 2^-(m c - mc).  0 stays 0.
__device__ __forceinline__ float exact_sum(float m, float mc, float s, float c) {
  return s > 0.f ? s * ex2_approx(-fmaf(m, c, -mc)) : 0.f;
}

// The hot path: one 2 KiB slice (four vectors per lane; a partial slice at
// the end of a row holds nvec < 128 vectors, the rest read as -inf, whose
// terms are exactly 0).  Updates the lane's (max, sum) and, when some vector
// reaches tau, appends those vectors to the row's ring.
template <int DT, bool FULL>
__device__ __forceinline__ void reduce_slice(RowCtx& rc, const uint4* src, int nvec, float c, uint32_t id_base,
                                             const VecRing& vr) {
  using E = Elem<DT>;
  constexpr int EPV = E::kPerVec;
  constexpr int U = kVecPerLane;
  const int lane = threadIdx.x & 31;
  uint4 raw[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    if (FULL) raw[u] = src[u * 32 + lane];
    else raw[u] = (u * 32 + lane < nvec) ? src[u * 32 + lane] : E::neg_inf();
  }
  const float vm = E::vmax4(raw);
  raise_max(rc.m, rc.mc, rc.s, vm, c);
  const float2 nmc2 = make_float2(-rc.mc, -rc.mc);
  const float2 c2 = make_float2(c, c);
  float2 acc[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    acc[u] = make_float2(0.f, 0.f);
#pragma unroll
    for (int p = 0; p < EPV / 2; ++p) {
      const float2 t = __ffma2_rn(E::pair(raw[u], p), c2, nmc2);
      acc[u] = __fadd2_rn(acc[u], make_float2(ex2_approx(t.x), ex2_approx(t.y)));
    }
  }
  const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
  rc.s += a.x + a.y;
  // absent vectors hold -inf, which must not pass while tau is still -inf
  const bool lane_hit = (FULL || lane < nvec) && vm >= rc.tau;
  if (__ballot_sync(0xFFFFFFFFu, lane_hit) != 0u) push_vectors<DT, FULL>(raw, nvec, id_base, rc.tau, vr);
}

// The end of a row: up to NSUB partial-or-full 2 KiB steps of nvec vectors.
template <int DT, int NSUB>
__device__ __forceinline__ void reduce_tail_stage(RowCtx* rcp, const uint4* src, int nvec, uint32_t id_base, int SH,
                                               float c, const VecRing& vr) {
  RowCtx rc = *rcp;
#pragma unroll 1
  for (int j = 0; j < NSUB; ++j) {
    const int nv = min(nvec - j * (kSlice / 16), kSlice / 16);
    if (nv <= 0) break;
    reduce_slice<DT, false>(rc, src + j * (kSlice / 16), nv, c, id_base + uint32_t((j * kSlice) >> SH), vr);
  }
  *rcp = rc;
}

// Unaligned elements [b0, b1) of a segment (its head or tail), one per lane.
template <int DT>
__device__ __noinline__ float2 reduce_scalars(const uint8_t* logits, unsigned long long b0, unsigned long long b1,
                                              int es, uint32_t id0, float c, float m, float s, float tau,
                                              const VecRing vr) {
  const int lane = threadIdx.x & 31;
  const int cnt = int((b1 - b0) / es);
  for (int base = 0; base < cnt; base += 32) {
    const int i = base + lane;
    bool hit = false;
    float z = 0.f;
    if (i < cnt) {
      z = Elem<DT>::scalar(logits + b0 + (unsigned long long)i * es);
      float mc = scaled_max(m, c);
      raise_max(m, mc, s, z, c);
      s += ex2_approx(fmaf(z, c, -mc));
      hit = z >= tau;
    }
    uint32_t pos;
    if (warp_reserve(vr, hit ? 1u : 0u, &pos) && hit) ring_put(vr, pos, Elem<DT>::single(z), (1u << 24) | (id0 + uint32_t(i) + 1u));
  }
  __syncwarp();
  return make_float2(m, s);
}

struct Seg {
  unsigned long long s0, s1;  // flat element range
  unsigned long long a, b;    // aligned interior, bytes (a == b: none)
};

// The part of row r (its V valid elements; padding up to the row stride is
// never read) that lies in the span [e0, e1).
__device__ __forceinline__ Seg segment(const RowsParams& P, unsigned long long e0, unsigned long long e1,
                                       long long r) {
  Seg g;
  const unsigned long long rs = (unsigned long long)r * P.stride;
  g.s0 = e0 > rs ? e0 : rs;
  const unsigned long long re = rs + P.V;
  g.s1 = e1 < re ? e1 : re;
  if (g.s1 < g.s0) g.s1 = g.s0;
  g.a = (g.s0 * P.es + 15) & ~15ull;
  g.b = (g.s1 * P.es) & ~15ull;
  if (g.a >= g.b) g.a = g.b = g.s1 * P.es;  // nothing aligned: all scalars
  return g;
}

// ------------------------------------------------------------------ row end
// Writes a row's results from its maximum M, its sum S of 2^((z - M) c) and
// its best keys (lanes 0..k-1 hold them, descending).
__device__ __forceinline__ void finish_row(const RowsParams& P, long long r, float M, double S, uint64_t list) {
  const int lane = threadIdx.x & 31;
  const int k = P.k;
  const float zmax = key_value(__shfl_sync(0xFFFFFFFFu, list, 0));
  if (lane == 0 && zmax != M) set_dev_error(P.ctrl, DART_DEVERR_ROW_MAX);
  // log S = e ln 2 + log f with S = f 2^e, f in [0.5, 1): one float log of
  // the mantissa keeps the slow double unit to a multiply and an add
  int e2;
  const double f = frexp(S, &e2);
  const double logS = double(e2) * 0.6931471805599453 + double(logf(float(f)));
  if (lane < k) {
    const float z = key_value(list);
    const int32_t id = int32_t(key_id(list));
    P.row_ids[(size_t)r * k + lane] = id;
    P.row_base[(size_t)r * k + lane] = double(z);
    if (P.out_ids) P.out_ids[(size_t)r * k + lane] = id;
    if (P.out_logp) P.out_logp[(size_t)r * k + lane] = float((double(z) - double(zmax)) * P.invT - logS);
  }
  if (lane == 0) {
    const double lse = double(zmax) * P.invT + logS;
    P.row_off[r] = lse;
    if (P.out_lse) P.out_lse[r] = float(lse);
  }
}

// Global partial of one CTA for one row: [f32 max][4 pad][f64 sum][k keys].
// The last CTA to finish a row merges all of that row's partials.
__device__ __forceinline__ void merge_row(const RowsParams& P, long long r, int nseg) {
  const int lane = threadIdx.x & 31;
  const int k = P.k;
  const uint8_t* base = P.partials + (size_t)r * P.pmax * P.pstride;
  float M = -FLT_MAX;
  uint64_t tstar = 0;
  for (int p = lane; p < nseg; p += 32) {
    const uint8_t* q = base + (size_t)p * P.pstride;
    M = fmaxf(M, __ldcg(reinterpret_cast<const float*>(q)));
    const uint64_t kth = __ldcg(reinterpret_cast<const unsigned long long*>(q + 16) + (k - 1));
    tstar = kth > tstar ? kth : tstar;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    const uint64_t t = __shfl_xor_sync(0xFFFFFFFFu, tstar, o);
    tstar = t > tstar ? t : tstar;
  }
  double S = 0.0;
  for (int p = lane; p < nseg; p += 32) {
    const uint8_t* q = base + (size_t)p * P.pstride;
    const float mp = __ldcg(reinterpret_cast<const float*>(q));
    const double sp = __ldcg(reinterpret_cast<const double*>(q + 8));
    S += sp * double(ex2_approx((mp - M) * P.c));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xFFFFFFFFu, S, o);
  // keys >= tstar (the largest k-th key of any partial) contain the row's best k
  uint64_t list = 0;
  const int total = nseg * k;
  for (int b0 = 0; b0 < total; b0 += 32) {
    const int idx = b0 + lane;
    uint64_t key = 0;
    if (idx < total) {
      const int p = idx / k, e = idx - p * k;
      key = __ldcg(reinterpret_cast<const unsigned long long*>(base + (size_t)p * P.pstride + 16) + e);
      if (key < tstar) key = 0;
    }
    if (__any_sync(0xFFFFFFFFu, key != 0)) list = warp_merge_top32(list, key);
  }
  finish_row(P, r, M, S, list);
}

// Adds up to 32 keys (one per lane, 0 = none) to the best-32 list.  Keys not
// above the list's k-th key cannot reach the row's best k and are dropped; a
// few survivors are inserted one at a time (a vote finds the position), more
// go through a bitonic merge.  Returns whether the list changed.
__device__ __forceinline__ bool merge_keys(uint64_t& list, uint64_t key, int k) {
  const int lane = threadIdx.x & 31;
  const uint64_t kth = __shfl_sync(0xFFFFFFFFu, list, k - 1);
  const bool keep = key > kth;   // keys are distinct; 0 never passes
  uint32_t bal = __ballot_sync(0xFFFFFFFFu, keep);
  if (bal == 0u) return false;
  if (__popc(bal) > 4) {
    list = warp_merge_top32(list, keep ? key : 0ull);
    return true;
  }
  while (bal) {
    const int src = __ffs(bal) - 1;
    bal &= bal - 1u;
    const uint64_t x = __shfl_sync(0xFFFFFFFFu, key, src);
    const int pos = __popc(__ballot_sync(0xFFFFFFFFu, list > x));   // < k: x beats the k-th
    const uint64_t up = __shfl_up_sync(0xFFFFFFFFu, list, 1);
    list = lane < pos ? list : (lane == pos ? x : up);
  }
  return true;
}

// The merger warp: per row of the span, drains the row's key ring into the
// CTA's best-32 list (publishing its k-th value as the row's threshold) until
// every consumer lane is done with the row, then combines the consumer warps'
// (max, sum) and finishes the row or leaves the CTA's partial.
template <int DT>
__device__ __forceinline__ void merge_span_rows(const RowsParams& P, RowSmem& S, long long r_first,
                                                long long r_last) {
  using E = Elem<DT>;
  constexpr int EPV = E::kPerVec;
  const int lane = threadIdx.x & 31;
  const int k = P.k;
  for (long long r = r_first; r <= r_last; ++r) {
    const int rowseq = int(r - r_first);
    const int rslot = rowseq % kRowSlots;
    const uint32_t parity = uint32_t(rowseq / kRowSlots) & 1u;
    volatile uint32_t* vid = S.vid[rslot];
    uint32_t head = 0;
    uint64_t list = 0;
    long long t0 = clock64();
    for (;;) {
      // read "done" before the tail: once done, the tail read after it is final
      const bool done = __shfl_sync(0xFFFFFFFFu, mbar_test_wait(&S.row_full[rslot], parity) ? 1 : 0, 0) != 0;
      const uint32_t tail = __shfl_sync(0xFFFFFFFFu, *reinterpret_cast<volatile uint32_t*>(&S.tail[rslot]), 0);
      if (tail != head) {
        const uint32_t n = (tail - head) < 32u ? (tail - head) : 32u;
        uint32_t tag = 0;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (uint32_t(lane) < n) {
          const uint32_t i = (head + uint32_t(lane)) & uint32_t(kRingVecs - 1);
          tag = vid[i];
          if (tag == 0u) {
            const long long t1 = clock64();
            while ((tag = vid[i]) == 0u) {
              if (aborted(S)) break;
              if (clock64() - t1 > P.wait_limit) {
                raise_abort(S, P.ctrl);
                break;
              }
            }
          }
          __threadfence_block();   // the vector was stored before its tag
          v = lds_v4_volatile(S.vdata[rslot] + i);
          vid[i] = 0u;
        }
        if (__any_sync(0xFFFFFFFFu, aborted(S))) return;
        head += n;
        __threadfence_block();
        if (lane == 0) *reinterpret_cast<volatile uint32_t*>(&S.head[rslot]) = head;
        // expand the vectors: element e of lane's vector is id (tag & 0xFFFFFF) - 1 + e;
        // elements below the row's published threshold (seed or k-th so far)
        // cannot reach the row's best k and are dropped before any merging
        const uint32_t id0 = (tag & 0xFFFFFFu) - 1u;
        const uint32_t tau_o = __shfl_sync(0xFFFFFFFFu, *reinterpret_cast<volatile uint32_t*>(&S.tau[rslot]), 0);
        // survivors: above the threshold and above the list's current k-th key
        const uint64_t kth0 = __shfl_sync(0xFFFFFFFFu, list, k - 1);
        uint64_t cand[EPV];
        uint32_t cnt = 0;
#pragma unroll
        for (int p = 0; p < EPV / 2; ++p) {
          const float2 z = E::pair(v, p);
          const bool q0 = ((tag >> (24 + 2 * p)) & 1u) && ord_f32(z.x) >= tau_o;
          const bool q1 = ((tag >> (25 + 2 * p)) & 1u) && ord_f32(z.y) >= tau_o;
          cand[2 * p] = q0 ? elem_key(z.x, id0 + 2 * p) : 0ull;
          cand[2 * p + 1] = q1 ? elem_key(z.y, id0 + 2 * p + 1) : 0ull;
          if (cand[2 * p] <= kth0) cand[2 * p] = 0ull;
          if (cand[2 * p + 1] <= kth0) cand[2 * p + 1] = 0ull;
          cnt += (cand[2 * p] != 0ull) + (cand[2 * p + 1] != 0ull);
        }
        // compact them into shared memory (prefix sum of counts <= 8 by ballots)
        const uint32_t c0 = __ballot_sync(0xFFFFFFFFu, cnt & 1u), c1 = __ballot_sync(0xFFFFFFFFu, cnt & 2u);
        const uint32_t c2 = __ballot_sync(0xFFFFFFFFu, cnt & 4u), c3 = __ballot_sync(0xFFFFFFFFu, cnt & 8u);
        const int total = __popc(c0) + 2 * __popc(c1) + 4 * __popc(c2) + 8 * __popc(c3);
        const bool changed = total > 0;
        if (changed) {
          const uint32_t below = (1u << lane) - 1u;
          int at = __popc(c0 & below) + 2 * __popc(c1 & below) + 4 * __popc(c2 & below) + 8 * __popc(c3 & below);
#pragma unroll
          for (int e = 0; e < EPV; ++e)
            if (cand[e] != 0ull) S.mkeys[at++] = cand[e];
          __syncwarp();
          if (total <= 4) {
            // a few: insert one at a time (a vote finds the position)
            for (int t = 0; t < total; ++t) {
              const uint64_t x = S.mkeys[t];
              const int pos = __popc(__ballot_sync(0xFFFFFFFFu, list > x));
              const uint64_t up = __shfl_up_sync(0xFFFFFFFFu, list, 1);
              list = lane < pos ? list : (lane == pos ? x : up);
            }
          } else {
            for (int b0 = 0; b0 < total; b0 += 32)
              list = warp_merge_top32(list, b0 + lane < total ? S.mkeys[b0 + lane] : 0ull);
          }
          __syncwarp();
        }
        if (changed) {
          const uint64_t kth = __shfl_sync(0xFFFFFFFFu, list, k - 1);
          if (kth != 0 && lane == 0) atomicMax(&S.tau[rslot], uint32_t(kth >> 32));
        }
        t0 = clock64();
        continue;
      }
      if (done) break;
      __nanosleep(1000);   // an idle merger must not take issue slots from the consumers
      if (__any_sync(0xFFFFFFFFu, aborted(S))) return;
      if (__any_sync(0xFFFFFFFFu, clock64() - t0 > P.wait_limit)) {
        raise_abort(S, P.ctrl);
        return;
      }
    }
    // every lane acquires the completed phase (it cannot move on before the
    // slot is handed back)
    (void)mbar_test_wait(&S.row_full[rslot], parity);
    // the consumer warps' (max, sum) of the row
    const float2 pw = lane < kConsumers ? S.part[rslot][lane] : make_float2(-FLT_MAX, 0.f);
    float M = pw.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    float Sf = pw.y * ex2_approx((pw.x - M) * P.c);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Sf += __shfl_xor_sync(0xFFFFFFFFu, Sf, o);
    const double Ssum = double(Sf);
    // hand the slot back (its ring is all zeros again)
    if (lane == 0) {
      S.tail[rslot] = 0u;
      S.head[rslot] = 0u;
      S.tau[rslot] = 0u;
    }
    __syncwarp();
    __threadfence_block();
    mbar_arrive(&S.row_free[rslot]);

    const unsigned long long rb0 = (unsigned long long)r * P.stride * P.es;
    const long long cfirst = (long long)(rb0 / P.span);
    const long long clast = (long long)((rb0 + (unsigned long long)P.V * P.es - 1) / P.span);
    if (cfirst == clast) {
      finish_row(P, r, M, Ssum, list);
      continue;
    }
    const int nseg = int(clast - cfirst + 1);
    uint8_t* part = P.partials + ((size_t)r * P.pmax + (blockIdx.x - cfirst)) * P.pstride;
    if (lane == 0) {
      reinterpret_cast<float*>(part)[0] = M;
      reinterpret_cast<double*>(part)[1] = Ssum;
    }
    if (lane < k) reinterpret_cast<unsigned long long*>(part + 16)[lane] = list;
    __threadfence();
    __syncwarp();
    uint32_t old = 0;
    if (lane == 0) old = atomicAdd(P.row_cnt + r, 1u);
    old = __shfl_sync(0xFFFFFFFFu, old, 0);
    if (int(old) == nseg - 1) {
      __threadfence();
      merge_row(P, r, nseg);
      if (lane == 0) P.row_cnt[r] = 0u;   // every CTA of the row has arrived: ready for the next call
    }
  }
}

// -------------------------------------------------------------------- kernel
template <int DT, int NSUB>
__global__ void __launch_bounds__(kRowThreads, 1)
row_stream_kernel(const RowsParams P) {
  constexpr int SH = Elem<DT>::kShift;
  constexpr uint32_t SB = uint32_t(kConsumers * NSUB * kSlice);   // stage bytes
  constexpr int NST = kMaxStages / NSUB;                          // stages in the ring
  extern __shared__ __align__(128) uint8_t smem_raw[];
  RowSmem& S = *reinterpret_cast<RowSmem*>(smem_raw);
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;          // 0 producer, 1..kConsumers consumers, then the merger

  const unsigned long long B0 = (unsigned long long)blockIdx.x * P.span;
  const unsigned long long B1 = (B0 + P.span < P.total) ? B0 + P.span : P.total;
  const unsigned long long e0 = B0 / P.es, e1 = B1 / P.es;
  // the rows whose valid elements meet the span (none when it holds padding only)
  long long r_first = (long long)(e0 / P.stride);
  if (e0 - (unsigned long long)r_first * P.stride >= (unsigned long long)P.V) ++r_first;
  const long long r_last = (long long)((e1 - 1) / P.stride);

  if (blockIdx.x == 0 && threadIdx.x == 0) {
    // rows of this call, for clearing the counters after a failed call
    P.ctrl[2] = uint32_t((unsigned long long)P.R);
    P.ctrl[3] = uint32_t((unsigned long long)P.R >> 32);
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxStages; ++i) {
      mbar_init(&S.full[i], 1);
      mbar_init(&S.empty[i], kConsumers);
    }
    for (int i = 0; i < kRowSlots; ++i) {
      mbar_init(&S.row_full[i], kConsumers * 32);
      mbar_init(&S.row_free[i], 32);
    }
    mbar_init(&S.seed_bar[0], kConsumers * 32);
    mbar_init(&S.seed_bar[1], kConsumers * 32);
    fence_mbar_init();
  }
  {
    uint32_t* vz = &S.vid[0][0];
    for (int i = threadIdx.x; i < kRowSlots * kRingVecs; i += blockDim.x) vz[i] = 0u;
    if (threadIdx.x < kRowSlots) {
      S.tail[threadIdx.x] = 0u;
      S.head[threadIdx.x] = 0u;
      S.tau[threadIdx.x] = 0u;
    }
    if (threadIdx.x == 0) S.abort = 0u;
  }
  __syncthreads();

  // ---------------------------------------------------------------- producer
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int slot = 0;
      uint32_t round = 0;   // fills of `slot` so far
      int issued = 0;
      bool ok = true;
      for (long long r = r_first; r <= r_last && ok; ++r) {
        const Seg g = segment(P, e0, e1, r);
        for (unsigned long long off = g.a; off < g.b; off += SB) {
          if (round > 0 && !wait_phase(S, &S.empty[slot], (round - 1) & 1u, P.wait_limit, P.ctrl)) {
            ok = false;
            break;
          }
          const uint32_t bytes = uint32_t((g.b - off) < (unsigned long long)SB ? (g.b - off) : SB);
          mbar_expect_tx(&S.full[slot], bytes);
          bulk_g2s(S.ring + size_t(slot) * SB, P.logits + off, bytes, &S.full[slot], pol);
          ++issued;
          if (++slot == NST) {
            slot = 0;
            ++round;
          }
        }
      }
      // the CTA may not retire while a copy still writes its shared memory;
      // these waits are bounded by the clock alone
      for (int j = 0; j < NST && j < issued; ++j) {
        // the last fill of each slot used so far
        const int sl = (slot + NST - 1 - j) % NST;
        const uint32_t rd = (sl < slot) ? round : round - 1;
        if (!mbar_wait_bounded(&S.full[sl], rd & 1u, kDrainLimit)) {
          set_dev_error(P.ctrl, DART_DEVERR_WAIT_TIMEOUT);
          break;
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------------ merger
  if (warp == kMergerWarp) {
    merge_span_rows<DT>(P, S, r_first, r_last);
    return;
  }

  // --------------------------------------------------------------- consumers
  const int w = warp - 1;
  const long long lim = P.wait_limit;
  int slot = 0;         // ring stage of the next stage
  uint32_t round = 0;   // fills of `slot` before this one
  int nseed = 0;   // seeds taken so far (rows with an aligned interior), the same in every consumer warp
  for (long long r = r_first; r <= r_last; ++r) {
    const int rowseq = int(r - r_first);
    const int rslot = rowseq % kRowSlots;
    if (rowseq >= kRowSlots &&
        !__all_sync(0xFFFFFFFFu, wait_phase(S, &S.row_free[rslot], uint32_t(rowseq / kRowSlots - 1) & 1u, lim, P.ctrl)))
      return;
    const Seg g = segment(P, e0, e1, r);
    const unsigned long long rs = (unsigned long long)r * P.stride;
    RowCtx rc;
    rc.m = -FLT_MAX;
    rc.mc = scaled_max(rc.m, P.c);
    rc.s = 0.f;
    rc.tau_ord = 0u;
    rc.tau = -INFINITY;
    rc.tau_slot = &S.tau[rslot];
    VecRing vr;
    vr.tail = &S.tail[rslot];
    vr.head = &S.head[rslot];
    vr.vdata = S.vdata[rslot];
    vr.vid = S.vid[rslot];
    vr.S = &S;
    vr.ctrl = P.ctrl;
    vr.limit = lim;

    // head: [s0, a) (or the whole segment when nothing is aligned), warp 0 only
    if (w == 0) {
      const unsigned long long hb0 = g.s0 * P.es;
      const unsigned long long hb1 = (g.a < g.b) ? g.a : g.s1 * P.es;
      if (hb1 > hb0) {
        refresh_tau(rc);
        const float2 ms = reduce_scalars<DT>(P.logits, hb0, hb1, P.es, uint32_t(g.s0 - rs), P.c, rc.m, rc.s, rc.tau, vr);
        rc.m = ms.x;
        rc.mc = scaled_max(rc.m, P.c);
        rc.s = ms.y;
      }
    }
    // aligned interior: this warp's slice of every stage
    const uint32_t ilen = uint32_t(g.b - g.a);
    const uint32_t id_a = uint32_t((g.a >> SH) - rs);
    constexpr uint32_t kMine = uint32_t(NSUB * kSlice);   // bytes of a full stage per warp
    const uint32_t s0 = uint32_t(w) * kMine;
    for (uint32_t o = 0; o < ilen; o += SB) {
      if (!__all_sync(0xFFFFFFFFu, wait_phase(S, &S.full[slot], round & 1u, lim, P.ctrl))) return;
      const uint4* src = reinterpret_cast<const uint4*>(S.ring + size_t(slot) * SB + s0);
      const uint32_t rem = ilen - o;
      const int nvec = s0 < rem ? int(min(rem - s0, kMine) / 16) : 0;
      if (o == 0) {
        const uint32_t kth = seed_stage<DT>(src, nvec, &S, nseed, w, P.k, lim, P.ctrl);
        if (__any_sync(0xFFFFFFFFu, aborted(S))) return;
        raise_tau(rc, kth);
        if (lane == 0 && kth != 0u) atomicMax(rc.tau_slot, kth);
        ++nseed;
      }
      refresh_tau(rc);
      if (rem >= SB) {
#pragma unroll
        for (int j = 0; j < NSUB; ++j) {
          const uint4* sj = src + j * (kSlice / 16);
          reduce_slice<DT, true>(rc, sj, kSlice / 16, P.c, id_a + ((o + s0 + uint32_t(j * kSlice)) >> SH), vr);
        }
      } else if (nvec > 0) {
        reduce_tail_stage<DT, NSUB>(&rc, src, nvec, id_a + ((o + s0) >> SH), SH, P.c, vr);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[slot]);
      if (++slot == NST) {
        slot = 0;
        ++round;
      }
    }
    // tail: [b, s1), warp 0 only
    if (w == 0 && g.a < g.b && g.s1 * P.es > g.b) {
      refresh_tau(rc);
      const float2 ms = reduce_scalars<DT>(P.logits, g.b, g.s1 * P.es, P.es, uint32_t((g.b >> SH) - rs), P.c, rc.m,
                                           rc.s, rc.tau, vr);
      rc.m = ms.x;
      rc.mc = scaled_max(rc.m, P.c);
      rc.s = ms.y;
    }
    // the warp's (max, sum) of the row
    float m = rc.m, s = exact_sum(rc.m, rc.mc, rc.s, P.c);
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) {
      const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o2);
      const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o2);
      const float M = fmaxf(m, m2);
      s = s * ex2_approx((m - M) * P.c) + s2 * ex2_approx((m2 - M) * P.c);
      m = M;
    }
    if (lane == 0) S.part[rslot][w] = make_float2(m, s);
    __syncwarp();
    mbar_arrive(&S.row_full[rslot]);
  }
}

// ------------------------------------------------------------------ launch
size_t rows_smem_bytes() { return sizeof(RowSmem); }

// Clock cycles any one wait of the row pass may take before the pass gives
// up (default about two seconds; tests of the timeout path shorten it).
static std::atomic<long long> g_wait_limit{kDefaultWaitLimit};
long long rows_wait_limit() { return g_wait_limit.load(std::memory_order_relaxed); }
void set_rows_wait_limit(long long cycles) {
  g_wait_limit.store(cycles > 0 ? cycles : kDefaultWaitLimit, std::memory_order_relaxed);
}

cudaError_t launch_rows(const void* logits, long long R, int V, long long stride, int dtype, float T, int k,
                        void* ws, const WsLayout& L, int sms,
                        int32_t* out_ids, float* out_logp, float* out_lse, cudaStream_t stream) {
  RowsParams P;
  const int es = dtype == DART_F32 ? 4 : 2;
  P.logits = static_cast<const uint8_t*>(logits);
  P.R = R;
  P.V = V;
  P.stride = (unsigned long long)stride;
  P.k = k;
  P.es = es;
  P.T = double(T);
  P.invT = 1.0 / double(T);
  P.c = float(1.4426950408889634 / double(T));
  // the stream ends at the last valid element (the last row's padding may be absent)
  P.total = R > 0 ? ((unsigned long long)(R - 1) * P.stride + (unsigned long long)V) * (unsigned long long)es : 0ull;
  // one span per SM, whole 16-byte units, at least kMinSpanBytes
  const unsigned long long want = (P.total + (unsigned long long)sms - 1) / (unsigned long long)sms;
  unsigned long long span = (want + 15) & ~15ull;
  if (span < kMinSpanBytes) span = kMinSpanBytes;
  if (span >= (1ull << 31)) return cudaErrorInvalidValue;   // 32-bit offsets inside a span
  P.span = span;
  P.grid = int((P.total + span - 1) / span);
  // long rows take 48 KiB stages (less loop overhead per byte); rows shorter
  // than about five of those take 24 KiB stages (less idle tail per row)
  const unsigned long long row_bytes = (unsigned long long)V * (unsigned long long)es;
  P.nsub = row_bytes >= 262144ull ? 2 : 1;
  P.pmax = L.pmax;
  P.pstride = L.pstride;
  uint8_t* w = static_cast<uint8_t*>(ws);
  P.ctrl = reinterpret_cast<uint32_t*>(w + L.ctrl);
  P.row_cnt = reinterpret_cast<uint32_t*>(w + L.row_cnt);
  P.partials = w + L.partials;
  P.row_off = reinterpret_cast<double*>(w + L.row_off);
  P.row_ids = reinterpret_cast<int32_t*>(w + L.row_ids);
  P.row_base = reinterpret_cast<double*>(w + L.row_base);
  P.out_ids = out_ids;
  P.out_logp = out_logp;
  P.out_lse = out_lse;
  P.wait_limit = rows_wait_limit();
  if (P.total == 0) return cudaSuccess;
  const size_t smem = rows_smem_bytes();
  cudaError_t e = cudaSuccess;
  auto go = [&](auto kernel) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e == cudaSuccess) kernel<<<P.grid, kRowThreads, smem, stream>>>(P);
  };
  if (P.nsub == 2) {
    if (dtype == DART_F32) go(row_stream_kernel<DART_F32, 2>);
    else if (dtype == DART_F16) go(row_stream_kernel<DART_F16, 2>);
    else go(row_stream_kernel<DART_BF16, 2>);
  } else {
    if (dtype == DART_F32) go(row_stream_kernel<DART_F32, 1>);
    else if (dtype == DART_F16) go(row_stream_kernel<DART_F16, 1>);
    else go(row_stream_kernel<DART_BF16, 1>);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dart
