// dart_rows.cu -- K1: one streaming pass over the logits computing, per row,
// the temperature log-sum-exp and the k best candidates.
//
// DART, Figure 3 caption: each of the d logit vectors of a sequence supplies
// the candidates of one depth.  Here every row z[b][j][:] is read exactly once
// from HBM and reduced to (max, sum of exp((z - max) / T), k best (z, id)).
//
// Work split.  The logits are one flat byte stream cut into equal,
// contiguous, 16-byte-aligned spans, one per warp (twelve warps per CTA, one
// CTA per SM).  Warps never wait for one another: each one streams its own
// span through its own ring of three 4 KiB shared-memory stages, filled by
// bulk copies (cp.async.bulk, L2 evict-first) that its lane 0 issues three
// stages ahead of the stage being reduced.  A span may cover the end of one
// row and the start of the next; each (warp, row) overlap is a piece.  Spans
// are at least 8 KiB; an input with fewer spans than 152 x 12 warps deals
// them round-robin over one CTA per SM, so that every SM streams a share.
//
// Per stage a lane holds eight 16-byte vectors.  One packed maximum per
// vector (bf16x2 / f16x2 max on 16-bit types) feeds one running-max update
// per stage; each element then costs one fused multiply-add, one ex2.approx
// and one add.
//
// Top-k.  The streaming warps keep no sorted list.  Each lane's running
// maximum over its elements of the piece is already at hand, and the lanes
// hold disjoint elements, so the k-th largest of the 32 lane maxima is a lower
// bound tau of the row's k-th value (k elements of the row reach it).  It only
// rises; it is recomputed when k lanes have risen above it (one redux.sync
// min per lane dropped), and warps of one CTA that work on the same row share
// it through a word in shared memory (atomic max).  A stage's vectors whose
// maximum reaches tau are copied, 16 bytes and an id with an element mask,
// into the warp's candidate buffer in shared memory: a vote and a few stores,
// no chain of shuffles.  Should the buffer fill up (inputs with very many
// near-equal values), the warp replaces its candidates by their k best.
//
// Piece and row ends.  At a piece's end the warp writes its (max, sum), its
// bound and its candidates to the piece's slot in the workspace (plain
// stores, nothing waits).  The row merge, a second kernel with one CTA per
// row, then merges the pieces' (max, sum) in piece order, takes the row's
// bound (the largest of the pieces' bounds and, with k or more pieces, the
// k-th largest piece maximum), keeps the candidate elements that reach it and
// ranks them (each key counts the keys above it) to get the row's k best.
// When one round of loads holds every slot entry of the row, headers and
// entries are read together; otherwise the headers come first and only the
// pieces whose maximum reaches the bound have their entries gathered.
//
// Every wait (a stage landing) is bounded: on a timeout the warp records the
// error bit, lets its copies in flight land and returns; the call's results
// are then invalid.
#include "dart_common.cuh"
#include "dart_launch.h"

#include <atomic>
#include <cfloat>

namespace dart {

constexpr int kRowWarps = 12;                     // warps per CTA, one CTA per SM
constexpr int kRowStages = 3;                     // bulk-copy stages in flight per warp
constexpr int kStageBytes = 4096;                 // one stage: eight 16-byte vectors per lane
constexpr int kStageVecs = kStageBytes / 16;
constexpr int kVecPerLane = kStageVecs / 32;
constexpr int kRowSlots = 64;                     // rows per CTA with a shared bound
constexpr int kCandCap = 200;                     // candidate vectors a warp can buffer (slot_capacity <= this)
constexpr int kKeyStage = 288;                    // keys a warp stages: one round of 32 x 8 plus k
constexpr int kRowThreads = kRowWarps * 32;
// Copies in flight always land before their warp retires: that drain is
// bounded by about two seconds of SM clock whatever limit the other waits have.
constexpr long long kDrainLimit = 4000000000LL;
constexpr long long kDefaultWaitLimit = 4000000000LL;
constexpr uint32_t kFull = 0xFFFFFFFFu;
static_assert(kVecPerLane == 8, "stage_reduce reduces exactly eight vectors per lane");
static_assert(kKeyStage >= 32 * 8 + kMaxK, "a stage must take one round of keys after keeping k");
static_assert(kCandCap < 256, "piece counts must fit the row merge's 8-bit prefix sums");

struct RowsParams {
  const uint8_t* logits;
  long long R;
  int V, k, es;
  unsigned long long stride;  // elements from one row's start to the next (>= V; the rest is padding)
  float c;                    // log2(e) / T
  double invT;                // 1 / T
  unsigned long long total;   // bytes from the first element to the last valid one
  unsigned long long wspan;   // bytes per warp, multiple of 16
  int pmax, cp;               // slots per row, candidate vectors per slot
  unsigned long long slot_bytes;
  uint32_t* ctrl;
  uint8_t* slots;
  double* row_off;
  int32_t* row_ids;
  double* row_base;
  int32_t* out_ids;   // optional [R][k]
  float* out_logp;    // optional [R][k]
  float* out_lse;     // optional [R]
  long long wait_limit;
  int spread;         // warps dealt round-robin over the CTAs (inputs too small to fill every SM)
};

// A warp's candidates: vectors of logits and their tags (element mask << 24
// | row index of the vector's first element; the mask says which elements
// are real logits).
struct WarpCands {
  uint4 vecs[kCandCap];
  uint32_t tags[kCandCap];
  uint64_t keys[kKeyStage];   // keys while the warp ranks them
  uint64_t best[kMaxK];
};

struct __align__(128) RowSmem {
  uint8_t ring[kRowWarps][kRowStages][kStageBytes];
  WarpCands cand[kRowWarps];
  uint64_t full[kRowWarps][kRowStages];   // bytes of a stage have landed
  uint32_t tau[kRowSlots];                // ordered form of each row's best published bound
};

// ------------------------------------------------------------- element types
// Two floats in one 64-bit register pair, for the packed f32x2 operations
// (each lane of fma.rn.f32x2 / add.rn.f32x2 rounds as fma.rn.f32 / add.rn.f32).
__device__ __forceinline__ uint64_t pack_f32x2(float x, float y) {
  uint64_t v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "f"(x), "f"(y));
  return v;
}
__device__ __forceinline__ float2 unpack_f32x2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
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

// Per type: elements per vector, a packed maximum of a vector (vpack), the
// maximum of two packed maxima (pcombine), its float value (punpack), element
// e of a vector, element pair p as two floats, one scalar load.
template <int DT> struct Elem;
template <> struct Elem<DART_F32> {
  static constexpr int kPerVec = 4;
  static constexpr int kShift = 2;      // log2 of the element size
  __device__ static uint4 neg_inf() { return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u); }
  __device__ static float2 pair(const uint4& r, int p) {
    return make_float2(__uint_as_float(word(r, 2 * p)), __uint_as_float(word(r, 2 * p + 1)));
  }
  __device__ static float elem(const uint4& r, int e) { return __uint_as_float(word(r, e)); }
  __device__ static uint32_t vpack(const uint4& r) {
    return __float_as_uint(fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)),
                                 fmaxf(__uint_as_float(r.z), __uint_as_float(r.w))));
  }
  __device__ static uint32_t pcombine(uint32_t a, uint32_t b) {
    return __float_as_uint(fmaxf(__uint_as_float(a), __uint_as_float(b)));
  }
  __device__ static float punpack(uint32_t p) { return __uint_as_float(p); }
  __device__ static float scalar(const uint8_t* p) { return __ldg(reinterpret_cast<const float*>(p)); }
};
template <> struct Elem<DART_BF16> {
  static constexpr int kPerVec = 8;
  static constexpr int kShift = 1;
  __device__ static uint4 neg_inf() { return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u); }
  __device__ static float2 pair(const uint4& r, int p) {
    const uint32_t w = word(r, p);
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  }
  __device__ static float elem(const uint4& r, int e) {
    const uint32_t w = word(r, e >> 1);
    return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
  __device__ static uint32_t vpack(const uint4& r) { return bmax2(bmax2(r.x, r.y), bmax2(r.z, r.w)); }
  __device__ static uint32_t pcombine(uint32_t a, uint32_t b) { return bmax2(a, b); }
  __device__ static float punpack(uint32_t m) {
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
  }
  // tau (a bf16 value, or -inf) in both halves; 1 when a half of m reaches it
  __device__ static uint32_t pack_tau(float tau) {
    const uint32_t t = __float_as_uint(tau) >> 16;
    return t | (t << 16);
  }
  __device__ static uint32_t any_ge(uint32_t m, uint32_t t2) {
    uint32_t r;
    asm("{\n .reg .pred p, q;\n setp.ge.bf16x2 p|q, %1, %2;\n or.pred p, p, q;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(r) : "r"(m), "r"(t2));
    return r;
  }
  __device__ static float scalar(const uint8_t* p) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(p));
    return __uint_as_float(uint32_t(h) << 16);
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
  __device__ static float elem(const uint4& r, int e) {
    const uint32_t w = word(r, e >> 1);
    return __half2float(__ushort_as_half((unsigned short)((e & 1) ? (w >> 16) : (w & 0xFFFFu))));
  }
  __device__ static uint32_t vpack(const uint4& r) { return hmax2(hmax2(r.x, r.y), hmax2(r.z, r.w)); }
  __device__ static uint32_t pcombine(uint32_t a, uint32_t b) { return hmax2(a, b); }
  __device__ static float punpack(uint32_t m) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&m));
    return fmaxf(f.x, f.y);
  }
  __device__ static uint32_t pack_tau(float tau) {
    const uint32_t t = uint32_t(__half_as_ushort(__float2half_rn(tau)));   // exact: tau is an f16 value or -inf
    return t | (t << 16);
  }
  __device__ static uint32_t any_ge(uint32_t m, uint32_t t2) {
    uint32_t r;
    asm("{\n .reg .pred p, q;\n setp.ge.f16x2 p|q, %1, %2;\n or.pred p, p, q;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(r) : "r"(m), "r"(t2));
    return r;
  }
  __device__ static float scalar(const uint8_t* p) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(p));
    return __half2float(__ushort_as_half(h));
  }
};


// A vector whose element 0 is z (from a logit of this type, so exact) and
// whose other elements are -inf; its tag mask is 1.
template <int DT>
__device__ __forceinline__ uint4 single_vec(float z) {
  uint4 v = Elem<DT>::neg_inf();
  if (DT == DART_F32) v.x = __float_as_uint(z);
  else if (DT == DART_BF16) v.x = (__float_as_uint(z) >> 16) | 0xFF800000u;
  else v.x = uint32_t(__half_as_ushort(__float2half_rn(z))) | 0xFC000000u;
  return v;
}

// ----------------------------------------------------------- piece state
// A lane's sum s is kept against mc = fl(m c) rather than m c: each term is
// 2^fma(z, c, -mc), one fused multiply-add per element.  Since m c - mc is
// exact in float (fma(m, c, -mc)), the piece end turns s back into the sum of
// 2^((z - m) c).
struct Acc {
  float m, mc, s;     // per lane: running max of z, fl(m c), sum of 2^(z c - mc)
};

__device__ __forceinline__ float tau_value(uint32_t o) { return o != 0u ? unord_f32(o) : -INFINITY; }

// fl(m c), kept finite (-FLT_MAX before the first element) so that
// fma(-inf, c, -mc) stays -inf.
__device__ __forceinline__ float scaled_max(float m, float c) { return fmaxf(m * c, -FLT_MAX); }
// Raises the lane's running max to v (if larger), rescaling its sum.
__device__ __forceinline__ void raise_max(Acc& a, float v, float c) {
  if (v > a.m) {
    const float mcn = scaled_max(v, c);
    a.s *= ex2_approx(a.mc - mcn);
    a.m = v;
    a.mc = mcn;
  }
}
// s against exact m c: s * 2^-(m c - mc).  0 stays 0.
__device__ __forceinline__ float exact_sum(const Acc& a, float c) {
  return a.s > 0.f ? a.s * ex2_approx(-fmaf(a.m, c, -a.mc)) : 0.f;
}

// Exclusive prefix and total over the warp of a per-lane count in 0..255:
// one ballot per bit, all independent.
__device__ __forceinline__ int warp_prefix8(uint32_t cnt, int* total) {
  const uint32_t below = (1u << (threadIdx.x & 31)) - 1u;
  int pre = 0, tot = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t q = __ballot_sync(kFull, (cnt >> j) & 1u);
    pre += __popc(q & below) << j;
    tot += __popc(q) << j;
  }
  *total = tot;
  return pre;
}

// Exclusive prefix and total over the warp of a per-lane count in 0..15.
__device__ __forceinline__ int warp_prefix4(uint32_t cnt, int* total) {
  const int lane = threadIdx.x & 31;
  const uint32_t below = (1u << lane) - 1u;
  const uint32_t q0 = __ballot_sync(kFull, cnt & 1u), q1 = __ballot_sync(kFull, cnt & 2u);
  const uint32_t q2 = __ballot_sync(kFull, cnt & 4u), q3 = __ballot_sync(kFull, cnt & 8u);
  *total = __popc(q0) + 2 * __popc(q1) + 4 * __popc(q2) + 8 * __popc(q3);
  return __popc(q0 & below) + 2 * __popc(q1 & below) + 4 * __popc(q2 & below) + 8 * __popc(q3 & below);
}

// The k-th largest of the lanes' values v (ordered floats, 0 = a lane
// without elements) among those above `above`, or `above` when fewer than k
// lanes are above it: the values below the k-th are dropped one lane at a
// time (a redux.sync min each).
__device__ __forceinline__ uint32_t kth_above(uint32_t v, uint32_t above, int k) {
  const int lane = threadIdx.x & 31;
  bool cand = v > above;
  const int c = __popc(__ballot_sync(kFull, cand));
  if (c < k) return above;
  for (int i = c - k; i > 0; --i) {
    const uint32_t mn = __reduce_min_sync(kFull, cand ? v : 0xFFFFFFFFu);
    const uint32_t b = __ballot_sync(kFull, cand && v == mn);
    if (lane == __ffs(b) - 1) cand = false;
  }
  return __reduce_min_sync(kFull, cand ? v : 0xFFFFFFFFu);
}

// The same for a piece's first stage, where most lanes are above `above`:
// a bitonic sort of the 32 values (fifteen exchange steps) instead of one
// removal per excess lane.
__device__ __forceinline__ uint32_t kth_sorted(uint32_t v, uint32_t above, int k) {
  const int lane = threadIdx.x & 31;
  uint32_t x = v > above ? v : 0u;
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint32_t y = __shfl_xor_sync(kFull, x, stride);
      const bool keep_max = ((lane & stride) == 0) == ((lane & size) == 0);
      x = keep_max ? max(x, y) : min(x, y);
    }
  }
  const uint32_t kth = __shfl_sync(kFull, x, k - 1);   // descending: lane k-1 holds the k-th largest
  return kth > above ? kth : above;
}

// Real elements of a tagged vector that reach tau (bit e = element e).
template <int DT>
__device__ __forceinline__ uint32_t vec_hits(const uint4& v, uint32_t tag, float tau) {
  uint32_t cm = 0;
#pragma unroll
  for (int e = 0; e < Elem<DT>::kPerVec; ++e)
    if (((tag >> (24 + e)) & 1u) && Elem<DT>::elem(v, e) >= tau) cm |= 1u << e;
  return cm;
}

// Keeps the k best of a warp's n staged keys (distinct) in keys[0..min(n,k)),
// best first: each key counts the keys above it.  Returns min(n, k).
__device__ __forceinline__ int keep_best(WarpCands& C, int n, int k) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  for (int i = lane; i < n; i += 32) {
    const uint64_t key = C.keys[i];
    int rank = 0;
    for (int q = 0; q < n; ++q) rank += C.keys[q] > key ? 1 : 0;
    if (rank < k) C.best[rank] = key;
  }
  __syncwarp();
  const int kept = n < k ? n : k;
  for (int i = lane; i < kept; i += 32) C.keys[i] = C.best[i];
  __syncwarp();
  return kept;
}

// Stages the keys of the elements in cm (element e of vector v has id
// id0 + e; one vector per lane), keeping only the k best whenever the stage
// could overflow.  Every lane takes part.
template <int DT>
__device__ __forceinline__ void stage_keys(WarpCands& C, int& n, int k, const uint4& v, uint32_t cm, uint32_t id0) {
  int added;
  const int pre = warp_prefix4(uint32_t(__popc(cm)), &added);
  if (added == 0) return;
  if (n + added > kKeyStage) n = keep_best(C, n, k);
  int at = n + pre;
  while (cm) {
    const int e = __ffs(cm) - 1;
    cm &= cm - 1u;
    C.keys[at++] = elem_key(Elem<DT>::elem(v, e), id0 + uint32_t(e));
  }
  n += added;
  __syncwarp();
}

// The k best keys of the warp's cnt candidates (elements reaching tau), best
// first in C.keys; returns their number.
template <int DT>
__device__ __forceinline__ int cands_best(WarpCands& C, int cnt, float tau, int k) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  int n = 0;
  for (int b0 = 0; b0 < cnt; b0 += 32) {
    const int i = b0 + lane;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    uint32_t tag = 0;
    if (i < cnt) {
      v = C.vecs[i];
      tag = C.tags[i];
    }
    stage_keys<DT>(C, n, k, v, i < cnt ? vec_hits<DT>(v, tag, tau) : 0u, tag & 0xFFFFFFu);
  }
  return keep_best(C, n, k);
}

// A full buffer: its candidates are replaced by their k best (tau rises to
// the k-th of them when there are k).  Rare: only inputs with very many
// near-equal values get here.
template <int DT>
__device__ __forceinline__ void compact_cands(WarpCands& C, int& cnt, uint32_t& tau_o, int k) {
  const int lane = threadIdx.x & 31;
  const int kept = cands_best<DT>(C, cnt, tau_value(tau_o), k);
  if (lane < kept) {
    const uint64_t key = C.keys[lane];
    C.vecs[lane] = single_vec<DT>(key_value(key));
    C.tags[lane] = (1u << 24) | key_id(key);
  }
  cnt = kept;
  if (kept == k) {
    const uint32_t o = uint32_t(C.keys[k - 1] >> 32);
    if (o > tau_o) tau_o = o;
  }
  __syncwarp();
}

// Appends the lanes' candidate vectors (vector u of the lane when bit u of
// hm is set; r holds them, and src, the stage buffer, holds vector u of the
// lane at u * 32 + lane), compacting whenever the buffer is full.
template <int DT>
__device__ __forceinline__ void cands_append(WarpCands& C, int cap, int& cnt, uint32_t& tau_o, int k,
                                             const uint4 (&r)[kVecPerLane], const uint4* src, uint32_t hm,
                                             uint32_t id0) {
  constexpr int EPV = Elem<DT>::kPerVec;
  constexpr uint32_t kMask = ((1u << EPV) - 1u) << 24;
  const int lane = threadIdx.x & 31;
  int total, first;
  if (!__any_sync(kFull, (hm & (hm - 1u)) != 0u)) {
    // the usual case, no lane with more than one vector: one ballot, and the
    // vector copied from the stage buffer (still intact) by its index
    const uint32_t b = __ballot_sync(kFull, hm != 0u);
    total = __popc(b);
    first = __popc(b & ((1u << lane) - 1u));
    if (cnt + total <= cap) {
      if (hm) {
        const int u = __ffs(hm) - 1;
        C.vecs[cnt + first] = src[u * 32 + lane];
        C.tags[cnt + first] = kMask | (id0 + uint32_t((u * 32 + lane) * EPV));
      }
      cnt += total;
      __syncwarp();
      return;
    }
  } else {
    first = warp_prefix4(uint32_t(__popc(hm)), &total);
  }
  if (cnt + total <= cap) {
    int pos = cnt + first;
#pragma unroll
    for (int u = 0; u < kVecPerLane; ++u) {
      if ((hm >> u) & 1u) {
        C.vecs[pos] = r[u];
        C.tags[pos] = kMask | (id0 + uint32_t((u * 32 + lane) * EPV));
        ++pos;
      }
    }
    cnt += total;
    __syncwarp();
    return;
  }
  int done = 0;
  while (done < total) {
    if (cnt == cap) compact_cands<DT>(C, cnt, tau_o, k);
    const int take = min(cap - cnt, total - done);
    int q = first;
#pragma unroll
    for (int u = 0; u < kVecPerLane; ++u) {
      if ((hm >> u) & 1u) {
        if (q >= done && q < done + take) {
          C.vecs[cnt + q - done] = r[u];
          C.tags[cnt + q - done] = kMask | (id0 + uint32_t((u * 32 + lane) * EPV));
        }
        ++q;
      }
    }
    cnt += take;
    done += take;
    __syncwarp();
  }
}

// The hot path: one stage of nv vectors (nv <= 256; vectors past nv read as
// -inf, whose terms are exactly 0).  id0 = row index of the stage's first
// element.  SEED: the stage opens a piece (its lanes' maxima are all new).
template <int DT, bool SEED>
__device__ __forceinline__ void stage_reduce(Acc& a, uint32_t& tau_o, int& cnt, WarpCands& C, int cap,
                                             const uint4* src, int nv, uint32_t id0, float c, int k,
                                             uint32_t* tau_slot) {
  using E = Elem<DT>;
  constexpr int EPV = E::kPerVec;
  constexpr int U = kVecPerLane;
  const int lane = threadIdx.x & 31;
  const bool whole = nv == kStageVecs;
  uint4 r[U];
  uint32_t pm[U];
#pragma unroll
  for (int u = 0; u < U; ++u) r[u] = src[u * 32 + lane];   // a stage buffer is always 4 KiB
  if (!whole) {
    // a row's last stage: vectors past nv hold stale bytes; read them as -inf
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (u * 32 + lane >= nv) r[u] = E::neg_inf();
  }
#pragma unroll
  for (int u = 0; u < U; ++u) pm[u] = E::vpack(r[u]);
  uint32_t pa = pm[0];
#pragma unroll
  for (int u = 1; u < U; ++u) pa = E::pcombine(pa, pm[u]);
  const float vm = E::punpack(pa);
  raise_max(a, vm, c);
  // the bound: k-th largest lane maximum of the piece so far (lanes without
  // an element post 0), raised only when k lanes are above it
  {
    const uint32_t post = a.m > -FLT_MAX ? ord_f32(a.m) : 0u;
    uint32_t o = tau_o;
    if (SEED) o = kth_sorted(post, o, k);
    else if (__popc(__ballot_sync(kFull, post > o)) >= k) o = kth_above(post, o, k);
    if (tau_slot) {
      if (o > tau_o && lane == 0) atomicMax(tau_slot, o);
      const uint32_t so = *reinterpret_cast<volatile uint32_t*>(tau_slot);
      if (so > o) o = so;
    }
    tau_o = o;
  }
  // one fused multiply-add, one exponential and one add per element, the
  // multiply-adds and adds two elements to an instruction (f32x2), into
  // eight independent sums (element e of every vector goes to sum e)
  const uint64_t c2 = pack_f32x2(c, c), nmc2 = pack_f32x2(-a.mc, -a.mc);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int u = 0; u < U; ++u) {
#pragma unroll
    for (int p = 0; p < EPV / 2; ++p) {
      const float2 z = E::pair(r[u], p);
      const float2 t = unpack_f32x2(fma_f32x2(pack_f32x2(z.x, z.y), c2, nmc2));
      acc[p & 3] = add_f32x2(acc[p & 3], pack_f32x2(ex2_approx(t.x), ex2_approx(t.y)));
    }
  }
  const float2 s01 = unpack_f32x2(acc[0]), s23 = unpack_f32x2(acc[1]);
  const float2 s45 = unpack_f32x2(acc[2]), s67 = unpack_f32x2(acc[3]);
  a.s += ((s01.x + s01.y) + (s23.x + s23.y)) + ((s45.x + s45.y) + (s67.x + s67.y));
  // candidates: absent vectors hold -inf, which must not pass while tau is -inf
  const float tau = tau_value(tau_o);
  if (__ballot_sync(kFull, lane < nv && vm >= tau) != 0u) {
    // vectors past nv are -inf and tau is finite here unless no bound
    // exists yet, so the index test only matters in partial stages
    uint32_t hm = 0;
    if constexpr (DT == DART_F32) {
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (E::punpack(pm[u]) >= tau) hm |= 1u << u;
    } else {
      // 16-bit elements: the bound is one of them (or -inf), so a packed
      // compare of each vector's two-half maximum decides exactly
      const uint32_t t2 = E::pack_tau(tau);
#pragma unroll
      for (int u = 0; u < U; ++u) hm |= E::any_ge(pm[u], t2) << u;
    }
    if (!whole) {
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (u * 32 + lane >= nv) hm &= ~(1u << u);
    }
    cands_append<DT>(C, cap, cnt, tau_o, k, r, src, hm, id0);
  }
}

// Unaligned elements [b0, b1) of a piece (its head or tail), one per lane;
// a candidate becomes a one-element vector.
template <int DT>
__device__ __forceinline__ void piece_scalars(Acc& a, uint32_t& tau_o, int& cnt, WarpCands& C, int cap,
                                              const uint8_t* logits, unsigned long long b0, unsigned long long b1,
                                              int es, uint32_t id0, float c, int k) {
  const int lane = threadIdx.x & 31;
  const int n = int((b1 - b0) / es);
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    float z = -INFINITY;
    if (i < n) {
      z = Elem<DT>::scalar(logits + b0 + (unsigned long long)i * es);
      raise_max(a, z, c);
      a.s += ex2_approx(fmaf(z, c, -a.mc));
    }
    const bool hit = i < n && z >= tau_value(tau_o);
    int total;
    const int at = warp_prefix4(hit ? 1u : 0u, &total);
    if (total == 0) continue;
    if (cnt + total > cap) compact_cands<DT>(C, cnt, tau_o, k);
    if (hit) {
      C.vecs[cnt + at] = single_vec<DT>(z);
      C.tags[cnt + at] = (1u << 24) | (id0 + uint32_t(i));
    }
    cnt += total;
    __syncwarp();
  }
}

struct Seg {
  unsigned long long s0, s1;  // flat element range
  unsigned long long a, b;    // aligned interior, bytes (a == b: none)
};

// The part of row r (its V valid elements; padding up to the row stride is
// never read) that lies in the element range [e0, e1).
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
// A piece slot: {f32 max; u32 count; f32 sum; pad; u32 bound; pad}, then cp
// vectors, then cp tags.
__device__ __forceinline__ uint8_t* slot_of(const RowsParams& P, long long r, long long p) {
  return P.slots + ((size_t)r * P.pmax + (size_t)p) * P.slot_bytes;
}
__device__ __forceinline__ uint4* slot_vecs(const RowsParams& P, uint8_t* q) {
  return reinterpret_cast<uint4*>(q + kSlotHeader);
}
__device__ __forceinline__ uint32_t* slot_tags(const RowsParams& P, uint8_t* q) {
  return reinterpret_cast<uint32_t*>(q + kSlotHeader + 16 * (size_t)P.cp);
}

// First warp whose span meets row r; returns the row's number of pieces.
__device__ __forceinline__ int row_pieces(const RowsParams& P, long long r, long long* wa) {
  const unsigned long long rb0 = (unsigned long long)r * P.stride * P.es;
  const long long a = (long long)(rb0 / P.wspan);
  const long long b = (long long)((rb0 + (unsigned long long)P.V * P.es - 1) / P.wspan);
  *wa = a;
  return int(b - a + 1);
}

// The end of a piece of row r: the warp's (max, sum), bound and candidates
// into the piece's slot.  Plain stores; nothing waits.
__device__ __forceinline__ void piece_end(const RowsParams& P, const WarpCands& C, const Acc& a, int cnt,
                                          uint32_t tau_o, long long r, long long gwarp) {
  const int lane = threadIdx.x & 31;
  float m = a.m, s = exact_sum(a, P.c);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(kFull, m, o);
    const float s2 = __shfl_xor_sync(kFull, s, o);
    const float Mx = fmaxf(m, m2);
    s = s * ex2_approx((m - Mx) * P.c) + s2 * ex2_approx((m2 - Mx) * P.c);
    m = Mx;
  }
  long long wa;
  (void)row_pieces(P, r, &wa);
  uint8_t* q = slot_of(P, r, gwarp - wa);
  if (lane == 0) {
    *reinterpret_cast<float*>(q) = m;
    *reinterpret_cast<uint32_t*>(q + 4) = uint32_t(cnt);
    *reinterpret_cast<float*>(q + 8) = s;
    *reinterpret_cast<uint32_t*>(q + 16) = tau_o;
  }
  __syncwarp();
  uint4* vv = slot_vecs(P, q);
  uint32_t* tt = slot_tags(P, q);
  for (int i = lane; i < cnt; i += 32) {
    vv[i] = C.vecs[i];
    tt[i] = C.tags[i];
  }
  __syncwarp();
}

// Next stage of a warp's span after byte `off` of row r (a stage starts at
// off, covers min(4 KiB, end of the row's interior - off)); moves on to later
// rows when the row's interior is used up.  valid = false past the span.
struct Cursor {
  long long r;
  unsigned long long off, b;   // stage start, end of the row's interior (bytes)
  bool valid;
};
__device__ __forceinline__ void cursor_seek(const RowsParams& P, Cursor& cu, unsigned long long e0,
                                            unsigned long long e1, long long r_last) {
  while (cu.r <= r_last) {
    const Seg g = segment(P, e0, e1, cu.r);
    if (g.a < g.b) {
      cu.off = g.a;
      cu.b = g.b;
      cu.valid = true;
      return;
    }
    ++cu.r;
  }
  cu.valid = false;
}
__device__ __forceinline__ void cursor_next(const RowsParams& P, Cursor& cu, unsigned long long e0,
                                            unsigned long long e1, long long r_last) {
  cu.off += kStageBytes;
  if (cu.off < cu.b) return;
  ++cu.r;
  cursor_seek(P, cu, e0, e1, r_last);
}

// Waits for a stage to land until `limit` clock cycles have passed (false).
// Probes may suspend the thread until the phase completes; short limits
// (tests of the timeout path) probe without suspending, so that the clock
// decides.
constexpr long long kSuspendingWaitMin = 100000;
__device__ __forceinline__ bool stage_wait(uint64_t* bar, uint32_t parity, long long limit) {
  if (mbar_test_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (limit >= kSuspendingWaitMin ? mbar_try_wait(bar, parity) : mbar_test_wait(bar, parity)) return true;
    if (clock64() - t0 > limit) return false;
  }
}

// -------------------------------------------------------------------- kernel
template <int DT>
__global__ void __launch_bounds__(kRowThreads, 1)
row_stream_kernel(const __grid_constant__ RowsParams P) {
  constexpr int SH = Elem<DT>::kShift;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  RowSmem& S = *reinterpret_cast<RowSmem*>(smem_raw);
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  // spans are numbered CTA by CTA; a small input deals them round-robin so
  // that every SM streams a share
  const long long gwarp = P.spread ? (long long)w * gridDim.x + blockIdx.x : (long long)blockIdx.x * kRowWarps + w;

  for (int i = threadIdx.x; i < kRowSlots; i += blockDim.x) S.tau[i] = 0u;
  if (lane == 0) {
    for (int s = 0; s < kRowStages; ++s) mbar_init(&S.full[w][s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // the warp's span and the rows whose valid elements meet it
  const unsigned long long B0 = (unsigned long long)gwarp * P.wspan;
  if (B0 >= P.total) return;
  const unsigned long long B1 = (B0 + P.wspan < P.total) ? B0 + P.wspan : P.total;
  const unsigned long long e0 = B0 / P.es, e1 = B1 / P.es;
  long long r_first = (long long)(e0 / P.stride);
  if (e0 - (unsigned long long)r_first * P.stride >= (unsigned long long)P.V) ++r_first;
  const long long r_last = (long long)((e1 - 1) / P.stride);
  // rows of the CTA that share a bound word
  const unsigned long long cta_e0 = ((unsigned long long)blockIdx.x * kRowWarps * P.wspan) / P.es;
  const long long cta_r0 = (long long)(cta_e0 / P.stride);

  const uint64_t pol = policy_evict_first();
  uint8_t* ring = &S.ring[w][0][0];
  uint64_t* full = &S.full[w][0];
  WarpCands& C = S.cand[w];
  // lane 0 issues the stages; every lane follows the same sequence to consume them
  Cursor iss;
  iss.r = r_first;
  cursor_seek(P, iss, e0, e1, r_last);
  // stages issued (counted by lane 0, the only lane that reads it) and
  // consumed so far; a stage's ring slot and phase follow from its number
  // (slot = n mod kRowStages, phase parity = (n / kRowStages) & 1)
  uint32_t issued = 0, consumed = 0;
  int islot = 0, cslot = 0;
  uint32_t cpar = 0;
  auto issue = [&]() {
    const uint32_t bytes = uint32_t((iss.b - iss.off) < (unsigned long long)kStageBytes ? (iss.b - iss.off)
                                                                                        : kStageBytes);
    mbar_expect_tx(&full[islot], bytes);
    bulk_g2s(ring + (size_t)islot * kStageBytes, P.logits + iss.off, bytes, &full[islot], pol);
    ++issued;
    if (++islot == kRowStages) islot = 0;
    cursor_next(P, iss, e0, e1, r_last);
  };
  if (lane == 0)
    for (int s = 0; s < kRowStages && iss.valid; ++s) issue();

  bool ok = true;
  for (long long r = r_first; r <= r_last && ok; ++r) {
    const Seg g = segment(P, e0, e1, r);
    if (g.s1 <= g.s0) continue;
    const unsigned long long rs = (unsigned long long)r * P.stride;
    const long long slot_i = r - cta_r0;
    uint32_t* tau_slot = (!P.spread && slot_i >= 0 && slot_i < kRowSlots) ? &S.tau[slot_i] : nullptr;
    Acc a;
    a.m = -FLT_MAX;
    a.mc = scaled_max(a.m, P.c);
    a.s = 0.f;
    uint32_t tau_o = tau_slot ? *reinterpret_cast<volatile uint32_t*>(tau_slot) : 0u;
    int cnt = 0;
    // head: [s0, a) (or the whole piece when nothing is aligned)
    {
      const unsigned long long hb0 = g.s0 * P.es;
      const unsigned long long hb1 = (g.a < g.b) ? g.a : g.s1 * P.es;
      if (hb1 > hb0)
        piece_scalars<DT>(a, tau_o, cnt, C, P.cp, P.logits, hb0, hb1, P.es, uint32_t(g.s0 - rs), P.c, P.k);
    }
    // aligned interior, stage by stage (offsets within the interior fit 32 bits)
    const uint32_t ilen = uint32_t(g.b - g.a);
    const uint32_t id_a = uint32_t((g.a >> SH) - rs);
    for (uint32_t o = 0; o < ilen; o += kStageBytes) {
      if (!__all_sync(kFull, stage_wait(&full[cslot], cpar, P.wait_limit))) {
        ok = false;
        break;
      }
      const uint4* src = reinterpret_cast<const uint4*>(ring + cslot * kStageBytes);
      const uint32_t rem = ilen - o;
      const int nv = int((rem < uint32_t(kStageBytes) ? rem : uint32_t(kStageBytes)) >> 4);
      const uint32_t id0 = id_a + (o >> SH);
      if (o == 0) stage_reduce<DT, true>(a, tau_o, cnt, C, P.cp, src, nv, id0, P.c, P.k, tau_slot);
      else stage_reduce<DT, false>(a, tau_o, cnt, C, P.cp, src, nv, id0, P.c, P.k, tau_slot);
      __syncwarp();
      ++consumed;
      if (++cslot == kRowStages) {
        cslot = 0;
        cpar ^= 1u;
      }
      if (lane == 0 && iss.valid) issue();
    }
    if (!ok) break;
    // tail: [b, s1)
    if (g.a < g.b && g.s1 * P.es > g.b)
      piece_scalars<DT>(a, tau_o, cnt, C, P.cp, P.logits, g.b, g.s1 * P.es, P.es, uint32_t((g.b >> SH) - rs), P.c,
                        P.k);
    piece_end(P, C, a, cnt, tau_o, r, gwarp);
  }
  if (!ok) {
    set_dev_error(lane == 0 ? P.ctrl : nullptr, DART_DEVERR_WAIT_TIMEOUT);
    // the warp may not retire while a copy still writes its ring; these
    // waits are bounded by the clock alone
    if (lane == 0) {
      for (uint32_t q = consumed; q < issued; ++q) {
        if (!mbar_wait_bounded(&full[q % kRowStages], (q / kRowStages) & 1u, kDrainLimit)) break;
      }
    }
    __syncwarp();
  }
}

// ---------------------------------------------------------------- row merge
constexpr int kMergeThreads = 128;
constexpr int kMergePieces = 64;     // pieces a row merges from shared memory (more: the loop below)
constexpr int kMergeKeys = 1024;     // candidate keys a row keeps in shared memory (more: one warp merges)

// Writes a row's results from its maximum M, its sum S of 2^((z - M) c) and
// its best keys (keys[0..kept), descending); one warp.
__device__ __forceinline__ void finish_row(const RowsParams& P, long long r, float M, float S, const uint64_t* keys,
                                           int kept) {
  const int lane = threadIdx.x & 31;
  const int k = P.k;
  const float zmax = kept > 0 ? key_value(keys[0]) : -INFINITY;
  if (lane == 0 && (kept < k || zmax != M)) set_dev_error(P.ctrl, DART_DEVERR_ROW_MAX);
  // log S = e ln 2 + log f with S = f 2^e, f in [0.5, 1): the float log of
  // the mantissa is within about 1e-7 of its value
  int e2;
  const float f = frexpf(S, &e2);
  const double logS = fma(double(e2), 0.6931471805599453, double(logf(f)));
  if (lane < k) {
    const uint64_t key = lane < kept ? keys[lane] : 0ull;
    const float z = key_value(key);
    const int32_t id = int32_t(key_id(key));
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

// A whole row merged by one warp (rows beyond what one CTA merges from shared
// memory).  The headers come first: the pieces' (max, sum)
// combine into the row's (a fixed shuffle tree over the pieces' running
// pairs), and the bound is the largest piece bound or, with k or more pieces
// (up to 64), the k-th largest piece maximum if that is higher.  Only pieces
// whose maximum reaches the bound can hold one of the k best; their entries
// are gathered (eight per lane per round trip) and the keys of the elements
// that reach the bound go through the warp's key stage, the k best kept
// whenever it could overflow.  `lists` holds 2 * kMergeSel + 1 ints.
// The k-th largest of the warp's values (two per lane, ordered floats; 0 =
// no value), or 0 when fewer than k are nonzero: k rounds of a warp maximum,
// each removing one occurrence of the value it found.  Registers only.
__device__ __forceinline__ uint32_t warp_kth_largest2(uint32_t v0, uint32_t v1, int k) {
  const int lane = threadIdx.x & 31;
  uint32_t m = 0;
  for (int i = 0; i < k; ++i) {
    m = __reduce_max_sync(kFull, v0 > v1 ? v0 : v1);
    if (m == 0u) return 0u;
    const uint32_t holder = __ballot_sync(kFull, v0 == m || v1 == m);
    if (lane == __ffs(holder) - 1) {
      if (v0 == m) v0 = 0u;
      else v1 = 0u;
    }
  }
  return m;
}

constexpr int kMergeSel = 256;   // selected pieces per gathering round

template <int DT>
__device__ __forceinline__ void stage_keys_of(uint64_t* wstage, uint64_t* best, int& nk, int k, const uint4& vv,
                                              uint32_t tag, uint32_t cm) {
  const int lane = threadIdx.x & 31;
  int added;
  const int pre = warp_prefix4(uint32_t(__popc(cm)), &added);
  if (added == 0) return;
  if (nk + added > kKeyStage) {
    // keep the k best of the stage (ranking), best first
    __syncwarp();
    for (int x = lane; x < nk; x += 32) {
      const uint64_t key = wstage[x];
      int rank = 0;
      for (int y = 0; y < nk; ++y) rank += wstage[y] > key ? 1 : 0;
      if (rank < k) best[rank] = key;
    }
    __syncwarp();
    nk = nk < k ? nk : k;
    for (int x = lane; x < nk; x += 32) wstage[x] = best[x];
    __syncwarp();
  }
  int at = nk + pre;
  while (cm) {
    const int el = __ffs(cm) - 1;
    cm &= cm - 1u;
    wstage[at++] = elem_key(Elem<DT>::elem(vv, el), (tag & 0xFFFFFFu) + uint32_t(el));
  }
  nk += added;
  __syncwarp();
}

template <int DT>
__device__ __noinline__ void merge_row_warp(const RowsParams& P, long long r, uint64_t* wstage, uint64_t* best,
                                            int* lists) {
  const long long v = r;
  const int lane = threadIdx.x & 31;
  const int k = P.k;
  long long wa;
  const int nseg = row_pieces(P, v, &wa);
  // headers: running (max, sum) per lane over its pieces, the largest bound;
  // pieces lane and lane + 32 keep their maxima for the k-th largest
  float mp = -FLT_MAX, sp = 0.f;
  uint32_t b = 0;
  uint32_t om[2] = {0u, 0u};
  for (int p0 = 0; p0 < nseg; p0 += 32) {
    const int p = p0 + lane;
    if (p < nseg) {
      const uint8_t* q = slot_of(P, v, p);
      const float m2 = __ldcg(reinterpret_cast<const float*>(q));
      const float s2 = __ldcg(reinterpret_cast<const float*>(q + 8));
      const uint32_t b2 = __ldcg(reinterpret_cast<const uint32_t*>(q + 16));
      const float M2 = fmaxf(mp, m2);
      sp = sp * ex2_approx((mp - M2) * P.c) + s2 * ex2_approx((m2 - M2) * P.c);
      mp = M2;
      b = max(b, b2);
      if (p0 < 64) om[p0 >> 5] = ord_f32(m2);
    }
  }
  // mp > -FLT_MAX only for lanes with a piece, so the ordered maximum is a real one
  const float Mx = unord_f32(__reduce_max_sync(kFull, ord_f32(mp)));
  b = __reduce_max_sync(kFull, b);
  float Sx = sp * ex2_approx((mp - Mx) * P.c);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Sx += __shfl_xor_sync(kFull, Sx, o);
  if (nseg >= k && nseg <= 64) {
    // the k-th largest piece maximum: k pieces each hold an element that high
    b = max(b, warp_kth_largest2(om[0], om[1], k));
  }
  const float tau = tau_value(b);
  const uint32_t otau = b;
  int* sel = lists;                    // selected pieces
  int* start = lists + kMergeSel;      // their first entry in the gathered range
  int nk = 0;
  int p0 = 0;
  while (p0 < nseg) {
    // select pieces whose maximum reaches the bound, up to kMergeSel of them
    int ns = 0, E = 0;
    for (; p0 < nseg && ns + 32 <= kMergeSel; p0 += 32) {
      const int p = p0 + lane;
      int cnt = 0;
      bool take = false;
      if (p < nseg) {
        const uint8_t* q = slot_of(P, v, p);
        cnt = int(min(__ldcg(reinterpret_cast<const uint32_t*>(q + 4)), uint32_t(P.cp)));
        take = cnt > 0 && ord_f32(__ldcg(reinterpret_cast<const float*>(q))) >= otau;
      }
      const uint32_t tm = __ballot_sync(kFull, take);
      // prefix of the taken pieces' counts (exclusive), lanes in order
      int incl = take ? cnt : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      const int excl = incl - (take ? cnt : 0);
      if (take) {
        const int at = ns + __popc(tm & ((1u << lane) - 1u));
        sel[at] = p;
        start[at] = E + excl;
      }
      ns += __popc(tm);
      E += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) start[ns] = E;
    __syncwarp();
    // gather the selected pieces' entries, eight per lane per round trip
    for (int e0 = 0; e0 < E; e0 += 256) {
      uint4 vv[8];
      uint32_t tg[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = e0 + u * 32 + lane;
        vv[u] = make_uint4(0u, 0u, 0u, 0u);
        tg[u] = 0u;
        if (e < E) {
          int lo = 0, hi = ns - 1;     // the selected piece holding entry e
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (start[mid] <= e) lo = mid;
            else hi = mid - 1;
          }
          const uint8_t* q = slot_of(P, v, sel[lo]);
          const int i = e - start[lo];
          vv[u] = __ldcg(slot_vecs(P, const_cast<uint8_t*>(q)) + i);
          tg[u] = __ldcg(slot_tags(P, const_cast<uint8_t*>(q)) + i);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int e = e0 + u * 32 + lane;
        const uint32_t cm = e < E ? vec_hits<DT>(vv[u], tg[u], tau) : 0u;
        stage_keys_of<DT>(wstage, best, nk, k, vv[u], tg[u], cm);
      }
    }
    __syncwarp();
  }
  for (int x = lane; x < nk; x += 32) {
    const uint64_t key = wstage[x];
    int rank = 0;
    for (int y = 0; y < nk; ++y) rank += wstage[y] > key ? 1 : 0;
    if (rank < k) best[rank] = key;
  }
  __syncwarp();
  finish_row(P, r, Mx, Sx, best, nk < k ? nk : k);
}

struct MergeSmem {
  float m[kMergePieces];
  float s[kMergePieces];
  uint32_t end[kMergePieces];   // the pieces' candidate counts
  uint32_t pb[kMergePieces];    // the pieces' bounds
  uint32_t bound;
  uint32_t nkeys;
  float M;
  float S;
  uint64_t keys[kMergeKeys];
  uint64_t best[kMaxK];
  int sel[kMergePieces];          // pieces whose maximum reaches the bound (rows of many entries)
  int start[kMergePieces + 1];    // their first entry in the gathered range
  int E;                          // entries of the selected pieces
  int nsel;                       // selected pieces
};

// One CTA per row: every piece's header and every candidate slot entry are
// loaded in one round (entries past a piece's count are dropped after), the
// row's bound follows from the headers, the keys of the candidate elements
// that reach it are appended in shared memory, and the row's k best are found
// by ranking (each key counts the keys above it).  A row with more than
// kMergePieces pieces, more entries than one round holds, or more than
// kMergeKeys such keys, is merged by one warp instead (inputs far from the
// streamed shapes).
template <int DT, int MINB>
__global__ void __launch_bounds__(kMergeThreads, MINB)
row_merge_kernel(const __grid_constant__ RowsParams P) {
  __shared__ MergeSmem M;
  __shared__ uint64_t wstage[kKeyStage];
  constexpr int kPer = 8;   // slot entries per thread in the one round
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long long r = blockIdx.x;
  long long wa;
  const int nseg = row_pieces(P, r, &wa);
  const int k = P.k;
  if (nseg <= kMergePieces) {
    // one round: headers (threads < nseg) and slot entries e = tid + u * T,
    // when one round holds them all; else the headers first, and then only
    // the entries of pieces whose maximum reaches the row's bound
    const bool one_round = nseg * P.cp <= kMergeThreads * kPer;
    if (tid < nseg) {
      uint8_t* q = slot_of(P, r, tid);
      M.m[tid] = __ldcg(reinterpret_cast<const float*>(q));
      M.s[tid] = __ldcg(reinterpret_cast<const float*>(q + 8));
      M.end[tid] = min(__ldcg(reinterpret_cast<const uint32_t*>(q + 4)), uint32_t(P.cp));
      M.pb[tid] = __ldcg(reinterpret_cast<const uint32_t*>(q + 16));
    }
    uint4 v[kPer];
    uint32_t tag[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = tid + u * kMergeThreads;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      tag[u] = 0u;
      if (one_round && e < nseg * P.cp) {
        const int p = e / P.cp, i = e - p * P.cp;
        uint8_t* q = slot_of(P, r, p);
        v[u] = __ldcg(slot_vecs(P, q) + i);
        tag[u] = __ldcg(slot_tags(P, q) + i);
      }
    }
    if (tid == 0) M.nkeys = 0u;
    __syncthreads();
    if (warp == 0) {
      // max, sum (a fixed shuffle tree) and the bound: the largest piece
      // bound, and the k-th largest piece maximum; pieces lane and lane + 32
      const bool h0 = lane < nseg, h1 = lane + 32 < nseg;
      const float m0 = h0 ? M.m[lane] : -FLT_MAX, m1 = h1 ? M.m[lane + 32] : -FLT_MAX;
      uint32_t b = max(h0 ? M.pb[lane] : 0u, h1 ? M.pb[lane + 32] : 0u);
      // (every row has a piece, so the ordered maximum is a real one)
      const float mx = unord_f32(__reduce_max_sync(kFull, ord_f32(fmaxf(m0, m1))));
      float sum = (h0 ? M.s[lane] * ex2_approx((m0 - mx) * P.c) : 0.f) +
                  (h1 ? M.s[lane + 32] * ex2_approx((m1 - mx) * P.c) : 0.f);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
      if (nseg >= k) {
        // the k-th largest piece maximum: of the lane's two maxima, one with
        // fewer than k pieces above it and at least k at or above it (the
        // lane counts over all the maxima, broadcast reads of shared memory)
        const uint32_t o0 = h0 ? ord_f32(m0) : 0u, o1 = h1 ? ord_f32(m1) : 0u;
        int a0 = 0, t0 = 0, a1 = 0, t1 = 0;
        for (int q = 0; q < nseg; ++q) {
          const uint32_t y = ord_f32(M.m[q]);
          a0 += y > o0 ? 1 : 0;
          t0 += y >= o0 ? 1 : 0;
          a1 += y > o1 ? 1 : 0;
          t1 += y >= o1 ? 1 : 0;
        }
        if (h0 && a0 < k && t0 >= k) b = max(b, o0);
        if (h1 && a1 < k && t1 >= k) b = max(b, o1);
      }
      b = __reduce_max_sync(kFull, b);
      if (lane == 0) {
        M.M = mx;
        M.S = sum;
        M.bound = b;
      }
      if (!one_round) {
        // the pieces that can hold one of the k best, in piece order, and
        // where their entries start in the gathered range: bit-sliced
        // prefix sums of the counts (independent ballots, no scan chain)
        const bool t0 = h0 && M.end[lane] > 0u && ord_f32(m0) >= b;
        const bool t1 = h1 && M.end[lane + 32] > 0u && ord_f32(m1) >= b;
        int tot0, tot1;
        const int i0 = warp_prefix8(t0 ? M.end[lane] : 0u, &tot0);
        const int i1 = warp_prefix8(t1 ? M.end[lane + 32] : 0u, &tot1);
        const uint32_t bm0 = __ballot_sync(kFull, t0), bm1 = __ballot_sync(kFull, t1);
        const uint32_t below = (1u << lane) - 1u;
        if (t0) {
          const int at = __popc(bm0 & below);
          M.sel[at] = lane;
          M.start[at] = i0;
        }
        if (t1) {
          const int at = __popc(bm0) + __popc(bm1 & below);
          M.sel[at] = lane + 32;
          M.start[at] = tot0 + i1;
        }
        if (lane == 0) {
          const int ns = __popc(bm0) + __popc(bm1);
          M.E = tot0 + tot1;
          M.start[ns] = tot0 + tot1;
          M.nsel = ns;
        }
      }
    }
    __syncthreads();
    const float tau = tau_value(M.bound);
    const int entries = one_round ? nseg * P.cp : M.E;
    for (int base = 0; base < entries; base += kMergeThreads * kPer) {
      if (!one_round) {   // gathered entries of the selected pieces
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int e = base + tid + u * kMergeThreads;
          v[u] = make_uint4(0u, 0u, 0u, 0u);
          tag[u] = 0u;
          if (e < entries) {
            int lo = 0, hi = M.nsel - 1;    // the selected piece holding entry e
            while (lo < hi) {
              const int mid = (lo + hi + 1) >> 1;
              if (M.start[mid] <= e) lo = mid;
              else hi = mid - 1;
            }
            uint8_t* q = slot_of(P, r, M.sel[lo]);
            const int i = e - M.start[lo];
            v[u] = __ldcg(slot_vecs(P, q) + i);
            tag[u] = __ldcg(slot_tags(P, q) + i);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int e = base + tid + u * kMergeThreads;
        if (e >= entries) continue;
        if (one_round) {
          const int p = e / P.cp, i = e - p * P.cp;
          if (uint32_t(i) >= M.end[p]) continue;   // past the piece's count
        }
        uint32_t cm = vec_hits<DT>(v[u], tag[u], tau);
        if (cm) {
          uint32_t at = atomicAdd(&M.nkeys, uint32_t(__popc(cm)));
          while (cm) {
            const int el = __ffs(cm) - 1;
            cm &= cm - 1u;
            if (at < uint32_t(kMergeKeys))
              M.keys[at] = elem_key(Elem<DT>::elem(v[u], el), (tag[u] & 0xFFFFFFu) + uint32_t(el));
            ++at;
          }
        }
      }
    }
    __syncthreads();
    const uint32_t n = M.nkeys;
    if (n <= uint32_t(kMergeKeys)) {
      for (uint32_t i = tid; i < n; i += kMergeThreads) {
        const uint64_t key = M.keys[i];
        int rank = 0;
        for (uint32_t q2 = 0; q2 < n; ++q2) rank += M.keys[q2] > key ? 1 : 0;
        if (rank < k) M.best[rank] = key;
      }
      __syncthreads();
      if (warp == 0) finish_row(P, r, M.M, M.S, M.best, int(n < uint32_t(k) ? n : uint32_t(k)));
      return;
    }
  }
  // one warp, any number of pieces and keys
  if (warp != 0) return;
  merge_row_warp<DT>(P, r, wstage, M.best, reinterpret_cast<int*>(M.keys));
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

static bool rows_params(RowsParams* Pp, const void* logits, long long R, int V, long long stride, int dtype, float T,
                        int k, void* ws, const WsLayout& L, int32_t* out_ids, float* out_logp, float* out_lse) {
  RowsParams& P = *Pp;
  const int es = dtype == DART_F32 ? 4 : 2;
  P.logits = static_cast<const uint8_t*>(logits);
  P.R = R;
  P.V = V;
  P.stride = (unsigned long long)stride;
  P.k = k;
  P.es = es;
  P.invT = 1.0 / double(T);
  P.c = float(1.4426950408889634 / double(T));
  // the stream ends at the last valid element (the last row's padding may be absent)
  P.total = R > 0 ? ((unsigned long long)(R - 1) * P.stride + (unsigned long long)V) * (unsigned long long)es : 0ull;
  // spans of the fixed nominal grid; padded rows only make them longer, so
  // a row never has more pieces than the layout's slots
  P.wspan = row_pass_span(P.total);
  if (P.wspan < L.wspan) return false;
  P.pmax = L.pmax;
  P.cp = L.cp;
  P.slot_bytes = L.slot_bytes;
  uint8_t* w = static_cast<uint8_t*>(ws);
  P.ctrl = reinterpret_cast<uint32_t*>(w + L.ctrl);
  P.slots = w + L.slots;
  P.row_off = reinterpret_cast<double*>(w + L.row_off);
  P.row_ids = reinterpret_cast<int32_t*>(w + L.row_ids);
  P.row_base = reinterpret_cast<double*>(w + L.row_base);
  P.out_ids = out_ids;
  P.out_logp = out_logp;
  P.out_lse = out_lse;
  P.wait_limit = rows_wait_limit();
  P.spread = 0;
  return true;
}

cudaError_t launch_row_pass(const void* logits, long long R, int V, long long stride, int dtype, float T, int k,
                            void* ws, const WsLayout& L, cudaStream_t stream) {
  RowsParams P;
  if (!rows_params(&P, logits, R, V, stride, dtype, T, k, ws, L, nullptr, nullptr, nullptr))
    return cudaErrorInvalidValue;
  if (P.total == 0) return cudaSuccess;
  const unsigned long long warps = (P.total + P.wspan - 1) / P.wspan;
  unsigned long long grid = (warps + kRowWarps - 1) / kRowWarps;
  constexpr unsigned long long kSMs = kRowPassWarps / kRowWarps;   // the grid the spans are sized for
  if (grid < kSMs) {
    // fewer spans than CTAs x warps: one CTA per SM, the spans dealt round-robin
    P.spread = 1;
    grid = warps < kSMs ? warps : kSMs;
  }
  const size_t smem = rows_smem_bytes();
  cudaError_t e = cudaSuccess;
  auto go = [&](auto kernel) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e == cudaSuccess) kernel<<<unsigned(grid), kRowThreads, smem, stream>>>(P);
  };
  if (dtype == DART_F32) go(row_stream_kernel<DART_F32>);
  else if (dtype == DART_F16) go(row_stream_kernel<DART_F16>);
  else go(row_stream_kernel<DART_BF16>);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_row_merge(long long R, int V, long long stride, int dtype, float T, int k, void* ws,
                             const WsLayout& L, int32_t* out_ids, float* out_logp, float* out_lse,
                             cudaStream_t stream) {
  RowsParams P;
  if (!rows_params(&P, nullptr, R, V, stride, dtype, T, k, ws, L, out_ids, out_logp, out_lse))
    return cudaErrorInvalidValue;
  if (R == 0) return cudaSuccess;
  // more rows than four CTAs per SM: the build held to 64 registers, so that
  // eight CTAs share an SM and the rows take fewer waves (a few spilled
  // registers make it slower when the rows fit one wave anyway)
  const int sms = device_sms();
  const bool dense = sms > 0 && R > 4LL * sms;
  auto go = [&](auto kernel) { kernel<<<unsigned(R), kMergeThreads, 0, stream>>>(P); };
  if (dtype == DART_F32) dense ? go(row_merge_kernel<DART_F32, 8>) : go(row_merge_kernel<DART_F32, 1>);
  else if (dtype == DART_F16) dense ? go(row_merge_kernel<DART_F16, 8>) : go(row_merge_kernel<DART_F16, 1>);
  else dense ? go(row_merge_kernel<DART_BF16, 8>) : go(row_merge_kernel<DART_BF16, 1>);
  return cudaGetLastError();
}

cudaError_t launch_rows(const void* logits, long long R, int V, long long stride, int dtype, float T, int k,
                        void* ws, const WsLayout& L,
                        int32_t* out_ids, float* out_logp, float* out_lse, cudaStream_t stream) {
  cudaError_t e = launch_row_pass(logits, R, V, stride, dtype, T, k, ws, L, stream);
  if (e != cudaSuccess) return e;
  return launch_row_merge(R, V, stride, dtype, T, k, ws, L, out_ids, out_logp, out_lse, stream);
}

}  // namespace dart
