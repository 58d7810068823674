// dart_rows.cu -- K1: one streaming pass over the logits computing, per row,
// the temperature log-sum-exp and the k best candidates.
//
// DART, Figure 3 caption: each of the d logit vectors of a sequence supplies
// the candidates of one depth.  Here every row z[b][j][:] is read exactly once
// from HBM and reduced to (max, sum of exp((z - max) / T), k best (z, id)).
//
// Work split.  The logits are one flat byte stream.  Each warp owns one
// contiguous, 16-byte-aligned span of it (equal spans, so every warp moves the
// same number of bytes) and streams that span through its own ring of shared
// memory stages filled by cp.async.bulk (one elected lane issues, an mbarrier
// per stage counts the bytes).  A span cuts rows into segments; every segment
// yields a partial (running max, scaled sum, top-k keys).  The last warp to
// finish a row (an arrival counter, no waiting) merges that row's partials and
// writes the row's results.  No warp ever waits on another warp.
//
// Per stage a lane holds four 16-byte vectors.  One running-max update covers
// all of them (maxima taken on packed bf16x2 / f16x2 words), the exponentials
// use packed f32x2 subtract / multiply and accumulate, and one warp vote
// decides whether any element can enter the top-k.
//
// Top-k.  Candidates are 64-bit keys (ordered value, then inverted id), so a
// larger key is a better candidate and equal values fall back to the lower id.
// A warp keeps its best 32 keys spread over its lanes.  An element can only
// matter if it is >= tau, a lower bound of the row's k-th value: the k-th best
// key value the warp has merged, the k-th largest of the 32 lane maxima of the
// segment's first stage, or any value another warp of the same row published.
// Qualifying elements are appended to a per-warp buffer (slots from a shared
// counter); every 32 buffered keys are bitonic-sorted and merged into the list.
#include "dart_common.cuh"

#include <cfloat>

namespace dart {

constexpr int kRowWarps = 16;                   // 16 independent streams per CTA, one CTA per SM
constexpr int kStageBytes = 2048;               // one stage = 4 vectors of 16 B per lane
constexpr int kStages = 4;                      // 8 KB in flight per warp, 128 KB per SM
constexpr int kVecPerLane = kStageBytes / 16 / 32;
constexpr int kBufCap = 32 + 256 + 32;

struct RowsParams {
  const uint8_t* logits;
  long long R;
  int V, k, es;
  float c;                    // log2(e) / T
  double T;
  unsigned long long total;   // R * V * es bytes
  unsigned long long span;    // bytes per warp, multiple of 16
  int nwarps, grid;
  int pmax, pstride;
  uint32_t* ctrl;
  uint32_t* row_cnt;
  uint32_t* row_tau;
  uint8_t* partials;
  double* row_off;
  int32_t* row_ids;
  double* row_base;
  int32_t* out_ids;   // optional [R][k]
  float* out_logp;    // optional [R][k]
  float* out_lse;     // optional [R]
  long long wait_limit;
};

struct __align__(128) WarpSmem {
  uint8_t ring[kStages][kStageBytes];
  uint64_t buf[kBufCap];
  uint64_t bar[kStages];
  int nbuf;
};

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
  __device__ static uint4 neg_inf() { return make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u); }
  __device__ static float2 pair(const uint4& r, int p) {
    return make_float2(__uint_as_float(word(r, 2 * p)), __uint_as_float(word(r, 2 * p + 1)));
  }
  __device__ static float vmax(const uint4& r) {
    return fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)),
                 fmaxf(__uint_as_float(r.z), __uint_as_float(r.w)));
  }
  __device__ static float scalar(const uint8_t* p) { return __ldg(reinterpret_cast<const float*>(p)); }
};
template <> struct Elem<DART_BF16> {
  static constexpr int kPerVec = 8;
  __device__ static uint4 neg_inf() { return make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u); }
  __device__ static float2 pair(const uint4& r, int p) {
    const uint32_t w = word(r, p);
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  }
  __device__ static float vmax(const uint4& r) {
    const uint32_t m = bmax2(bmax2(r.x, r.y), bmax2(r.z, r.w));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
  }
  __device__ static float scalar(const uint8_t* p) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(p));
    return __uint_as_float(uint32_t(h) << 16);
  }
};
template <> struct Elem<DART_F16> {
  static constexpr int kPerVec = 8;
  __device__ static uint4 neg_inf() { return make_uint4(0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u); }
  __device__ static float2 pair(const uint4& r, int p) {
    const uint32_t w = word(r, p);
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
  }
  __device__ static float vmax(const uint4& r) {
    const uint32_t m = hmax2(hmax2(r.x, r.y), hmax2(r.z, r.w));
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&m));
    return fmaxf(f.x, f.y);
  }
  __device__ static float scalar(const uint8_t* p) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(p));
    return __half2float(__ushort_as_half(h));
  }
};

// Per-warp running state for one row segment.
struct SegState {
  float m, s;        // per lane: running max of z and sum of 2^((z - m) c)
  uint64_t list;     // per lane: entry `lane` of the warp's best 32 keys (desc)
  uint32_t tau_ord;  // ordered form of the filter threshold (0 = none yet)
  float tau;         // filter threshold value (-inf = none yet)
  int nbuf;          // keys waiting in the buffer (warp-uniform copy of WarpSmem::nbuf)
};

__device__ __forceinline__ void update_tau(SegState& st, int k, uint32_t* tau_slot) {
  const uint64_t kth = __shfl_sync(0xFFFFFFFFu, st.list, k - 1);
  const uint32_t o = uint32_t(kth >> 32);
  if (kth != 0 && o > st.tau_ord) {
    uint32_t old = 0;
    if ((threadIdx.x & 31) == 0) old = atomicMax(tau_slot, o);
    old = __shfl_sync(0xFFFFFFFFu, old, 0);
    st.tau_ord = o > old ? o : old;
    st.tau = unord_f32(st.tau_ord);
  }
}

// After lanes appended keys through the shared counter: pick up the count and
// merge whole chunks of 32 into the list.
__device__ __forceinline__ void after_push(SegState& st, WarpSmem& S, int k, uint32_t* tau_slot) {
  const int lane = threadIdx.x & 31;
  __syncwarp();
  st.nbuf = *reinterpret_cast<volatile int*>(&S.nbuf);
  if (st.nbuf >= 32) {
    while (st.nbuf >= 32) {
      const uint64_t chunk = S.buf[st.nbuf - 32 + lane];
      st.list = warp_merge_top32(st.list, chunk);
      st.nbuf -= 32;
    }
    __syncwarp();
    if (lane == 0) S.nbuf = st.nbuf;
    __syncwarp();
    update_tau(st, k, tau_slot);
  }
}

// k-th largest of the lanes' maxima: k distinct elements of this row are at
// least that large, so it is a lower bound of the row's k-th value.
__device__ __forceinline__ void seed_tau(SegState& st, float vm, bool valid, int k, uint32_t* tau_slot) {
  uint64_t key = valid ? (uint64_t(ord_f32(vm)) << 32) : 0ull;
  key = warp_sort_desc_u64(key);
  const uint64_t kth = __shfl_sync(0xFFFFFFFFu, key, k - 1);
  const uint32_t o = uint32_t(kth >> 32);
  if (kth != 0 && o > st.tau_ord) {
    st.tau_ord = o;
    st.tau = unord_f32(o);
    if ((threadIdx.x & 31) == 0) atomicMax(tau_slot, o);
  }
}

// One unaligned element per lane (head or tail of a segment).
__device__ __forceinline__ void consume_scalar(SegState& st, WarpSmem& S, float z, bool valid,
                                               uint32_t id, float c, int k, uint32_t* tau_slot) {
  if (valid) {
    if (z > st.m) {
      st.s *= ex2_approx((st.m - z) * c);
      st.m = z;
    }
    st.s += ex2_approx((z - st.m) * c);
  }
  const bool h = valid && z >= st.tau;
  if (__any_sync(0xFFFFFFFFu, h)) {
    if (h) {
      const int pos = atomicAdd(&S.nbuf, 1);
      S.buf[pos] = elem_key(z, id);
    }
    after_push(st, S, k, tau_slot);
  }
}

// One stage from shared memory: vector v = u*32 + lane (u < kVecPerLane) holds
// elements id_base + v*EPV ...; vectors at or past nvec are absent.
template <int DT>
__device__ __forceinline__ void consume_stage(SegState& st, WarpSmem& S, const uint4* ring, int nvec,
                                              uint32_t id_base, float c, int k, uint32_t* tau_slot,
                                              bool seed) {
  using E = Elem<DT>;
  constexpr int EPV = E::kPerVec;
  constexpr int U = kVecPerLane;
  const int lane = threadIdx.x & 31;
  uint4 raw[U];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int v = u * 32 + lane;
    raw[u] = v < nvec ? ring[v] : E::neg_inf();
  }
  float vmu[U];
#pragma unroll
  for (int u = 0; u < U; ++u) vmu[u] = E::vmax(raw[u]);
  float vm = vmu[0];
#pragma unroll
  for (int u = 1; u < U; ++u) vm = fmaxf(vm, vmu[u]);
  const bool lane_valid = lane < nvec;
  if (seed) seed_tau(st, vm, lane_valid, k, tau_slot);
  if (vm > st.m) {
    st.s *= ex2_approx((st.m - vm) * c);
    st.m = vm;
  }
  const float2 nm2 = make_float2(-st.m, -st.m);
  const float2 c2 = make_float2(c, c);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int u = 0; u < U; ++u) {
#pragma unroll
    for (int p = 0; p < EPV / 2; ++p) {
      const float2 t = __fmul2_rn(__fadd2_rn(E::pair(raw[u], p), nm2), c2);
      acc = __fadd2_rn(acc, make_float2(ex2_approx(t.x), ex2_approx(t.y)));
    }
  }
  st.s += acc.x + acc.y;
  // absent vectors hold -inf, which must not pass while tau is still -inf
  if (__any_sync(0xFFFFFFFFu, lane_valid && vm >= st.tau)) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const bool h = (u * 32 + lane < nvec) && vmu[u] >= st.tau;
      if (__any_sync(0xFFFFFFFFu, h)) {
        if (h) {
          const uint32_t id0 = id_base + uint32_t((u * 32 + lane) * EPV);
#pragma unroll
          for (int p = 0; p < EPV / 2; ++p) {
            const float2 z = E::pair(raw[u], p);
            if (z.x >= st.tau) {
              const int pos = atomicAdd(&S.nbuf, 1);
              S.buf[pos] = elem_key(z.x, id0 + 2 * p);
            }
            if (z.y >= st.tau) {
              const int pos = atomicAdd(&S.nbuf, 1);
              S.buf[pos] = elem_key(z.y, id0 + 2 * p + 1);
            }
          }
        }
        after_push(st, S, k, tau_slot);
      }
    }
  }
}

struct Seg {
  unsigned long long s0, s1;  // flat element range
  unsigned long long a, b;    // aligned interior, bytes (a == b: none)
};

__device__ __forceinline__ Seg segment(const RowsParams& P, unsigned long long e0, unsigned long long e1,
                                       long long r) {
  Seg g;
  const unsigned long long rs = (unsigned long long)r * P.V;
  g.s0 = e0 > rs ? e0 : rs;
  const unsigned long long re = rs + P.V;
  g.s1 = e1 < re ? e1 : re;
  g.a = (g.s0 * P.es + 15) & ~15ull;
  g.b = (g.s1 * P.es) & ~15ull;
  if (g.a >= g.b) g.a = g.b = g.s1 * P.es;  // nothing aligned: all scalars
  return g;
}

__device__ __forceinline__ void merge_row(const RowsParams& P, long long r, int nseg) {
  const int lane = threadIdx.x & 31;
  const int k = P.k;
  const uint8_t* base = P.partials + (size_t)r * P.pmax * P.pstride;
  // maximum over the partials
  float M = -FLT_MAX;
  for (int p = lane; p < nseg; p += 32)
    M = fmaxf(M, __ldcg(reinterpret_cast<const float*>(base + (size_t)p * P.pstride)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
  // sum of the partial sums rescaled to M, accumulated in double
  double S = 0.0;
  uint64_t tstar = 0;
  for (int p = lane; p < nseg; p += 32) {
    const uint8_t* q = base + (size_t)p * P.pstride;
    const float mp = __ldcg(reinterpret_cast<const float*>(q));
    const float sp = __ldcg(reinterpret_cast<const float*>(q + 4));
    S += double(sp) * double(ex2_approx((mp - M) * P.c));
    const uint64_t kth = __ldcg(reinterpret_cast<const unsigned long long*>(q + 16) + (k - 1));
    tstar = kth > tstar ? kth : tstar;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    S += __shfl_xor_sync(0xFFFFFFFFu, S, o);
    const uint64_t t = __shfl_xor_sync(0xFFFFFFFFu, tstar, o);
    tstar = t > tstar ? t : tstar;
  }
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
  const float zmax = key_value(__shfl_sync(0xFFFFFFFFu, list, 0));
  if (lane == 0 && zmax != M) set_dev_error(P.ctrl, DART_DEVERR_ROW_MAX);
  const double logS = log(S);
  if (lane < k) {
    const float z = key_value(list);
    const int32_t id = int32_t(key_id(list));
    P.row_ids[(size_t)r * k + lane] = id;
    P.row_base[(size_t)r * k + lane] = double(z);
    if (P.out_ids) P.out_ids[(size_t)r * k + lane] = id;
    if (P.out_logp) P.out_logp[(size_t)r * k + lane] = float((double(z) - double(zmax)) / P.T - logS);
  }
  if (lane == 0) {
    const double lse = double(zmax) / P.T + logS;
    P.row_off[r] = lse;
    if (P.out_lse) P.out_lse[r] = float(lse);
  }
}

template <int DT>
__global__ void __launch_bounds__(kRowWarps * 32, 1)
row_stream_kernel(const RowsParams P) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int gw = wib * P.grid + blockIdx.x;
  if (gw >= P.nwarps) return;
  WarpSmem& S = reinterpret_cast<WarpSmem*>(smem_raw)[wib];

  const unsigned long long B0 = (unsigned long long)gw * P.span;
  const unsigned long long B1 = (B0 + P.span < P.total) ? B0 + P.span : P.total;
  const unsigned long long e0 = B0 / P.es, e1 = B1 / P.es;
  const long long r_first = (long long)(e0 / P.V);
  const long long r_last = (long long)((e1 - 1) / P.V);

  if (lane == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&S.bar[i], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t pol = policy_evict_first();

  // producer cursor over (row segment, stage) in stream order
  long long pr = r_first;
  unsigned long long poff = 0, pend = 0;
  bool pvalid = false;
  auto prod_seek = [&](long long r) {
    pvalid = false;
    for (; r <= r_last; ++r) {
      const Seg g = segment(P, e0, e1, r);
      if (g.a < g.b) { pr = r; poff = g.a; pend = g.b; pvalid = true; return; }
    }
  };
  long long issued = 0;
  auto prod_issue = [&]() {
    const int slot = int(issued % kStages);
    const uint32_t bytes = uint32_t((pend - poff) < (unsigned long long)kStageBytes ? (pend - poff) : kStageBytes);
    if (lane == 0) {
      mbar_expect_tx(&S.bar[slot], bytes);
      bulk_g2s(S.ring[slot], P.logits + poff, bytes, &S.bar[slot], pol);
    }
    ++issued;
    poff += bytes;
    if (poff >= pend) prod_seek(pr + 1);
  };
  prod_seek(r_first);
  for (int i = 0; i < kStages && pvalid; ++i) prod_issue();

  long long consumed = 0;
  bool aborted = false;
  for (long long r = r_first; r <= r_last && !aborted; ++r) {
    const Seg g = segment(P, e0, e1, r);
    const unsigned long long rs = (unsigned long long)r * P.V;
    uint32_t* tau_slot = P.row_tau + r;
    SegState st;
    st.m = -FLT_MAX;
    st.s = 0.f;
    st.list = 0;
    st.nbuf = 0;
    st.tau_ord = __ldcg(tau_slot);
    st.tau = st.tau_ord ? unord_f32(st.tau_ord) : -INFINITY;
    if (lane == 0) S.nbuf = 0;
    __syncwarp();

    // head: [s0, a) (or the whole segment when nothing is aligned)
    {
      const unsigned long long hb0 = g.s0 * P.es;
      const unsigned long long hb1 = (g.a < g.b) ? g.a : g.s1 * P.es;
      const int cnt = int((hb1 - hb0) / P.es);
      for (int base = 0; base < cnt; base += 32) {
        const int i = base + lane;
        const bool valid = i < cnt;
        const float z = valid ? Elem<DT>::scalar(P.logits + hb0 + (unsigned long long)i * P.es) : -INFINITY;
        consume_scalar(st, S, z, valid, uint32_t(g.s0 - rs) + uint32_t(i), P.c, P.k, tau_slot);
      }
    }
    // aligned interior through the ring
    bool first_stage = true;
    for (unsigned long long off = g.a; off < g.b; off += kStageBytes) {
      const uint32_t bytes = uint32_t((g.b - off) < (unsigned long long)kStageBytes ? (g.b - off) : kStageBytes);
      const int slot = int(consumed % kStages);
      const uint32_t parity = uint32_t((consumed / kStages) & 1);
      if (!mbar_wait_bounded(&S.bar[slot], parity, P.wait_limit)) {
        aborted = true;
        break;
      }
      consume_stage<DT>(st, S, reinterpret_cast<const uint4*>(S.ring[slot]), int(bytes / 16),
                        uint32_t(off / P.es - rs), P.c, P.k, tau_slot, first_stage);
      first_stage = false;
      __syncwarp();
      ++consumed;
      if (pvalid) prod_issue();
    }
    if (aborted) break;
    // tail: [b, s1)
    if (g.a < g.b) {
      const unsigned long long tb0 = g.b, tb1 = g.s1 * P.es;
      const int cnt = int((tb1 - tb0) / P.es);
      for (int base = 0; base < cnt; base += 32) {
        const int i = base + lane;
        const bool valid = i < cnt;
        const float z = valid ? Elem<DT>::scalar(P.logits + tb0 + (unsigned long long)i * P.es) : -INFINITY;
        consume_scalar(st, S, z, valid, uint32_t(tb0 / P.es - rs) + uint32_t(i), P.c, P.k, tau_slot);
      }
    }
    // finish the segment: remaining buffer, cross-lane (max, sum)
    __syncwarp();
    st.nbuf = *reinterpret_cast<volatile int*>(&S.nbuf);
    if (st.nbuf > 0) {
      const uint64_t chunk = lane < st.nbuf ? S.buf[lane] : 0ull;
      st.list = warp_merge_top32(st.list, chunk);
      st.nbuf = 0;
    }
    float m = st.m, s = st.s;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
      const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
      const float M = fmaxf(m, m2);
      s = s * ex2_approx((m - M) * P.c) + s2 * ex2_approx((m2 - M) * P.c);
      m = M;
    }
    const unsigned long long rb0 = rs * P.es;
    const long long wfirst = (long long)(rb0 / P.span);
    const long long wlast = (long long)((rb0 + (unsigned long long)P.V * P.es - 1) / P.span);
    const int p = int(gw - wfirst);
    const int nseg = int(wlast - wfirst + 1);
    uint8_t* part = P.partials + ((size_t)r * P.pmax + p) * P.pstride;
    if (lane == 0) {
      reinterpret_cast<float*>(part)[0] = m;
      reinterpret_cast<float*>(part)[1] = s;
    }
    if (lane < P.k) reinterpret_cast<unsigned long long*>(part + 16)[lane] = st.list;
    __threadfence();
    __syncwarp();
    uint32_t old = 0;
    if (lane == 0) old = atomicAdd(P.row_cnt + r, 1u);
    old = __shfl_sync(0xFFFFFFFFu, old, 0);
    if (int(old) == nseg - 1) {
      __threadfence();
      merge_row(P, r, nseg);
    }
  }
  if (aborted) {
    if (lane == 0) set_dev_error(P.ctrl, DART_DEVERR_WAIT_TIMEOUT);
    // let copies still in flight land before the warp's shared memory is released
    for (long long q = consumed; q < issued; ++q) {
      const int slot = int(q % kStages);
      (void)mbar_wait_bounded(&S.bar[slot], uint32_t((q / kStages) & 1), P.wait_limit);
    }
  }
}

// ------------------------------------------------------------------ launch
size_t rows_smem_bytes() { return sizeof(WarpSmem) * kRowWarps; }

cudaError_t launch_rows(const void* logits, long long R, int V, int dtype, float T, int k,
                        void* ws, const WsLayout& L, int sms,
                        int32_t* out_ids, float* out_logp, float* out_lse, cudaStream_t stream) {
  RowsParams P;
  const int es = dtype == DART_F32 ? 4 : 2;
  P.logits = static_cast<const uint8_t*>(logits);
  P.R = R;
  P.V = V;
  P.k = k;
  P.es = es;
  P.T = double(T);
  P.c = float(1.4426950408889634 / double(T));
  P.total = (unsigned long long)R * (unsigned long long)V * (unsigned long long)es;
  const unsigned long long want = (P.total + (unsigned long long)sms * kRowWarps - 1) /
                                  ((unsigned long long)sms * kRowWarps);
  unsigned long long span = (want + 15) & ~15ull;
  if (span < kMinSpanBytes) span = kMinSpanBytes;
  P.span = span;
  P.nwarps = int((P.total + span - 1) / span);
  P.grid = P.nwarps < sms ? P.nwarps : sms;
  P.pmax = L.pmax;
  P.pstride = L.pstride;
  uint8_t* w = static_cast<uint8_t*>(ws);
  P.ctrl = reinterpret_cast<uint32_t*>(w + L.ctrl);
  P.row_cnt = reinterpret_cast<uint32_t*>(w + L.row_cnt);
  P.row_tau = reinterpret_cast<uint32_t*>(w + L.row_tau);
  P.partials = w + L.partials;
  P.row_off = reinterpret_cast<double*>(w + L.row_off);
  P.row_ids = reinterpret_cast<int32_t*>(w + L.row_ids);
  P.row_base = reinterpret_cast<double*>(w + L.row_base);
  P.out_ids = out_ids;
  P.out_logp = out_logp;
  P.out_lse = out_lse;
  P.wait_limit = 4000000000LL;  // about two seconds of SM clock
  if (P.total == 0) return cudaSuccess;
  const size_t smem = rows_smem_bytes();
  cudaError_t e = cudaSuccess;
  switch (dtype) {
    case DART_F32:
      e = cudaFuncSetAttribute(row_stream_kernel<DART_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (e == cudaSuccess) row_stream_kernel<DART_F32><<<P.grid, kRowWarps * 32, smem, stream>>>(P);
      break;
    case DART_F16:
      e = cudaFuncSetAttribute(row_stream_kernel<DART_F16>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (e == cudaSuccess) row_stream_kernel<DART_F16><<<P.grid, kRowWarps * 32, smem, stream>>>(P);
      break;
    default:
      e = cudaFuncSetAttribute(row_stream_kernel<DART_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
      if (e == cudaSuccess) row_stream_kernel<DART_BF16><<<P.grid, kRowWarps * 32, smem, stream>>>(P);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dart
