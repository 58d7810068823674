// dart_tree.cu -- K2: per-depth frontier expansion, n-gram scoring and top-W
// pruning (one CTA per tree), with the ancestor masks written as nodes are
// emitted; K3: ancestor masks from a parent array; the n-gram lookup kernel.
//
// DARTree, Method / Tree Construction: every frontier node is expanded in one
// batch and only the W best children of the whole frontier survive each depth.
// DART, Figure 3 caption: the N-gram model scores the continuity of each
// expanded token; the result feeds tree attention, which needs each node's
// ancestors (here one bit per node, LSB-first in 32-bit words).
//
// Per depth the CTA scores all n_j * k children at once (one thread per
// child: one hash probe, a few double adds), turns each into a 96-bit key
// (ordered ranking key, then inverted (parent rank, token rank)), sorts 32- or
// 64-key runs with warp bitonic networks and merges runs pairwise, keeping
// only the best run length, until one run holds the survivors in order.
#include <atomic>
#include "dart_launch.h"

namespace dart {

#include "dart_select.cuh"

constexpr int kTreeThreads = 512;
constexpr uint32_t kTieMax = 0xFFFFFu;      // (parent rank << 5 | token rank) < 2^11

struct CKey {
  uint64_t s;   // ordered ranking key
  uint32_t t;   // kTieMax - (parent rank << 5 | token rank): larger = lower parent, lower token
};

__device__ __forceinline__ bool ck_gt(const CKey& a, const CKey& b) {
  return a.s > b.s || (a.s == b.s && a.t > b.t);
}
__device__ __forceinline__ CKey ck_shfl_xor(const CKey& a, int m) {
  CKey r;
  r.s = __shfl_xor_sync(0xFFFFFFFFu, a.s, m);
  r.t = __shfl_xor_sync(0xFFFFFFFFu, a.t, m);
  return r;
}

// Bitonic sort of 32*R keys held R per lane (element e = r*32 + lane), descending.
template <int R>
__device__ __forceinline__ void run_sort(CKey (&v)[R]) {
  const int lane = threadIdx.x & 31;
  constexpr int n = 32 * R;
#pragma unroll
  for (int size = 2; size <= n; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 32) {
        // partner lives in the other register of this lane (R == 2, size == 64)
        if (R == 2) {
          CKey& lo = v[0];
          CKey& hi = v[R - 1];
          if (ck_gt(hi, lo)) { CKey t = lo; lo = hi; hi = t; }
        }
      } else {
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int e = r * 32 + lane;
          const CKey o = ck_shfl_xor(v[r], stride);
          const bool desc = (e & size) == 0;
          const bool lower = (e & stride) == 0;
          const bool keep_max = (lower == desc);
          const bool og = ck_gt(o, v[r]);
          if (keep_max == og) v[r] = o;
        }
      }
    }
  }
}

// Finishes a bitonic sequence of 32*R keys into descending order.
template <int R>
__device__ __forceinline__ void run_merge_desc(CKey (&v)[R]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int stride = 16 * R; stride > 0; stride >>= 1) {
    if (stride >= 32) {
      if (R == 2) {
        CKey& lo = v[0];
        CKey& hi = v[R - 1];
        if (ck_gt(hi, lo)) { CKey t = lo; lo = hi; hi = t; }
      }
    } else {
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const CKey o = ck_shfl_xor(v[r], stride);
        const bool lower = (lane & stride) == 0;
        const bool og = ck_gt(o, v[r]);
        if (lower == og) v[r] = o;
      }
    }
  }
}

// A lookup reads the key's two buckets (four slots, 64 bytes) at once, one
// 32-byte load each: one memory round trip whether the key is present or
// not.  probe_issue starts the loads; probe_match, called once the caller has
// done other work, compares.
static_assert(kBucketSlots == 2, "a bucket is one 32-byte load");
struct Probe { uint4 s[2 * kBucketSlots]; };
__device__ __forceinline__ void probe_issue(const uint4* slots, unsigned long long nb, Key96 key, Probe& pr) {
  const Buckets bk = key_buckets(key, nb);
  ldg_nc_v8(slots + kBucketSlots * bk.b1, pr.s[0], pr.s[1]);
  ldg_nc_v8(slots + kBucketSlots * bk.b2, pr.s[2], pr.s[3]);
}
__device__ __forceinline__ bool probe_match(const Probe& pr, Key96 key, float* val) {
  bool hit = false;
#pragma unroll
  for (int t = 0; t < 2 * kBucketSlots; ++t) {
    if (pr.s[t].x == key.w0 && pr.s[t].y == key.w1 && pr.s[t].z == key.w2) {
      *val = __uint_as_float(pr.s[t].w);
      hit = true;
    }
  }
  return hit;
}
__device__ __forceinline__ bool probe(const uint4* slots, unsigned long long nb, Key96 key, float* val) {
  Probe pr;
  probe_issue(slots, nb, key, pr);
  return probe_match(pr, key, val);
}

__host__ __device__ inline int tree_run_len(int W) { return W <= 32 ? 32 : 64; }
__host__ __device__ inline int tree_pad(int W, int k) {
  const int run = tree_run_len(W);
  return (W * k + run - 1) / run * run;
}
constexpr int kRankMax = 128;   // up to this many children a depth selects by ranking (more: sorted runs)
constexpr int kGroup = 2;       // sorted runs one warp folds together per merge round
// Threads per tree: one per child of a full frontier, 32..512; two per child
// when every depth selects by ranking and the trees fit one CTA per SM (then
// two threads rank each key against half of the keys).  Doubling for more
// trees than SMs would cost a second wave: at about 120 registers a thread
// an SM holds one CTA of 320 threads.
inline int tree_threads(int W, int k, int B, int sms) {
  int t = (W * k + 31) / 32 * 32;
  t = t < 32 ? 32 : (t > kTreeThreads ? kTreeThreads : t);
  if (W * k <= kRankMax && 2 * t <= kTreeThreads && B <= sms) t *= 2;
  return t;
}

int device_sms() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cache[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

inline size_t tree_smem_bytes(int d, int W, int k, int MW, int N, bool select) {
  const size_t np = size_t(tree_pad(W, k));
  const size_t dk = size_t(d) * k;
  size_t b = 0;
  b += 4 * kMaxW * sizeof(double);                // frontier Z and G (ping-pong)
  b += align_up(dk * sizeof(double), 16);         // candidate base values of every row
  b += align_up(size_t(d) * sizeof(double), 16);  // row offsets
  b += 4 * np * sizeof(uint64_t);                 // keys (ping-pong), candidate G (ping-pong)
  b += kMaxW * sizeof(uint64_t);                  // selected keys
  b += 2 * np * sizeof(uint32_t);                 // tie keys (ping-pong)
  b += kMaxW * sizeof(uint32_t);                  // selected tie keys
  b += 2 * kMaxW * sizeof(int);                   // frontier node ids
  b += 2 * kMaxW * 3 * sizeof(int);               // frontier n-gram contexts
  b += 2 * size_t(kMaxW) * MW * sizeof(uint32_t); // frontier mask rows
  b += 3 * align_up(dk * sizeof(int), 16);        // ids, token ranks, inverse ranks of every row
  if (select) b += select_shared_bytes(N);          // the verification tree's selection
  return b + 64;
}

// One row's candidate lists, with each candidate's rank by token id (ties on
// the ranking key fall to the lower token id, which is the lower token rank).
struct RowBuf {
  const int* rid;      // [k] token ids in list order
  const double* rb;    // [k] base values
  const int* rrank;    // [k] rank of rid[c] among the row's ids
  const int* rinv;     // [k] list position of the id with a given rank
};

// One CTA per tree.  A frontier node carries Z (sum of its candidates' base
// values) and G (sum of its continuity terms: n-gram values, or the caller's
// pair scores of (parent column, child column)); a child's ranking key is
// Z * invT + lam * G, accumulated in double exactly as the oracle does it, so
// equal keys (ties the inputs hold exactly) stay equal.  The reported score
// subtracts the rows' offsets (their log-sum-exp), which every node of one
// depth shares.  All d candidate rows are read once at the start.  A depth
// then selects its W best children -- by ranking (each child counts the keys
// that beat it) when there are at most kRankMax, else by sorting runs and
// merging them -- and each thread decodes one survivor's child straight from
// the selected list, writes that node's outputs and frontier state, and scores
// the child (one probe).
template <int R>
__global__ void __launch_bounds__(kTreeThreads)
tree_kernel(const TreeArgs A) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  constexpr int RUN = 32 * R;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int b = blockIdx.x;
  const int k = A.k, W = A.W, N = A.N, MW = A.MW, n = A.n, d = A.d;
  const int npad_max = tree_pad(W, k);
  const int dk = d * k;

  // carve shared memory (8-byte members first); every size is a multiple of 16
  uint8_t* p = smem_raw;
  auto take = [&](size_t bytes) { uint8_t* q = p; p += (bytes + 15) & ~size_t(15); return q; };
  double* fZ_a = reinterpret_cast<double*>(take(kMaxW * sizeof(double)));
  double* fZ_b = reinterpret_cast<double*>(take(kMaxW * sizeof(double)));
  double* fG_a = reinterpret_cast<double*>(take(kMaxW * sizeof(double)));
  double* fG_b = reinterpret_cast<double*>(take(kMaxW * sizeof(double)));
  double* rows_b = reinterpret_cast<double*>(take(size_t(dk) * sizeof(double)));
  double* offs = reinterpret_cast<double*>(take(size_t(d) * sizeof(double)));
  uint64_t* ks_a = reinterpret_cast<uint64_t*>(take(size_t(npad_max) * 8));
  uint64_t* ks_b = reinterpret_cast<uint64_t*>(take(size_t(npad_max) * 8));
  double* cG_a = reinterpret_cast<double*>(take(size_t(npad_max) * 8));
  double* cG_b = reinterpret_cast<double*>(take(size_t(npad_max) * 8));
  uint64_t* sel_s = reinterpret_cast<uint64_t*>(take(kMaxW * sizeof(uint64_t)));
  uint32_t* kt_a = reinterpret_cast<uint32_t*>(take(size_t(npad_max) * 4));
  uint32_t* kt_b = reinterpret_cast<uint32_t*>(take(size_t(npad_max) * 4));
  uint32_t* sel_t = reinterpret_cast<uint32_t*>(take(kMaxW * sizeof(uint32_t)));
  int* fnode_a = reinterpret_cast<int*>(take(kMaxW * sizeof(int)));
  int* fnode_b = reinterpret_cast<int*>(take(kMaxW * sizeof(int)));
  int* fctx_a = reinterpret_cast<int*>(take(kMaxW * 3 * sizeof(int)));
  int* fctx_b = reinterpret_cast<int*>(take(kMaxW * 3 * sizeof(int)));
  uint32_t* fmask_a = reinterpret_cast<uint32_t*>(take(size_t(kMaxW) * MW * 4));
  uint32_t* fmask_b = reinterpret_cast<uint32_t*>(take(size_t(kMaxW) * MW * 4));
  int* rows_id = reinterpret_cast<int*>(take(size_t(dk) * sizeof(int)));
  int* rows_rank = reinterpret_cast<int*>(take(size_t(dk) * sizeof(int)));
  int* rows_inv = reinterpret_cast<int*>(take(size_t(dk) * sizeof(int)));
  // the verification tree's selection (only with a budget)
  SelectShared S{nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  float* sel_score = nullptr;
  int32_t* sel_par = nullptr;
  if (A.M > 0) {
    S.key = reinterpret_cast<uint64_t*>(take(size_t(N) * 8));
    sel_score = reinterpret_cast<float*>(take(size_t(N) * 4));
    sel_par = reinterpret_cast<int32_t*>(take(size_t(N) * 4));
    S.fresh = reinterpret_cast<int32_t*>(take(size_t(N) * 4));
    S.npar = reinterpret_cast<int32_t*>(take(size_t(N) * 4));
    S.chunk = reinterpret_cast<uint32_t*>(take(size_t(kMaxN / 32) * 4));
    S.score = sel_score;
    S.parent = sel_par;
  }
  auto row = [&](int j) {
    RowBuf r;
    r.rid = rows_id + j * k;
    r.rb = rows_b + j * k;
    r.rrank = rows_rank + j * k;
    r.rinv = rows_inv + j * k;
    return r;
  };

  const uint4* slots = static_cast<const uint4*>(A.slots);
  const unsigned long long nbuckets = A.capacity / kBucketSlots;
  const int nctx = n > 1 ? n - 1 : 0;
  const double invT = A.invT, lam = A.lam;
  const bool unit_T = invT == 1.0;   // Z * 1 is Z itself: the multiply is skipped, the bits are the same
  // caller pair scores of this tree: [d][k][k], the parent's column first
  const float* pair = A.pair ? A.pair + (size_t)b * dk * k : nullptr;

  // child key of frontier entry (Zp, Gp, context ctx) with candidate c of row R
  auto child = [&](double Zp, double Gp, int x0, int x1, int x2, const RowBuf& Rw, int c, double* Gout) {
    const int tok = Rw.rid[c];
    const double Z = __dadd_rn(Zp, Rw.rb[c]);
    double G = Gp;
    if (n > 0) {
      int32_t t[4] = {x0, x1, x2, 0};
      if (nctx == 1) t[1] = tok;
      else if (nctx == 2) t[2] = tok;
      else t[3] = tok;
      float g = 0.f;
      const double gg = probe(slots, nbuckets, pack_ngram(t, n), &g) ? double(g) : A.beta;
      G = __dadd_rn(G, gg);
    } else if (pair) {
      G = __dadd_rn(G, double(__ldg(pair + c)));   // row 0: the root is column 0
    }
    *Gout = G;
    return __dadd_rn(unit_T ? Z : __dmul_rn(Z, invT), __dmul_rn(lam, G));
  };

  // ---- every row's candidates and offset, then their token ranks
  const size_t row0 = (size_t)b * dk;
  int rootctx[3] = {0, 0, 0};
#pragma unroll
  for (int f = 0; f < 3; ++f)
    if (f < nctx) rootctx[f] = A.ctx[(size_t)b * nctx + f];
  int tok0 = 0;   // thread q < k: candidate q of row 0, the root's child q
  for (int e = tid; e < dk; e += blockDim.x) {
    const int id = A.ids[row0 + e];
    rows_id[e] = id;
    rows_b[e] = A.base[row0 + e];
    if (e == tid) tok0 = id;
  }
  for (int j = tid; j < d; j += blockDim.x) offs[j] = A.off ? A.off[(size_t)b * d + j] : 0.0;
  // the root's children's lookups start now and land while the ranks are made
  Probe rp;
  Key96 rkey{0u, 0u, 0u};
  const bool root_probe = n > 0 && tid < k;
  if (root_probe) {
    int32_t t[4] = {rootctx[0], rootctx[1], rootctx[2], 0};
    if (nctx == 1) t[1] = tok0;
    else if (nctx == 2) t[2] = tok0;
    else t[3] = tok0;
    rkey = pack_ngram(t, n);
    probe_issue(slots, nbuckets, rkey, rp);
  }
  __syncthreads();
  for (int e = tid; e < dk; e += blockDim.x) {
    const int j = e / k, c = e - j * k;
    const int* ids = rows_id + j * k;
    const int t = ids[c];
    // equal ids (which valid inputs never hold) fall to their list order, so
    // the ranks stay a permutation and every child keeps a distinct tie key
    int r = 0;
    for (int c2 = 0; c2 < k; ++c2) r += (ids[c2] < t || (ids[c2] == t && c2 < c)) ? 1 : 0;
    rows_rank[e] = r;
    rows_inv[j * k + r] = c;
  }
  if (tid == 0) {
    // each depth's sum of row offsets, accumulated in depth order
    double acc = 0.0;
    for (int j = 0; j < d; ++j) {
      acc = __dadd_rn(acc, offs[j]);
      offs[j] = acc;
    }
  }
  __syncthreads();

  // ---- depth 1: the root's children
  uint64_t* keys = ks_a;     // unsorted keys of the current depth
  uint32_t* ties = kt_a;
  double* cG = cG_a;         // G of each current candidate
  {
    const RowBuf R0 = row(0);
    const int npad = (k + RUN - 1) / RUN * RUN;
    for (int q = tid; q < npad; q += blockDim.x) {
      uint64_t ks = 0;
      uint32_t kt = 0;
      if (q < k) {
        double G, key;
        if (root_probe && q == tid) {
          // as child() for the root (Z = 0 + base, G = 0 + g), on the lookup started above
          float g = 0.f;
          const double Z = __dadd_rn(0.0, R0.rb[q]);
          G = __dadd_rn(0.0, probe_match(rp, rkey, &g) ? double(g) : A.beta);
          key = __dadd_rn(unit_T ? Z : __dmul_rn(Z, invT), __dmul_rn(lam, G));
        } else {
          key = child(0.0, 0.0, rootctx[0], rootctx[1], rootctx[2], R0, q, &G);
        }
        cG[q] = G;
        ks = ord_f64(key);
        kt = kTieMax - uint32_t(R0.rrank[q]);             // parent rank 0
      }
      keys[q] = ks;
      ties[q] = kt;
    }
  }
  // frontier of the current depth: the root (only its context and mask are read)
  double* fZ_cur = fZ_a;
  double* fZ_nxt = fZ_b;
  double* fG_cur = fG_a;
  double* fG_nxt = fG_b;
  int* fnode_cur = fnode_a;
  int* fnode_nxt = fnode_b;
  int* fctx_cur = fctx_a;
  int* fctx_nxt = fctx_b;
  uint32_t* fmask_cur = fmask_a;
  uint32_t* fmask_nxt = fmask_b;
  if (tid == 0) {
    fZ_cur[0] = 0.0;
    fG_cur[0] = 0.0;
    fnode_cur[0] = -1;
    for (int f = 0; f < nctx; ++f) fctx_cur[f] = rootctx[f];
  }
  int nf = 1, node_base = 0;
  double Lsum = 0.0;   // sum of the row offsets down to this depth
  __syncthreads();

  for (int j = 0; j < d; ++j) {
    const RowBuf Rc = row(j);                      // row j: candidates of the children selected now
    const RowBuf Rn = row(j + 1 < d ? j + 1 : j);  // row j+1: candidates of the next depth
    Lsum = offs[j];
    const int m = nf * k;
    const int nsel = m < W ? m : W;
    const uint64_t* src_s;     // the nsel survivors, best first
    const uint32_t* src_t;
    uint64_t* ks_dst;          // keys of the next depth go here
    uint32_t* kt_dst;
    if (m <= kRankMax) {
      // rank: the number of keys better than mine (keys are distinct); at
      // depths with at most half as many children as threads, each key is
      // ranked by two threads against one half of the keys each
      const int parts = int(blockDim.x) >= 2 * m ? 2 : 1;
      if (warp * 32 < parts * m) {
        const int q0 = parts == 2 ? (tid >> 1) : tid;
        const int part = parts == 2 ? (tid & 1) : 0;
        const bool live = q0 < m;
        const uint64_t sq = live ? keys[q0] : 0ull;
        const uint32_t tq = live ? ties[q0] : 0u;
        int rank = 0;
        // eight keys per step from 16-byte loads; the zero padding up to a
        // multiple of 32 never beats a real key
        const ulonglong2* k2 = reinterpret_cast<const ulonglong2*>(keys);
        const uint4* t4 = reinterpret_cast<const uint4*>(ties);
        const int half = parts == 2 ? (m + 15) / 16 * 8 : m;
        const int lo = live ? part * half : 0, hi = live ? (part == 0 ? half : m) : 0;
        for (int q = lo; q < hi; q += 8) {
          const ulonglong2 a0 = k2[(q >> 1) + 0], a1 = k2[(q >> 1) + 1];
          const ulonglong2 a2 = k2[(q >> 1) + 2], a3 = k2[(q >> 1) + 3];
          const uint4 b0 = t4[(q >> 2) + 0], b1 = t4[(q >> 2) + 1];
          rank += (a0.x > sq || (a0.x == sq && b0.x > tq)) ? 1 : 0;
          rank += (a0.y > sq || (a0.y == sq && b0.y > tq)) ? 1 : 0;
          rank += (a1.x > sq || (a1.x == sq && b0.z > tq)) ? 1 : 0;
          rank += (a1.y > sq || (a1.y == sq && b0.w > tq)) ? 1 : 0;
          rank += (a2.x > sq || (a2.x == sq && b1.x > tq)) ? 1 : 0;
          rank += (a2.y > sq || (a2.y == sq && b1.y > tq)) ? 1 : 0;
          rank += (a3.x > sq || (a3.x == sq && b1.z > tq)) ? 1 : 0;
          rank += (a3.y > sq || (a3.y == sq && b1.w > tq)) ? 1 : 0;
        }
        if (parts == 2) rank += __shfl_xor_sync(0xFFFFFFFFu, rank, 1);
        if (live && part == 0 && rank < nsel) {
          sel_s[rank] = sq;
          sel_t[rank] = tq;
        }
      }
      __syncthreads();
      src_s = sel_s;
      src_t = sel_t;
      ks_dst = (keys == ks_a) ? ks_b : ks_a;
      kt_dst = (ties == kt_a) ? kt_b : kt_a;
    } else {
      const int npad = (m + RUN - 1) / RUN * RUN;
      // sort runs of RUN keys, one warp per run
      int nr = npad / RUN;
      for (int run = warp; run < nr; run += nwarps) {
        CKey v[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int e = run * RUN + r * 32 + lane;
          v[r].s = keys[e];
          v[r].t = ties[e];
        }
        run_sort<R>(v);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int e = run * RUN + r * 32 + lane;
          keys[e] = v[r].s;
          ties[e] = v[r].t;
        }
      }
      __syncthreads();
      // merge runs in groups of kGroup: each warp folds a group's runs into
      // one run in registers (the best RUN keys so far, merged with the next
      // run reversed), so a round costs one barrier for kGroup runs
      uint64_t* ks_src = keys;
      uint32_t* kt_src = ties;
      ks_dst = (keys == ks_a) ? ks_b : ks_a;
      kt_dst = (ties == kt_a) ? kt_b : kt_a;
      while (nr > 1) {
        const int nout = (nr + kGroup - 1) / kGroup;
        for (int t = warp; t < nout; t += nwarps) {
          CKey v[R];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int e = r * 32 + lane;
            v[r].s = ks_src[(t * kGroup) * RUN + e];
            v[r].t = kt_src[(t * kGroup) * RUN + e];
          }
          for (int f = 1; f < kGroup && t * kGroup + f < nr; ++f) {
            const int run = t * kGroup + f;
#pragma unroll
            for (int r = 0; r < R; ++r) {
              const int e = r * 32 + lane;
              CKey y;
              y.s = ks_src[run * RUN + (RUN - 1 - e)];
              y.t = kt_src[run * RUN + (RUN - 1 - e)];
              if (ck_gt(y, v[r])) v[r] = y;
            }
            run_merge_desc<R>(v);
          }
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int e = r * 32 + lane;
            ks_dst[t * RUN + e] = v[r].s;
            kt_dst[t * RUN + e] = v[r].t;
          }
        }
        __syncthreads();
        uint64_t* ts = ks_src; ks_src = ks_dst; ks_dst = ts;
        uint32_t* tt = kt_src; kt_src = kt_dst; kt_dst = tt;
        nr = nout;
      }
      src_s = ks_src;
      src_t = kt_src;
    }
    // survivors of depth j+1 are src[0..nsel); decode each one, emit it and
    // (unless this is the last depth) score its k children of row j+1
    const bool last = (j + 1 == d);
    const int kk = last ? 1 : k;
    const int m2 = nsel * kk;
    const int npad2 = last ? m2 : (m2 + RUN - 1) / RUN * RUN;
    double* cG_next = (cG == cG_a) ? cG_b : cG_a;
    for (int q = tid; q < npad2; q += blockDim.x) {
      uint64_t ks2 = 0;
      uint32_t kt2 = 0;
      if (q < m2) {
        const int x = q / kk;             // survivor rank = node index within the depth
        const int c2 = q - x * kk;        // its child column in row j+1
        const uint64_t ks = src_s[x];
        const uint32_t tie = kTieMax - src_t[x];
        int i = int(tie >> 5);
        int c = (i < nf) ? Rc.rinv[tie & 31u] : 0;
        if (ks == 0 || i >= nf) {
          set_dev_error(A.ctrl, DART_DEVERR_SELECT);
          i = 0;
          c = 0;
        }
        const int tok = Rc.rid[c];
        const int node = node_base + x;
        int ctx[3] = {0, 0, 0};
#pragma unroll
        for (int f = 0; f + 1 < 3; ++f)
          if (f + 1 < nctx) ctx[f] = fctx_cur[i * 3 + f + 1];
        if (nctx > 0) {
          if (nctx == 1) ctx[0] = tok;
          else if (nctx == 2) ctx[1] = tok;
          else ctx[2] = tok;
        }
        // start the lookup of child (x, c2) before the rest of the work
        Probe pr;
        Key96 ckey{0u, 0u, 0u};
        float pg = 0.f;
        if (!last && pair) pg = __ldg(pair + ((size_t)(j + 1) * k + c) * k + c2);
        if (!last && n > 0) {
          const int ctok = Rn.rid[c2];
          int32_t t[4] = {ctx[0], ctx[1], ctx[2], 0};
          if (nctx == 1) t[1] = ctok;
          else if (nctx == 2) t[2] = ctok;
          else t[3] = ctok;
          ckey = pack_ngram(t, n);
          probe_issue(slots, nbuckets, ckey, pr);
        }
        const double Zp = __dadd_rn(fZ_cur[i], Rc.rb[c]);
        const double Gp = cG[i * k + c];
        // ancestor-mask words of the node, spread over its k child threads
        for (int w = c2; w < MW; w += kk) {
          uint32_t val = (j == 0) ? 0u : fmask_cur[i * MW + w];
          if (w == (node >> 5)) val |= 1u << (node & 31);
          fmask_nxt[x * MW + w] = val;
          A.out_mask[((size_t)b * N + node) * MW + w] = val;
        }
        if (c2 == 0) {
          const size_t o = (size_t)b * N + node;
          A.out_tokens[o] = tok;
          A.out_parents[o] = j == 0 ? -1 : fnode_cur[i];
          A.out_pos[o] = j + 1;
          if (A.out_scores || A.M > 0) {
            const float sc = float(__dsub_rn(unord_f64(ks), Lsum));
            if (A.out_scores) A.out_scores[o] = sc;
            if (A.M > 0) {
              sel_score[node] = sc;
              sel_par[node] = j == 0 ? -1 : fnode_cur[i];
            }
          }
          fZ_nxt[x] = Zp;
          fG_nxt[x] = Gp;
          fnode_nxt[x] = node;
#pragma unroll
          for (int f = 0; f < 3; ++f)
            if (f < nctx) fctx_nxt[x * 3 + f] = ctx[f];
        }
        if (!last) {
          // key of child (x, c2): (Zp + base) * invT + lam * (Gp + g), as in child()
          const double Zc = __dadd_rn(Zp, Rn.rb[c2]);
          const double ZinvT = unit_T ? Zc : __dmul_rn(Zc, invT);
          double G = Gp;
          if (n > 0) {
            float g = 0.f;
            G = __dadd_rn(G, probe_match(pr, ckey, &g) ? double(g) : A.beta);
          } else if (pair) {
            G = __dadd_rn(G, double(pg));
          }
          cG_next[q] = G;
          ks2 = ord_f64(__dadd_rn(ZinvT, __dmul_rn(lam, G)));
          kt2 = kTieMax - ((uint32_t(x) << 5) | uint32_t(Rn.rrank[c2]));
        }
      }
      if (!last) {
        ks_dst[q] = ks2;
        kt_dst[q] = kt2;
      }
    }
    if (last) break;
    keys = ks_dst;
    ties = kt_dst;
    cG = cG_next;
    { double* t = fZ_cur; fZ_cur = fZ_nxt; fZ_nxt = t; }
    { double* t = fG_cur; fG_cur = fG_nxt; fG_nxt = t; }
    { int* t = fnode_cur; fnode_cur = fnode_nxt; fnode_nxt = t; }
    { int* t = fctx_cur; fctx_cur = fctx_nxt; fctx_nxt = t; }
    { uint32_t* t = fmask_cur; fmask_cur = fmask_nxt; fmask_nxt = t; }
    nf = nsel;
    node_base += nsel;
    __syncthreads();
  }
  if (A.M > 0) {
    // the verification tree chosen best-first from the tree just built
    __syncthreads();
    const int Mp = A.M < N ? A.M : N;
    const size_t ob = (size_t)b * Mp;
    const size_t tb = (size_t)b * N;
    select_best_first(N, Mp, S, A.out_tokens + tb, A.out_pos + tb, A.v_index + ob, A.v_tokens + ob,
                      A.v_parents + ob, A.v_pos + ob, A.v_mask + ob * ((Mp + 31) / 32),
                      A.v_scores ? A.v_scores + ob : nullptr, A.ctrl);
  }
}

cudaError_t launch_tree(const TreeArgs& a, cudaStream_t stream) {
  if (a.B == 0) return cudaSuccess;
  const size_t smem = tree_smem_bytes(a.d, a.W, a.k, a.MW, a.N, a.M > 0);
  const int threads = tree_threads(a.W, a.k, a.B, device_sms());
  cudaError_t e;
  if (a.W <= 32) {
    e = cudaFuncSetAttribute(tree_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    tree_kernel<1><<<a.B, threads, smem, stream>>>(a);
  } else {
    e = cudaFuncSetAttribute(tree_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    tree_kernel<2><<<a.B, threads, smem, stream>>>(a);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------ K3: masks
__global__ void mask_pack_kernel(const int32_t* __restrict__ parents, int N, int MW,
                                 uint32_t* __restrict__ out, uint32_t* err) {
  const int b = blockIdx.y;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= N * MW) return;
  const int x = idx / MW;
  const int w = idx - x * MW;
  const int32_t* par = parents + (size_t)b * N;
  uint32_t val = 0;
  int a = x;
  for (int steps = 0; a >= 0 && steps <= N; ++steps) {
    if ((a >> 5) == w) val |= 1u << (a & 31);
    const int q = __ldg(par + a);
    if (q >= a || q < -1) {
      set_dev_error(err, DART_DEVERR_PARENT);
      break;
    }
    a = q;
  }
  out[((size_t)b * N + x) * MW + w] = val;
}

cudaError_t launch_mask_pack(const int32_t* parents, int B, int N, uint32_t* out_mask,
                             uint32_t* err, cudaStream_t stream) {
  if (B == 0 || N == 0) return cudaSuccess;
  const int MW = (N + 31) / 32;
  const int threads = 256;
  dim3 grid((N * MW + threads - 1) / threads, B);
  mask_pack_kernel<<<grid, threads, 0, stream>>>(parents, N, MW, out_mask, err);
  return cudaGetLastError();
}

// ----------------------------------------------------- n-gram batch lookup
__global__ void ngram_lookup_kernel(const uint4* __restrict__ slots, unsigned long long nb, int n,
                                    const int32_t* __restrict__ keys, long long Q,
                                    float* __restrict__ vals, int32_t* __restrict__ found) {
  const long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= Q) return;
  int32_t t[4] = {0, 0, 0, 0};
#pragma unroll
  for (int f = 0; f < 4; ++f)
    if (f < n) t[f] = keys[q * n + f];
  float v = 0.f;
  const bool hit = probe(slots, nb, pack_ngram(t, n), &v);
  vals[q] = hit ? v : 0.f;
  found[q] = hit ? 1 : 0;
}

cudaError_t launch_ngram_lookup(const void* slots, unsigned long long capacity, int n,
                                const int32_t* keys, long long Q, float* vals, int32_t* found,
                                cudaStream_t stream) {
  if (Q == 0) return cudaSuccess;
  const int threads = 256;
  const long long blocks = (Q + threads - 1) / threads;
  ngram_lookup_kernel<<<unsigned(blocks), threads, 0, stream>>>(
      static_cast<const uint4*>(slots), capacity / kBucketSlots, n, keys, Q, vals, found);
  return cudaGetLastError();
}

}  // namespace dart
