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
// (ordered ranking key, then inverted (parent rank, token)), sorts 32- or
// 64-key runs with warp bitonic networks and merges runs pairwise, keeping
// only the best run length, until one run holds the survivors in order.
#include "dart_launch.h"

namespace dart {

constexpr int kTreeThreads = 512;
constexpr uint32_t kTieMax = 0x3FFFFFFFu;   // (rank << 24 | token) < 2^30

struct CKey {
  uint64_t s;   // ordered ranking key
  uint32_t t;   // kTieMax - (parent rank << 24 | token): larger = lower rank, lower token
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

// Linear probing from the key's home slot.  Each round trip reads the aligned
// pair of 32-byte sectors around the current slot (4 slots) at once, so most
// lookups (load factor <= 1/2) finish after one memory latency.
__device__ __forceinline__ bool probe(const uint4* slots, unsigned long long mask, Key96 key, float* val) {
  unsigned long long idx = hash_key(key) & mask;
  for (unsigned long long done = 0; done <= mask;) {
    const unsigned long long base = idx & ~1ull;
    uint4 s[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) s[t] = ldg_nc_v4(slots + ((base + t) & mask));
    const int start = int(idx - base);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (t < start) continue;
      if (s[t].x == key.w0 && s[t].y == key.w1 && s[t].z == key.w2) {
        *val = __uint_as_float(s[t].w);
        return true;
      }
      if (s[t].x == kEmpty && s[t].y == kEmpty && s[t].z == kEmpty) return false;
      ++done;
    }
    idx = (base + 4) & mask;
  }
  return false;
}

__host__ __device__ inline int tree_run_len(int W) { return W <= 32 ? 32 : 64; }
__host__ __device__ inline int tree_pad(int W, int k) {
  const int run = tree_run_len(W);
  return (W * k + run - 1) / run * run;
}
// Threads per tree: one per child of a full frontier, 32..512.
inline int tree_threads(int W, int k) {
  int t = (W * k + 31) / 32 * 32;
  return t < 32 ? 32 : (t > kTreeThreads ? kTreeThreads : t);
}
inline size_t tree_smem_bytes(int W, int k, int MW) {
  const size_t np = size_t(tree_pad(W, k));
  size_t b = 0;
  b += 4 * kMaxW * sizeof(double);                // frontier Z and G (ping-pong)
  b += kMaxK * sizeof(double);                    // candidate base values
  b += 3 * np * sizeof(uint64_t);                 // sort keys (ping-pong), candidate G
  b += 2 * np * sizeof(uint32_t);                 // tie keys (ping-pong)
  b += 2 * kMaxW * sizeof(int);                   // frontier node ids
  b += 2 * kMaxW * 3 * sizeof(int);               // frontier n-gram contexts
  b += 2 * size_t(kMaxW) * MW * sizeof(uint32_t); // frontier mask rows
  b += kMaxK * sizeof(int);                       // candidate ids
  b += kMaxW * sizeof(int);                       // chosen parent ranks
  return b + 64;
}

// One CTA per tree.  A frontier node carries Z (sum of its candidates' base
// values) and G (sum of its n-gram terms); a child's ranking key is
// Z * invT + lam * G, accumulated in double exactly as the oracle does it, so
// equal keys (ties the inputs hold exactly) stay equal.  The reported score
// subtracts the rows' offsets (their log-sum-exp), which every node of one
// depth shares.
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
  const int k = A.k, W = A.W, N = A.N, MW = A.MW, n = A.n;
  const int npad_max = tree_pad(W, k);

  // carve shared memory (8-byte members first); every size is a multiple of 16
  uint8_t* p = smem_raw;
  auto take = [&](size_t bytes) { uint8_t* q = p; p += (bytes + 15) & ~size_t(15); return q; };
  double* fZ_a = reinterpret_cast<double*>(take(kMaxW * sizeof(double)));
  double* fZ_b = reinterpret_cast<double*>(take(kMaxW * sizeof(double)));
  double* fG_a = reinterpret_cast<double*>(take(kMaxW * sizeof(double)));
  double* fG_b = reinterpret_cast<double*>(take(kMaxW * sizeof(double)));
  double* rbase = reinterpret_cast<double*>(take(kMaxK * sizeof(double)));
  uint64_t* ks_a = reinterpret_cast<uint64_t*>(take(size_t(npad_max) * 8));
  uint64_t* ks_b = reinterpret_cast<uint64_t*>(take(size_t(npad_max) * 8));
  double* cG = reinterpret_cast<double*>(take(size_t(npad_max) * 8));
  uint32_t* kt_a = reinterpret_cast<uint32_t*>(take(size_t(npad_max) * 4));
  uint32_t* kt_b = reinterpret_cast<uint32_t*>(take(size_t(npad_max) * 4));
  int* fnode_a = reinterpret_cast<int*>(take(kMaxW * sizeof(int)));
  int* fnode_b = reinterpret_cast<int*>(take(kMaxW * sizeof(int)));
  int* fctx_a = reinterpret_cast<int*>(take(kMaxW * 3 * sizeof(int)));
  int* fctx_b = reinterpret_cast<int*>(take(kMaxW * 3 * sizeof(int)));
  uint32_t* fmask_a = reinterpret_cast<uint32_t*>(take(size_t(kMaxW) * MW * 4));
  uint32_t* fmask_b = reinterpret_cast<uint32_t*>(take(size_t(kMaxW) * MW * 4));
  int* rid = reinterpret_cast<int*>(take(kMaxK * sizeof(int)));
  int* sel = reinterpret_cast<int*>(take(kMaxW * sizeof(int)));

  const uint4* slots = static_cast<const uint4*>(A.slots);
  const unsigned long long cmask = A.capacity - 1;
  const int nctx = n > 1 ? n - 1 : 0;
  const double invT = A.invT, lam = A.lam;

  // frontier of the current depth (cur) and of the next (nxt)
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
  }
  if (tid < nctx) fctx_cur[tid] = A.ctx[(size_t)b * nctx + tid];
  if (tid < k) {
    rid[tid] = A.ids[(size_t)b * A.d * k + tid];
    rbase[tid] = A.base[(size_t)b * A.d * k + tid];
  }
  int nf = 1, node_base = 0;
  double Lsum = 0.0;   // sum of the row offsets down to this depth (same in every thread)
  __syncthreads();

  for (int j = 0; j < A.d; ++j) {
    if (A.off) Lsum = __dadd_rn(Lsum, A.off[(size_t)b * A.d + j]);
    const int m = nf * k;
    const int npad = (m + RUN - 1) / RUN * RUN;
    // expand and score every child of the frontier: one probe per child
    for (int q = tid; q < npad; q += blockDim.x) {
      uint64_t ks = 0;
      uint32_t kt = 0;
      if (q < m) {
        const int i = q / k;
        const int c = q - i * k;
        const int tok = rid[c];
        const double Z = __dadd_rn(fZ_cur[i], rbase[c]);
        double G = fG_cur[i];
        if (n > 0) {
          int32_t t[4] = {0, 0, 0, 0};
#pragma unroll
          for (int f = 0; f < 3; ++f)
            if (f < nctx) t[f] = fctx_cur[i * 3 + f];
          if (nctx == 1) t[1] = tok;
          else if (nctx == 2) t[2] = tok;
          else t[3] = tok;
          float g = 0.f;
          const double gg = probe(slots, cmask, pack_ngram(t, n), &g) ? double(g) : A.beta;
          G = __dadd_rn(G, gg);
        }
        cG[q] = G;
        const double key = __dadd_rn(__dmul_rn(Z, invT), __dmul_rn(lam, G));
        ks = ord_f64(key);
        kt = kTieMax - ((uint32_t(i) << 24) | (uint32_t(tok) & 0xFFFFFFu));
      }
      ks_a[q] = ks;
      kt_a[q] = kt;
    }
    __syncthreads();
    // sort runs of RUN keys, one warp per run
    int nr = npad / RUN;
    for (int run = warp; run < nr; run += nwarps) {
      CKey v[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int e = run * RUN + r * 32 + lane;
        v[r].s = ks_a[e];
        v[r].t = kt_a[e];
      }
      run_sort<R>(v);
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int e = run * RUN + r * 32 + lane;
        ks_a[e] = v[r].s;
        kt_a[e] = v[r].t;
      }
    }
    __syncthreads();
    // merge runs pairwise, keeping the best RUN keys of each pair
    uint64_t* ks_src = ks_a;
    uint32_t* kt_src = kt_a;
    uint64_t* ks_dst = ks_b;
    uint32_t* kt_dst = kt_b;
    while (nr > 1) {
      const int nout = (nr + 1) >> 1;
      for (int t = warp; t < nout; t += nwarps) {
        CKey v[R];
        if (2 * t + 1 < nr) {
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int e = r * 32 + lane;
            CKey x, y;
            x.s = ks_src[(2 * t) * RUN + e];
            x.t = kt_src[(2 * t) * RUN + e];
            y.s = ks_src[(2 * t + 1) * RUN + (RUN - 1 - e)];
            y.t = kt_src[(2 * t + 1) * RUN + (RUN - 1 - e)];
            v[r] = ck_gt(y, x) ? y : x;
          }
          run_merge_desc<R>(v);
        } else {
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int e = r * 32 + lane;
            v[r].s = ks_src[(2 * t) * RUN + e];
            v[r].t = kt_src[(2 * t) * RUN + e];
          }
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
    // the survivors, best first
    const int nsel = m < W ? m : W;
    for (int x = tid; x < nsel; x += blockDim.x) {
      const uint64_t ks = ks_src[x];
      const uint32_t tie = kTieMax - kt_src[x];
      int i = int(tie >> 24);
      const int tok = int(tie & 0xFFFFFFu);
      int c = 0;
      while (c < k && rid[c] != tok) ++c;
      if (ks == 0 || i >= nf || c == k) {
        set_dev_error(A.ctrl, DART_DEVERR_SELECT);
        i = 0;
        c = 0;
      }
      const double key = unord_f64(ks);
      const int node = node_base + x;
      const size_t o = (size_t)b * N + node;
      A.out_tokens[o] = tok;
      A.out_parents[o] = j == 0 ? -1 : fnode_cur[i];
      A.out_pos[o] = j + 1;
      if (A.out_scores) A.out_scores[o] = float(__dsub_rn(key, Lsum));
      fZ_nxt[x] = __dadd_rn(fZ_cur[i], rbase[c]);
      fG_nxt[x] = cG[i * k + c];
      fnode_nxt[x] = node;
      if (nctx > 0) {
        for (int f = 0; f + 1 < nctx; ++f) fctx_nxt[x * 3 + f] = fctx_cur[i * 3 + f + 1];
        fctx_nxt[x * 3 + nctx - 1] = tok;
      }
      sel[x] = i;
    }
    __syncthreads();
    // ancestor masks: the parent's row plus the node's own bit; the next
    // depth's candidate lists are fetched in the same phase
    for (int w = tid; w < nsel * MW; w += blockDim.x) {
      const int x = w / MW;
      const int word = w - x * MW;
      const int node = node_base + x;
      uint32_t val = (j == 0) ? 0u : fmask_cur[sel[x] * MW + word];
      if (word == (node >> 5)) val |= 1u << (node & 31);
      fmask_nxt[x * MW + word] = val;
      A.out_mask[((size_t)b * N + node) * MW + word] = val;
    }
    if (j + 1 < A.d && tid < k) {
      rid[tid] = A.ids[((size_t)b * A.d + j + 1) * k + tid];
      rbase[tid] = A.base[((size_t)b * A.d + j + 1) * k + tid];
    }
    __syncthreads();
    { double* t = fZ_cur; fZ_cur = fZ_nxt; fZ_nxt = t; }
    { double* t = fG_cur; fG_cur = fG_nxt; fG_nxt = t; }
    { int* t = fnode_cur; fnode_cur = fnode_nxt; fnode_nxt = t; }
    { int* t = fctx_cur; fctx_cur = fctx_nxt; fctx_nxt = t; }
    { uint32_t* t = fmask_cur; fmask_cur = fmask_nxt; fmask_nxt = t; }
    nf = nsel;
    node_base += nsel;
  }
}

cudaError_t launch_tree(const TreeArgs& a, cudaStream_t stream) {
  if (a.B == 0) return cudaSuccess;
  const size_t smem = tree_smem_bytes(a.W, a.k, a.MW);
  const int threads = tree_threads(a.W, a.k);
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
__global__ void ngram_lookup_kernel(const uint4* __restrict__ slots, unsigned long long mask, int n,
                                    const int32_t* __restrict__ keys, long long Q,
                                    float* __restrict__ vals, int32_t* __restrict__ found) {
  const long long q = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= Q) return;
  int32_t t[4] = {0, 0, 0, 0};
#pragma unroll
  for (int f = 0; f < 4; ++f)
    if (f < n) t[f] = keys[q * n + f];
  float v = 0.f;
  const bool hit = probe(slots, mask, pack_ngram(t, n), &v);
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
      static_cast<const uint4*>(slots), capacity - 1, n, keys, Q, vals, found);
  return cudaGetLastError();
}

}  // namespace dart
