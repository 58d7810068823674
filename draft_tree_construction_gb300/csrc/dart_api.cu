// dart_api.cu -- the C ABI declared in include/darttree.h: argument checks,
// workspace layout, kernel launches, and the host-side n-gram table packer.
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>

#include "dart_launch.h"

using namespace dart;

namespace {

bool finite(float x) { return std::isfinite(x); }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
int elem_bytes(int dtype) { return dtype == DART_F32 ? 4 : 2; }
bool valid_dtype(int dtype) { return dtype == DART_F32 || dtype == DART_F16 || dtype == DART_BF16; }
bool pow2(uint64_t x) { return x >= 2 && (x & (x - 1)) == 0; }

// Temperature check.  T = 0 is greedy decoding (DART, Figure 2 caption reports
// results at T = 0 and T = 1): it names how the target samples, and
// log_softmax(z / 0) is undefined, so the candidates (chosen on the raw
// logits whatever T is) are scored with the draft's own log-probabilities,
// the T = 1 values.  A negative or non-finite T is an argument error.
bool score_temperature(float* T) {
  if (!finite(*T) || *T < 0.f) return false;
  if (*T == 0.f) *T = 1.f;
  return true;
}

int num_nodes(int d, int k, int W) {
  if (d < 1 || k < 1 || W < 1) return -1;
  long long total = 0, width = 1;
  for (int j = 1; j <= d; ++j) {
    width *= k;
    if (width > W) width = W;
    total += width;
    if (total > (1LL << 30)) return -1;
  }
  return int(total);
}

int check_table(const dart_ngram_table_t* t, const int32_t* ctx, int B) {
  if (!t) return DART_OK;
  if (t->n < 2 || t->n > 4 || t->reserved != 0) return DART_ERR_INVALID_ARG;
  if (!pow2(t->capacity) || t->capacity < kMinTableSlots || !t->slots || !aligned(t->slots, 64))
    return DART_ERR_INVALID_ARG;
  if (B > 0 && !ctx) return DART_ERR_INVALID_ARG;
  return DART_OK;
}

// Shared checks of the tree-shape arguments.
int check_tree_shape(int B, int d, int k, int W, float lambda, float beta) {
  if (B < 0 || d < 1 || d > kMaxD || k < 1 || k > kMaxK || W < 1 || W > kMaxW) return DART_ERR_INVALID_ARG;
  const int N = num_nodes(d, k, W);
  if (N < 1 || N > kMaxN) return DART_ERR_INVALID_ARG;
  if (!finite(lambda) || !finite(beta)) return DART_ERR_INVALID_ARG;
  return DART_OK;
}

TreeArgs tree_args(int B, int d, int k, int W, float lambda, float beta,
                   const dart_ngram_table_t* t, const int32_t* ctx,
                   int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                   uint32_t* out_mask, float* out_scores) {
  TreeArgs a;
  a.B = B; a.d = d; a.k = k; a.W = W;
  a.N = num_nodes(d, k, W);
  a.MW = (a.N + 31) / 32;
  a.n = t ? t->n : 0;
  a.lam = double(lambda);
  a.beta = double(beta);
  a.ids = nullptr;
  a.base = nullptr;
  a.off = nullptr;
  a.invT = 1.0;
  a.ctx = ctx;
  a.slots = t ? t->slots : nullptr;
  a.capacity = t ? t->capacity : 0;
  a.pair = nullptr;
  a.out_tokens = out_tokens;
  a.out_parents = out_parents;
  a.out_pos = out_pos;
  a.out_mask = out_mask;
  a.out_scores = out_scores;
  a.ctrl = nullptr;
  a.M = 0;
  a.v_index = a.v_tokens = a.v_parents = a.v_pos = nullptr;
  a.v_mask = nullptr;
  a.v_scores = nullptr;
  return a;
}

// The verification tree's outputs of dart_tree_build_verify.
struct VerifyOut {
  int M;
  int32_t* index;
  int32_t* tokens;
  int32_t* parents;
  int32_t* pos;
  uint32_t* mask;
  float* scores;
};

// The whole path on a workspace: the row pass, then the tree kernel.
int launch_path(const void* logits, int B, int d, int V, int64_t row_stride, int dtype, float T, int k, int W,
                float lambda, float beta, const dart_ngram_table_t* ngram_table, const int32_t* ctx_tokens,
                int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos, uint32_t* out_mask,
                float* out_scores, uint8_t* ws, const WsLayout& L, cudaStream_t s,
                const VerifyOut* verify = nullptr) {
  const long long R = (long long)B * d;
  if (launch_rows(logits, R, V, row_stride, dtype, T, k, ws, L, nullptr, nullptr, nullptr, s) != cudaSuccess)
    return DART_ERR_CUDA;
  TreeArgs a = tree_args(B, d, k, W, lambda, beta, ngram_table, ctx_tokens, out_tokens, out_parents,
                         out_pos, out_mask, out_scores);
  a.ids = reinterpret_cast<const int32_t*>(ws + L.row_ids);
  a.base = reinterpret_cast<const double*>(ws + L.row_base);
  a.off = reinterpret_cast<const double*>(ws + L.row_off);
  a.invT = 1.0 / double(T);
  a.ctrl = reinterpret_cast<uint32_t*>(ws + L.ctrl);
  if (verify) {
    a.M = verify->M;
    a.v_index = verify->index;
    a.v_tokens = verify->tokens;
    a.v_parents = verify->parents;
    a.v_pos = verify->pos;
    a.v_mask = verify->mask;
    a.v_scores = verify->scores;
  }
  if (launch_tree(a, s) != cudaSuccess) return DART_ERR_CUDA;
  return DART_OK;
}

}  // namespace

// ---------------------------------------------------- fixed device scratch
// Scratch for dart_tree_build_noalloc: the workspace that dart_tree_build
// takes from its caller lives here instead.  Every device that loads the
// library holds these bytes until the process exits.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

// The CUDA runtime gives a __device__ variable one address per context, and a
// context replaced by cudaDeviceReset (or a driver-API caller's own context)
// may place it elsewhere, so the cache is keyed by the current context's
// unique id.  cuCtxGetCurrent and cuCtxGetId come through the runtime's
// driver entry-point query, which keeps the library free of a link-time
// dependency on the driver library.
using CtxGetCurrentFn = int (*)(void** ctx);
using CtxGetIdFn = int (*)(void* ctx, unsigned long long* id);

struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
constexpr int kMaxScratchContexts = 64;
std::mutex g_scratch_mutex;
ScratchEntry g_scratch_cache[kMaxScratchContexts] = {};
int g_scratch_used = 0;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

bool driver_entry(const char* name, void** fn) {
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  return cudaGetDriverEntryPointByVersion(name, fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
         q == cudaDriverEntryPointSuccess && *fn;
}

// Device address of g_static_scratch in the current context.  The first call
// in a context binds the runtime's primary context if none is current yet and
// looks the address up; later calls in that context use the cached address.
int static_scratch(void** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_ctx_get_current || !g_ctx_get_id) {
    void* a = nullptr;
    void* b = nullptr;
    if (!driver_entry("cuCtxGetCurrent", &a) || !driver_entry("cuCtxGetId", &b)) return DART_ERR_CUDA;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(a);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(b);
  }
  void* ctx = nullptr;
  void* addr = nullptr;
  if (g_ctx_get_current(&ctx) != 0) return DART_ERR_CUDA;
  if (!ctx) {
    // no context current on this thread yet: the lookup binds the device's primary context
    if (cudaGetSymbolAddress(&addr, g_static_scratch) != cudaSuccess || !addr) return DART_ERR_CUDA;
    if (g_ctx_get_current(&ctx) != 0 || !ctx) return DART_ERR_CUDA;
  }
  unsigned long long id = 0;
  if (g_ctx_get_id(ctx, &id) != 0) return DART_ERR_CUDA;
  for (int i = 0; i < g_scratch_used; ++i)
    if (g_scratch_cache[i].ctx_id == id) {
      *out = g_scratch_cache[i].addr;
      return DART_OK;
    }
  if (!addr && (cudaGetSymbolAddress(&addr, g_static_scratch) != cudaSuccess || !addr)) return DART_ERR_CUDA;
  // a full cache forgets its oldest entry (contexts that old are usually gone)
  if (g_scratch_used == kMaxScratchContexts) {
    for (int i = 1; i < kMaxScratchContexts; ++i) g_scratch_cache[i - 1] = g_scratch_cache[i];
    --g_scratch_used;
  }
  g_scratch_cache[g_scratch_used++] = ScratchEntry{id, addr};
  *out = addr;
  return DART_OK;
}

// Copies the control block's error word (word 0) to *out_flags and clears the
// block when the word is nonzero.  The caller has synchronised the stream.
int read_error_word(void* ctrl, uint32_t* out_flags) {
  uint32_t word = 0;
  if (cudaMemcpy(&word, ctrl, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return DART_ERR_CUDA;
  *out_flags = word;
  if (word != 0u && cudaMemset(ctrl, 0, kCtrlBytes) != cudaSuccess) return DART_ERR_CUDA;
  return DART_OK;
}

}  // namespace

extern "C" {

int dart_tree_num_nodes(int d, int k, int W) { return num_nodes(d, k, W); }

int dart_tree_mask_words(int num_nodes_) { return num_nodes_ < 0 ? -1 : (num_nodes_ + 31) / 32; }

size_t dart_tree_workspace_bytes(int B, int d, int V, int dtype, int k) {
  if (B < 0 || d < 1 || V < 1 || !valid_dtype(dtype) || k < 1 || k > kMaxK) return 0;
  WsLayout L;
  if (!ws_layout((long long)B * d, V, elem_bytes(dtype), k, &L)) return 0;
  return L.total;
}

int dart_tree_build(const void* logits, int B, int d, int V, int dtype,
                    float T, int k, int W, float lambda, float beta,
                    const dart_ngram_table_t* ngram_table, const int32_t* ctx_tokens,
                    int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                    uint32_t* out_mask, float* out_scores,
                    void* workspace, size_t workspace_bytes, void* stream) {
  return dart_tree_build_strided(logits, B, d, V, V, dtype, T, k, W, lambda, beta, ngram_table, ctx_tokens,
                                 out_tokens, out_parents, out_pos, out_mask, out_scores, workspace,
                                 workspace_bytes, stream);
}

namespace {
// The argument checks of dart_tree_build_strided; on DART_OK with B > 0,
// *L holds the workspace layout and *T the scoring temperature.
int prepare_build(const void* logits, int B, int d, int V, int64_t row_stride, int dtype, float* T, int k, int W,
                  float lambda, float beta, const dart_ngram_table_t* ngram_table, const int32_t* ctx_tokens,
                  int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos, uint32_t* out_mask,
                  void* workspace, size_t workspace_bytes, WsLayout* L) {
  int rc = check_tree_shape(B, d, k, W, lambda, beta);
  if (rc) return rc;
  if (V < 2 || V > kMaxV || k > V || !valid_dtype(dtype)) return DART_ERR_INVALID_ARG;
  if (row_stride < V || row_stride > kMaxRowStride) return DART_ERR_INVALID_ARG;
  if (!score_temperature(T)) return DART_ERR_INVALID_ARG;
  if ((rc = check_table(ngram_table, ctx_tokens, B))) return rc;
  if (B == 0) return DART_OK;
  if (!logits || !aligned(logits, 16)) return DART_ERR_INVALID_ARG;
  if (!out_tokens || !out_parents || !out_pos || !out_mask) return DART_ERR_INVALID_ARG;
  const long long R = (long long)B * d;
  if (!ws_layout(R, V, elem_bytes(dtype), k, L)) return DART_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L->total) return DART_ERR_WORKSPACE;
  return DART_OK;
}
}  // namespace

int dart_tree_build_strided(const void* logits, int B, int d, int V, int64_t row_stride, int dtype,
                            float T, int k, int W, float lambda, float beta,
                            const dart_ngram_table_t* ngram_table, const int32_t* ctx_tokens,
                            int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                            uint32_t* out_mask, float* out_scores,
                            void* workspace, size_t workspace_bytes, void* stream) {
  WsLayout L;
  const int rc = prepare_build(logits, B, d, V, row_stride, dtype, &T, k, W, lambda, beta, ngram_table, ctx_tokens,
                               out_tokens, out_parents, out_pos, out_mask, workspace, workspace_bytes, &L);
  if (rc || B == 0) return rc;
  return launch_path(logits, B, d, V, row_stride, dtype, T, k, W, lambda, beta, ngram_table, ctx_tokens,
                     out_tokens, out_parents, out_pos, out_mask, out_scores, static_cast<uint8_t*>(workspace), L,
                     static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------- plans
struct dart_tree_plan_s {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  int device;
  // the call's arguments, for launches into a stream that is itself being
  // captured (the kernels are then launched as dart_tree_build_strided would)
  const void* logits;
  int B, d, V, dtype, k, W;
  int64_t row_stride;
  float T, lambda, beta;
  bool has_table;
  dart_ngram_table_t table;
  const int32_t* ctx;
  int32_t *tokens, *parents, *pos;
  uint32_t* mask;
  float* scores;
  uint8_t* ws;
  WsLayout L;
};

int dart_tree_plan_create(dart_tree_plan_t* out_plan, const void* logits, int B, int d, int V, int64_t row_stride,
                          int dtype, float T, int k, int W, float lambda, float beta,
                          const dart_ngram_table_t* ngram_table, const int32_t* ctx_tokens,
                          int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                          uint32_t* out_mask, float* out_scores, void* workspace, size_t workspace_bytes) {
  if (!out_plan) return DART_ERR_INVALID_ARG;
  *out_plan = nullptr;
  WsLayout L;
  int rc = prepare_build(logits, B, d, V, row_stride, dtype, &T, k, W, lambda, beta, ngram_table, ctx_tokens,
                         out_tokens, out_parents, out_pos, out_mask, workspace, workspace_bytes, &L);
  if (rc) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DART_ERR_CUDA;
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return DART_ERR_CUDA;
  // the launches are recorded on a stream of the plan's own, none of them runs
  cudaGraph_t graph = nullptr;
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaStreamDestroy(s);
    return DART_ERR_CUDA;
  }
  if (B > 0)
    rc = launch_path(logits, B, d, V, row_stride, dtype, T, k, W, lambda, beta, ngram_table, ctx_tokens,
                     out_tokens, out_parents, out_pos, out_mask, out_scores, static_cast<uint8_t*>(workspace), L, s);
  const cudaError_t ec = cudaStreamEndCapture(s, &graph);
  cudaStreamDestroy(s);
  if (rc == DART_OK && ec != cudaSuccess) rc = DART_ERR_CUDA;
  cudaGraphExec_t exec = nullptr;
  if (rc == DART_OK && cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) rc = DART_ERR_CUDA;
  if (rc != DART_OK) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    return rc;
  }
  dart_tree_plan_s* plan = new (std::nothrow) dart_tree_plan_s{};
  if (plan) {
    plan->graph = graph;
    plan->exec = exec;
    plan->device = dev;
    plan->logits = logits;
    plan->B = B;
    plan->d = d;
    plan->V = V;
    plan->dtype = dtype;
    plan->k = k;
    plan->W = W;
    plan->row_stride = row_stride;
    plan->T = T;
    plan->lambda = lambda;
    plan->beta = beta;
    plan->has_table = ngram_table != nullptr;
    if (ngram_table) plan->table = *ngram_table;
    plan->ctx = ctx_tokens;
    plan->tokens = out_tokens;
    plan->parents = out_parents;
    plan->pos = out_pos;
    plan->mask = out_mask;
    plan->scores = out_scores;
    plan->ws = static_cast<uint8_t*>(workspace);
    plan->L = L;
  }
  if (!plan) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(graph);
    return DART_ERR_INTERNAL;
  }
  *out_plan = plan;
  return DART_OK;
}

int dart_tree_plan_launch(dart_tree_plan_t plan, void* stream) {
  if (!plan) return DART_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DART_ERR_CUDA;
  if (dev != plan->device) return DART_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) return DART_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) {
    // a caller capturing its own graph: record the kernels themselves
    if (plan->B == 0) return DART_OK;
    return launch_path(plan->logits, plan->B, plan->d, plan->V, plan->row_stride, plan->dtype, plan->T, plan->k,
                       plan->W, plan->lambda, plan->beta, plan->has_table ? &plan->table : nullptr, plan->ctx,
                       plan->tokens, plan->parents, plan->pos, plan->mask, plan->scores, plan->ws, plan->L, s);
  }
  return cudaGraphLaunch(plan->exec, s) == cudaSuccess ? DART_OK : DART_ERR_CUDA;
}

int dart_tree_plan_destroy(dart_tree_plan_t plan) {
  if (!plan) return DART_OK;
  const bool ok = cudaGraphExecDestroy(plan->exec) == cudaSuccess && cudaGraphDestroy(plan->graph) == cudaSuccess;
  delete plan;
  return ok ? DART_OK : DART_ERR_CUDA;
}

int dart_tree_build_verify(const void* logits, int B, int d, int V, int64_t row_stride, int dtype,
                           float T, int k, int W, float lambda, float beta,
                           const dart_ngram_table_t* ngram_table, const int32_t* ctx_tokens,
                           int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                           uint32_t* out_mask, float* out_scores, int M, int32_t* out_vindex,
                           int32_t* out_vtokens, int32_t* out_vparents, int32_t* out_vpos,
                           uint32_t* out_vmask, float* out_vscores,
                           void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_tree_shape(B, d, k, W, lambda, beta);
  if (rc) return rc;
  if (V < 2 || V > kMaxV || k > V || !valid_dtype(dtype)) return DART_ERR_INVALID_ARG;
  if (row_stride < V || row_stride > kMaxRowStride) return DART_ERR_INVALID_ARG;
  if (!score_temperature(&T)) return DART_ERR_INVALID_ARG;
  if (M < 1) return DART_ERR_INVALID_ARG;
  if ((rc = check_table(ngram_table, ctx_tokens, B))) return rc;
  if (B == 0) return DART_OK;
  if (!logits || !aligned(logits, 16)) return DART_ERR_INVALID_ARG;
  if (!out_tokens || !out_parents || !out_pos || !out_mask) return DART_ERR_INVALID_ARG;
  if (!out_vindex || !out_vtokens || !out_vparents || !out_vpos || !out_vmask) return DART_ERR_INVALID_ARG;
  WsLayout L;
  const long long R = (long long)B * d;
  if (!ws_layout(R, V, elem_bytes(dtype), k, &L)) return DART_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return DART_ERR_WORKSPACE;
  const VerifyOut verify{M, out_vindex, out_vtokens, out_vparents, out_vpos, out_vmask, out_vscores};
  return launch_path(logits, B, d, V, row_stride, dtype, T, k, W, lambda, beta, ngram_table, ctx_tokens,
                     out_tokens, out_parents, out_pos, out_mask, out_scores, static_cast<uint8_t*>(workspace), L,
                     static_cast<cudaStream_t>(stream), &verify);
}

int dart_tree_build_noalloc(const void* logits, int B, int d, int V, int dtype,
                            float T, int k, int W, float lambda, float beta,
                            const dart_ngram_table_t* ngram_table, const int32_t* ctx_tokens,
                            int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                            uint32_t* out_mask, float* out_scores, void* stream) {
  int rc = check_tree_shape(B, d, k, W, lambda, beta);
  if (rc) return rc;
  if (V < 2 || V > kMaxV || k > V || !valid_dtype(dtype)) return DART_ERR_INVALID_ARG;
  if (!score_temperature(&T)) return DART_ERR_INVALID_ARG;
  if ((rc = check_table(ngram_table, ctx_tokens, B))) return rc;
  if (B == 0) return DART_OK;
  if (!logits || !aligned(logits, 16)) return DART_ERR_INVALID_ARG;
  if (!out_tokens || !out_parents || !out_pos || !out_mask) return DART_ERR_INVALID_ARG;
  WsLayout L;
  const long long R = (long long)B * d;
  if (!ws_layout(R, V, elem_bytes(dtype), k, &L)) return DART_ERR_INVALID_ARG;
  if (L.total > kStaticScratchBytes) return DART_ERR_WORKSPACE;   // sizes beyond the fixed scratch
  void* scratch = nullptr;
  if ((rc = static_scratch(&scratch))) return rc;
  // Nothing in the buffer has to start at zero for a call except the device
  // error word, which starts at zero when the module loads and is cleared by
  // dart_noalloc_device_error; every other byte a call reads it wrote itself.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(scratch);
  return launch_path(logits, B, d, V, V, dtype, T, k, W, lambda, beta, ngram_table, ctx_tokens, out_tokens,
                     out_parents, out_pos, out_mask, out_scores, ws, L, s);
}

int dart_tree_from_topk(const int32_t* cand_ids, const double* cand_logp,
                        int B, int d, int k, int W, float lambda, float beta,
                        const dart_ngram_table_t* ngram_table, const int32_t* ctx_tokens,
                        int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                        uint32_t* out_mask, float* out_scores, void* stream) {
  int rc = check_tree_shape(B, d, k, W, lambda, beta);
  if (rc) return rc;
  if ((rc = check_table(ngram_table, ctx_tokens, B))) return rc;
  if (B == 0) return DART_OK;
  if (!cand_ids || !cand_logp || !out_tokens || !out_parents || !out_pos || !out_mask)
    return DART_ERR_INVALID_ARG;
  TreeArgs a = tree_args(B, d, k, W, lambda, beta, ngram_table, ctx_tokens, out_tokens, out_parents,
                         out_pos, out_mask, out_scores);
  a.ids = cand_ids;
  a.base = cand_logp;
  if (launch_tree(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return DART_ERR_CUDA;
  return DART_OK;
}

int dart_tree_from_topk_pairs(const int32_t* cand_ids, const double* cand_logp, const float* pair_scores,
                              int B, int d, int k, int W, float lambda,
                              int32_t* out_tokens, int32_t* out_parents, int32_t* out_pos,
                              uint32_t* out_mask, float* out_scores, void* stream) {
  int rc = check_tree_shape(B, d, k, W, lambda, 0.f);
  if (rc) return rc;
  if (B == 0) return DART_OK;
  if (!cand_ids || !cand_logp || !pair_scores || !out_tokens || !out_parents || !out_pos || !out_mask)
    return DART_ERR_INVALID_ARG;
  TreeArgs a = tree_args(B, d, k, W, lambda, 0.f, nullptr, nullptr, out_tokens, out_parents, out_pos,
                         out_mask, out_scores);
  a.ids = cand_ids;
  a.base = cand_logp;
  a.pair = pair_scores;
  if (launch_tree(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return DART_ERR_CUDA;
  return DART_OK;
}

int dart_tree_from_rows_pairs(int B, int d, int V, int dtype, float T, int k, int W, float lambda,
                              const float* pair_scores, int32_t* out_tokens, int32_t* out_parents,
                              int32_t* out_pos, uint32_t* out_mask, float* out_scores,
                              const void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_tree_shape(B, d, k, W, lambda, 0.f);
  if (rc) return rc;
  if (V < 2 || V > kMaxV || k > V || !valid_dtype(dtype)) return DART_ERR_INVALID_ARG;
  if (!score_temperature(&T)) return DART_ERR_INVALID_ARG;
  if (B == 0) return DART_OK;
  if (!pair_scores || !out_tokens || !out_parents || !out_pos || !out_mask) return DART_ERR_INVALID_ARG;
  WsLayout L;
  if (!ws_layout((long long)B * d, V, elem_bytes(dtype), k, &L)) return DART_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return DART_ERR_WORKSPACE;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  TreeArgs a = tree_args(B, d, k, W, lambda, 0.f, nullptr, nullptr, out_tokens, out_parents, out_pos,
                         out_mask, out_scores);
  a.ids = reinterpret_cast<const int32_t*>(ws + L.row_ids);
  a.base = reinterpret_cast<const double*>(ws + L.row_base);
  a.off = reinterpret_cast<const double*>(ws + L.row_off);
  a.invT = 1.0 / double(T);
  a.pair = pair_scores;
  a.ctrl = reinterpret_cast<uint32_t*>(const_cast<uint8_t*>(ws) + L.ctrl);
  if (launch_tree(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return DART_ERR_CUDA;
  return DART_OK;
}

int dart_row_topk(const void* logits, int rows, int V, int dtype, float T, int k,
                  int32_t* out_ids, float* out_logp, float* out_lse,
                  void* workspace, size_t workspace_bytes, void* stream) {
  return dart_row_topk_strided(logits, rows, V, V, dtype, T, k, out_ids, out_logp, out_lse, workspace,
                               workspace_bytes, stream);
}

int dart_row_topk_strided(const void* logits, int rows, int V, int64_t row_stride, int dtype, float T, int k,
                          int32_t* out_ids, float* out_logp, float* out_lse,
                          void* workspace, size_t workspace_bytes, void* stream) {
  if (rows < 0 || V < 2 || V > kMaxV || !valid_dtype(dtype) || k < 1 || k > kMaxK || k > V)
    return DART_ERR_INVALID_ARG;
  if (row_stride < V || row_stride > kMaxRowStride) return DART_ERR_INVALID_ARG;
  if (!score_temperature(&T)) return DART_ERR_INVALID_ARG;
  if (rows == 0) return DART_OK;
  if (!logits || !aligned(logits, 16)) return DART_ERR_INVALID_ARG;
  WsLayout L;
  if (!ws_layout(rows, V, elem_bytes(dtype), k, &L)) return DART_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total) return DART_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_rows(logits, rows, V, row_stride, dtype, T, k, workspace, L, out_ids, out_logp, out_lse, s) !=
      cudaSuccess)
    return DART_ERR_CUDA;
  return DART_OK;
}

namespace {
int check_rows(const void* logits, bool need_logits, int rows, int V, int64_t row_stride, int dtype, float T, int k,
               const void* workspace, size_t workspace_bytes, WsLayout* L) {
  if (rows < 0 || V < 2 || V > kMaxV || !valid_dtype(dtype) || k < 1 || k > kMaxK || k > V)
    return DART_ERR_INVALID_ARG;
  if (row_stride < V || row_stride > kMaxRowStride) return DART_ERR_INVALID_ARG;
  if (!score_temperature(&T)) return DART_ERR_INVALID_ARG;
  if (rows == 0) return DART_OK;
  if (need_logits && (!logits || !aligned(logits, 16))) return DART_ERR_INVALID_ARG;
  if (!ws_layout(rows, V, elem_bytes(dtype), k, L)) return DART_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L->total) return DART_ERR_WORKSPACE;
  return DART_OK;
}
}  // namespace

int dart_row_pass(const void* logits, int rows, int V, int64_t row_stride, int dtype, float T, int k,
                  void* workspace, size_t workspace_bytes, void* stream) {
  WsLayout L;
  const int rc = check_rows(logits, true, rows, V, row_stride, dtype, T, k, workspace, workspace_bytes, &L);
  if (rc || rows == 0) return rc;
  if (launch_row_pass(logits, rows, V, row_stride, dtype, T, k, workspace, L, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return DART_ERR_CUDA;
  return DART_OK;
}

int dart_row_finish(int rows, int V, int64_t row_stride, int dtype, float T, int k, int32_t* out_ids,
                    float* out_logp, float* out_lse, void* workspace, size_t workspace_bytes, void* stream) {
  WsLayout L;
  const int rc = check_rows(nullptr, false, rows, V, row_stride, dtype, T, k, workspace, workspace_bytes, &L);
  if (rc || rows == 0) return rc;
  if (launch_row_merge(rows, V, row_stride, dtype, T, k, workspace, L, out_ids, out_logp, out_lse,
                       static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DART_ERR_CUDA;
  return DART_OK;
}

int dart_mask_pack(const int32_t* parents, int B, int N, uint32_t* out_mask, uint32_t* device_err,
                   void* stream) {
  if (B < 0 || N < 0 || N > (1 << 20)) return DART_ERR_INVALID_ARG;
  if (B == 0 || N == 0) return DART_OK;
  if (!parents || !out_mask) return DART_ERR_INVALID_ARG;
  if (launch_mask_pack(parents, B, N, out_mask, device_err, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DART_ERR_CUDA;
  return DART_OK;
}

uint64_t dart_ngram_capacity_for(uint64_t M) {
  if (M > (1ull << 62)) return 0;
  uint64_t c = kMinTableSlots;
  while (c < 2 * M) c <<= 1;
  return c;
}

namespace {
bool slot_is(const uint32_t* slot, const Key96& k) { return slot[0] == k.w0 && slot[1] == k.w1 && slot[2] == k.w2; }
bool slot_empty(const uint32_t* slot) { return slot[0] == kEmpty && slot[1] == kEmpty && slot[2] == kEmpty; }
uint32_t* free_slot(uint32_t* s, uint64_t bucket) {
  for (int t = 0; t < kBucketSlots; ++t)
    if (slot_empty(s + 4 * (kBucketSlots * bucket + t))) return s + 4 * (kBucketSlots * bucket + t);
  return nullptr;
}
void put(uint32_t* slot, const Key96& k, uint32_t v) {
  slot[0] = k.w0;
  slot[1] = k.w1;
  slot[2] = k.w2;
  slot[3] = v;
}
}  // namespace

int dart_ngram_table_pack_host(int n, const int32_t* keys, const float* vals, uint64_t M,
                               uint64_t capacity, void* host_slots, uint64_t* out_distinct) {
  if (n < 1 || n > 4 || !pow2(capacity) || capacity < kMinTableSlots || !host_slots) return DART_ERR_INVALID_ARG;
  if (M > 0 && (!keys || !vals)) return DART_ERR_INVALID_ARG;
  uint32_t* s = static_cast<uint32_t*>(host_slots);
  for (uint64_t i = 0; i < capacity; ++i) put(s + 4 * i, Key96{kEmpty, kEmpty, kEmpty}, 0u);
  const uint64_t nb = capacity / kBucketSlots;
  uint64_t distinct = 0;
  int rc = DART_OK;
  for (uint64_t i = 0; i < M && rc == DART_OK; ++i) {
    const int32_t* t = keys + i * n;
    for (int f = 0; f < n; ++f)
      if (t[f] < 0 || t[f] >= kMaxV) rc = DART_ERR_INVALID_ARG;
    if (rc) break;
    Key96 key = pack_ngram(t, n);
    uint32_t val;
    memcpy(&val, &vals[i], 4);
    const Buckets bk = key_buckets(key, nb);
    bool present = false;
    for (int tt = 0; tt < 2 * kBucketSlots && !present; ++tt)
      present = slot_is(s + 4 * (kBucketSlots * (tt < kBucketSlots ? bk.b1 : bk.b2) + tt % kBucketSlots), key);
    if (present) continue;   // the first value of a key is kept
    if (distinct >= capacity / 2) {
      rc = DART_ERR_TABLE_FULL;
      break;
    }
    uint32_t* slot = free_slot(s, bk.b1);
    if (!slot) slot = free_slot(s, bk.b2);
    // both buckets full: displace along the chain b -> the victim's other bucket
    uint64_t b = bk.b1;
    for (int kick = 0; !slot && kick < 500; ++kick) {
      uint32_t* victim = s + 4 * (kBucketSlots * b + uint64_t(kick % kBucketSlots));
      const Key96 vk{victim[0], victim[1], victim[2]};
      const uint32_t vv = victim[3];
      put(victim, key, val);
      key = vk;
      val = vv;
      const Buckets vb = key_buckets(key, nb);
      b = (vb.b1 == b) ? vb.b2 : vb.b1;
      slot = free_slot(s, b);
    }
    if (!slot) {
      rc = DART_ERR_TABLE_FULL;
      break;
    }
    put(slot, key, val);
    ++distinct;
  }
  if (out_distinct) *out_distinct = distinct;
  return rc;
}

int dart_ngram_lookup(const dart_ngram_table_t* table, const int32_t* keys, int64_t Q,
                      float* vals, int32_t* found, void* stream) {
  if (!table || table->n < 1 || table->n > 4 || !pow2(table->capacity) || table->capacity < kMinTableSlots ||
      !table->slots || !aligned(table->slots, 64) || Q < 0)
    return DART_ERR_INVALID_ARG;
  if (Q == 0) return DART_OK;
  if (!keys || !vals || !found) return DART_ERR_INVALID_ARG;
  if (launch_ngram_lookup(table->slots, table->capacity, table->n, keys, Q, vals, found,
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DART_ERR_CUDA;
  return DART_OK;
}

void dart_set_wait_limit(int64_t cycles) { set_rows_wait_limit((long long)cycles); }

int dart_device_error(const void* workspace, uint32_t* out_flags, void* stream) {
  if (!workspace || !out_flags) return DART_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return DART_ERR_CUDA;
  return read_error_word(const_cast<void*>(workspace), out_flags);
}

int dart_noalloc_device_error(uint32_t* out_flags, void* stream) {
  if (!out_flags) return DART_ERR_INVALID_ARG;
  void* scratch = nullptr;
  int rc = static_scratch(&scratch);
  if (rc) return rc;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DART_ERR_CUDA;
  return read_error_word(scratch, out_flags);
}

const char* dart_status_string(int status) {
  switch (status) {
    case DART_OK: return "ok";
    case DART_ERR_INVALID_ARG: return "invalid argument";
    case DART_ERR_UNSUPPORTED: return "unsupported";
    case DART_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case DART_ERR_CUDA: return "CUDA runtime error";
    case DART_ERR_INTERNAL: return "internal inconsistency reported by a kernel";
    case DART_ERR_TIMEOUT: return "bounded device wait ran out";
    case DART_ERR_TABLE_FULL: return "n-gram table full (more than capacity/2 keys)";
    default: return "unknown status";
  }
}

}  // extern "C"
