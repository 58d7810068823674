// dart_launch.h -- host-side launchers shared between the C-ABI layer and the
// kernel translation units (internal; not part of the public header).
#pragma once

#include "dart_common.cuh"

namespace dart {

long long rows_wait_limit();
// Multiprocessors of the current device (cached per device; 0 if unknown).
int device_sms();
void set_rows_wait_limit(long long cycles);

// The streaming pass over R rows (per-piece results in the workspace).
cudaError_t launch_row_pass(const void* logits, long long R, int V, long long stride, int dtype, float T, int k,
                            void* ws, const WsLayout& L, cudaStream_t stream);
// The row merge: each row's results (row_off / row_ids / row_base in the
// workspace, and the optional outputs) from the pass's per-piece results.
cudaError_t launch_row_merge(long long R, int V, long long stride, int dtype, float T, int k, void* ws,
                             const WsLayout& L, int32_t* out_ids, float* out_logp, float* out_lse,
                             cudaStream_t stream);
// Both.
cudaError_t launch_rows(const void* logits, long long R, int V, long long stride, int dtype, float T, int k,
                        void* ws, const WsLayout& L,
                        int32_t* out_ids, float* out_logp, float* out_lse, cudaStream_t stream);

struct TreeArgs {
  int B, d, k, W, N, MW, n;    // n = 0: no n-gram term
  double lam, beta;
  const int32_t* ids;          // [B][d][k] candidate tokens
  const double* base;          // [B][d][k] candidate base values (logits, or log-probabilities)
  const double* off;           // [B][d] per-row offset subtracted from reported scores, or nullptr
  double invT;                 // ranking key = (sum of base) * invT + lam * (sum of n-gram terms)
  const int32_t* ctx;          // [B][n-1]
  const void* slots;
  unsigned long long capacity;
  const float* pair;           // [B][d][k][k] caller pair scores (with n = 0), or nullptr
  int32_t* out_tokens;
  int32_t* out_parents;
  int32_t* out_pos;
  uint32_t* out_mask;
  float* out_scores;
  uint32_t* ctrl;              // device error word or nullptr
  // the best-first verification tree of budget M (M = 0: none), [B][min(M, N)]
  int M;
  int32_t* v_index;
  int32_t* v_tokens;
  int32_t* v_parents;
  int32_t* v_pos;
  uint32_t* v_mask;            // [B][min(M, N)][ceil(min(M, N) / 32)]
  float* v_scores;             // or nullptr
};

cudaError_t launch_tree(const TreeArgs& a, cudaStream_t stream);

cudaError_t launch_mask_pack(const int32_t* parents, int B, int N, uint32_t* out_mask,
                             uint32_t* err, cudaStream_t stream);

cudaError_t launch_ngram_lookup(const void* slots, unsigned long long capacity, int n,
                                const int32_t* keys, long long Q, float* vals, int32_t* found,
                                cudaStream_t stream);

}  // namespace dart
