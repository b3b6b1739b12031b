// Host-side declarations shared by the translation units of libdomino.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/domino.h"

namespace domino {

struct Ctl;

// Process-wide bound of device-side waits (ns).
uint64_t wait_timeout_ns();

// Number of SMs of the current device (cached per device).
int num_sms();

// One A operand of a batched GEMM sharing its B operand:
//   out[n * ldo + m] = sum_k A[m * lda + k] * B[n * ldb + k] (+ bias[m])
// for m < M, n < N, k < K. A, B and bias have the head's element type.
struct GemmA {
  const void* A;
  int64_t lda;
  int M;
  float* out;
  int64_t ldo;
  const void* bias;  // may be null
};

// bf16 operands on tcgen05 tensor cores (TMA-fed, TMEM accumulators).
cudaError_t gemm_bf16_tc(const GemmA* probs, int nprob, const void* B, int64_t ldb, int N, int K,
                         Ctl* ctl, cudaStream_t stream);
// fp32 operands on CUDA cores.
cudaError_t gemm_f32_simt(const GemmA* probs, int nprob, const void* B, int64_t ldb, int N, int K,
                          cudaStream_t stream);

struct ChainArgs {
  int dtype, bs, P, d, g, r, V;
  const float* gate_table;
  const void* w_hh;
  const void* b_hh;
  const void* w1;
  const void* w2;
  const float* L_base;
  const float* P_h;
  const int32_t* anchor;
  float temperature;
  const float* gumbel;
  int64_t gumbel_bstride;
  const int32_t* force;
  int32_t* tokens;
  float* logits_out;
  // Draft statistics in place of the logits (batched kernel only): u_i
  // [bs][P][r] and logsumexp_v L_i[v] / T' [bs][P], per-CTA partials in
  // lse_part [P][bs][num_sms] (float2). Null when not wanted.
  float* u_out = nullptr;
  float* lse_out = nullptr;
  float2* lse_part = nullptr;
  // workspace pieces
  Ctl* ctl;
  unsigned long long* keys;  // [P][bs]
  float* S;                  // [2][bs][g] floats; small-batch kernel: [2][bs][g] tagged u64 words
  long long* uacc;           // [2][bs*r] padded to 16 per entry
  float* uglob;              // [bs][r]
  // batched (tensor-core) chain only; null when not provided
  __nv_bfloat16* s16;        // [128][g]
  __nv_bfloat16* u16;        // [128][r]
  unsigned int* ctr;         // [3][P + 1] counters, 32 bytes apart
  uint8_t* bimg;             // per-CTA operand images
};
// Zero up to kMaxZeroRanges byte ranges (8-byte aligned, sizes multiples of
// 8) in one launch: the per-call scratch reset before a chain.
constexpr int kMaxZeroRanges = 5;
cudaError_t zero_ranges(void* const* ptrs, const size_t* bytes, int n, cudaStream_t stream);
size_t chain_ws_bytes(int bs, int P, int g, int r);
bool chain_fits(int dtype, int bs, int g, int r);
cudaError_t launch_chain(const ChainArgs& a, cudaStream_t stream);
// Small-batch specialisation (bf16, rank 256, batch <= 4) with W2 resident on chip.
bool chain_small_applies(const ChainArgs& a);
cudaError_t launch_chain_small(const ChainArgs& a, cudaStream_t stream);
// Batched specialisation (bf16, rank 256, 5 <= batch <= 64) on tcgen05 tensor cores.
size_t batched_ws_bytes(int g);
bool chain_batched_applies(const ChainArgs& a);
bool chain_batched_shape_ok(int dtype, int bs, int P, int g, int r, int V);
cudaError_t launch_chain_batched(const ChainArgs& a, cudaStream_t stream);

cudaError_t launch_verify(const int32_t* draft, const int32_t* target, int bs, int P,
                          int32_t* accept, int32_t* advanced, cudaStream_t stream);

size_t topm_ws_bytes(int rows, int n, int M);
cudaError_t launch_topm(const float* values, int rows, int n, int M, int32_t* ids, float* vals,
                        void* scratch, cudaStream_t stream);

struct TreeArgs {
  int dtype, bs, P, d, g, r, V, N, M;
  float inv_tau;  // 1 / scoring temperature (1 for greedy decoding)
  const float* gate_table;
  const void* w_hh;
  const void* b_hh;
  const void* w1;
  const void* w2;
  const float* L_base;
  const float* P_h;
  const int32_t* anchor;
  int32_t* node_token;
  int32_t* node_parent;
  int32_t* node_depth;
  float* node_score;
  Ctl* ctl;
  const int32_t* cand;  // [bs][P][M]
  float* states;        // [bs][N][g] node states (nonzero bits once written), zeroed per build
  long long* uacc;      // [bs][N][r] W1_s S per node (counted fixed-point sums), zeroed per build
  int32_t* cur;         // [bs][N + 1][4] published nodes
};
size_t tree_ws_bytes(int bs, int P, int g, int r, int N, int M);
bool tree_fits(int dtype, int bs, int g, int r, int N, int M);
cudaError_t launch_tree(const TreeArgs& a, cudaStream_t stream);

cudaError_t launch_wait_selftest(Ctl* ctl, uint64_t timeout_ns, cudaStream_t stream);
cudaError_t launch_rate_selftest(int which, int arg, long long* out, Ctl* ctl, void* scratch,
                                 cudaStream_t stream);

// Tree acceptance: mask and accepted path of a drafted tree.
cudaError_t launch_tree_verify(const int32_t* tok, const int32_t* par, const int32_t* tgt, int bs, int n1,
                               int32_t* accept, int32_t* advanced, int32_t* path, uint8_t* mask,
                               cudaStream_t stream);
// Verification at T > 0: row logsumexps, accept decisions, residual draw.
size_t sampled_verify_ws_bytes(int bs, int P);
cudaError_t launch_sampled_verify(const int32_t* draft, const float* L, const float* Z, const float* U,
                                  const float* G, int bs, int P, int V, float temperature, int32_t* accept,
                                  int32_t* advanced, int32_t* next_token, Ctl* ctl, void* scratch,
                                  cudaStream_t stream);
// Verification at T > 0 from the head (draft statistics, no draft logits):
// the walk in head form, then the residual draw that rebuilds the rejected
// rows from W2 for all rejected requests at once.
struct SampledHeadArgs {
  const int32_t* draft;
  const float* L_base;
  const void* w2;  // bf16 [V, 256]
  const float* u;
  const float* lse;
  const float* Z;
  const float* U;
  const float* G;
  int bs, P, V;
  float temperature;
  int32_t* accept;
  int32_t* advanced;
  int32_t* next_token;
  Ctl* ctl;
  int32_t* rej_j;               // [bs]
  float* rej_norm;              // [bs][2]
  unsigned long long* rd_keys;  // [bs], zero between calls
  unsigned int* rd_done;        // one counter per 64-request window, 32 bytes apart, zero between calls
};
size_t sampled_head_ws_bytes(int bs);
cudaError_t launch_sampled_verify_head(const SampledHeadArgs& a, cudaStream_t stream);
cudaError_t launch_residual_draw(const SampledHeadArgs& a, cudaStream_t stream);
// Head-off baselines: per-row argmax of L_base (self-cleaning row scratch),
// and the marginal best-first tree from the top-M candidates.
size_t headoff_chain_ws_bytes(int rows);
cudaError_t launch_headoff_chain(const float* L_base, int bs, int P, int V, float temperature, const float* gumbel,
                                 int64_t gstride, int32_t* tokens, Ctl* ctl, void* scratch, cudaStream_t stream);
size_t tree_marginal_smem_bytes(int P, int N, int M);
cudaError_t launch_tree_marginal(const float* cand_val, const int32_t* cand_id, const int32_t* anchor, int bs,
                                 int P, int V, int N, int M, float inv_tau, int32_t* node_token,
                                 int32_t* node_parent, int32_t* node_depth, float* node_score, Ctl* ctl,
                                 cudaStream_t stream);

}  // namespace domino
