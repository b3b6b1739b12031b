// C ABI of libdomino: argument validation, workspace layout and dispatch to
// the kernels. Declarations and the meaning of every argument: domino.h.
#include <math.h>
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace domino {

namespace {
std::atomic<uint64_t> g_timeout_ns{2000000000ull};

inline size_t al256(size_t x) { return (x + 255) & ~(size_t)255; }

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

struct WsLayout {
  size_t ctl = 0;
  size_t keys = 0, S = 0, uacc = 0, uglob = 0, bat = 0, lsep = 0;
  size_t cand = 0, states = 0, cur = 0, tuacc = 0, topm = 0;
  size_t total = 0;
};

WsLayout layout(const domino_head* h, int bs, int P, int N, int M) {
  WsLayout L;
  size_t off = 256;
  // Argmax keys: one slot per (step, request, CTA) for the small-batch chain.
  L.keys = off; off += al256((size_t)P * bs * num_sms() * 8);
  L.S = off; off += al256((size_t)2 * bs * h->g * 8);
  L.uacc = off; off += al256((size_t)2 * bs * h->r * 16 * 8);
  L.uglob = off; off += al256((size_t)bs * h->r * 4);
  L.bat = off; off += al256(batched_ws_bytes(h->g));
  // Per-CTA log-sum-exp partials of the draft statistics [P][bs][num_sms] (float2).
  L.lsep = off; off += al256((size_t)P * bs * num_sms() * 8);
  if (N > 0 && M > 0) {
    L.cand = off; off += al256((size_t)bs * P * M * 4);
    L.states = off; off += al256((size_t)bs * N * h->g * 4);
    L.cur = off; off += al256((size_t)bs * (N + 1) * 4 * 4);
    L.tuacc = off; off += al256((size_t)bs * N * h->r * 8);
    L.topm = off; off += al256(topm_ws_bytes(bs * P, h->V, M));
  }
  L.total = off;
  return L;
}

domino_status check_head(const domino_head* h, bool need_table) {
  if (!h) return DOMINO_ERR_INVALID_ARG;
  if (h->dtype != DOMINO_F32 && h->dtype != DOMINO_BF16) return DOMINO_ERR_INVALID_ARG;
  if (h->d <= 0 || h->e <= 0 || h->g <= 0 || h->r <= 0 || h->V <= 0) return DOMINO_ERR_INVALID_ARG;
  const void* ptrs[] = {h->w_lm, h->emb, h->w_ih, h->w_hh, h->b_ih, h->b_hh, h->w1, h->w2};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return DOMINO_ERR_INVALID_ARG;
  if (need_table && (!h->gate_table || !aligned16(h->gate_table))) return DOMINO_ERR_INVALID_ARG;
  if (h->dtype == DOMINO_BF16 && ((h->d | h->e | h->g | h->r) & 7)) return DOMINO_ERR_UNSUPPORTED;
  if (h->dtype == DOMINO_F32 && ((h->d | h->e | h->g | h->r) & 3)) return DOMINO_ERR_UNSUPPORTED;
  if (h->r > 256) return DOMINO_ERR_UNSUPPORTED;
  return DOMINO_OK;
}

domino_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws || ((uintptr_t)ws & 255u) || ws_bytes < need) return DOMINO_ERR_WORKSPACE;
  return DOMINO_OK;
}

inline domino_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DOMINO_OK;
  if (e == cudaErrorInvalidConfiguration || e == cudaErrorCooperativeLaunchTooLarge) return DOMINO_ERR_UNSUPPORTED;
  return DOMINO_ERR_CUDA;
}


}  // namespace

struct ZeroArgs {
  unsigned long long* p[kMaxZeroRanges];
  size_t n8[kMaxZeroRanges];
  int n;
};

__global__ void zero_ranges_kernel(const __grid_constant__ ZeroArgs z) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (int r = 0; r < z.n; ++r)
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < z.n8[r]; i += stride) z.p[r][i] = 0ull;
}

cudaError_t zero_ranges(void* const* ptrs, const size_t* bytes, int n, cudaStream_t stream) {
  if (n < 0 || n > kMaxZeroRanges) return cudaErrorInvalidValue;
  ZeroArgs z;
  z.n = n;
  size_t most = 0;
  for (int r = 0; r < n; ++r) {
    if (((uintptr_t)ptrs[r] & 7u) || (bytes[r] & 7u)) return cudaErrorInvalidValue;
    z.p[r] = (unsigned long long*)ptrs[r];
    z.n8[r] = bytes[r] / 8;
    most = z.n8[r] > most ? z.n8[r] : most;
  }
  const int threads = 256;
  size_t blocks = (most + threads - 1) / threads;
  const size_t cap = (size_t)num_sms() * 4;
  blocks = blocks < 1 ? 1 : (blocks > cap ? cap : blocks);
  zero_ranges_kernel<<<(unsigned)blocks, threads, 0, stream>>>(z);
  return cudaGetLastError();
}

uint64_t wait_timeout_ns() { return g_timeout_ns.load(); }

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace domino

using namespace domino;

extern "C" {

int domino_abi_version(void) { return DOMINO_ABI_VERSION; }

const char* domino_status_str(int s) {
  switch (s) {
    case DOMINO_OK: return "DOMINO_OK";
    case DOMINO_ERR_INVALID_ARG: return "DOMINO_ERR_INVALID_ARG";
    case DOMINO_ERR_UNSUPPORTED: return "DOMINO_ERR_UNSUPPORTED";
    case DOMINO_ERR_CUDA: return "DOMINO_ERR_CUDA";
    case DOMINO_ERR_TIMEOUT: return "DOMINO_ERR_TIMEOUT";
    case DOMINO_ERR_WORKSPACE: return "DOMINO_ERR_WORKSPACE";
    case DOMINO_ERR_DEVICE_DATA: return "DOMINO_ERR_DEVICE_DATA";
    case DOMINO_ERR_INDEX: return "DOMINO_ERR_INDEX";
    default: return "DOMINO_ERR_UNKNOWN";
  }
}

size_t domino_workspace_bytes(const domino_head* head, int batch, int P, int n_nodes, int top_m) {
  if (!head || batch < 0 || P < 0 || n_nodes < 0 || top_m < 0 || head->g <= 0 || head->r <= 0) return 0;
  return layout(head, batch, P, n_nodes, top_m).total;
}

void domino_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1ull); }

domino_status domino_prepare_gate_table(const domino_head* h, float* table, void* ws, size_t ws_bytes,
                                        void* stream) {
  domino_status st = check_head(h, false);
  if (st != DOMINO_OK) return st;
  if (!table || !aligned16(table)) return DOMINO_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, 256)) != DOMINO_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  GemmA a{h->w_ih, h->e, 3 * h->g, table, (int64_t)3 * h->g, h->b_ih};
  cudaError_t e = h->dtype == DOMINO_BF16 ? gemm_bf16_tc(&a, 1, h->emb, h->e, h->V, h->e, (Ctl*)ws, s)
                                          : gemm_f32_simt(&a, 1, h->emb, h->e, h->V, h->e, s);
  return cuda_status(e);
}

domino_status domino_base_logits(const domino_head* h, const void* H, int batch, int P, float* L_base,
                                 float* P_h, void* ws, size_t ws_bytes, void* stream) {
  domino_status st = check_head(h, false);
  if (st != DOMINO_OK) return st;
  if (batch < 0 || P < 0) return DOMINO_ERR_INVALID_ARG;
  if (batch == 0 || P == 0) return DOMINO_OK;
  if (!H || !aligned16(H) || !L_base || !aligned16(L_base) || (P_h && !aligned16(P_h)))
    return DOMINO_ERR_INVALID_ARG;
  if ((st = check_ws(ws, ws_bytes, 256)) != DOMINO_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  GemmA probs[2] = {{h->w_lm, h->d, h->V, L_base, h->V, nullptr},
                    {h->w1, (int64_t)h->d + h->g, h->r, P_h, h->r, nullptr}};
  const int nprob = P_h ? 2 : 1;
  const int N = batch * P;
  cudaError_t e = h->dtype == DOMINO_BF16 ? gemm_bf16_tc(probs, nprob, H, h->d, N, h->d, (Ctl*)ws, s)
                                          : gemm_f32_simt(probs, nprob, H, h->d, N, h->d, s);
  return cuda_status(e);
}

static domino_status run_chain(const domino_head* h, const float* L_base, const float* P_h,
                               const int32_t* anchor, int batch, int P, float temperature, const float* gumbel,
                               int64_t gumbel_batch_stride, const int32_t* force_tokens, int32_t* tokens,
                               float* logits_out, float* u_out, float* lse_out, void* ws, size_t ws_bytes,
                               void* stream) {
  domino_status st = check_head(h, true);
  if (st != DOMINO_OK) return st;
  if (batch < 0 || P < 0) return DOMINO_ERR_INVALID_ARG;
  if (batch == 0 || P == 0) return DOMINO_OK;
  if (!L_base || !P_h || !anchor || !tokens) return DOMINO_ERR_INVALID_ARG;
  if (!(temperature >= 0.0f) || !isfinite(temperature)) return DOMINO_ERR_INVALID_ARG;
  if (temperature > 0.0f) {
    if (!gumbel || gumbel_batch_stride < (int64_t)P * h->V) return DOMINO_ERR_INVALID_ARG;
  }
  const WsLayout L = layout(h, batch, P, 0, 0);
  if ((st = check_ws(ws, ws_bytes, L.total)) != DOMINO_OK) return st;
  if (batch > 1024) return DOMINO_ERR_UNSUPPORTED;
  if (!chain_fits(h->dtype, batch, h->g, h->r)) return DOMINO_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* w = (uint8_t*)ws;
  // What the kernels expect at zero: the barrier counter and abort flag (not
  // the sticky status), the per-step argmax keys, the first bottleneck
  // accumulator buffer, the batched kernel's arrival counters and the
  // small-batch kernel's step-tagged GRU state words. The S16 / U16 operands
  // need no clearing: rows past 2 x batch only reach outputs the batched
  // kernel never reads.
  const size_t ctr_off = L.bat + (size_t)128 * h->g * 2 + (size_t)128 * 256 * 2;
  void* zp[5] = {ws, w + L.keys, w + L.uacc, w + ctr_off, w + L.S};
  const size_t zb[5] = {8, (size_t)P * batch * num_sms() * 8, (size_t)batch * h->r * 16 * 8, (size_t)3 * 256 * 32,
                        (size_t)2 * batch * h->g * 8};
  ChainArgs a;
  a.dtype = h->dtype; a.bs = batch; a.P = P; a.d = h->d; a.g = h->g; a.r = h->r; a.V = h->V;
  a.gate_table = h->gate_table; a.w_hh = h->w_hh; a.b_hh = h->b_hh; a.w1 = h->w1; a.w2 = h->w2;
  a.L_base = L_base; a.P_h = P_h; a.anchor = anchor;
  a.temperature = temperature; a.gumbel = temperature > 0.0f ? gumbel : nullptr;
  a.gumbel_bstride = gumbel_batch_stride;
  a.force = force_tokens; a.tokens = tokens; a.logits_out = logits_out;
  a.u_out = u_out; a.lse_out = lse_out; a.lse_part = (float2*)(w + L.lsep);
  a.ctl = (Ctl*)ws;
  a.keys = (unsigned long long*)(w + L.keys);
  a.S = (float*)(w + L.S);
  a.uacc = (long long*)(w + L.uacc);
  a.uglob = (float*)(w + L.uglob);
  a.s16 = (__nv_bfloat16*)(w + L.bat);
  a.u16 = (__nv_bfloat16*)(w + L.bat + (size_t)128 * h->g * 2);
  a.ctr = (unsigned int*)(w + L.bat + (size_t)128 * h->g * 2 + (size_t)128 * 256 * 2);
  a.bimg = w + L.bat + (size_t)128 * h->g * 2 + (size_t)128 * 256 * 2 + (size_t)3 * 256 * 32;
  if (lse_out && !chain_batched_applies(a)) return DOMINO_ERR_UNSUPPORTED;
  if (zero_ranges(zp, zb, 5, s) != cudaSuccess) return DOMINO_ERR_CUDA;
  return cuda_status(launch_chain(a, s));
}

domino_status domino_draft_chain(const domino_head* h, const float* L_base, const float* P_h,
                                 const int32_t* anchor, int batch, int P, float temperature,
                                 const float* gumbel, int64_t gumbel_batch_stride,
                                 const int32_t* force_tokens, int32_t* tokens, float* logits_out, void* ws,
                                 size_t ws_bytes, void* stream) {
  return run_chain(h, L_base, P_h, anchor, batch, P, temperature, gumbel, gumbel_batch_stride, force_tokens, tokens,
                   logits_out, nullptr, nullptr, ws, ws_bytes, stream);
}

int domino_draft_chain_stats_supported(const domino_head* h, int batch, int P) {
  if (check_head(h, false) != DOMINO_OK || batch < 1 || P < 1) return 0;
  return chain_batched_shape_ok(h->dtype, batch, P, h->g, h->r, h->V) ? 1 : 0;
}

domino_status domino_draft_chain_stats(const domino_head* h, const float* L_base, const float* P_h,
                                       const int32_t* anchor, int batch, int P, float temperature,
                                       const float* gumbel, int64_t gumbel_batch_stride,
                                       const int32_t* force_tokens, int32_t* tokens, float* u_out,
                                       float* lse_out, void* ws, size_t ws_bytes, void* stream) {
  if (batch > 0 && P > 0 && (!u_out || !lse_out || !aligned16(u_out))) return DOMINO_ERR_INVALID_ARG;
  return run_chain(h, L_base, P_h, anchor, batch, P, temperature, gumbel, gumbel_batch_stride, force_tokens, tokens,
                   nullptr, u_out, lse_out, ws, ws_bytes, stream);
}

domino_status domino_verify(const int32_t* draft, const int32_t* target, int batch, int P,
                            int32_t* accept_len, int32_t* advanced, void* stream) {
  if (batch < 0 || P < 0) return DOMINO_ERR_INVALID_ARG;
  if (batch == 0) return DOMINO_OK;
  if (!accept_len || !advanced) return DOMINO_ERR_INVALID_ARG;
  if (P > 0 && (!draft || !target)) return DOMINO_ERR_INVALID_ARG;
  return cuda_status(launch_verify(draft, target, batch, P, accept_len, advanced, (cudaStream_t)stream));
}

size_t domino_topm_workspace_bytes(int rows, int n, int top_m) {
  if (rows <= 0 || n <= 0 || top_m <= 0) return 0;
  return al256(topm_ws_bytes(rows, n, top_m));
}

domino_status domino_topm_select(const float* values, int rows, int n, int top_m, int32_t* ids_out,
                                 float* vals_out, void* ws, size_t ws_bytes, void* stream) {
  if (rows < 0 || n <= 0 || top_m < 1 || top_m > 256 || top_m > n) return DOMINO_ERR_INVALID_ARG;
  if (rows == 0) return DOMINO_OK;
  if (!values || !ids_out) return DOMINO_ERR_INVALID_ARG;
  if (rows > 65535) return DOMINO_ERR_UNSUPPORTED;
  domino_status st = check_ws(ws, ws_bytes, domino_topm_workspace_bytes(rows, n, top_m));
  if (st != DOMINO_OK) return st;
  return cuda_status(launch_topm(values, rows, n, top_m, ids_out, vals_out, ws, (cudaStream_t)stream));
}

// Scoring temperature of the trees: temperature 0 (greedy decoding) ranks by
// the draft's own log-softmax; T > 0 by log-softmax(l / T).
static bool tree_inv_tau(float temperature, float* inv_tau) {
  if (!(temperature >= 0.0f) || !isfinite(temperature)) return false;
  *inv_tau = temperature > 0.0f ? 1.0f / temperature : 1.0f;
  return isfinite(*inv_tau);
}

domino_status dominotree_build(const domino_head* h, const float* L_base, const float* P_h,
                               const int32_t* anchor, int batch, int P, int n_nodes, int top_m,
                               float temperature, int32_t* node_token, int32_t* node_parent,
                               int32_t* node_depth, float* node_score, void* ws, size_t ws_bytes,
                               void* stream) {
  domino_status st = check_head(h, true);
  if (st != DOMINO_OK) return st;
  if (batch < 0 || P < 0 || n_nodes < 1 || n_nodes > 64 || top_m < 1 || top_m > 256 || top_m > h->V)
    return DOMINO_ERR_INVALID_ARG;
  float inv_tau = 1.0f;
  if (!tree_inv_tau(temperature, &inv_tau)) return DOMINO_ERR_INVALID_ARG;
  if (batch == 0) return DOMINO_OK;
  if (!anchor || !node_token || !node_parent || !node_depth || !node_score) return DOMINO_ERR_INVALID_ARG;
  if (P > 0 && (!L_base || !P_h)) return DOMINO_ERR_INVALID_ARG;
  const WsLayout L = layout(h, batch, P, n_nodes, top_m);
  if ((st = check_ws(ws, ws_bytes, L.total)) != DOMINO_OK) return st;
  if (!tree_fits(h->dtype, batch, h->g, h->r, n_nodes, top_m)) return DOMINO_ERR_UNSUPPORTED;
  if (batch * P > 65535) return DOMINO_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* w = (uint8_t*)ws;
  // Barrier counter and abort flag, the published-node tags, the per-node
  // bottleneck accumulators and state words (nonzero once written) start at
  // zero.
  void* zp[4] = {ws, w + L.cur, w + L.tuacc, w + L.states};
  const size_t zb[4] = {8, (size_t)batch * (n_nodes + 1) * 4 * 4, (size_t)batch * n_nodes * h->r * 8,
                        (size_t)batch * n_nodes * h->g * 4};
  cudaError_t e = zero_ranges(zp, zb, 4, s);
  if (e != cudaSuccess) return DOMINO_ERR_CUDA;
  if (P > 0) {
    e = launch_topm(L_base, batch * P, h->V, top_m, (int32_t*)(w + L.cand), nullptr, w + L.topm, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  TreeArgs a;
  a.dtype = h->dtype; a.bs = batch; a.P = P; a.d = h->d; a.g = h->g; a.r = h->r; a.V = h->V;
  a.N = n_nodes; a.M = top_m; a.inv_tau = inv_tau;
  a.gate_table = h->gate_table; a.w_hh = h->w_hh; a.b_hh = h->b_hh; a.w1 = h->w1; a.w2 = h->w2;
  a.L_base = L_base; a.P_h = P_h; a.anchor = anchor;
  a.node_token = node_token; a.node_parent = node_parent; a.node_depth = node_depth;
  a.node_score = node_score;
  a.ctl = (Ctl*)ws;
  a.cand = (const int32_t*)(w + L.cand);
  a.states = (float*)(w + L.states);
  a.cur = (int32_t*)(w + L.cur);
  a.uacc = (long long*)(w + L.tuacc);
  return cuda_status(launch_tree(a, s));
}

domino_status dominotree_verify(const int32_t* node_token, const int32_t* node_parent, const int32_t* target_next,
                                int batch, int n_nodes, int32_t* accept_len, int32_t* advanced,
                                int32_t* accepted_path, uint8_t* mask, void* stream) {
  if (batch < 0 || n_nodes < 0 || n_nodes > 4096) return DOMINO_ERR_INVALID_ARG;
  if (batch == 0) return DOMINO_OK;
  if (!node_token || !node_parent || !target_next || !accept_len || !advanced) return DOMINO_ERR_INVALID_ARG;
  if (batch > (1 << 24)) return DOMINO_ERR_UNSUPPORTED;
  return cuda_status(launch_tree_verify(node_token, node_parent, target_next, batch, n_nodes + 1, accept_len,
                                        advanced, accepted_path, mask, (cudaStream_t)stream));
}

namespace {

struct HoLayout {
  size_t chain = 0, cand = 0, vals = 0, topm = 0, total = 0;
};

HoLayout ho_layout(int batch, int P, int V, int n_nodes, int top_m) {
  HoLayout L;
  size_t off = 256;  // control block
  L.chain = off; off += al256(headoff_chain_ws_bytes(batch * P));
  if (n_nodes > 0 && top_m > 0 && P > 0) {
    L.cand = off; off += al256((size_t)batch * P * top_m * 4);
    L.vals = off; off += al256((size_t)batch * P * top_m * 4);
    L.topm = off; off += al256(topm_ws_bytes(batch * P, V, top_m));
  }
  L.total = off;
  return L;
}

}  // namespace

size_t domino_headoff_workspace_bytes(int batch, int P, int V, int n_nodes, int top_m) {
  if (batch < 0 || P < 0 || V <= 0 || n_nodes < 0 || top_m < 0) return 0;
  return ho_layout(batch, P, V, n_nodes, top_m).total;
}

domino_status domino_draft_chain_headoff(const float* L_base, int batch, int P, int V, float temperature,
                                         const float* gumbel, int64_t gumbel_batch_stride, int32_t* tokens,
                                         void* ws, size_t ws_bytes, void* stream) {
  if (batch < 0 || P < 0 || V <= 0) return DOMINO_ERR_INVALID_ARG;
  if (batch == 0 || P == 0) return DOMINO_OK;
  if (!L_base || !tokens) return DOMINO_ERR_INVALID_ARG;
  if (!(temperature >= 0.0f) || !isfinite(temperature)) return DOMINO_ERR_INVALID_ARG;
  if (temperature > 0.0f && (!gumbel || gumbel_batch_stride < (int64_t)P * V)) return DOMINO_ERR_INVALID_ARG;
  const HoLayout L = ho_layout(batch, P, V, 0, 0);
  domino_status st = check_ws(ws, ws_bytes, L.total);
  if (st != DOMINO_OK) return st;
  if ((int64_t)batch * P > 65535) return DOMINO_ERR_UNSUPPORTED;
  uint8_t* w = (uint8_t*)ws;
  return cuda_status(launch_headoff_chain(L_base, batch, P, V, temperature, gumbel, gumbel_batch_stride, tokens,
                                          (Ctl*)ws, w + L.chain, (cudaStream_t)stream));
}

domino_status dominotree_build_marginal(const float* L_base, const int32_t* anchor, int batch, int P, int V,
                                        int n_nodes, int top_m, float temperature, int32_t* node_token,
                                        int32_t* node_parent, int32_t* node_depth, float* node_score, void* ws,
                                        size_t ws_bytes, void* stream) {
  if (batch < 0 || P < 0 || V <= 0 || n_nodes < 1 || n_nodes > 64 || top_m < 1 || top_m > 256 || top_m > V)
    return DOMINO_ERR_INVALID_ARG;
  float inv_tau = 1.0f;
  if (!tree_inv_tau(temperature, &inv_tau)) return DOMINO_ERR_INVALID_ARG;
  if (batch == 0) return DOMINO_OK;
  if (!anchor || !node_token || !node_parent || !node_depth || !node_score) return DOMINO_ERR_INVALID_ARG;
  if (P > 0 && !L_base) return DOMINO_ERR_INVALID_ARG;
  const HoLayout L = ho_layout(batch, P, V, n_nodes, top_m);
  domino_status st = check_ws(ws, ws_bytes, L.total);
  if (st != DOMINO_OK) return st;
  if ((int64_t)batch * P > 65535 || batch > 65535) return DOMINO_ERR_UNSUPPORTED;
  if (tree_marginal_smem_bytes(P, n_nodes, top_m) > 227 * 1024) return DOMINO_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* w = (uint8_t*)ws;
  if (P > 0) {
    const cudaError_t e = launch_topm(L_base, batch * P, V, top_m, (int32_t*)(w + L.cand), (float*)(w + L.vals),
                                      w + L.topm, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return cuda_status(launch_tree_marginal((const float*)(w + L.vals), (const int32_t*)(w + L.cand), anchor, batch,
                                          P, V, n_nodes, top_m, inv_tau, node_token, node_parent, node_depth,
                                          node_score, (Ctl*)ws, s));
}

size_t domino_verify_sampled_workspace_bytes(int batch, int P) {
  if (batch < 0 || P < 0) return 0;
  return 256 + al256(sampled_verify_ws_bytes(batch, P));
}

domino_status domino_verify_sampled(const int32_t* draft, const float* draft_logits, const float* target_logits,
                                    const float* uniform, const float* gumbel, int batch, int P, int V,
                                    float temperature, int32_t* accept_len, int32_t* advanced, int32_t* next_token,
                                    void* ws, size_t ws_bytes, void* stream) {
  if (batch < 0 || P < 0 || V <= 0) return DOMINO_ERR_INVALID_ARG;
  if (batch == 0) return DOMINO_OK;
  if (!(temperature > 0.0f) || !isfinite(temperature)) return DOMINO_ERR_INVALID_ARG;
  if (!target_logits || !gumbel || !accept_len || !advanced || !next_token) return DOMINO_ERR_INVALID_ARG;
  if (P > 0 && (!draft || !draft_logits || !uniform)) return DOMINO_ERR_INVALID_ARG;
  domino_status st = check_ws(ws, ws_bytes, domino_verify_sampled_workspace_bytes(batch, P));
  if (st != DOMINO_OK) return st;
  if (batch > 65535 || (int64_t)batch * (2 * P + 1) > (1 << 30)) return DOMINO_ERR_UNSUPPORTED;
  return cuda_status(launch_sampled_verify(draft, draft_logits, target_logits, uniform, gumbel, batch, P, V,
                                           temperature, accept_len, advanced, next_token, (Ctl*)ws,
                                           (uint8_t*)ws + 256, (cudaStream_t)stream));
}

size_t domino_verify_sampled_head_workspace_bytes(int batch, int P) {
  if (batch < 0 || P < 0) return 0;
  return 256 + al256(sampled_head_ws_bytes(batch));
}

domino_status domino_verify_sampled_head(const domino_head* h, const int32_t* draft, const float* L_base,
                                         const float* u, const float* lse, const float* target_logits,
                                         const float* uniform, const float* gumbel, int batch, int P,
                                         float temperature, int32_t* accept_len, int32_t* advanced,
                                         int32_t* next_token, void* ws, size_t ws_bytes, void* stream) {
  domino_status st = check_head(h, false);
  if (st != DOMINO_OK) return st;
  if (batch < 0 || P < 0) return DOMINO_ERR_INVALID_ARG;
  if (batch == 0) return DOMINO_OK;
  if (!(temperature > 0.0f) || !isfinite(temperature)) return DOMINO_ERR_INVALID_ARG;
  if (!target_logits || !gumbel || !accept_len || !advanced || !next_token) return DOMINO_ERR_INVALID_ARG;
  if (P > 0 && (!draft || !L_base || !u || !lse || !uniform || !aligned16(u))) return DOMINO_ERR_INVALID_ARG;
  if (h->dtype != DOMINO_BF16 || h->r != 256) return DOMINO_ERR_UNSUPPORTED;
  if ((st = check_ws(ws, ws_bytes, domino_verify_sampled_head_workspace_bytes(batch, P))) != DOMINO_OK) return st;
  if (batch > 65535 || (int64_t)batch * (2 * P + 1) > (1 << 30)) return DOMINO_ERR_UNSUPPORTED;
  uint8_t* w = (uint8_t*)ws + 256;
  SampledHeadArgs a;
  a.draft = draft; a.L_base = L_base; a.w2 = h->w2; a.u = u; a.lse = lse;
  a.Z = target_logits; a.U = uniform; a.G = gumbel;
  a.bs = batch; a.P = P; a.V = h->V; a.temperature = temperature;
  a.accept = accept_len; a.advanced = advanced; a.next_token = next_token;
  a.ctl = (Ctl*)ws;
  a.rej_j = (int32_t*)w;
  w += al256((size_t)batch * 4);
  a.rej_norm = (float*)w;
  w += al256((size_t)batch * 8);
  a.rd_keys = (unsigned long long*)w;
  w += al256((size_t)batch * 8);
  a.rd_done = (unsigned int*)w;
  return cuda_status(launch_sampled_verify_head(a, (cudaStream_t)stream));
}

domino_status domino_last_status(void* ws, void* stream) {
  if (!ws || ((uintptr_t)ws & 255u)) return DOMINO_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  unsigned int host = 0;
  uint8_t* w = (uint8_t*)ws;
  if (cudaMemcpyAsync(&host, w + offsetof(Ctl, status), 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DOMINO_ERR_CUDA;
  if (cudaMemsetAsync(w + offsetof(Ctl, status), 0, 4, s) != cudaSuccess) return DOMINO_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DOMINO_ERR_CUDA;
  if (host & DEV_ERR_TIMEOUT) return DOMINO_ERR_TIMEOUT;
  if (host & DEV_ERR_INDEX) return DOMINO_ERR_INDEX;
  if (host & DEV_ERR_DATA) return DOMINO_ERR_DEVICE_DATA;
  return DOMINO_OK;
}

domino_status domino_selftest_wait_timeout(uint64_t timeout_ns, void* ws, size_t ws_bytes, void* stream) {
  domino_status st = check_ws(ws, ws_bytes, 256);
  if (st != DOMINO_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemsetAsync((uint8_t*)ws + offsetof(Ctl, never), 0, 8, s) != cudaSuccess) return DOMINO_ERR_CUDA;
  return cuda_status(launch_wait_selftest((Ctl*)ws, timeout_ns, s));
}

domino_status domino_selftest_rates(int which, int arg, int64_t* out, void* ws, size_t ws_bytes, void* stream) {
  if (!out || ((uintptr_t)out & 7u)) return DOMINO_ERR_INVALID_ARG;
  domino_status st = check_ws(ws, ws_bytes, 512);
  if (st != DOMINO_OK) return st;
  if (which == 0) {
    if (arg < 1 || arg >= num_sms()) return DOMINO_ERR_INVALID_ARG;
  } else if (which == 1 || which == 2) {
    if (arg < 1 || arg > (1 << 20)) return DOMINO_ERR_INVALID_ARG;
  } else {
    return DOMINO_ERR_INVALID_ARG;
  }
  return cuda_status(launch_rate_selftest(which, arg, (long long*)out, (Ctl*)ws, (uint8_t*)ws + 256,
                                          (cudaStream_t)stream));
}

}  // extern "C"
