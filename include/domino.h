/*
 * domino.h -- C ABI of the GB300 (sm_103a) Domino drafting hot path.
 *
 * The method (sources, by page title):
 *  - "Technische Samenvatting: Domino" (gist.science), "Methodologie: Domino":
 *    a parallel backbone yields hidden states H_i for a whole draft block; base
 *    logits come from the frozen target LM head; a GRU causal encoder summarises
 *    the preceding drafted tokens into S_{i-1}; a low-rank head maps [H_i; S_{i-1}]
 *    through W1, SiLU and W2 to correction logits; L_i = L_base_i + dL_i and the
 *    token is drawn from L_i.
 *  - "上交大突破：多米诺推理策略实现AI推理速度近6倍能力提升" (163.com), section 四:
 *    GRU hidden 1024, bottleneck 256, correction in logit space.
 *  - "Domino: Decoupling Causal Modeling from Autoregressive Drafting in
 *    Speculative Decoding Review", sections 1-1 and 3-2: anchor + masked block,
 *    tokens advanced per cycle.
 *  - "DominoTree: Conditional Tree-Structured Drafting with Domino for
 *    Speculative Decoding" (gist.science), "核心组件": best-first heap keyed by
 *    cumulative log-probability, per-path GRU correction, top-M candidates.
 *
 * Conventions for every entry point:
 *  - Pointers named as device pointers are CUDA device memory owned by the
 *    caller; the library never allocates, frees or keeps them.
 *  - `stream` is a cudaStream_t passed as void*. Every call only enqueues work
 *    on it and returns; the host never waits inside a call.
 *  - Host-side argument errors return DOMINO_ERR_INVALID_ARG or
 *    DOMINO_ERR_UNSUPPORTED before anything is enqueued. A failed launch returns
 *    DOMINO_ERR_CUDA.
 *  - Errors found on the device (a bounded wait that ran out, an out-of-range
 *    token id, a bottleneck partial sum too large for the fixed-point
 *    accumulators) set a sticky status word inside the
 *    workspace `ws`; domino_last_status() synchronises the stream, returns it and
 *    clears it. Kernels never trap: they record the error and return.
 *  - Row-major layouts; weights use the nn.Linear layout [out, in].
 *  - L_base, P_h and the noise are expected finite; in greedy drafting an
 *    -inf or +inf entry of L_base ranks as the extreme it is. With a NaN among
 *    them the drafted token is unspecified (a valid id; no error is reported).
 *  - A block has B positions: the anchor (position 0) plus P = B - 1 drafted
 *    positions. Arrays with a position axis hold the P drafted rows; row i is
 *    block position i + 1.
 *  - Calls that share one workspace must be ordered on one stream.
 */
#ifndef DOMINO_H
#define DOMINO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DOMINO_ABI_VERSION 3

typedef enum {
  DOMINO_OK = 0,
  DOMINO_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer */
  DOMINO_ERR_UNSUPPORTED = 2,  /* valid but outside what the kernels implement */
  DOMINO_ERR_CUDA = 3,         /* a CUDA call or launch failed */
  DOMINO_ERR_TIMEOUT = 4,      /* a device-side bounded wait ran out */
  DOMINO_ERR_WORKSPACE = 5,    /* workspace null, too small or misaligned */
  DOMINO_ERR_DEVICE_DATA = 6,  /* device found a token id out of range or an out-of-range
                                  fixed-point partial */
  DOMINO_ERR_INDEX = 7         /* checked build (libdomino_checked.so) only: a device-side index
                                  check failed; the access was skipped */
} domino_status;

typedef enum { DOMINO_F32 = 0, DOMINO_BF16 = 1 } domino_dtype;

/*
 * The Domino head plus the frozen target LM head and token embedding.
 * All weight pointers are device pointers of element type `dtype`.
 *   w_lm [V, d]      frozen target LM head (base logits L_base = H W_lm^T)
 *   emb  [V, e]      target token embedding (GRU input)
 *   w_ih [3g, e], w_hh [3g, g], b_ih [3g], b_hh [3g]
 *                    GRU cell, gate rows ordered r, z, n:
 *                    r = s(W_ir x + b_ir + W_hr h + b_hr), z = likewise,
 *                    n = tanh(W_in x + b_in + r * (W_hn h + b_hn)),
 *                    h' = (1 - z) n + z h
 *   w1   [r, d + g]  bottleneck; columns [0, d) act on H_i, [d, d + g) on S_{i-1}
 *   w2   [V, r]      low-rank map back to the vocabulary (no biases in W1, W2)
 *   gate_table [V, 3g] fp32 device buffer holding emb W_ih^T + b_ih, filled by
 *                    domino_prepare_gate_table(); the chain and tree read it
 *                    instead of projecting emb rows on every step.
 * bf16 requires d, e, g, r to be multiples of 8 and every pointer 16-byte
 * aligned (tensor-memory-access rules); f32 requires 16-byte alignment too.
 */
typedef struct {
  int32_t dtype;
  int32_t d, e, g, r, V;
  const void* w_lm;
  const void* emb;
  const void* w_ih;
  const void* w_hh;
  const void* b_ih;
  const void* b_hh;
  const void* w1;
  const void* w2;
  const float* gate_table;
} domino_head;

/* ABI version of the loaded library (DOMINO_ABI_VERSION). */
int domino_abi_version(void);

/* Human-readable name of a status code. Never NULL. */
const char* domino_status_str(int status);

/*
 * Bytes of device workspace needed by calls on (batch, P) and, for the tree,
 * (n_nodes, top_m); pass 0 for the tree sizes when no tree is built. The
 * workspace must be 256-byte aligned (cudaMalloc memory is). Zero it once
 * before its first use (its first 256 bytes hold the sticky status word);
 * after that every call resets the scratch it uses.
 */
size_t domino_workspace_bytes(const domino_head* head, int batch, int P, int n_nodes, int top_m);

/*
 * Fill table[v, q] = sum_k emb[v, k] W_ih[q, k] + b_ih[q] (fp32, [V, 3g]):
 * the input half of every GRU step, precomputed once per head. `table` is a
 * device buffer of V * 3g floats (it may be head->gate_table). Algebraically
 * identical to projecting the embedding row at each step (GRU input term,
 * "上交大突破…", section 四). ws may be any workspace of at least 256 bytes.
 */
domino_status domino_prepare_gate_table(const domino_head* head, float* table,
                                        void* ws, size_t ws_bytes, void* stream);

/*
 * Base pass over a draft block ("Technische Samenvatting: Domino",
 * "Parallel Draft-ruggengraat"): everything that depends on H only.
 *   H      [batch, P, d] device, head->dtype: backbone hidden states of the
 *          drafted positions.
 *   L_base [batch, P, V] device fp32 out: L_base = H W_lm^T.
 *   P_h    [batch, P, r] device fp32 out, or NULL: H W1[:, :d]^T, the H-half
 *          of the bottleneck pre-activation (exact split of W1 [H; S]).
 * fp32 accumulation; bf16 inputs are exact in fp32 products.
 */
domino_status domino_base_logits(const domino_head* head, const void* H, int batch, int P,
                                 float* L_base, float* P_h,
                                 void* ws, size_t ws_bytes, void* stream);

/*
 * The sequential Domino head chain ("Technische Samenvatting: Domino",
 * "Domino-head"), per request b, for i = 0..P-1:
 *   S_0 = GRU(emb[anchor[b]], 0)   (state after the anchor)
 *   u_i = SiLU(P_h[b, i] + W1[:, d:] S_i)
 *   L_i = L_base[b, i] + W2 u_i
 *   tokens[b, i] = argmax(L_i)                        if temperature == 0
 *                = argmax(L_i / temperature + G[b,i]) otherwise (Gumbel-max)
 *   (ties to the lowest token id)
 *   S_{i+1} = GRU(emb[x], S_i), x = force_tokens[b, i] if given, else tokens[b, i]
 * Arguments:
 *   L_base [batch, P, V], P_h [batch, P, r]  device fp32, from domino_base_logits
 *   anchor [batch] device int32 token ids
 *   temperature >= 0; when > 0, gumbel must be a device fp32 pointer with
 *     G[b, i, v] = gumbel[b * gumbel_batch_stride + i * V + v] (row i =
 *     block position i + 1); ignored when temperature == 0.
 *   force_tokens [batch, P] device int32 or NULL (teacher-forced GRU inputs;
 *     the last column is never read).
 *   tokens [batch, P] device int32 out.
 *   logits_out [batch, P, V] device fp32 out or NULL: the corrected logits L_i.
 * The chain runs as one persistent kernel (one CTA per SM); head->gate_table
 * must be prepared.
 */
domino_status domino_draft_chain(const domino_head* head, const float* L_base, const float* P_h,
                                 const int32_t* anchor, int batch, int P, float temperature,
                                 const float* gumbel, int64_t gumbel_batch_stride,
                                 const int32_t* force_tokens, int32_t* tokens, float* logits_out,
                                 void* ws, size_t ws_bytes, void* stream);

/*
 * The same chain, returning in place of the corrected logits what a
 * verification at temperature T needs of the draft (163.com report, section
 * 五, standard speculative-decoding verification; the draft distribution is
 * q_i = softmax(L_i / T)): from u_i any single logit follows as
 * L_i[v] = L_base[b, i, v] + W2[v] . u_i, and lse_out normalises them.
 *   u_out   [batch, P, r] device fp32 out (16-byte aligned): u_i of the chain
 *           (the bottleneck activations SiLU(P_h[b, i] + W1[:, d:] S_i)).
 *   lse_out [batch, P] device fp32 out: logsumexp_v L_i[v] / T' with T' = T
 *           when temperature > 0, else 1.
 * Other arguments, the tokens and the workspace as domino_draft_chain. Only
 * the tensor-core batched chain computes these (bf16 head, r = 256,
 * 1 <= batch <= 64, V % 4 == 0, g % 64 == 0, 16-byte aligned L_base and
 * noise): other shapes return DOMINO_ERR_UNSUPPORTED, and
 * domino_draft_chain_stats_supported(head, batch, P) says which (1 or 0;
 * buffer alignment is checked at the call). At batch <= 4 the plain chain
 * runs a faster kernel, and its full logits (logits_out of
 * domino_draft_chain) are the cheaper form there.
 * The pages define no such interface: it splits their verification step at
 * the point where the full logits would otherwise travel through memory.
 */
int domino_draft_chain_stats_supported(const domino_head* head, int batch, int P);
domino_status domino_draft_chain_stats(const domino_head* head, const float* L_base, const float* P_h,
                                       const int32_t* anchor, int batch, int P, float temperature,
                                       const float* gumbel, int64_t gumbel_batch_stride,
                                       const int32_t* force_tokens, int32_t* tokens, float* u_out,
                                       float* lse_out, void* ws, size_t ws_bytes, void* stream);

/*
 * Longest accepted prefix ("Domino: Decoupling … Review", section 1-1; the
 * target checks the block in one pass and A tokens are advanced per cycle):
 *   accept_len[b] = max k <= P with draft[b, 0..k-1] == target[b, 0..k-1]
 *   advanced[b]   = accept_len[b] + 1 (the target's own next token)
 * All arrays are device int32: draft, target [batch, P]; accept_len,
 * advanced [batch]. Uses no workspace.
 */
domino_status domino_verify(const int32_t* draft, const int32_t* target, int batch, int P,
                            int32_t* accept_len, int32_t* advanced, void* stream);

/*
 * Top-M candidate limit ("DominoTree…", "候选限制（Top-M）"): for each of `rows`
 * rows of `values` ([rows, n] device fp32), the ids of the top_m largest
 * values ordered by value descending, then id ascending; ids_out [rows, top_m]
 * device int32, vals_out [rows, top_m] device fp32 (may be NULL).
 * Requires 1 <= top_m <= 256 and top_m <= n. Values must not be NaN.
 * Workspace: domino_topm_workspace_bytes(rows, n, top_m) bytes, zeroed before
 * its first use; each call leaves it ready for the next.
 */
size_t domino_topm_workspace_bytes(int rows, int n, int top_m);
domino_status domino_topm_select(const float* values, int rows, int n, int top_m,
                                 int32_t* ids_out, float* vals_out,
                                 void* ws, size_t ws_bytes, void* stream);

/*
 * DominoTree best-first build ("DominoTree…", "条件评分的最佳优先堆"), per request:
 *   node 0 = root: token anchor[b], parent -1, depth 0, score 0,
 *            state GRU(emb[anchor], 0);
 *   C_t = top_m ids of L_base[b, t] (value desc, id asc), t = 0..P-1;
 *   expanding node n at depth t < P with state S_n: for c in C_t
 *     l_c = L_base[b, t, c] + W2[c] . SiLU(P_h[b, t] + W1[:, d:] S_n),
 *     logp_c = l_c / tau - logsumexp_{c' in C_t} l_{c'} / tau,
 *     child score = score(n) + logp_c (fp32);
 *   tau = temperature when temperature > 0 (the decoding temperatures the
 *   page evaluates the tree at, 实验结果: 0, 0.5, 1), tau = 1 when
 *   temperature == 0 (greedy decoding ranks by the draft's own
 *   log-probabilities); a negative or non-finite temperature is
 *   DOMINO_ERR_INVALID_ARG;
 *   pop the largest score (ties: smaller parent id, then smaller token id);
 *   node ids 1..n_nodes in pop order; a popped node k < n_nodes at depth < P
 *   gets S_k = GRU(emb[token_k], S_parent) and is expanded.
 * Outputs [batch, n_nodes + 1] device: node_token, node_parent, node_depth
 * (int32) and node_score (fp32); slots left when the candidate tree has fewer
 * than n_nodes nodes hold -1, -1, -1, -inf.
 * Requires 1 <= n_nodes <= 64, 1 <= top_m <= 256, batch < number of SMs (one
 * SM per request expands it; the others run the GRU steps), and a prepared
 * gate table.
 */
domino_status dominotree_build(const domino_head* head, const float* L_base, const float* P_h,
                               const int32_t* anchor, int batch, int P, int n_nodes, int top_m,
                               float temperature, int32_t* node_token, int32_t* node_parent,
                               int32_t* node_depth, float* node_score, void* ws, size_t ws_bytes,
                               void* stream);

/*
 * Tree acceptance ("DominoTree…", section 验证: tree-attention verification
 * with an ancestor-only causal mask, unchanged and lossless). The target pass
 * is the caller's: target_next[b, n] is the target's greedy next token after
 * node n's root path (node 0 = the anchor). Per request:
 *   walk from node 0; at node n move to the child c (node_parent[c] == n,
 *   node_token[c] >= 0) with node_token[c] == target_next[n] (siblings carry
 *   distinct tokens; the lowest such id if not); stop when none matches;
 *   accept_len[b] = depth of the last node reached, advanced[b] = accept_len + 1;
 *   accepted_path[b, k] = node id at depth k of that walk, -1 after it;
 *   mask[b, i, j] = 1 iff node j is node i or an ancestor of node i (the
 *   attention mask of the verification pass), rows of empty slots all 0.
 * Inputs [batch, n_nodes + 1] device int32 as dominotree_build writes them
 * (parents precede children; a parent outside [0, i) ends an ancestor walk);
 * outputs device: accept_len, advanced [batch] int32, accepted_path
 * [batch, n_nodes + 1] int32 (may be NULL), mask [batch, n_nodes + 1,
 * n_nodes + 1] uint8 (may be NULL). Uses no workspace.
 */
domino_status dominotree_verify(const int32_t* node_token, const int32_t* node_parent,
                                const int32_t* target_next, int batch, int n_nodes,
                                int32_t* accept_len, int32_t* advanced, int32_t* accepted_path,
                                uint8_t* mask, void* stream);

/*
 * Verification at temperature T > 0 (163.com report, section 五: drafts are
 * checked by the standard speculative-decoding procedure and the output keeps
 * the target's probabilities; "DominoTree…", 实验结果: lossless). With
 * q_i = softmax(draft_logits[b, i] / T), p_i = softmax(target_logits[b, i] / T):
 *   accept draft[b, i] while uniform[b, i] < p_i(x) / q_i(x); at the first
 *   rejection j, next_token[b] = argmax_v log max(0, p_j - q_j)_v + gumbel[b, v]
 *   (a draw from the normalised residual; from p_j if the residual is zero
 *   everywhere in fp32); if all P are accepted (j = P), next_token[b] =
 *   argmax_v log p_P(v) + gumbel[b, v];
 *   accept_len[b] = j, advanced[b] = j + 1.
 * Device arrays: draft [batch, P] int32; draft_logits [batch, P, V] fp32 (the
 * chain's logits_out); target_logits [batch, P + 1, V] fp32 (the target's
 * logits at the drafted positions and the one after); uniform [batch, P] fp32
 * in (0, 1); gumbel [batch, V] fp32 standard Gumbel noise; outputs
 * accept_len, advanced, next_token [batch] int32. Requires temperature > 0.
 * Positions are tested in order and the walk stops at the first rejection, so
 * the draft and target rows after it are not read.
 * Workspace: domino_verify_sampled_workspace_bytes(batch, P) bytes (it holds
 * the status word), zeroed before its first use; each call leaves it ready
 * for the next. Device-side data errors are reported by
 * domino_last_status(ws, stream).
 */
size_t domino_verify_sampled_workspace_bytes(int batch, int P);
domino_status domino_verify_sampled(const int32_t* draft, const float* draft_logits,
                                    const float* target_logits, const float* uniform, const float* gumbel,
                                    int batch, int P, int V, float temperature, int32_t* accept_len,
                                    int32_t* advanced, int32_t* next_token, void* ws, size_t ws_bytes,
                                    void* stream);

/*
 * The same verification with the draft given by the head and the chain's
 * statistics (domino_draft_chain_stats) instead of its logits:
 *   q_i(x) = exp(L_i[x] / T - lse[b, i]), L_i[x] = L_base[b, i, x] + W2[x] . u[b, i];
 * the residual draw at the first rejection j rebuilds row L_j in full, for
 * all rejected requests of the call in one pass over W2. Same decisions,
 * outputs and conditions as domino_verify_sampled; the draft-side rows read
 * are W2 and, per rejected request, L_base[b, j] (no [batch, P, V] draft
 * logits exist). head: bf16 with r = 256 (else DOMINO_ERR_UNSUPPORTED).
 * Device arrays: draft [batch, P] int32; L_base [batch, P, V] fp32 (from
 * domino_base_logits); u [batch, P, 256] fp32, 16-byte aligned; lse [batch, P]
 * fp32 (both from domino_draft_chain_stats at the same temperature);
 * target_logits, uniform, gumbel, accept_len, advanced, next_token as
 * domino_verify_sampled.
 * Workspace: domino_verify_sampled_head_workspace_bytes(batch, P) bytes,
 * 256-byte aligned, zeroed before its first use; each call leaves it ready
 * for the next. Device-side data errors are reported by domino_last_status.
 */
size_t domino_verify_sampled_head_workspace_bytes(int batch, int P);
domino_status domino_verify_sampled_head(const domino_head* head, const int32_t* draft, const float* L_base,
                                         const float* u, const float* lse, const float* target_logits,
                                         const float* uniform, const float* gumbel, int batch, int P,
                                         float temperature, int32_t* accept_len, int32_t* advanced,
                                         int32_t* next_token, void* ws, size_t ws_bytes, void* stream);

/*
 * The pages' baselines with the correction head off (the full method with
 * W2 = 0), which need no head weights:
 *
 * domino_draft_chain_headoff ("…Speculative Decoding Review" sections 1-1 and
 * 3-2, 163.com section 四: the parallel backbone alone drafts each position
 * from its marginal logits):
 *   tokens[b, i] = argmax_v L_base[b, i, v]              (temperature == 0)
 *   tokens[b, i] = argmax_v L_base[b, i, v] / T + G[b, i, v]  (T > 0)
 * ties to the lowest id; L_base [batch, P, V] and gumbel (row i at gumbel +
 * b * gumbel_batch_stride + i * V) device fp32; tokens [batch, P] int32.
 *
 * dominotree_build_marginal ("DominoTree…", 核心贡献, the marginal-scoring
 * ablation): dominotree_build with logp_c = L_base[b, t, c] / tau - logsumexp
 * over C_t of L_base / tau (no GRU, no correction; tau from temperature as in
 * dominotree_build); same outputs, same limits on n_nodes / top_m.
 *
 * Workspace for both: domino_headoff_workspace_bytes(batch, P, V, n_nodes,
 * top_m) bytes (n_nodes = top_m = 0 for the chain alone), 256-byte aligned,
 * zeroed before its first use; after a call it is left ready for the next
 * one. Requires batch * P <= 65535. Device-side data errors are reported by
 * domino_last_status(ws, stream).
 */
size_t domino_headoff_workspace_bytes(int batch, int P, int V, int n_nodes, int top_m);
domino_status domino_draft_chain_headoff(const float* L_base, int batch, int P, int V,
                                         float temperature, const float* gumbel,
                                         int64_t gumbel_batch_stride, int32_t* tokens, void* ws,
                                         size_t ws_bytes, void* stream);
domino_status dominotree_build_marginal(const float* L_base, const int32_t* anchor, int batch, int P,
                                        int V, int n_nodes, int top_m, float temperature,
                                        int32_t* node_token, int32_t* node_parent, int32_t* node_depth,
                                        float* node_score, void* ws, size_t ws_bytes, void* stream);

/*
 * domino_draft_chain without a workspace, for callers that cannot allocate
 * device memory themselves (a framework pool that hands out no raw memory, a
 * serving loop that must not allocate after warm-up, an embedder without an
 * allocator). The pages describe no such entry point; it is an interface
 * choice of this library. Arguments and results are those of
 * domino_draft_chain, without ws/ws_bytes; device_status (device int32, may
 * be NULL) receives the DOMINO_* code of the device-side checks of this call.
 * The scratch is one fixed device array inside the library (659,712 bytes per
 * GPU that loads it, held until the process exits), so the sizes are capped:
 * batch <= 4, P <= 32, g <= 2048, r <= 256, at most 256 SMs; larger sizes return
 * DOMINO_ERR_UNSUPPORTED. The first call on a device looks up and zeroes that
 * array synchronously, so make it before any stream capture. The array's
 * device address is kept for the life of the process: do not use this entry
 * point across a cudaDeviceReset(). All calls share the array: calls that
 * overlap on the GPU race, on the scratch and on the status word that
 * device_status is read from (it may then report another call's error);
 * order them on one stream.
 */
domino_status domino_draft_chain_noalloc(const domino_head* head, const float* L_base,
                                         const float* P_h, const int32_t* anchor, int batch, int P,
                                         float temperature, const float* gumbel,
                                         int64_t gumbel_batch_stride, const int32_t* force_tokens,
                                         int32_t* tokens, float* logits_out, int32_t* device_status,
                                         void* stream);

/*
 * Synchronise `stream`, return the sticky device status recorded in `ws` by
 * earlier calls (DOMINO_OK if none) and clear it.
 */
domino_status domino_last_status(void* ws, void* stream);

/*
 * Upper bound, in nanoseconds, of every device-side wait (grid barriers,
 * pipeline barriers, the polls on exchanged sums, keys and published nodes)
 * in kernels launched after this call. Default 2e9 (2 s).
 * Process-wide.
 */
void domino_set_wait_timeout_ns(uint64_t ns);

/*
 * Diagnostic: launch one CTA that waits on a flag in `ws` which nothing sets,
 * bounded by `timeout_ns`; the wait runs out and records DOMINO_ERR_TIMEOUT,
 * which the next domino_last_status() returns. Exercises the error path of
 * bounded waits without hanging the GPU.
 */
domino_status domino_selftest_wait_timeout(uint64_t timeout_ns, void* ws, size_t ws_bytes,
                                           void* stream);

/*
 * Diagnostic measurements behind the chain's latency floor (the pages have no
 * counterpart; the benchmark reports the floor next to the step time). All
 * enqueue on `stream` and write device int64 out[2] (8-byte aligned); the
 * caller synchronises before reading it. ws: a workspace of at least 512
 * bytes (its status word records a wait that ran out).
 *   which = 0: a flag passed back and forth between CTA 0 and CTA `arg`
 *              (1 <= arg < number of SMs) of a grid of one CTA per SM,
 *              through L2 with release stores and acquire loads, 2000 times:
 *              out[0] = cycles, out[1] = round trips completed (bounded waits).
 *   which = 1: 16 warps per SM each issue `arg` x 4 bf16 tensor-core MMAs of
 *              shape m16n8k16 (fp32 accumulate, operands in registers):
 *              out[0] = cycles on the slowest SM.
 *   which = 2: the same with `arg` x 16 packed fp32x2 FMAs on bf16 pairs
 *              unpacked to fp32 (64 multiply-adds per warp instruction).
 * 1 <= arg <= 2^20 for which 1 and 2.
 */
domino_status domino_selftest_rates(int which, int arg, int64_t* out, void* ws, size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DOMINO_H */
