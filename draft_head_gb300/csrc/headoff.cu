// The pages' ablation baselines with the correction head switched off.
//
// Head-off chain: "Domino: Decoupling Causal Modeling from Autoregressive
// Drafting in Speculative Decoding Review" (sections 1-1, 3-2) and the 163.com
// report (section 四) describe the parallel backbone alone drafting every
// position from its marginal logits, the DFlash baseline Domino corrects:
//   tokens[b, i] = argmax_v L_base[b, i, v]            (T = 0)
//   tokens[b, i] = argmax_v L_base[b, i, v] / T + G     (T > 0, Gumbel-max)
// ties to the lowest id. One pass over L_base: each CTA reduces a chunk of one
// row to a (value, id) key, folds it into the row's key with atomicMax, and
// the CTA that completes a row writes its token and clears the row's scratch.
//
// Marginal tree: "DominoTree: Conditional Tree-Structured Drafting with Domino
// for Speculative Decoding" (核心贡献, the ablation) scores the same
// best-first tree with path-independent marginal log-probabilities:
//   logp_c = L_base[t, c] - logsumexp_{c' in C_t} L_base[t, c'],
// C_t the top-M candidates of depth t, child score = parent score + logp_c,
// pop order (score desc, parent asc, token asc). With no GRU and no
// correction a request needs no other CTA: one CTA per request keeps every
// node's sorted sibling group in shared memory.
#include "common.cuh"

namespace domino {

namespace {

constexpr int kHoThreads = 256;
constexpr int kHoChunk = 8192;  // vocabulary ids per CTA

__global__ void __launch_bounds__(kHoThreads) headoff_chain_kernel(
    const float* __restrict__ L_base, int P, int V, float inv_T, const float* __restrict__ gumbel,
    int64_t gstride, int nch, unsigned long long* keys, unsigned* cnt, int32_t* __restrict__ tokens, Ctl* ctl) {
  __shared__ unsigned long long red[kHoThreads / 32];
  const int row = blockIdx.y, ch = blockIdx.x;
  const int b = row / P, i = row - b * P;
  const int v0 = ch * kHoChunk, v1 = min(V, v0 + kHoChunk);
  const float* Lr = L_base + (size_t)row * V;
  const float* Gr = gumbel ? gumbel + (int64_t)b * gstride + (int64_t)i * V : nullptr;
  unsigned long long best = 0ull;
  for (int v = v0 + (int)threadIdx.x; v < v1; v += kHoThreads) {
    const float l = __ldcs(Lr + v);
    const float dec = Gr ? l * inv_T + __ldcs(Gr + v) : l;
    const unsigned long long k = value_id_key(dec, (uint32_t)v);
    best = k > best ? k : best;
  }
  best = warp_max_u64(best);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kHoThreads / 32; ++w) best = red[w] > best ? red[w] : best;
    if (best) atomicMax(keys + row, best);
    __threadfence();
    const unsigned before = atomicAdd(cnt + row, 1u);
    if (before == (unsigned)nch - 1u) {  // this CTA completed the row
      __threadfence();
      const unsigned long long k = atomicExch(keys + row, 0ull);
      cnt[row] = 0u;
      int tok = 0;
      if (k == 0ull) dev_error(ctl, DEV_ERR_DATA);  // every value NaN
      else tok = (int)key_id(k);
      tokens[row] = tok;
    }
  }
}

constexpr int kMtThreads = 256;
constexpr int kMtWarps = kMtThreads / 32;

// Sort np (power of two) keys descending in shared memory.
__device__ void bitonic_desc(unsigned long long* s, int np) {
  for (int k = 2; k <= np; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int x = threadIdx.x; x < np; x += kMtThreads) {
        const int y = x ^ j;
        if (y > x) {
          const bool desc = (x & k) == 0;
          const unsigned long long a = s[x], c = s[y];
          if (desc ? (a < c) : (a > c)) { s[x] = c; s[y] = a; }
        }
      }
      __syncthreads();
    }
  }
}

struct MargP {
  int P, N, M, Mp, V;
  float inv_tau;           // 1 / scoring temperature
  const float* cand_val;   // [bs * P][M] L_base values of the candidates
  const int32_t* cand_id;  // [bs * P][M] candidate ids, value desc then id asc
  const int32_t* anchor;
  int32_t* node_token;
  int32_t* node_parent;
  int32_t* node_depth;
  float* node_score;
  Ctl* ctl;
};

__global__ void __launch_bounds__(kMtThreads) tree_marginal_kernel(const __grid_constant__ MargP p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = p.P, N = p.N, M = p.M, Mp = p.Mp;
  unsigned long long* grp_s = (unsigned long long*)smem;           // [N][M] sibling groups
  unsigned long long* key_s = grp_s + (size_t)N * M;               // [Mp]
  float* lse_s = (float*)(key_s + Mp);                             // [P]
  int* head_s = (int*)(lse_s + P);                                 // [N + 1]
  int* ndep_s = head_s + (N + 1);                                  // [N + 1]
  float* nsc_s = (float*)(ndep_s + (N + 1));                       // [N + 1]
  int* live_s = (int*)(nsc_s + (N + 1));

  // logsumexp over each depth's M-slice of l / tau (fp32, max-shifted).
  const float it = p.inv_tau;
  for (int t = warp; t < P; t += kMtWarps) {
    const float* l = p.cand_val + ((size_t)b * P + t) * M;
    float mx = -INFINITY;
    for (int m = lane; m < M; m += 32) mx = fmaxf(mx, l[m] * it);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float se = 0.0f;
    for (int m = lane; m < M; m += 32) se += expf(l[m] * it - mx);
    se = warp_sum(se);
    if (lane == 0) lse_s[t] = mx + logf(se);
  }
  const size_t o0 = (size_t)b * (N + 1);
  for (int k = threadIdx.x; k <= N; k += kMtThreads) {
    head_s[k] = M;
    ndep_s[k] = -1;
    nsc_s[k] = -INFINITY;
    if (k > 0) {
      p.node_token[o0 + k] = -1;
      p.node_parent[o0 + k] = -1;
      p.node_depth[o0 + k] = -1;
      p.node_score[o0 + k] = -INFINITY;
    }
  }
  if (threadIdx.x == 0) {
    int a = p.anchor[b];
    if (a < 0 || a >= p.V) { dev_error(p.ctl, DEV_ERR_DATA); a = 0; }
    p.node_token[o0] = a;
    p.node_parent[o0] = -1;
    p.node_depth[o0] = 0;
    p.node_score[o0] = 0.0f;
    *live_s = 1;
  }
  __syncthreads();
  if (threadIdx.x == 0) { ndep_s[0] = 0; nsc_s[0] = 0.0f; }
  __syncthreads();

  for (int t = 0; t < N && *live_s; ++t) {
    // Expand node t: its children, sorted by (score desc, token asc).
    const int dep = ndep_s[t];
    if (dep >= 0 && dep < P) {
      const float base = nsc_s[t];
      const float lse = lse_s[dep];
      const float* l = p.cand_val + ((size_t)b * P + dep) * M;
      const int32_t* C = p.cand_id + ((size_t)b * P + dep) * M;
      for (int m = threadIdx.x; m < Mp; m += kMtThreads)
        key_s[m] = m < M ? value_id_key(base + (l[m] * it - lse), (uint32_t)C[m]) : 0ull;
      __syncthreads();
      bitonic_desc(key_s, Mp);
      for (int m = threadIdx.x; m < M; m += kMtThreads) grp_s[(size_t)t * M + m] = key_s[m];
      if (threadIdx.x == 0) head_s[t] = 0;
    }
    __syncthreads();
    // Pop node t + 1: the best group head under (score desc, parent asc).
    if (warp == 0) {
      unsigned long long best = 0ull, bestchild = 0ull;
      int bestg = -1;
      for (int gi = lane; gi <= t; gi += 32) {
        const int h = head_s[gi];
        if (h < M) {
          const unsigned long long ck = grp_s[(size_t)gi * M + h];
          const unsigned long long cmp = value_id_key(key_value(ck), (uint32_t)gi);
          if (cmp > best) { best = cmp; bestg = gi; bestchild = ck; }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int og = __shfl_xor_sync(0xffffffffu, bestg, o);
        const unsigned long long oc = __shfl_xor_sync(0xffffffffu, bestchild, o);
        if (ob > best) { best = ob; bestg = og; bestchild = oc; }
      }
      if (lane == 0) {
        if (bestg < 0) {
          *live_s = 0;  // the candidate tree is exhausted
        } else {
          const int k = t + 1;
          head_s[bestg] += 1;
          const int dk = ndep_s[bestg] + 1;
          const float sc = key_value(bestchild);
          ndep_s[k] = dk;
          nsc_s[k] = sc;
          p.node_token[o0 + k] = (int)key_id(bestchild);
          p.node_parent[o0 + k] = bestg;
          p.node_depth[o0 + k] = dk;
          p.node_score[o0 + k] = sc;
        }
      }
    }
    __syncthreads();
  }
}

int pow2_ceil(int x) {
  int n = 1;
  while (n < x) n <<= 1;
  return n;
}

}  // namespace

size_t headoff_chain_ws_bytes(int rows) { return (size_t)rows * 8 + (size_t)rows * 4; }

cudaError_t launch_headoff_chain(const float* L_base, int bs, int P, int V, float temperature, const float* gumbel,
                                 int64_t gstride, int32_t* tokens, Ctl* ctl, void* scratch, cudaStream_t stream) {
  const int rows = bs * P;
  const int nch = (V + kHoChunk - 1) / kHoChunk;
  unsigned long long* keys = (unsigned long long*)scratch;
  unsigned* cnt = (unsigned*)(keys + rows);
  const float inv_T = temperature > 0.0f ? 1.0f / temperature : 0.0f;
  headoff_chain_kernel<<<dim3(nch, rows), kHoThreads, 0, stream>>>(
      L_base, P, V, inv_T, temperature > 0.0f ? gumbel : nullptr, gstride, nch, keys, cnt, tokens, ctl);
  return cudaGetLastError();
}

size_t tree_marginal_smem_bytes(int P, int N, int M) {
  return (size_t)N * M * 8 + (size_t)pow2_ceil(M) * 8 + (size_t)P * 4 + (size_t)3 * (N + 1) * 4 + 16;
}

cudaError_t launch_tree_marginal(const float* cand_val, const int32_t* cand_id, const int32_t* anchor, int bs,
                                 int P, int V, int N, int M, float inv_tau, int32_t* node_token,
                                 int32_t* node_parent, int32_t* node_depth, float* node_score, Ctl* ctl,
                                 cudaStream_t stream) {
  MargP p;
  p.P = P; p.N = N; p.M = M; p.Mp = pow2_ceil(M); p.V = V;
  p.inv_tau = inv_tau;
  p.cand_val = cand_val; p.cand_id = cand_id; p.anchor = anchor;
  p.node_token = node_token; p.node_parent = node_parent; p.node_depth = node_depth; p.node_score = node_score;
  p.ctl = ctl;
  const size_t smem = tree_marginal_smem_bytes(P, N, M);
  if (smem > 227 * 1024) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(tree_marginal_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  tree_marginal_kernel<<<bs, kMtThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace domino
