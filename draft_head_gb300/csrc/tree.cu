// DominoTree on sm_103a ("DominoTree: Conditional Tree-Structured Drafting with
// Domino for Speculative Decoding", "核心组件").
//
// 1. Top-M candidate select ("候选限制（Top-M）"): per row of L_base, the M best
//    (value desc, id asc). Each (value, id) pair becomes one distinct 64-bit
//    key, so the selection is an exact k-th-largest search: an 8-bit radix
//    select over the keys in shared memory. Stage 1 keeps the top M of each
//    4096-wide chunk of the row (one CTA per chunk, the row is read from HBM
//    once); stage 2 selects among the chunk winners and sorts them (bitonic).
//
// 2. Best-first build ("条件评分的最佳优先堆"), one persistent kernel, all
//    requests in lockstep. Node ids are assigned in pop order and node t is
//    expanded right after it is popped, so iteration t of every request
//    expands its node t:
//      G  every CTA runs the GRU for its slice of hidden units (W_hh slice in
//         shared memory, input gates from the prepared table) for each
//         request's node t, from the parent's stored state, and writes its
//         share of W1_s S_t to a per-CTA partial;
//      -- grid barrier --
//      E  CTA b (one per request) sums the partials in a fixed order,
//         u = SiLU(P_h[depth] + .), scores its M candidates
//         l_c = L_base[depth, c] + W2[c] u, log-softmax over the slice, and
//         stores the children sorted by (score desc, token asc) as the sibling
//         group of node t. The best-first heap is the set of group heads: the
//         pop takes the best head under (score desc, parent asc), which is the
//         same order a binary heap over all pushed children gives.
//      -- grid barrier --
#include "common.cuh"

namespace domino {

namespace {

constexpr int kChunk = 4096;  // 32 KB of keys in static shared memory
constexpr int kSelThreads = 512;

// k largest of n distinct 64-bit keys in shared memory -> out[0..k) (unordered).
__device__ void block_topk_u64(const unsigned long long* keys, int n, int k, unsigned long long* out,
                               unsigned* hist, unsigned* misc) {
  const int tid = threadIdx.x, nt = blockDim.x, warp = tid >> 5, lane = tid & 31;
  unsigned long long prefix = 0ull, mask = 0ull;
  unsigned remaining = (unsigned)k;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += nt) hist[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += nt) {
      const unsigned long long key = keys[i];
      if ((key & mask) == prefix) atomicAdd(&hist[(unsigned)(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      unsigned local[8];
      unsigned s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        local[j] = hist[lane * 8 + j];
        s += local[j];
      }
      unsigned suf = s;  // sum over lanes >= lane
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned t = __shfl_down_sync(0xffffffffu, suf, o);
        if (lane + o < 32) suf += t;
      }
      const unsigned above = suf - s;
      if (above < remaining && remaining <= suf) {
        unsigned cum = above;
        for (int j = 7; j >= 0; --j) {
          if (cum + local[j] >= remaining) {
            misc[0] = (unsigned)(lane * 8 + j);
            misc[1] = remaining - cum;
            break;
          }
          cum += local[j];
        }
      }
    }
    __syncthreads();
    const unsigned digit = misc[0];
    remaining = misc[1];
    prefix |= (unsigned long long)digit << shift;
    mask |= 0xFFull << shift;
    __syncthreads();
  }
  if (tid == 0) misc[2] = 0u;
  __syncthreads();
  for (int i = tid; i < n; i += nt) {
    const unsigned long long key = keys[i];
    if (key >= prefix) out[atomicAdd(&misc[2], 1u)] = key;
  }
  __syncthreads();
}

// Sort np (power of two) keys descending in shared memory.
__device__ void block_bitonic_desc(unsigned long long* s, int np) {
  for (int k = 2; k <= np; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < np; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = s[i], b = s[ixj];
          const bool desc = (i & k) == 0;
          if (desc ? (a < b) : (a > b)) {
            s[i] = b;
            s[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

__global__ void __launch_bounds__(kSelThreads) topm_stage1(const float* __restrict__ values, int n, int M,
                                                          unsigned long long* __restrict__ cand) {
  __shared__ unsigned long long keys[kChunk];
  __shared__ unsigned long long outk[256];
  __shared__ unsigned hist[256];
  __shared__ unsigned misc[4];
  const int row = blockIdx.y, chunk = blockIdx.x, nchunks = gridDim.x;
  const int begin = chunk * kChunk;
  const int len = min(kChunk, n - begin);
  const int k = min(M, len);
  const float* src = values + (size_t)row * n + begin;
  for (int i = threadIdx.x; i < len; i += kSelThreads)
    keys[i] = value_id_key(__ldcs(src + i), (uint32_t)(begin + i));
  __syncthreads();
  block_topk_u64(keys, len, k, outk, hist, misc);
  unsigned long long* dst = cand + ((size_t)row * nchunks + chunk) * M;
  for (int i = threadIdx.x; i < M; i += kSelThreads) dst[i] = (i < k) ? outk[i] : 0ull;
}

__global__ void __launch_bounds__(kSelThreads) topm_stage2(const unsigned long long* __restrict__ cand,
                                                          int nchunks, int M, int32_t* __restrict__ ids,
                                                          float* __restrict__ vals) {
  extern __shared__ unsigned long long sh2[];
  __shared__ unsigned hist[256];
  __shared__ unsigned misc[4];
  int np = 1;
  while (np < M) np <<= 1;
  const int total = nchunks * M;
  unsigned long long* keys = sh2;          // [total]
  unsigned long long* outk = sh2 + total;  // [np]
  const int row = blockIdx.x;
  // Zero keys (short last chunks) are never selected: at least M real keys exist.
  for (int i = threadIdx.x; i < total; i += kSelThreads) keys[i] = cand[(size_t)row * total + i];
  for (int i = threadIdx.x; i < np; i += kSelThreads) outk[i] = 0ull;
  __syncthreads();
  block_topk_u64(keys, total, M, outk, hist, misc);
  block_bitonic_desc(outk, np);
  for (int i = threadIdx.x; i < M; i += kSelThreads) {
    const unsigned long long key = outk[i];
    ids[(size_t)row * M + i] = (int32_t)key_id(key);
    if (vals) vals[(size_t)row * M + i] = key_value(key);
  }
}

// ---------------------------------------------------------------------------
// Best-first build.
// ---------------------------------------------------------------------------
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

template <typename WT>
struct TreeP {
  int bs, P, d, g, r, V, N, M, Mp, nu_max;
  const float* gate_table;
  const WT* w_hh;
  const WT* b_hh;
  const WT* w1;
  const WT* w2;
  const float* L_base;
  const float* P_h;
  const int32_t* anchor;
  int32_t* node_token;
  int32_t* node_parent;
  int32_t* node_depth;
  float* node_score;
  Ctl* ctl;
  const int32_t* cand;
  float* states;
  float* part;
  int32_t* cur;
  unsigned long long* grp;
  uint64_t timeout_ns;
};

template <typename WT>
__global__ void __launch_bounds__(kThreads, 1) tree_kernel(const __grid_constant__ TreeP<WT> p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int G = gridDim.x, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bs = p.bs, g = p.g, r = p.r, P = p.P, N = p.N, M = p.M;
  const int j0 = (int)((int64_t)g * c / G), j1 = (int)((int64_t)g * (c + 1) / G), nu = j1 - j0;
  const int nu_max = p.nu_max;

  WT* whh_s = (WT*)smem;
  size_t off = ((size_t)3 * nu_max * g * sizeof(WT) + 15) & ~(size_t)15;
  float* w1s_s = (float*)(smem + off); off += (size_t)r * nu_max * 4;
  float* bhh_s = (float*)(smem + off); off += (size_t)3 * nu_max * 4;
  float* snew_s = (float*)(smem + off); off += (size_t)bs * nu_max * 4;
  float* u_s = (float*)(smem + off); off += (size_t)r * 4;
  float* u2_s = (float*)(smem + off); off += (size_t)r * 4;
  float* lg_s = (float*)(smem + off); off += (size_t)p.Mp * 4;
  float* red_f = (float*)(smem + off); off += 64 * 4;
  int* head_s = (int*)(smem + off); off += (size_t)(N + 1) * 4;
  int* ndep_s = (int*)(smem + off); off += (size_t)(N + 1) * 4;
  float* nsc_s = (float*)(smem + off); off += (size_t)(N + 1) * 4;
  int* misc_s = (int*)(smem + off); off += 16 * 4;
  off = (off + 7) & ~(size_t)7;
  unsigned long long* key_s = (unsigned long long*)(smem + off);  // [Mp]

  for (int idx = threadIdx.x; idx < 3 * nu * g; idx += kThreads) {
    const int row = idx / g, k = idx - row * g;
    const int q = row / nu, jj = row - q * nu;
    whh_s[(size_t)(q * nu + jj) * g + k] = p.w_hh[(size_t)(q * g + j0 + jj) * g + k];
  }
  for (int idx = threadIdx.x; idx < r * nu; idx += kThreads) {
    const int k = idx / nu, jj = idx - k * nu;
    w1s_s[k * nu + jj] = to_f(p.w1[(size_t)k * (p.d + g) + p.d + j0 + jj]);
  }
  for (int idx = threadIdx.x; idx < 3 * nu; idx += kThreads) {
    const int q = idx / nu, jj = idx - q * nu;
    bhh_s[idx] = to_f(p.b_hh[q * g + j0 + jj]);
  }
  // Request state lives with CTA b (b < bs): root = node 0.
  const bool owner = c < bs;
  const int b_own = c;
  if (owner) {
    for (int k = threadIdx.x; k <= N; k += kThreads) {
      head_s[k] = 0;
      ndep_s[k] = -1;
      nsc_s[k] = -INFINITY;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int a = p.anchor[b_own];
      if (a < 0 || a >= p.V) { dev_error(p.ctl, DEV_ERR_DATA); a = 0; }
      ndep_s[0] = 0;
      nsc_s[0] = 0.0f;
      misc_s[0] = 1;  // request still active
      const size_t o = (size_t)b_own * (N + 1);
      p.node_token[o] = a;
      p.node_parent[o] = -1;
      p.node_depth[o] = 0;
      p.node_score[o] = 0.0f;
      for (int k = 1; k <= N; ++k) {
        p.node_token[o + k] = -1;
        p.node_parent[o + k] = -1;
        p.node_depth[o + k] = -1;
        p.node_score[o + k] = -INFINITY;
      }
    }
  }
  __syncthreads();

  unsigned epoch = 0;
  for (int t = 0; t < N; ++t) {
    // ---------------- G: GRU for node t of every request.
    for (int item = warp; item < bs * nu; item += kWarps) {
      const int b = item / nu, jj = item - b * nu, j = j0 + jj;
      int tok, parent, expand;
      if (t == 0) {
        tok = p.anchor[b];
        if (tok < 0 || tok >= p.V) tok = 0;
        parent = -1;
        expand = P > 0;
      } else {
        tok = __ldcg(p.cur + b * 4 + 0);
        parent = __ldcg(p.cur + b * 4 + 1);
        expand = __ldcg(p.cur + b * 4 + 2);
      }
      if (!expand) continue;  // warp-uniform
      const float* Sp = parent >= 0 ? p.states + ((size_t)b * N + parent) * g : nullptr;
      float a0 = 0.f, a1 = 0.f, a2 = 0.f;
      if (Sp) {
        const WT* wr0 = whh_s + (size_t)(0 * nu + jj) * g;
        const WT* wr1 = whh_s + (size_t)(1 * nu + jj) * g;
        const WT* wr2 = whh_s + (size_t)(2 * nu + jj) * g;
        for (int k = lane; k < g; k += 32) {
          const float s = __ldcg(Sp + k);
          a0 = fmaf(to_f(wr0[k]), s, a0);
          a1 = fmaf(to_f(wr1[k]), s, a1);
          a2 = fmaf(to_f(wr2[k]), s, a2);
        }
        a0 = warp_sum(a0);
        a1 = warp_sum(a1);
        a2 = warp_sum(a2);
      }
      if (lane == 0) {
        const float* gi = p.gate_table + (size_t)tok * 3 * g;
        const float rg = sigmoidf_(__ldg(gi + j) + a0 + bhh_s[jj]);
        const float zg = sigmoidf_(__ldg(gi + g + j) + a1 + bhh_s[nu + jj]);
        const float ng = tanhf(__ldg(gi + 2 * g + j) + rg * (a2 + bhh_s[2 * nu + jj]));
        const float h = Sp ? __ldcg(Sp + j) : 0.0f;
        const float hn = (1.0f - zg) * ng + zg * h;
        p.states[((size_t)b * N + t) * g + j] = hn;
        snew_s[b * nu_max + jj] = hn;
      }
    }
    __syncthreads();
    // Partial W1_s S for the owned units (zeros when this CTA owns none, or
    // the request does not expand: the owner then ignores them).
    for (int idx = threadIdx.x; idx < bs * r; idx += kThreads) {
      const int b = idx / r, k = idx - b * r;
      float s = 0.0f;
      for (int jj = 0; jj < nu; ++jj) s = fmaf(w1s_s[k * nu + jj], snew_s[b * nu_max + jj], s);
      p.part[((size_t)c * bs + b) * r + k] = s;
    }
    if (!grid_barrier(p.ctl, epoch, G, p.timeout_ns)) return;

    // ---------------- E: expand node t, then pop node t + 1 (owner CTAs).
    if (owner && misc_s[0]) {
      const int b = b_own;
      const int dep = ndep_s[t];
      const bool expand = (dep >= 0 && dep < P);
      if (expand) {
        // u = SiLU(P_h[b, dep] + sum_c part[c, b]), summed in a fixed order
        // (even CTAs, odd CTAs, then the two halves).
        for (int idx = threadIdx.x; idx < 2 * r; idx += kThreads) {
          const int k = idx % r, half = idx / r;
          float s = 0.0f;
          for (int cc = half; cc < G; cc += 2) s += __ldcg(p.part + ((size_t)cc * bs + b) * r + k);
          (half == 0 ? u_s : u2_s)[k] = s;
        }
        __syncthreads();
        for (int k = threadIdx.x; k < r; k += kThreads)
          u_s[k] = siluf_(__ldg(p.P_h + ((size_t)b * P + dep) * r + k) + (u_s[k] + u2_s[k]));
        __syncthreads();
        // Candidate logits l_c = L_base[b, dep, c] + W2[c] . u.
        const int32_t* C = p.cand + ((size_t)b * P + dep) * M;
        for (int m = warp; m < M; m += kWarps) {
          int v = C[m];
          if (v < 0 || v >= p.V) {  // never expected: candidate ids come from the select
            if (lane == 0) dev_error(p.ctl, DEV_ERR_DATA);
            v = 0;
          }
          float s = 0.0f;
          for (int k = lane; k < r; k += 32) s = fmaf(to_f(p.w2[(size_t)v * r + k]), u_s[k], s);
          s = warp_sum(s);
          if (lane == 0) lg_s[m] = __ldg(p.L_base + ((size_t)b * P + dep) * p.V + v) + s;
        }
        __syncthreads();
        // logsumexp over the M-slice (fp32, max-shifted).
        if (warp == 0) {
          float mx = -INFINITY;
          for (int m = lane; m < M; m += 32) mx = fmaxf(mx, lg_s[m]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          float se = 0.0f;
          for (int m = lane; m < M; m += 32) se += expf(lg_s[m] - mx);
          se = warp_sum(se);
          if (lane == 0) red_f[1] = mx + logf(se);
        }
        __syncthreads();
        const float lse = red_f[1];
        const float base = nsc_s[t];
        for (int m = threadIdx.x; m < p.Mp; m += kThreads) {
          if (m < M) {
            const float logp = lg_s[m] - lse;
            key_s[m] = value_id_key(base + logp, (uint32_t)C[m]);
          } else {
            key_s[m] = 0ull;
          }
        }
        __syncthreads();
        block_bitonic_desc(key_s, p.Mp);
        unsigned long long* gdst = p.grp + ((size_t)b * N + t) * M;
        for (int m = threadIdx.x; m < M; m += kThreads) gdst[m] = key_s[m];
        if (threadIdx.x == 0) head_s[t] = 0;
      } else if (threadIdx.x == 0) {
        head_s[t] = M;  // no children
      }
      __syncthreads();
      // Pop: best group head under (score desc, parent asc).
      if (warp == 0) {
        unsigned long long best = 0ull;
        int bestg = -1;
        unsigned long long bestchild = 0ull;
        for (int gi = lane; gi <= t; gi += 32) {
          const int h = head_s[gi];
          if (h < M) {
            const unsigned long long ck = __ldcg(p.grp + ((size_t)b * N + gi) * M + h);
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
          const int k = t + 1;
          if (bestg < 0) {
            misc_s[0] = 0;  // candidate tree exhausted
            p.cur[b * 4 + 2] = 0;
          } else {
            head_s[bestg] += 1;
            const int tok = (int)key_id(bestchild);
            const float sc = key_value(bestchild);
            const int dk = ndep_s[bestg] + 1;
            ndep_s[k] = dk;
            nsc_s[k] = sc;
            const size_t o = (size_t)b * (N + 1) + k;
            p.node_token[o] = tok;
            p.node_parent[o] = bestg;
            p.node_depth[o] = dk;
            p.node_score[o] = sc;
            p.cur[b * 4 + 0] = tok;
            p.cur[b * 4 + 1] = bestg;
            p.cur[b * 4 + 2] = (k < N && dk < P) ? 1 : 0;
            p.cur[b * 4 + 3] = dk;
          }
        }
      }
      __syncthreads();
    } else if (owner && threadIdx.x == 0) {
      p.cur[b_own * 4 + 2] = 0;
    }
    if (t + 1 < N) {
      if (!grid_barrier(p.ctl, epoch, G, p.timeout_ns)) return;
    }
  }
}

template <typename WT>
size_t tree_smem_bytes(int bs, int g, int r, int N, int Mp, int nu_max) {
  size_t off = ((size_t)3 * nu_max * g * sizeof(WT) + 15) & ~(size_t)15;
  off += (size_t)r * nu_max * 4 + (size_t)3 * nu_max * 4 + (size_t)bs * nu_max * 4 + (size_t)2 * r * 4 +
         (size_t)Mp * 4 + 64 * 4 + 3 * (size_t)(N + 1) * 4 + 16 * 4;
  off = (off + 7) & ~(size_t)7;
  return off + (size_t)Mp * 8;
}

int pow2_at_least(int x) {
  int n = 1;
  while (n < x) n <<= 1;
  return n;
}

template <typename WT>
cudaError_t launch_tree_t(const TreeArgs& a, cudaStream_t stream) {
  const int G = num_sms();
  TreeP<WT> p;
  p.bs = a.bs; p.P = a.P; p.d = a.d; p.g = a.g; p.r = a.r; p.V = a.V; p.N = a.N; p.M = a.M;
  p.Mp = pow2_at_least(a.M);
  p.nu_max = (a.g + G - 1) / G;
  p.gate_table = a.gate_table;
  p.w_hh = (const WT*)a.w_hh; p.b_hh = (const WT*)a.b_hh; p.w1 = (const WT*)a.w1; p.w2 = (const WT*)a.w2;
  p.L_base = a.L_base; p.P_h = a.P_h; p.anchor = a.anchor;
  p.node_token = a.node_token; p.node_parent = a.node_parent; p.node_depth = a.node_depth;
  p.node_score = a.node_score;
  p.ctl = a.ctl; p.cand = a.cand; p.states = a.states; p.part = a.part; p.cur = a.cur;
  p.grp = a.grp;
  p.timeout_ns = wait_timeout_ns();
  const size_t smem = tree_smem_bytes<WT>(a.bs, a.g, a.r, a.N, p.Mp, p.nu_max);
  if (smem > 227 * 1024) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(tree_kernel<WT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void* args[] = {(void*)&p};
  return cudaLaunchCooperativeKernel((const void*)tree_kernel<WT>, dim3(G), dim3(kThreads), args, smem, stream);
}

}  // namespace

size_t topm_ws_bytes(int rows, int n, int M) {
  const size_t nchunks = ((size_t)n + kChunk - 1) / kChunk;
  return (size_t)rows * nchunks * M * 8;
}

cudaError_t launch_topm(const float* values, int rows, int n, int M, int32_t* ids, float* vals,
                        void* scratch, cudaStream_t stream) {
  const int nchunks = (n + kChunk - 1) / kChunk;
  if (rows > 65535) return cudaErrorInvalidValue;
  topm_stage1<<<dim3(nchunks, rows), kSelThreads, 0, stream>>>(values, n, M, (unsigned long long*)scratch);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int np = pow2_at_least(M);
  const size_t smem = ((size_t)nchunks * M + np) * 8;
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(topm_stage2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topm_stage2<<<rows, kSelThreads, smem, stream>>>((const unsigned long long*)scratch, nchunks, M, ids, vals);
  return cudaGetLastError();
}

size_t tree_ws_bytes(int bs, int P, int g, int r, int N, int M) {
  const int G = num_sms();
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al((size_t)bs * P * M * 4) + al((size_t)bs * N * g * 4) + al((size_t)bs * 4 * 4) +
         al((size_t)G * bs * r * 4) + al((size_t)bs * N * M * 8);
}

bool tree_fits(int dtype, int bs, int g, int r, int N, int M) {
  const int G = num_sms();
  const int nu_max = (g + G - 1) / G;
  const int Mp = pow2_at_least(M);
  const size_t smem = dtype == DOMINO_BF16 ? tree_smem_bytes<__nv_bfloat16>(bs, g, r, N, Mp, nu_max)
                                           : tree_smem_bytes<float>(bs, g, r, N, Mp, nu_max);
  return smem <= 227 * 1024 && bs <= G;
}

cudaError_t launch_tree(const TreeArgs& a, cudaStream_t stream) {
  if (a.dtype == DOMINO_BF16) return launch_tree_t<__nv_bfloat16>(a, stream);
  return launch_tree_t<float>(a, stream);
}

}  // namespace domino
