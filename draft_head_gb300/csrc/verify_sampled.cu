// Verification at temperature T > 0: the standard speculative-decoding
// procedure the 163.com report names (section 五; the output keeps the
// target's probabilities), lossless as the DominoTree page states (实验结果).
// With q_i = softmax(L_i / T) the draft distribution and p_i = softmax(Z_i / T)
// the target's:
//   accept x_i while U_i < p_i(x_i) / q_i(x_i); at the first rejection j draw
//   the next token from norm(max(0, p_j - q_j)), after P acceptances from p_P.
// The draw is Gumbel-max with given noise G: argmax_v log r_v + G_v (from p_j
// when the residual is zero everywhere in fp32).
// Three kernels: the logsumexp of every draft and target row, one pass over
// V each (online: the running maximum rescales the running sum); the sequential accept decisions, one warp per request; the draw,
// chunks of the chosen row folded into the request's keys with atomicMax, the
// CTA that completes a request writing its token and clearing its scratch.
#include "common.cuh"

namespace domino {

namespace {

constexpr int kLseThreads = 512;
constexpr int kDrawThreads = 256;
constexpr int kDrawChunk = 8192;

__device__ __forceinline__ void lse_add(float& m, float& s, float y) {
  if (y > m) {
    s = s * expf(m - y) + 1.0f;
    m = y;
  } else {
    s += expf(y - m);
  }
}

__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  if (m2 > m) {
    s = s * expf(m - m2) + s2;
    m = m2;
  } else if (m2 > -INFINITY) {
    s += s2 * expf(m2 - m);
  }
}

// Four values at once: one rescale when the maximum moves, then four terms.
__device__ __forceinline__ void lse_add4(float& m, float& s, float4 x, float inv_T) {
  const float y0 = x.x * inv_T, y1 = x.y * inv_T, y2 = x.z * inv_T, y3 = x.w * inv_T;
  const float mx = fmaxf(fmaxf(y0, y1), fmaxf(y2, y3));
  if (mx > m) {
    s *= expf(m - mx);
    m = mx;
  }
  s += (expf(y0 - m) + expf(y1 - m)) + (expf(y2 - m) + expf(y3 - m));
}

// Row r < bs * P: draft row (b, i) of L; otherwise target row of Z. kVec:
// rows read as 16-byte vectors, four in flight per thread (V % 4 == 0 and
// 16-byte aligned bases).
template <bool kVec>
__global__ void __launch_bounds__(kLseThreads) sv_lse_kernel(const float* __restrict__ L, const float* __restrict__ Z,
                                                             int bsP, int V, float inv_T, float* __restrict__ lse) {
  __shared__ float sm[kLseThreads / 32], ss[kLseThreads / 32];
  const int r = blockIdx.x;
  const float* x = r < bsP ? L + (size_t)r * V : Z + (size_t)(r - bsP) * V;
  float m = -INFINITY, s = 0.0f;
  if (kVec) {
    const float4* x4 = (const float4*)x;
    const int n4 = V >> 2;
    for (int v = threadIdx.x; v < n4; v += 4 * kLseThreads) {
      float4 a[4];
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (v + t * kLseThreads < n4) a[t] = __ldcs(x4 + v + t * kLseThreads);
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (v + t * kLseThreads < n4) lse_add4(m, s, a[t], inv_T);
    }
  } else {
    for (int v = threadIdx.x; v < V; v += kLseThreads) lse_add(m, s, __ldcs(x + v) * inv_T);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_merge(m, s, m2, s2);
  }
  if ((threadIdx.x & 31) == 0) { sm[threadIdx.x >> 5] = m; ss[threadIdx.x >> 5] = s; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kLseThreads / 32; ++w) lse_merge(m, s, sm[w], ss[w]);
    lse[r] = m + logf(s);
  }
}

// One thread per request (the decisions are sequential in i).
__global__ void sv_decide_kernel(const int32_t* __restrict__ draft, const float* __restrict__ L,
                                 const float* __restrict__ Z, const float* __restrict__ U,
                                 const float* __restrict__ lse, int bs, int P, int V, float inv_T,
                                 int32_t* __restrict__ jpos, int32_t* __restrict__ accept,
                                 int32_t* __restrict__ advanced, Ctl* ctl) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= bs) return;
  const float* lse_q = lse + (size_t)b * P;
  const float* lse_p = lse + (size_t)bs * P + (size_t)b * (P + 1);
  int j = P;
  for (int i = 0; i < P; ++i) {
    int x = draft[(size_t)b * P + i];
    if (x < 0 || x >= V) { dev_error(ctl, DEV_ERR_DATA); x = 0; }
    const float lq = L[((size_t)b * P + i) * V + x] * inv_T - lse_q[i];
    const float lp = Z[((size_t)b * (P + 1) + i) * V + x] * inv_T - lse_p[i];
    const float ratio = fminf(1.0f, expf(lp - lq));
    if (!(U[(size_t)b * P + i] < ratio)) { j = i; break; }
  }
  jpos[b] = j;
  accept[b] = j;
  advanced[b] = j + 1;
}

// Keys per request: [0] residual draw, [1] draw from p; cnt counts chunks.
__global__ void __launch_bounds__(kDrawThreads) sv_draw_kernel(const float* __restrict__ L, const float* __restrict__ Z,
                                                               const float* __restrict__ G,
                                                               const float* __restrict__ lse,
                                                               const int32_t* __restrict__ jpos, int bs, int P, int V,
                                                               float inv_T, int nch, unsigned long long* keys,
                                                               unsigned* cnt, int32_t* __restrict__ next_token, Ctl* ctl) {
  __shared__ unsigned long long red[2][kDrawThreads / 32];
  const int b = blockIdx.y, ch = blockIdx.x;
  const int j = jpos[b];
  const int v0 = ch * kDrawChunk, v1 = min(V, v0 + kDrawChunk);
  const float lp0 = lse[(size_t)bs * P + (size_t)b * (P + 1) + j];
  const float* z = Z + ((size_t)b * (P + 1) + j) * V;
  const float* g = G + (size_t)b * V;
  const bool resid = j < P;
  const float lq0 = resid ? lse[(size_t)b * P + j] : 0.0f;
  const float* l = resid ? L + ((size_t)b * P + j) * V : nullptr;
  unsigned long long kr = 0ull, kp = 0ull;
  for (int v = v0 + (int)threadIdx.x; v < v1; v += kDrawThreads) {
    const float logp = z[v] * inv_T - lp0;
    const float gv = g[v];
    const unsigned long long a = value_id_key(logp + gv, (uint32_t)v);
    kp = a > kp ? a : kp;
    if (resid) {
      const float r = expf(logp) - expf(l[v] * inv_T - lq0);
      if (r > 0.0f) {
        const unsigned long long c = value_id_key(logf(r) + gv, (uint32_t)v);
        kr = c > kr ? c : kr;
      }
    }
  }
  kr = warp_max_u64(kr);
  kp = warp_max_u64(kp);
  if ((threadIdx.x & 31) == 0) { red[0][threadIdx.x >> 5] = kr; red[1][threadIdx.x >> 5] = kp; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kDrawThreads / 32; ++w) {
      kr = red[0][w] > kr ? red[0][w] : kr;
      kp = red[1][w] > kp ? red[1][w] : kp;
    }
    unsigned long long* k2 = keys + (size_t)b * 2;
    if (kr) atomicMax(k2, kr);
    if (kp) atomicMax(k2 + 1, kp);
    __threadfence();
    const unsigned before = atomicAdd(cnt + b, 1u);
    if (before == (unsigned)nch - 1u) {  // this CTA completed the request
      __threadfence();
      const unsigned long long r = atomicExch(k2, 0ull), pk = atomicExch(k2 + 1, 0ull);
      cnt[b] = 0u;
      const unsigned long long k = r ? r : pk;
      int tok = 0;
      if (k == 0ull) dev_error(ctl, DEV_ERR_DATA);
      else tok = (int)key_id(k);
      next_token[b] = tok;
    }
  }
}

}  // namespace

size_t sampled_verify_ws_bytes(int bs, int P) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al((size_t)bs * (2 * P + 1) * 4) + al((size_t)bs * 4) + al((size_t)bs * 16) + al((size_t)bs * 4);
}

cudaError_t launch_sampled_verify(const int32_t* draft, const float* L, const float* Z, const float* U,
                                  const float* G, int bs, int P, int V, float temperature, int32_t* accept,
                                  int32_t* advanced, int32_t* next_token, Ctl* ctl, void* scratch,
                                  cudaStream_t stream) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  uint8_t* w = (uint8_t*)scratch;
  float* lse = (float*)w; w += al((size_t)bs * (2 * P + 1) * 4);
  int32_t* jpos = (int32_t*)w; w += al((size_t)bs * 4);
  unsigned long long* keys = (unsigned long long*)w; w += al((size_t)bs * 16);
  unsigned* cnt = (unsigned*)w;
  const float inv_T = 1.0f / temperature;
  const int rows = bs * P + bs * (P + 1);
  const bool vec = (V % 4) == 0 && ((uintptr_t)L & 15u) == 0 && ((uintptr_t)Z & 15u) == 0;
  if (vec)
    sv_lse_kernel<true><<<rows, kLseThreads, 0, stream>>>(L, Z, bs * P, V, inv_T, lse);
  else
    sv_lse_kernel<false><<<rows, kLseThreads, 0, stream>>>(L, Z, bs * P, V, inv_T, lse);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  sv_decide_kernel<<<(bs + 127) / 128, 128, 0, stream>>>(draft, L, Z, U, lse, bs, P, V, inv_T, jpos, accept, advanced,
                                                         ctl);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int nch = (V + kDrawChunk - 1) / kDrawChunk;
  sv_draw_kernel<<<dim3(nch, bs), kDrawThreads, 0, stream>>>(L, Z, G, lse, jpos, bs, P, V, inv_T, nch, keys, cnt,
                                                             next_token, ctl);
  return cudaGetLastError();
}

}  // namespace domino
