// Verification at temperature T > 0: the standard speculative-decoding
// procedure the 163.com report names (section 五; the output keeps the
// target's probabilities), lossless as the DominoTree page states (实验结果).
// With q_i = softmax(L_i / T) the draft distribution and p_i = softmax(Z_i / T)
// the target's:
//   accept x_i while U_i < p_i(x_i) / q_i(x_i); at the first rejection j draw
//   the next token from norm(max(0, p_j - q_j)), after P acceptances from p_P.
// The draw is Gumbel-max with given noise G: argmax_v log r_v + G_v (from p_j
// when the residual is zero everywhere in fp32).
//
// One kernel. A thread-block cluster of K CTAs serves one request, each CTA a
// 1/K slice of the vocabulary, and walks the positions in order, as the
// procedure does: round i reads rows L_i and Z_i once (online logsumexp in
// base 2: the running maximum rescales the running sum), the CTAs exchange their (max,
// sum) pairs through distributed shared memory at one cluster barrier, and
// every CTA merges them in the same order and so takes the same decision.
// The walk stops at the first rejection, so only rows 0..j are read: the rows
// after it do not enter the result. The draw then folds row j (read again,
// mostly from L2) and the noise row into one (value, id) key per CTA, merged
// by CTA 0 of the cluster. Every branch that decides how far a CTA goes
// depends only on values all CTAs of the cluster compute identically, so
// they all meet at every cluster barrier.
//
// Head form (the chain's draft statistics instead of its logits): q_i(x_i)
// comes from L_i[x_i] = L_base[b, i, x_i] + W2[x_i] . u_i and the chain's
// log-partition of L_i / T, so the walk reads target rows only. A rejection
// at j leaves the draw to the residual kernel (residual.cu), which rebuilds
// the rejected rows L_j from W2 for all requests at once; the walk records j
// and the two normalisers for it.
#include <string.h>

#include "common.cuh"

namespace domino {

namespace {

constexpr int kSvThreads = 256;
constexpr int kSvWarps = kSvThreads / 32;
constexpr int kSvMaxCluster = 8;

// Online logsumexp in base 2: y = x log2(e) / T, m = the running maximum of
// y, s = sum of 2^(y - m); the natural logsumexp is (m + log2 s) ln 2. One
// exp2 per value (pre-scaled inputs), a rescale only when the maximum moves.
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void lse2_add(float& m, float& s, float y) {
  if (y > m) {
    s = s * exp2f(m - y) + 1.0f;
    m = y;
  } else {
    s += exp2f(y - m);
  }
}

__device__ __forceinline__ void lse2_merge(float& m, float& s, float m2, float s2) {
  if (m2 > m) {
    s = s * exp2f(m - m2) + s2;
    m = m2;
  } else if (m2 > -INFINITY) {
    s += s2 * exp2f(m2 - m);
  }
}

// Four values at once: one rescale when the maximum moves, then four terms.
__device__ __forceinline__ void lse2_add4(float& m, float& s, float4 x, float c) {
  const float y0 = x.x * c, y1 = x.y * c, y2 = x.z * c, y3 = x.w * c;
  const float mx = fmaxf(fmaxf(y0, y1), fmaxf(y2, y3));
  if (mx > m) {
    s *= exp2f(m - mx);
    m = mx;
  }
  s += (exp2f(y0 - m) + exp2f(y1 - m)) + (exp2f(y2 - m) + exp2f(y3 - m));
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster: shared-memory writes before it are
// visible to the cluster's CTAs after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The address of p's shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(p)), "r"(rank));
  return ra;
}
__device__ __forceinline__ float4 ld_dsmem_f32x4(const void* p, uint32_t rank) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(dsmem_addr(p, rank))
               : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long ld_dsmem_u64(const void* p, uint32_t rank) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(dsmem_addr(p, rank)) : "memory");
  return v;
}

struct SvP {
  const int32_t* draft;  // [bs, P]
  const float* L;        // [bs, P, V] (logits form)
  int head;              // 1: head form (Lb, w2, u, lse instead of L)
  const float* Lb;       // [bs, P, V] base logits
  const __nv_bfloat16* w2;  // [V, 256]
  const float* u;        // [bs, P, 256]
  const float* lse;      // [bs, P] logsumexp_v L_i[v] / T
  int32_t* rej_j;        // [bs] head form: the rejected position j < P, or -1
  float* rej_norm;       // [bs][2] head form: log2-unit normalisers (q, p) at j
  const float* Z;        // [bs, P + 1, V]
  const float* U;        // [bs, P]
  const float* G;        // [bs, V]
  int bs, P, V, K;       // K: CTAs per request (the cluster size)
  int vec;               // 1: rows read as 16-byte vectors (V % 4 == 0, 16-byte aligned bases)
  float inv_T;
  int32_t* accept;
  int32_t* advanced;
  int32_t* next_token;
  Ctl* ctl;
};

// Block-wide merge of the (m, s) pairs and of the (m2, s2) pairs; thread 0
// holds the result.
__device__ __forceinline__ void block_lse2(float& m, float& s, float& m2, float& s2, float4* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float a = __shfl_xor_sync(0xffffffffu, m, o), c = __shfl_xor_sync(0xffffffffu, s, o);
    const float a2 = __shfl_xor_sync(0xffffffffu, m2, o), c2 = __shfl_xor_sync(0xffffffffu, s2, o);
    lse2_merge(m, s, a, c);
    lse2_merge(m2, s2, a2, c2);
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = make_float4(m, s, m2, s2);
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kSvWarps; ++w) {
      const float4 q = red[w];
      lse2_merge(m, s, q.x, q.y);
      lse2_merge(m2, s2, q.z, q.w);
    }
  }
}

__global__ void __launch_bounds__(kSvThreads) sv_verify_kernel(const __grid_constant__ SvP p) {
  __shared__ float4 red[kSvWarps];
  __shared__ __align__(16) float4 part[2];  // this CTA's (m_q, s_q, m_p, s_p), by round parity
  __shared__ unsigned long long kred[2][kSvWarps];
  __shared__ unsigned long long keys[2];  // this CTA's best residual / p keys
  __shared__ int stop_s, j_s;
  __shared__ float lq_s, lp_s;
  __shared__ float dec_s[3];  // L_i[x_i], Z_i[x_i], U_i, loaded by thread 0 ahead of the merge
  const int K = p.K, P = p.P, V = p.V;
  const uint32_t rank = cluster_rank();
  const int b = blockIdx.x / K;
  const float inv_T = p.inv_T, c2 = p.inv_T * kLog2e;
  const int n = p.vec ? (V >> 2) : V;  // elements of a row, in vectors when vec
  const int e0 = (int)((int64_t)n * rank / K), e1 = (int)((int64_t)n * (rank + 1) / K);

  for (int i = 0;; ++i) {
    const bool has_q = i < P;
    const bool read_q = has_q && !p.head;  // draft rows read in the logits form only
    const float* zr = p.Z + ((size_t)b * (P + 1) + i) * V;
    const float* lr = read_q ? p.L + ((size_t)b * P + i) * V : nullptr;
    if (threadIdx.x < 32 && has_q) {
      int x = p.draft[(size_t)b * P + i];
      if (x < 0 || x >= V) {
        if (rank == 0 && threadIdx.x == 0) dev_error(p.ctl, DEV_ERR_DATA);
        x = 0;
      }
      float lx;
      if (p.head) {
        // L_i[x] = L_base[b, i, x] + W2[x] . u_i: eight products per lane.
        const int lane = threadIdx.x;
        const uint4 w = __ldg((const uint4*)(p.w2 + (size_t)x * 256) + lane);
        const float4* ur = (const float4*)(p.u + ((size_t)b * P + i) * 256) + 2 * lane;
        const float4 u0 = __ldg(ur), u1 = __ldg(ur + 1);
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
        const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        float acc = 0.0f;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          acc = fmaf(__uint_as_float(wv[t] << 16), uv[2 * t], acc);
          acc = fmaf(__uint_as_float(wv[t] & 0xFFFF0000u), uv[2 * t + 1], acc);
        }
        lx = warp_sum(acc) + __ldg(p.Lb + ((size_t)b * P + i) * V + x);
      } else {
        lx = threadIdx.x == 0 ? __ldg(lr + x) : 0.0f;
      }
      if (threadIdx.x == 0) {
        dec_s[0] = lx;
        dec_s[1] = __ldg(zr + x);
        dec_s[2] = __ldg(p.U + (size_t)b * P + i);
      }
    }
    float mq = -INFINITY, sq = 0.0f, mp = -INFINITY, sp = 0.0f;
    if (p.vec) {
      const float4* z4 = (const float4*)zr;
      const float4* l4 = (const float4*)lr;
      for (int v = e0 + (int)threadIdx.x; v < e1; v += 4 * kSvThreads) {
        float4 a[4], c[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int vt = v + t * kSvThreads;
          if (vt < e1) {
            a[t] = __ldg(z4 + vt);
            if (read_q) c[t] = __ldg(l4 + vt);
          }
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if (v + t * kSvThreads < e1) {
            lse2_add4(mp, sp, a[t], c2);
            if (read_q) lse2_add4(mq, sq, c[t], c2);
          }
        }
      }
    } else {
      for (int v = e0 + (int)threadIdx.x; v < e1; v += kSvThreads) {
        lse2_add(mp, sp, __ldg(zr + v) * c2);
        if (read_q) lse2_add(mq, sq, __ldg(lr + v) * c2);
      }
    }
    block_lse2(mq, sq, mp, sp, red);
    if (threadIdx.x == 0) part[i & 1] = make_float4(mq, sq, mp, sp);
    // Double-buffered by parity: a CTA writes this slot again two rounds on,
    // after the next barrier, which every CTA reaches only once it has read it.
    cluster_sync();
    if (threadIdx.x == 0) {
      // Every CTA merges the cluster's pairs in rank order: the same
      // normalisers, the same decision.
      float m1 = -INFINITY, s1 = 0.0f, m2 = -INFINITY, s2 = 0.0f;
      for (int k = 0; k < K; ++k) {
        const float4 q = ld_dsmem_f32x4(&part[i & 1], (uint32_t)k);
        lse2_merge(m1, s1, q.x, q.y);
        lse2_merge(m2, s2, q.z, q.w);
      }
      const float lse_q = !has_q ? 0.0f : p.head ? __ldg(p.lse + (size_t)b * P + i) : (m1 + log2f(s1)) * kLn2;
      const float lse_p = (m2 + log2f(s2)) * kLn2;
      int stop = 0;
      if (!has_q) {
        stop = 1;  // all P accepted: the draw is from p_P
      } else {
        const float lq = dec_s[0] * inv_T - lse_q;
        const float lp = dec_s[1] * inv_T - lse_p;
        const float ratio = fminf(1.0f, expf(lp - lq));
        if (!(dec_s[2] < ratio)) stop = 1;
      }
      stop_s = stop;
      j_s = i;
      lq_s = lse_q;
      lp_s = lse_p;
    }
    __syncthreads();
    if (stop_s) break;
  }

  // The draw at position j over this CTA's slice: residual keys (j < P) and
  // keys from p_j, folded to one pair per CTA.
  const int j = j_s;
  const bool resid = j < P;
  if (p.head && resid) {
    // The residual kernel draws for this request; the cluster's shared
    // memory stays until every CTA is done with the last round's pairs.
    if (rank == 0 && threadIdx.x == 0) {
      p.rej_j[b] = j;
      p.rej_norm[2 * b] = lq_s * kLog2e;
      p.rej_norm[2 * b + 1] = lp_s * kLog2e;
      p.accept[b] = j;
      p.advanced[b] = j + 1;
    }
    cluster_sync();
    return;
  }
  const float lp2 = lp_s * kLog2e, lq2 = lq_s * kLog2e;  // the normalisers in log2 units
  const float* z = p.Z + ((size_t)b * (P + 1) + j) * V;
  const float* l = resid ? p.L + ((size_t)b * P + j) * V : nullptr;
  const float* g = p.G + (size_t)b * V;
  unsigned long long kr = 0ull, kp = 0ull;
  auto fold = [&](int v, float zv, float lv, float gv) {
    const float t2 = zv * c2 - lp2;  // log2 p_v
    const unsigned long long a = value_id_key(t2 * kLn2 + gv, (uint32_t)v);
    kp = a > kp ? a : kp;
    if (resid) {
      const float r = exp2f(t2) - exp2f(lv * c2 - lq2);
      if (r > 0.0f) {
        const unsigned long long k2 = value_id_key(log2f(r) * kLn2 + gv, (uint32_t)v);
        kr = k2 > kr ? k2 : kr;
      }
    }
  };
  if (p.vec) {
    for (int v = e0 + (int)threadIdx.x; v < e1; v += kSvThreads) {
      const float4 zv = __ldg((const float4*)z + v), gv = __ldg((const float4*)g + v);
      const float4 lv = resid ? __ldg((const float4*)l + v) : make_float4(0.f, 0.f, 0.f, 0.f);
      fold(4 * v + 0, zv.x, lv.x, gv.x);
      fold(4 * v + 1, zv.y, lv.y, gv.y);
      fold(4 * v + 2, zv.z, lv.z, gv.z);
      fold(4 * v + 3, zv.w, lv.w, gv.w);
    }
  } else {
    for (int v = e0 + (int)threadIdx.x; v < e1; v += kSvThreads)
      fold(v, __ldg(z + v), resid ? __ldg(l + v) : 0.0f, __ldg(g + v));
  }
  kr = warp_max_u64(kr);
  kp = warp_max_u64(kp);
  if ((threadIdx.x & 31) == 0) {
    kred[0][threadIdx.x >> 5] = kr;
    kred[1][threadIdx.x >> 5] = kp;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kSvWarps; ++w) {
      kr = kred[0][w] > kr ? kred[0][w] : kr;
      kp = kred[1][w] > kp ? kred[1][w] : kp;
    }
    keys[0] = kr;
    keys[1] = kp;
  }
  cluster_sync();
  if (rank == 0 && threadIdx.x == 0) {
    unsigned long long r = 0ull, pk = 0ull;
    for (int k = 0; k < K; ++k) {
      const unsigned long long x = ld_dsmem_u64(&keys[0], (uint32_t)k), y = ld_dsmem_u64(&keys[1], (uint32_t)k);
      r = x > r ? x : r;
      pk = y > pk ? y : pk;
    }
    const unsigned long long k = r ? r : pk;
    int tok = 0;
    if (k == 0ull) dev_error(p.ctl, DEV_ERR_DATA);
    else tok = (int)key_id(k);
    p.next_token[b] = tok;
    p.accept[b] = j;
    p.advanced[b] = j + 1;
    if (p.head) p.rej_j[b] = -1;
  }
  cluster_sync();  // the other CTAs' shared memory stays until CTA 0 has read it
}

}  // namespace

size_t sampled_verify_ws_bytes(int, int) { return 0; }

namespace {

cudaError_t launch_walk(SvP& p, int bs, int P, int V, float temperature, cudaStream_t stream) {
  p.bs = bs; p.P = P; p.V = V;
  p.vec = (V % 4) == 0 && ((uintptr_t)p.Z & 15u) == 0 && ((uintptr_t)p.G & 15u) == 0 &&
          (P == 0 || p.head || ((uintptr_t)p.L & 15u) == 0);
  p.inv_T = 1.0f / temperature;
  // CTAs per request: the largest power of two up to 8 that keeps the grid
  // within four CTAs per SM (all resident) and each slice at least 4096
  // values. The walk's last rounds serve the few requests still accepting,
  // so their speed is that of one request's K CTAs.
  int K = 1;
  while (K < kSvMaxCluster && (int64_t)bs * (2 * K) <= 4 * (int64_t)num_sms() && V / (2 * K) >= 4096) K *= 2;
  p.K = K;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(bs * K));
  cfg.blockDim = dim3(kSvThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)K;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, sv_verify_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sampled_verify(const int32_t* draft, const float* L, const float* Z, const float* U,
                                  const float* G, int bs, int P, int V, float temperature, int32_t* accept,
                                  int32_t* advanced, int32_t* next_token, Ctl* ctl, void*, cudaStream_t stream) {
  SvP p;
  memset(&p, 0, sizeof(p));
  p.draft = draft; p.L = L; p.Z = Z; p.U = U; p.G = G;
  p.accept = accept; p.advanced = advanced; p.next_token = next_token; p.ctl = ctl;
  return launch_walk(p, bs, P, V, temperature, stream);
}

cudaError_t launch_sampled_verify_head(const SampledHeadArgs& a, cudaStream_t stream) {
  SvP p;
  memset(&p, 0, sizeof(p));
  p.draft = a.draft; p.Z = a.Z; p.U = a.U; p.G = a.G;
  p.head = 1; p.Lb = a.L_base; p.w2 = (const __nv_bfloat16*)a.w2; p.u = a.u; p.lse = a.lse;
  p.rej_j = a.rej_j; p.rej_norm = a.rej_norm;
  p.accept = a.accept; p.advanced = a.advanced; p.next_token = a.next_token; p.ctl = a.ctl;
  cudaError_t e = launch_walk(p, a.bs, a.P, a.V, a.temperature, stream);
  if (e != cudaSuccess) return e;
  return launch_residual_draw(a, stream);
}

}  // namespace domino
