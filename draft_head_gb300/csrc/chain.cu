// The Domino head chain as one persistent kernel ("Technische Samenvatting:
// Domino", "Domino-head"; "上交大突破…", section 四).
//
// One CTA per SM, all resident (cooperative launch). Per drafted position i:
//
//   A  GRU step. CTA c owns a contiguous slice of the g hidden units; its W_hh
//      rows (gates r, z, n) stay in shared memory for the whole chain. The
//      input half of the gates is a row of the prepared gate table
//      (emb W_ih^T + b_ih) for the token just drawn. S_i for the owned units
//      goes to global memory.
//   B  Bottleneck u_i = SiLU(P_h[i] + W1_s S_i).
//        small batch: each CTA adds its units' share W1_s[:, J_c] S_i[J_c]
//        into 64-bit fixed-point accumulators (integer adds are associative,
//        so the sum is bit-identical run to run), then reads all of u after
//        the barrier;
//        larger batch: after a barrier, the (b, k) outputs are split across
//        CTAs, then a second barrier publishes u.
//   C  Correction + residual + sample, fused: CTA c owns a contiguous range of
//      vocabulary rows, streams its W2 rows once, forms
//      L = L_base[i] + W2 u_i (+ Gumbel noise at T > 0) in registers and keeps
//      only the best (value, id) key; one atomicMax per CTA and request merges
//      the keys. Full correction logits never go to memory (unless requested
//      for parity checks).
//   D  After the barrier every CTA reads the merged keys: tokens[:, i].
//
// Every grid barrier is a bounded wait; on timeout the kernel records the
// error in the workspace status word and all CTAs leave.
#include "common.cuh"

namespace domino {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kUaccPad = 16;  // 64-bit accumulators 128 bytes apart
constexpr double kInvFix = 1.0 / 4294967296.0;

template <typename WT>
struct ChainP {
  int bs, P, d, g, r, V, direct_u, nu_max;
  const float* gate_table;
  const WT* w_hh;
  const WT* b_hh;
  const WT* w1;
  const WT* w2;
  const float* L_base;
  const float* P_h;
  const int32_t* anchor;
  float temperature, inv_temperature;
  const float* gumbel;
  int64_t gumbel_bstride;
  const int32_t* force;
  int32_t* tokens;
  float* logits_out;
  Ctl* ctl;
  unsigned long long* keys;
  float* S;
  long long* uacc;
  float* uglob;
  uint64_t timeout_ns;
};

__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <typename WT>
__device__ __forceinline__ int clamp_token(const ChainP<WT>& p, int t) {
  if (t < 0 || t >= p.V) {
    dev_error(p.ctl, DEV_ERR_DATA);
    return 0;
  }
  return t;
}

// Decision value of one logit (greedy, or Gumbel-max at temperature T).
template <typename WT>
__device__ __forceinline__ float decision(const ChainP<WT>& p, float logit, int b, int i, int v) {
  if (p.temperature > 0.0f)
    return logit * p.inv_temperature + __ldg(p.gumbel + (int64_t)b * p.gumbel_bstride + (int64_t)i * p.V + v);
  return logit;
}

template <typename WT>
__global__ void __launch_bounds__(kThreads, 1) chain_kernel(const __grid_constant__ ChainP<WT> p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int G = gridDim.x, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bs = p.bs, g = p.g, r = p.r, V = p.V, P = p.P;
  const int j0 = (int)((int64_t)g * c / G), j1 = (int)((int64_t)g * (c + 1) / G), nu = j1 - j0;
  const int v0 = (int)((int64_t)V * c / G), v1 = (int)((int64_t)V * (c + 1) / G);
  const int nu_max = p.nu_max;

  // Shared memory carve-up.
  WT* whh_s = (WT*)smem;                                                  // [3*nu_max][g]
  size_t off = ((size_t)3 * nu_max * g * sizeof(WT) + 15) & ~(size_t)15;
  float* w1s_s = (float*)(smem + off); off += (size_t)r * nu_max * 4;    // [r][nu_max]
  float* bhh_s = (float*)(smem + off); off += (size_t)3 * nu_max * 4;    // [3*nu_max]
  float* u_s = (float*)(smem + off); off += (size_t)bs * r * 4;          // [bs][r]
  float* snew_s = (float*)(smem + off); off += (size_t)bs * nu_max * 4;  // [bs][nu_max]
  int* tok_s = (int*)(smem + off); off += (size_t)bs * 4;                // [bs]
  off = (off + 7) & ~(size_t)7;
  unsigned long long* red_s = (unsigned long long*)(smem + off);         // [kWarps][bs]

  // Resident weights for the owned hidden units.
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
  for (int b = threadIdx.x; b < bs; b += kThreads) tok_s[b] = clamp_token(p, p.anchor[b]);
  __syncthreads();

  unsigned epoch = 0;
  const int bsr = bs * r;

  for (int i = 0; i < P; ++i) {
    // ---------------- A: S_i = GRU(x_i, S_{i-1}) for the owned units.
    const float* Sprev = (i == 0) ? nullptr : p.S + (size_t)((i - 1) & 1) * bs * g;
    float* Snew = p.S + (size_t)(i & 1) * bs * g;
    for (int item = warp; item < bs * nu; item += kWarps) {
      const int b = item / nu, jj = item - b * nu, j = j0 + jj;
      float a0 = 0.f, a1 = 0.f, a2 = 0.f;
      if (Sprev) {
        const float* sp = Sprev + (size_t)b * g;
        const WT* wr0 = whh_s + (size_t)(0 * nu + jj) * g;
        const WT* wr1 = whh_s + (size_t)(1 * nu + jj) * g;
        const WT* wr2 = whh_s + (size_t)(2 * nu + jj) * g;
        for (int k = lane; k < g; k += 32) {
          const float s = __ldcg(sp + k);
          a0 = fmaf(to_f(wr0[k]), s, a0);
          a1 = fmaf(to_f(wr1[k]), s, a1);
          a2 = fmaf(to_f(wr2[k]), s, a2);
        }
        a0 = warp_sum(a0);
        a1 = warp_sum(a1);
        a2 = warp_sum(a2);
      }
      if (lane == 0) {
        const float* gi = p.gate_table + (size_t)tok_s[b] * 3 * g;
        const float gh_r = a0 + bhh_s[0 * nu + jj];
        const float gh_z = a1 + bhh_s[1 * nu + jj];
        const float gh_n = a2 + bhh_s[2 * nu + jj];
        const float rg = sigmoidf_(__ldg(gi + j) + gh_r);
        const float zg = sigmoidf_(__ldg(gi + g + j) + gh_z);
        const float ng = tanhf(__ldg(gi + 2 * g + j) + rg * gh_n);
        const float h = Sprev ? __ldcg(Sprev + (size_t)b * g + j) : 0.0f;
        const float hn = (1.0f - zg) * ng + zg * h;
        Snew[(size_t)b * g + j] = hn;
        snew_s[b * nu_max + jj] = hn;
      }
    }
    __syncthreads();
    long long* uacc_cur = p.uacc + (size_t)(i & 1) * bsr * kUaccPad;
    if (p.direct_u && nu > 0) {
      for (int idx = threadIdx.x; idx < bsr; idx += kThreads) {
        const int b = idx / r, k = idx - b * r;
        float part = 0.0f;
        for (int jj = 0; jj < nu; ++jj) part = fmaf(w1s_s[k * nu + jj], snew_s[b * nu_max + jj], part);
        // Cleared every step: in range while the G partials sum below 2^31;
        // 2^30 / G per partial keeps a factor two.
        const long long fx = fix32_checked(part, 1073741824.0f / (float)G, p.ctl);
        atomicAdd((unsigned long long*)(uacc_cur + (size_t)idx * kUaccPad), (unsigned long long)fx);
      }
    }
    if (!grid_barrier(p.ctl, epoch, G, p.timeout_ns)) return;

    // ---------------- B: u_i.
    if (p.direct_u) {
      for (int idx = threadIdx.x; idx < bsr; idx += kThreads) {
        const int b = idx / r, k = idx - b * r;
        const long long fx = __ldcg(uacc_cur + (size_t)idx * kUaccPad);
        const float pre = __ldg(p.P_h + ((size_t)b * P + i) * r + k) + (float)((double)fx * kInvFix);
        u_s[idx] = siluf_(pre);
      }
      if (c == 0) {
        long long* nxt = p.uacc + (size_t)((i + 1) & 1) * bsr * kUaccPad;
        for (int idx = threadIdx.x; idx < bsr; idx += kThreads) nxt[(size_t)idx * kUaccPad] = 0;
      }
    } else {
      for (int item = c * kWarps + warp; item < bsr; item += G * kWarps) {
        const int b = item / r, k = item - b * r;
        const float* sp = Snew + (size_t)b * g;
        const WT* wr = p.w1 + (size_t)k * (p.d + g) + p.d;
        float a = 0.f;
        for (int kk = lane; kk < g; kk += 32) a = fmaf(to_f(wr[kk]), __ldcg(sp + kk), a);
        a = warp_sum(a);
        if (lane == 0) p.uglob[item] = siluf_(__ldg(p.P_h + ((size_t)b * P + i) * r + k) + a);
      }
      if (!grid_barrier(p.ctl, epoch, G, p.timeout_ns)) return;
      for (int idx = threadIdx.x; idx < bsr; idx += kThreads) u_s[idx] = __ldcg(p.uglob + idx);
    }
    for (int idx = threadIdx.x; idx < kWarps * bs; idx += kThreads) red_s[idx] = 0ull;
    __syncthreads();

    // ---------------- C: L = L_base + W2 u (+ noise), best key per request.
    const int nrows = v1 - v0;
    bool fast = false;
    if constexpr (sizeof(WT) == 2) {
      if (bs == 1 && r == 256) {
        fast = true;
        // Batch 1: a warp-load covers one 512-byte W2 row; 16 rows per
        // iteration are reduced across lanes with a transposing butterfly
        // (9 shuffles per 8 rows instead of 40).
        float ur[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) ur[t] = u_s[lane * 8 + t];
        const float* lrow = p.L_base + (size_t)i * V;
        unsigned long long best = 0ull;
        for (int base = warp * 16; base < nrows; base += kWarps * 16) {
          uint4 wv[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int rr = min(base + q, nrows - 1);
            wv[q] = ldg_stream_v4(p.w2 + (size_t)(v0 + rr) * 256 + lane * 8);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float pr[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float f[8];
              bf16x8_to_f32(wv[h * 8 + q], f);
              float s = 0.f;
#pragma unroll
              for (int t = 0; t < 8; ++t) s = fmaf(f[t], ur[t], s);
              pr[q] = s;
            }
            {
              const bool hi = lane & 16;
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                const float send = hi ? pr[t] : pr[t + 4];
                const float keep = hi ? pr[t + 4] : pr[t];
                pr[t] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
              }
            }
            {
              const bool hi = lane & 8;
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                const float send = hi ? pr[t] : pr[t + 2];
                const float keep = hi ? pr[t + 2] : pr[t];
                pr[t] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
              }
            }
            {
              const bool hi = lane & 4;
              const float send = hi ? pr[0] : pr[1];
              const float keep = hi ? pr[1] : pr[0];
              pr[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
            }
            pr[0] += __shfl_xor_sync(0xffffffffu, pr[0], 2);
            pr[0] += __shfl_xor_sync(0xffffffffu, pr[0], 1);
            const int rowq = ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
            const int rr = base + h * 8 + rowq;
            if ((lane & 3) == 0 && rr < nrows) {
              const int v = v0 + rr;
              const float logit = __ldg(lrow + v) + pr[0];
              if (p.logits_out) p.logits_out[(size_t)i * V + v] = logit;
              const unsigned long long key = value_id_key(decision(p, logit, 0, i, v), (uint32_t)v);
              best = key > best ? key : best;
            }
          }
        }
        best = warp_max_u64(best);
        if (lane == 0) red_s[warp] = best;
      }
    }
    if (!fast) {
      // General batch / element type: a warp per vocabulary row, W2 row held
      // in registers while every request's u is applied.
      for (int rr = warp; rr < nrows; rr += kWarps) {
        const int v = v0 + rr;
        float wreg[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const int k = lane + 32 * t;
          wreg[t] = (k < r) ? to_f(p.w2[(size_t)v * r + k]) : 0.0f;
        }
        for (int b = 0; b < bs; ++b) {
          const float* ub = u_s + (size_t)b * r;
          float s = 0.f;
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            const int k = lane + 32 * t;
            if (k < r) s = fmaf(wreg[t], ub[k], s);
          }
          s = warp_sum(s);
          if (lane == 0) {
            const float logit = __ldg(p.L_base + ((size_t)b * P + i) * V + v) + s;
            if (p.logits_out) p.logits_out[((size_t)b * P + i) * V + v] = logit;
            const unsigned long long key = value_id_key(decision(p, logit, b, i, v), (uint32_t)v);
            unsigned long long* slot = red_s + warp * bs + b;
            if (key > *slot) *slot = key;
          }
        }
      }
    }
    __syncthreads();
    for (int b = threadIdx.x; b < bs; b += kThreads) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kWarps; ++w) {
        const unsigned long long x = red_s[w * bs + b];
        m = x > m ? x : m;
      }
      if (m) atomicMax(p.keys + (size_t)i * bs + b, m);
    }
    if (!grid_barrier(p.ctl, epoch, G, p.timeout_ns)) return;

    // ---------------- D: tokens of position i; next GRU input.
    for (int b = threadIdx.x; b < bs; b += kThreads) {
      const unsigned long long key = __ldcg(p.keys + (size_t)i * bs + b);
      int tok = 0;
      if (key == 0ull) {
        dev_error(p.ctl, DEV_ERR_DATA);  // no finite decision value
      } else {
        tok = (int)key_id(key);
      }
      if (c == 0) p.tokens[(size_t)b * P + i] = tok;
      const int nxt = (p.force && i + 1 < P) ? p.force[(size_t)b * P + i] : tok;
      tok_s[b] = clamp_token(p, nxt);
    }
    __syncthreads();
  }
}

template <typename WT>
size_t chain_smem_bytes(int bs, int g, int r, int nu_max) {
  size_t off = ((size_t)3 * nu_max * g * sizeof(WT) + 15) & ~(size_t)15;
  off += (size_t)r * nu_max * 4 + (size_t)3 * nu_max * 4 + (size_t)bs * r * 4 + (size_t)bs * nu_max * 4 +
         (size_t)bs * 4;
  off = (off + 7) & ~(size_t)7;
  off += (size_t)kWarps * bs * 8;
  return off;
}

template <typename WT>
cudaError_t launch_chain_t(const ChainArgs& a, cudaStream_t stream) {
  const int G = num_sms();
  ChainP<WT> p;
  p.bs = a.bs; p.P = a.P; p.d = a.d; p.g = a.g; p.r = a.r; p.V = a.V;
  p.direct_u = (a.bs <= 4) ? 1 : 0;
  p.nu_max = (a.g + G - 1) / G;
  p.gate_table = a.gate_table;
  p.w_hh = (const WT*)a.w_hh; p.b_hh = (const WT*)a.b_hh; p.w1 = (const WT*)a.w1; p.w2 = (const WT*)a.w2;
  p.L_base = a.L_base; p.P_h = a.P_h; p.anchor = a.anchor;
  p.temperature = a.temperature;
  p.inv_temperature = a.temperature > 0.0f ? 1.0f / a.temperature : 0.0f;
  p.gumbel = a.gumbel; p.gumbel_bstride = a.gumbel_bstride;
  p.force = a.force; p.tokens = a.tokens; p.logits_out = a.logits_out;
  p.ctl = a.ctl; p.keys = a.keys; p.S = a.S; p.uacc = a.uacc; p.uglob = a.uglob;
  p.timeout_ns = wait_timeout_ns();
  const size_t smem = chain_smem_bytes<WT>(a.bs, a.g, a.r, p.nu_max);
  if (smem > 227 * 1024) return cudaErrorInvalidConfiguration;
  cudaError_t e = cudaFuncSetAttribute(chain_kernel<WT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void* args[] = {(void*)&p};
  return cudaLaunchCooperativeKernel((const void*)chain_kernel<WT>, dim3(G), dim3(kThreads), args, smem, stream);
}

}  // namespace

size_t chain_ws_bytes(int bs, int P, int g, int r) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al((size_t)P * bs * 8) + al((size_t)2 * bs * g * 8) + al((size_t)2 * bs * r * kUaccPad * 8) +
         al((size_t)bs * r * 4);
}

bool chain_fits(int dtype, int bs, int g, int r) {
  const int G = num_sms();
  const int nu_max = (g + G - 1) / G;
  const size_t smem = dtype == DOMINO_BF16 ? chain_smem_bytes<__nv_bfloat16>(bs, g, r, nu_max)
                                           : chain_smem_bytes<float>(bs, g, r, nu_max);
  return smem <= 227 * 1024;
}

cudaError_t launch_chain(const ChainArgs& a, cudaStream_t stream) {
  if (a.lse_out != nullptr)  // the draft statistics come from the batched kernel only
    return chain_batched_applies(a) ? launch_chain_batched(a, stream) : cudaErrorInvalidConfiguration;
  if (chain_small_applies(a)) return launch_chain_small(a, stream);
  if (chain_batched_applies(a)) return launch_chain_batched(a, stream);
  if (a.dtype == DOMINO_BF16) return launch_chain_t<__nv_bfloat16>(a, stream);
  return launch_chain_t<float>(a, stream);
}

}  // namespace domino
