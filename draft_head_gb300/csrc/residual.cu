// The draw at the first rejected position of a sampled verification when the
// draft is given by the head rather than by its logits (163.com report,
// section 五: the standard speculative-decoding procedure; the residual
// distribution norm(max(0, p_j - q_j)) at the first rejection j).
//
// The walk (verify_sampled.cu, head form) has found, per request, the
// rejected position j and the two normalisers. Here the rejected rows
//   L_j[v] = L_base[b, j, v] + W2[v] . u_j[b]
// are rebuilt for all rejected requests at once, so W2 is read once per call,
// not once per request: CTA c owns a contiguous vocabulary range, streams its
// W2 rows in 128-row tiles by TMA (128-byte swizzle, two stages), and each
// warp multiplies 16 rows by half of the requests' u columns on the tensor cores
// (bf16 m16n8k16 MMAs, fp32 accumulate; u as a bf16 high column and a bf16
// low column, hi + lo keeps ~16 mantissa bits, the chain's own split). The
// epilogue forms q_v and p_v in fp32 exactly as the logits form does and
// keeps the best (log r_v + G_v, v) key per request; one atomicMax per
// request and CTA. The last CTA to finish (an arrival counter, no waiting)
// writes the drawn tokens and leaves the keys and the counter at zero for the
// next call. If a request's residual is zero everywhere in fp32 that CTA
// draws from p_j instead.
#include <cuda.h>
#include <string.h>

#include "common.cuh"

namespace domino {

bool tmap_bf16_rows(CUtensorMap* tm, const void* base, int rows, int cols, int box_rows);

namespace {

constexpr int kRdThreads = 512;              // 16 warps: 8 row slices of 16 x 2 request halves
constexpr int kRdMaxReq = 64;                // requests per launch window (4 groups of 16)
constexpr uint32_t kTileBytes = 128u * 512u;  // 4 chunks of 128 rows x 64 bf16
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct RdP {
  CUtensorMap tm_w2;  // W2 [V, 256], boxes of 64 columns x 128 rows, 128-byte swizzle
  const float* Lb;    // [bs, P, V]
  const float* Z;     // [bs, P + 1, V]
  const float* G;     // [bs, V]
  const float* u;     // [bs, P, 256]
  const int32_t* rej_j;   // [bs] rejected position or -1
  const float* rej_norm;  // [bs][2] (q, p) normalisers, log2 units
  int bs, P, V, b0, nb;   // the window of requests [b0, b0 + nb)
  float c2;               // log2(e) / T
  unsigned long long* keys;  // [bs]
  unsigned int* done;        // this window's arrival counter
  int32_t* next_token;
  Ctl* ctl;
  uint64_t timeout_ns;
};

__device__ __forceinline__ int rd_vocab_begin(int V, int c, int G) {
  return c >= G ? V : (int)(((int64_t)V * c / G) & ~(int64_t)3);
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint2 b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b.x), "r"(b.y));
}

__device__ __forceinline__ uint32_t bf16_bits(float x) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}
// The high or the low bf16 part of x (x ~ hi + lo).
__device__ __forceinline__ uint32_t bf16_part(float x, int lo) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(x);
  return lo ? bf16_bits(x - __bfloat162float(hi)) : (uint32_t)__bfloat16_as_ushort(hi);
}

__global__ void __launch_bounds__(kRdThreads, 1) residual_kernel(const __grid_constant__ RdP p) {
  // Warp w: rows 16 (w % 8) .. + 16 of each tile, request groups 2 (w / 8)
  // and 2 (w / 8) + 1 (16 requests each).
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint2* bfrag = (uint2*)(smem + 2 * kTileBytes);  // [group 4][kk 16][n-tile 4][lane 32]
  __shared__ int rq_s[kRdMaxReq], rj_s[kRdMaxReq];
  __shared__ float lq_s[kRdMaxReq], lp_s[kRdMaxReq];
  __shared__ unsigned long long key_s[kRdMaxReq];
  __shared__ __align__(8) uint64_t full[2];
  __shared__ int nreq_s, last_s;
  __shared__ volatile int abort_s;
  const int G = gridDim.x, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g4 = lane >> 2, t4 = lane & 3;
  const int P = p.P, V = p.V;

  // The rejected requests of the window, in request order (every CTA builds
  // the same list).
  if (threadIdx.x == 0) {
    int n = 0;
    for (int b = p.b0; b < p.b0 + p.nb; ++b) {
      const int j = p.rej_j[b];
      if (j >= 0) {
        if (j >= P) { dev_error(p.ctl, DEV_ERR_DATA); continue; }
        rq_s[n] = b;
        rj_s[n] = j;
        lq_s[n] = p.rej_norm[2 * b];
        lp_s[n] = p.rej_norm[2 * b + 1];
        ++n;
      }
    }
    nreq_s = n;
    abort_s = 0;
  }
  for (int q = threadIdx.x; q < kRdMaxReq; q += kRdThreads) key_s[q] = 0ull;
  __syncthreads();
  const int nreq = nreq_s;
  if (nreq == 0) return;  // the same decision in every CTA: nothing to draw, no arrivals
  const int ngr = (nreq + 15) / 16;

  const int v0 = rd_vocab_begin(V, c, G), v1 = rd_vocab_begin(V, c + 1, G);
  const int ntiles = (v1 - v0 + 127) / 128;
  if (threadIdx.x == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_fence_init();
    for (int t = 0; t < 2 && t < ntiles; ++t) {
      mbar_expect_tx(&full[t], kTileBytes);
#pragma unroll
      for (int kc = 0; kc < 4; ++kc)
        tma_load_2d(smem + t * kTileBytes + kc * 16384u, &p.tm_w2, 64 * kc, v0 + 128 * t, &full[t]);
    }
  }
  // B fragments of the requests' u columns: n-tile nt of group gr holds
  // columns 8 nt .. 8 nt + 7 = requests 16 gr + 4 nt + (0..3), each as a high
  // and a low column; lane (g, t) holds column g's rows k = 16 kk + 2 t (+1)
  // and k + 8 (+1), the lower k in the lower half.
  for (int idx = threadIdx.x; idx < ngr * 16 * 4 * 32; idx += kRdThreads) {
    const int L = idx & 31, nt = (idx >> 5) & 3, kk = (idx >> 7) & 15, gr = idx >> 11;
    const int col = 8 * nt + (L >> 2), req = 16 * gr + (col >> 1), lo = col & 1;
    const int k = 16 * kk + 2 * (L & 3);
    uint2 f = make_uint2(0u, 0u);
    if (req < nreq) {
      const float* ur = p.u + ((size_t)rq_s[req] * P + rj_s[req]) * 256;
      f.x = bf16_part(__ldg(ur + k), lo) | (bf16_part(__ldg(ur + k + 1), lo) << 16);
      f.y = bf16_part(__ldg(ur + k + 8), lo) | (bf16_part(__ldg(ur + k + 9), lo) << 16);
    }
    bfrag[idx] = f;
  }
  __syncthreads();

  unsigned long long best[2][4];
#pragma unroll
  for (int g2 = 0; g2 < 2; ++g2)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) best[g2][nt] = 0ull;
  const float c2 = p.c2;
  const int slice = warp & 7, half = warp >> 3;

  for (int t = 0; t < ntiles; ++t) {
    const int s = t & 1;
    const bool got = mbar_wait(&full[s], (uint32_t)((t >> 1) & 1), &abort_s, p.ctl, p.timeout_ns);
    if (__syncthreads_or(!got)) break;  // the same decision in every thread
    // ldmatrix on the swizzled tile: lane L addresses row (L & 7) + 8 ((L >> 3) & 1)
    // of the warp's 16 rows and 16-byte column 2 (kk % 4) + (L >> 4) of chunk kk / 4.
    const int rr = 16 * slice + (lane & 7) + 8 * ((lane >> 3) & 1);
    const uint32_t abase = smem_u32(smem + s * kTileBytes) + (uint32_t)rr * 128u;
    const int va = v0 + 128 * t + 16 * slice + g4, vb = va + 8;  // this lane's two rows
#pragma unroll
    for (int g2 = 0; g2 < 2; ++g2) {
      const int gr = 2 * half + g2;
      if (gr < ngr) {
        // The epilogue's operands first, so their loads overlap the MMAs.
        float lb[4][2], zv[4][2], gv[4][2];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int req = 16 * gr + 4 * nt + t4;
          const bool rq = req < nreq;
          const int b = rq ? rq_s[req] : 0, j = rq ? rj_s[req] : 0;
          const float* lrow = p.Lb + ((size_t)b * P + j) * V;
          const float* zrow = p.Z + ((size_t)b * (P + 1) + j) * V;
          const float* grow = p.G + (size_t)b * V;
          const bool ia = rq && va < v1, ib = rq && vb < v1;
          lb[nt][0] = ia ? __ldg(lrow + va) : 0.0f;
          zv[nt][0] = ia ? __ldg(zrow + va) : 0.0f;
          gv[nt][0] = ia ? __ldg(grow + va) : 0.0f;
          lb[nt][1] = ib ? __ldg(lrow + vb) : 0.0f;
          zv[nt][1] = ib ? __ldg(zrow + vb) : 0.0f;
          gv[nt][1] = ib ? __ldg(grow + vb) : 0.0f;
        }
        float acc[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[nt][q] = 0.0f;
        const uint2* bf = bfrag + (size_t)gr * 16 * 4 * 32 + lane;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          uint32_t a[4];
          const int cu = 2 * (kk & 3) + (lane >> 4);
          const uint32_t addr = abase + (uint32_t)(kk >> 2) * 16384u + (uint32_t)((cu ^ (rr & 7)) << 4);
          asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                       : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                       : "r"(addr)
                       : "memory");
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) mma16816(acc[nt], a, bf[(kk * 4 + nt) * 32]);
        }
        // Lane (g, t): columns 2t (high) and 2t + 1 (low) of n-tile nt are
        // request 16 gr + 4 nt + t; accumulator pairs (0, 1) row g, (2, 3) row g + 8.
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const int req = 16 * gr + 4 * nt + t4;
          if (req < nreq) {
            const float lq2 = lq_s[req], lp2 = lp_s[req];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int v = h ? vb : va;
              if (v < v1) {
                const float lv = lb[nt][h] + (acc[nt][2 * h] + acc[nt][2 * h + 1]);
                const float t2 = zv[nt][h] * c2 - lp2;
                const float r = exp2f(t2) - exp2f(lv * c2 - lq2);
                if (r > 0.0f) {
                  const unsigned long long k2 = value_id_key(log2f(r) * kLn2 + gv[nt][h], (uint32_t)v);
                  best[g2][nt] = k2 > best[g2][nt] ? k2 : best[g2][nt];
                }
              }
            }
          }
        }
      }
    }
    __syncthreads();  // every warp is done with the stage: it can be refilled
    if (threadIdx.x == 0 && t + 2 < ntiles && !abort_s) {
      mbar_expect_tx(&full[s], kTileBytes);
#pragma unroll
      for (int kc = 0; kc < 4; ++kc)
        tma_load_2d(smem + s * kTileBytes + kc * 16384u, &p.tm_w2, 64 * kc, v0 + 128 * (t + 2), &full[s]);
    }
  }

  // Per request: the maximum over the eight lanes with the same t, then over
  // the warps (shared atomics), then one global atomicMax per CTA.
#pragma unroll
  for (int g2 = 0; g2 < 2; ++g2)
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int gr = 2 * half + g2;
      unsigned long long k = best[g2][nt];
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        const unsigned long long w = __shfl_xor_sync(0xffffffffu, k, o);
        k = w > k ? w : k;
      }
      const int req = 16 * gr + 4 * nt + t4;
      if (g4 == 0 && req < nreq && k) atomicMax(&key_s[req], k);
    }
  __syncthreads();
  for (int q = threadIdx.x; q < nreq; q += kRdThreads)
    if (key_s[q]) atomicMax(p.keys + rq_s[q], key_s[q]);
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last_s = atomicAdd(p.done, 1u) == (unsigned)(G - 1);
  }
  __syncthreads();
  if (!last_s) return;

  // The last CTA: every other CTA's keys are in. Read and clear them.
  __threadfence();
  for (int q = threadIdx.x; q < nreq; q += kRdThreads) key_s[q] = atomicExch(p.keys + rq_s[q], 0ull);
  __syncthreads();
  // A residual that is zero everywhere in fp32: the draw is from p_j.
  __shared__ unsigned long long red_s[kRdThreads / 32];
  for (int q = 0; q < nreq; ++q) {
    if (key_s[q] != 0ull) continue;  // uniform: shared value read after the barrier
    const int b = rq_s[q];
    const float* zrow = p.Z + ((size_t)b * (P + 1) + rj_s[q]) * V;
    const float* grow = p.G + (size_t)b * V;
    const float lp2 = lp_s[q];
    unsigned long long k = 0ull;
    for (int v = threadIdx.x; v < V; v += kRdThreads) {
      const unsigned long long a = value_id_key((__ldg(zrow + v) * c2 - lp2) * kLn2 + __ldg(grow + v), (uint32_t)v);
      k = a > k ? a : k;
    }
    k = warp_max_u64(k);
    if (lane == 0) red_s[warp] = k;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 0; w < kRdThreads / 32; ++w) k = red_s[w] > k ? red_s[w] : k;
      key_s[q] = k;
    }
    __syncthreads();
  }
  for (int q = threadIdx.x; q < nreq; q += kRdThreads) {
    const unsigned long long k = key_s[q];
    int tok = 0;
    if (k == 0ull) dev_error(p.ctl, DEV_ERR_DATA);
    else tok = (int)key_id(k);
    p.next_token[rq_s[q]] = tok;
  }
  if (threadIdx.x == 0) *p.done = 0u;
}

size_t residual_smem() { return 1024 + 2 * (size_t)kTileBytes + (size_t)4 * 16 * 4 * 32 * 8; }

}  // namespace

size_t sampled_head_ws_bytes(int bs) {
  // rej_j [bs] int32, rej_norm [bs][2] fp32, keys [bs] u64, one counter per
  // 64-request window (32 bytes apart); each piece 256-byte aligned.
  auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t nwin = ((size_t)bs + kRdMaxReq - 1) / kRdMaxReq;
  return a((size_t)bs * 4) + a((size_t)bs * 8) + a((size_t)bs * 8) + a(nwin * 32);
}

cudaError_t launch_residual_draw(const SampledHeadArgs& a, cudaStream_t stream) {
  RdP p;
  memset(&p, 0, sizeof(p));
  if (!tmap_bf16_rows(&p.tm_w2, a.w2, a.V, 256, 128)) return cudaErrorInvalidValue;
  p.Lb = a.L_base; p.Z = a.Z; p.G = a.G; p.u = a.u;
  p.rej_j = a.rej_j; p.rej_norm = a.rej_norm;
  p.bs = a.bs; p.P = a.P; p.V = a.V;
  p.c2 = kLog2e / a.temperature;
  p.keys = a.rd_keys; p.next_token = a.next_token; p.ctl = a.ctl;
  p.timeout_ns = wait_timeout_ns();
  const size_t smem = residual_smem();
  cudaError_t e = cudaFuncSetAttribute(residual_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  for (int b0 = 0; b0 < a.bs; b0 += kRdMaxReq) {
    p.b0 = b0;
    p.nb = a.bs - b0 < kRdMaxReq ? a.bs - b0 : kRdMaxReq;
    p.done = a.rd_done + (size_t)(b0 / kRdMaxReq) * 8;
    residual_kernel<<<num_sms(), kRdThreads, smem, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace domino
