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
//
// Two forms of the same computation. The tensor-memory form (V % 4 == 0,
// 16-byte aligned rows): the rejected requests' u_j as a bf16 high and low
// row each (at most 128 rows) are the A operand of tcgen05.mma in shared
// memory, W2 tiles (128 rows) the B operand, streamed by TMA through a
// four-stage ring; the accumulator D [request rows x 128 vocabulary rows]
// lives in tensor memory, double-buffered. An epilogue lane then holds one
// request's high or low products: the two lanes of a request swap halves,
// and each reads 16 consecutive entries of its request's L_base, target
// and noise rows with 16-byte loads. The warp-MMA form below serves the
// other shapes.
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

// ---------------------------------------------------------------------------
// Tensor-memory form.
constexpr int kRtThreads = 384;  // warp 0: TMA, warp 1: MMA, warps 4-11: epilogue
constexpr int kRtStages = 4;
constexpr uint32_t kRtChunk = 128u * 128u;  // 128 rows x 64 bf16

struct RtP {
  CUtensorMap tm_w2;  // W2 [V, 256], boxes of 64 columns x 128 rows, 128-byte swizzle
  const float* Lb;
  const float* Z;
  const float* G;
  const float* u;
  const int32_t* rej_j;
  const float* rej_norm;
  int bs, P, V, b0, nb;
  float c2;
  unsigned long long* keys;
  unsigned int* done;
  int32_t* next_token;
  Ctl* ctl;
  uint64_t timeout_ns;
};

// Byte offset of element (row, k) of a K-major operand of 64-column chunks of
// `rows` rows each, 128-byte swizzled (the layout TMA writes with SWIZZLE_128B).
// The larger of a and b, NaN if either is NaN.
__device__ __forceinline__ float fmax_nan_rt(float a, float b) {
  float y;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}

__device__ __forceinline__ uint32_t rt_sw128(int row, int k, int rows) {
  const int kc = k >> 6, kk = k & 63;
  return (uint32_t)(kc * rows * 128 + row * 128 + ((((kk >> 3) ^ (row & 7)) & 7) << 4) + (kk & 7) * 2);
}

__device__ __forceinline__ void rt_tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

__global__ void __launch_bounds__(kRtThreads, 1) residual_tc_kernel(const __grid_constant__ RtP p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t* ring = smem;                               // kRtStages x 16 KB of W2
  uint8_t* uop = ring + kRtStages * kRtChunk;         // U16: 4 chunks x 128 rows x 128 B
  __shared__ int rq_s[kRdMaxReq], rj_s[kRdMaxReq];
  __shared__ float lq_s[kRdMaxReq], lp_s[kRdMaxReq];
  __shared__ unsigned long long key_s[2][kRdMaxReq];
  __shared__ __align__(8) uint64_t full[kRtStages], empty[kRtStages], t_full[2], t_empty[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int nreq_s, last_s;
  __shared__ volatile int abort_s;
  __shared__ unsigned long long red_s[kRtThreads / 32];
  const int G = gridDim.x, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = p.P, V = p.V;

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
  for (int q = threadIdx.x; q < 2 * kRdMaxReq; q += kRtThreads) key_s[q >> 6][q & 63] = 0ull;
  __syncthreads();
  const int nreq = nreq_s;
  if (nreq == 0) return;  // the same in every CTA: nothing to draw, no arrivals

  // U16: row 2 q + h = the high (h = 0) or low (h = 1) bf16 part of u_j of
  // rejected request q; rows past 2 nreq zero.
  for (int idx = threadIdx.x; idx < 128 * 32; idx += kRtThreads) {  // 16-byte groups of 8 entries
    const int row = idx >> 5, k8 = (idx & 31) * 8;
    const int q = row >> 1, h = row & 1;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (q < nreq) {
      const float4* ur = (const float4*)(p.u + ((size_t)rq_s[q] * P + rj_s[q]) * 256 + k8);
      const float4 x0 = __ldg(ur), x1 = __ldg(ur + 1);
      const float xs[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t lo0 = bf16_part(xs[2 * e], h), hi0 = bf16_part(xs[2 * e + 1], h);
        w[e] = lo0 | (hi0 << 16);
      }
    }
    *(uint4*)(uop + rt_sw128(row, k8, 128)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes, then the MMA's reads

  const int v0 = rd_vocab_begin(V, c, G), v1 = rd_vocab_begin(V, c + 1, G);
  const int ntiles = (v1 - v0 + 127) / 128;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int a = 0; a < 2; ++a) { mbar_init(&t_full[a], 1); mbar_init(&t_empty[a], 8); }
    mbar_fence_init();
    tma_prefetch_desc(&p.tm_w2);
  }
  if (warp == 1) { tmem_alloc(&tmem_slot, 256); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t d_w = tmem_slot;
  const float c2 = p.c2;

  if (warp == 0 && lane == 0) {
    uint32_t st = 0, ph = 0;
    bool go = true;
    for (int t = 0; t < ntiles && go; ++t)
      for (int kc = 0; kc < 4; ++kc) {
        if (!mbar_wait(&empty[st], ph ^ 1u, &abort_s, p.ctl, p.timeout_ns)) { go = false; break; }
        mbar_expect_tx(&full[st], kRtChunk);
        tma_load_2d(ring + st * kRtChunk, &p.tm_w2, 64 * kc, v0 + 128 * t, &full[st]);
        if (++st == kRtStages) { st = 0; ph ^= 1u; }
      }
  } else if (warp == 1 && lane == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, 128);
    uint32_t st = 0, ph = 0;
    bool go = true;
    for (int t = 0; t < ntiles && go; ++t) {
      const int acc = t & 1;
      if (!mbar_wait(&t_empty[acc], (uint32_t)(((t >> 1) & 1) ^ 1), &abort_s, p.ctl, p.timeout_ns)) break;
      tc_fence_after();
      for (int kc = 0; kc < 4; ++kc) {
        if (!mbar_wait(&full[st], ph, &abort_s, p.ctl, p.timeout_ns)) { go = false; break; }
        tc_fence_after();
        const uint64_t ad = sdesc_k_sw128(smem_u32(uop + kc * kRtChunk));
        const uint64_t bd = sdesc_k_sw128(smem_u32(ring + st * kRtChunk));
#pragma unroll
        for (int k = 0; k < 4; ++k) umma_bf16(d_w + (uint32_t)(acc * 128), ad + 2 * k, bd + 2 * k, idesc, (kc | k) ? 1u : 0u);
        umma_commit(&empty[st]);
        if (++st == kRtStages) { st = 0; ph ^= 1u; }
      }
      if (go) umma_commit(&t_full[acc]);
    }
  } else if (warp >= 4) {
    // Lane 32 qd + l: U16 row 32 qd + l, request q = 16 qd + l / 2, part l % 2.
    // Team tm takes columns [64 tm, +64) of each tile, 32 at a time; the two
    // lanes of a request swap halves so each holds hi + lo for 16 columns.
    const int qd = warp & 3, tm = (warp - 4) >> 2;
    const int q = 16 * qd + (lane >> 1), part = lane & 1;
    const bool live = 32 * qd < 2 * nreq;  // warp-uniform
    const bool rq = q < nreq;
    const int b = rq ? rq_s[q] : 0, j = rq ? rj_s[q] : 0;
    const float lq2 = rq ? lq_s[q] : 0.0f, lp2 = rq ? lp_s[q] : 0.0f;
    const float* lrow = p.Lb + ((size_t)b * P + j) * V;
    const float* zrow = p.Z + ((size_t)b * (P + 1) + j) * V;
    const float* grow = p.G + (size_t)b * V;
    unsigned long long best = 0ull;  // exactly ranked groups (partial, or with a NaN)
    // Whole groups of 16 entries without a NaN are ranked by their largest
    // draw value alone; the lane keeps the values of its best such group
    // (the earliest on equal maxima) and ranks inside it once, at the end.
    // Entries with a zero residual do not take part: -inf here (the noise is
    // finite, so no present entry has that value).
    float gbest = -INFINITY, gvals[16];
    int gvb = -1;  // first vocabulary row of the best whole group (-1: none)
#pragma unroll
    for (int e = 0; e < 16; ++e) gvals[e] = -INFINITY;
    // The rows of half-tile h = 2 t + hh: 16 entries from vb(h) of this
    // request's L_base, target and noise rows. They do not depend on the
    // accumulator, so each half's are requested one half ahead.
    auto vbase = [&](int h) { return v0 + 128 * (h >> 1) + 64 * tm + 32 * (h & 1) + 16 * part; };
    float4 nL[4], nZ[4], nG[4];
    auto fetch = [&](int h) {
      const int vb = vbase(h);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const int v = vb + 4 * q4;
        const bool in = live && rq && h < 2 * ntiles && v < v1;  // v1 is a multiple of 4
        nL[q4] = in ? __ldg((const float4*)(lrow + v)) : make_float4(0.f, 0.f, 0.f, 0.f);
        nZ[q4] = in ? __ldg((const float4*)(zrow + v)) : make_float4(0.f, 0.f, 0.f, 0.f);
        nG[q4] = in ? __ldg((const float4*)(grow + v)) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    };
    fetch(0);
    for (int t = 0; t < ntiles; ++t) {
      const int acc = t & 1;
      if (!mbar_wait(&t_full[acc], (uint32_t)((t >> 1) & 1), &abort_s, p.ctl, p.timeout_ns)) break;
      tc_fence_after();
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = 2 * t + hh;
        float4 cL[4], cZ[4], cG[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) { cL[q4] = nL[q4]; cZ[q4] = nZ[q4]; cG[q4] = nG[q4]; }
        fetch(h + 1);
        if (live) {
          const int c0 = 64 * tm + 32 * hh;
          float dv[32];
          rt_tmem_ld32(d_w + (uint32_t)(acc * 128) + ((uint32_t)(32 * qd) << 16) + (uint32_t)c0, dv);
          float d[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float send = part ? dv[e] : dv[16 + e];
            const float keep = part ? dv[16 + e] : dv[e];
            d[e] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
          }
          const int vb = vbase(h);  // the lane's first vocabulary row (a multiple of 4)
          if (rq) {
            float dv16[16];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const float lv[4] = {cL[q4].x, cL[q4].y, cL[q4].z, cL[q4].w};
              const float zv[4] = {cZ[q4].x, cZ[q4].y, cZ[q4].z, cZ[q4].w};
              const float gv[4] = {cG[q4].x, cG[q4].y, cG[q4].z, cG[q4].w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float t2 = zv[e] * c2 - lp2;
                const float r = exp2f(t2) - exp2f((lv[e] + d[4 * q4 + e]) * c2 - lq2);
                dv16[4 * q4 + e] = r > 0.0f ? log2f(r) * kLn2 + gv[e] : -INFINITY;
              }
            }
            if (vb + 16 <= v1) {
              float mx = dv16[0];
#pragma unroll
              for (int e = 1; e < 16; ++e) mx = fmax_nan_rt(mx, dv16[e]);
              if (mx != mx) {  // a NaN: rank this group entry by entry
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  if (dv16[e] != -INFINITY) {
                    const unsigned long long k2 = value_id_key(dv16[e], (uint32_t)(vb + e));
                    best = k2 > best ? k2 : best;
                  }
              } else if (mx > gbest) {  // +0 and -0 compare equal, as their keys do
                gbest = mx;
                gvb = vb;
#pragma unroll
                for (int e = 0; e < 16; ++e) gvals[e] = dv16[e];
              }
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e)
                if (vb + e < v1 && dv16[e] != -INFINITY) {
                  const unsigned long long k2 = value_id_key(dv16[e], (uint32_t)(vb + e));
                  best = k2 > best ? k2 : best;
                }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&t_empty[acc]);
    }
    if (gvb >= 0) {
#pragma unroll
      for (int e = 0; e < 16; ++e)
        if (gvals[e] != -INFINITY) {
          const unsigned long long k2 = value_id_key(gvals[e], (uint32_t)(gvb + e));
          best = k2 > best ? k2 : best;
        }
    }
    const unsigned long long o = __shfl_xor_sync(0xffffffffu, best, 1);
    best = o > best ? o : best;
    if (live && rq && part == 0) key_s[tm][q] = best;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) { tc_fence_after(); tmem_dealloc(d_w, 256); }
  for (int q = threadIdx.x; q < nreq; q += kRtThreads) {
    const unsigned long long k = key_s[0][q] > key_s[1][q] ? key_s[0][q] : key_s[1][q];
    if (k) atomicMax(p.keys + rq_s[q], k);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last_s = atomicAdd(p.done, 1u) == (unsigned)(G - 1);
  }
  __syncthreads();
  if (!last_s) return;

  // The last CTA: every other CTA's keys are in. Read and clear them; a
  // residual zero everywhere in fp32 draws from p_j.
  __threadfence();
  for (int q = threadIdx.x; q < nreq; q += kRtThreads) key_s[0][q] = atomicExch(p.keys + rq_s[q], 0ull);
  __syncthreads();
  for (int q = 0; q < nreq; ++q) {
    if (key_s[0][q] != 0ull) continue;  // uniform: shared value read after the barrier
    const int b = rq_s[q];
    const float* zrow = p.Z + ((size_t)b * (P + 1) + rj_s[q]) * V;
    const float* grow = p.G + (size_t)b * V;
    const float lp2 = lp_s[q];
    unsigned long long k = 0ull;
    for (int v = threadIdx.x; v < V; v += kRtThreads) {
      const unsigned long long a = value_id_key((__ldg(zrow + v) * c2 - lp2) * kLn2 + __ldg(grow + v), (uint32_t)v);
      k = a > k ? a : k;
    }
    k = warp_max_u64(k);
    if (lane == 0) red_s[warp] = k;
    __syncthreads();
    if (threadIdx.x == 0) {
      for (int w = 0; w < kRtThreads / 32; ++w) k = red_s[w] > k ? red_s[w] : k;
      key_s[0][q] = k;
    }
    __syncthreads();
  }
  for (int q = threadIdx.x; q < nreq; q += kRtThreads) {
    const unsigned long long k = key_s[0][q];
    int tok = 0;
    if (k == 0ull) dev_error(p.ctl, DEV_ERR_DATA);
    else tok = (int)key_id(k);
    p.next_token[rq_s[q]] = tok;
  }
  if (threadIdx.x == 0) *p.done = 0u;
}

size_t residual_tc_smem() { return 1024 + (size_t)kRtStages * kRtChunk + 4 * (size_t)kRtChunk; }

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
  const bool tc = (a.V % 4) == 0 && ((uintptr_t)a.L_base & 15u) == 0 && ((uintptr_t)a.Z & 15u) == 0 &&
                  ((uintptr_t)a.G & 15u) == 0 && ((uintptr_t)a.u & 15u) == 0;
  if (tc) {
    RtP q;
    memset(&q, 0, sizeof(q));
    if (!tmap_bf16_rows(&q.tm_w2, a.w2, a.V, 256, 128)) return cudaErrorInvalidValue;
    q.Lb = a.L_base; q.Z = a.Z; q.G = a.G; q.u = a.u;
    q.rej_j = a.rej_j; q.rej_norm = a.rej_norm;
    q.bs = a.bs; q.P = a.P; q.V = a.V;
    q.c2 = kLog2e / a.temperature;
    q.keys = a.rd_keys; q.next_token = a.next_token; q.ctl = a.ctl;
    q.timeout_ns = wait_timeout_ns();
    const size_t smem = residual_tc_smem();
    cudaError_t e = cudaFuncSetAttribute(residual_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    for (int b0 = 0; b0 < a.bs; b0 += kRdMaxReq) {
      q.b0 = b0;
      q.nb = a.bs - b0 < kRdMaxReq ? a.bs - b0 : kRdMaxReq;
      q.done = a.rd_done + (size_t)(b0 / kRdMaxReq) * 8;
      residual_tc_kernel<<<num_sms(), kRtThreads, smem, stream>>>(q);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
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
