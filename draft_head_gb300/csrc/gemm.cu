// Base-logits GEMM family on sm_103a.
//
//   out[n * ldo + m] = sum_k A[m, k] * B[n, k] (+ bias[m])
//
// A is a weight with many rows (the LM head W_lm [V, d], the H-columns of W1,
// or W_ih for the gate table); B is the short list of activations (the draft
// block's hidden states H, or embedding rows). The tensor-core kernel puts the
// weight on the MMA's M side (128 rows per tile) and the activations on its N
// side (16..256 per tile), so one GEMM shape serves both the weight-streaming
// batch-1 case (N = 15) and the batched case (N = 960).
//
// Pipeline per CTA (persistent over output tiles, 6 warps):
//   warp 0      TMA producer: A tile 128x64 and B tile BNx64 per stage,
//               128-byte swizzle, completion on the stage's full barrier;
//   warp 1      allocates TMEM, one thread issues tcgen05.mma (M=128, N=BN,
//               K=16) into one of two TMEM accumulators; tcgen05.commit frees
//               the smem stage and, after the last K chunk, hands the
//               accumulator to the epilogue;
//   warps 2-5   epilogue: tcgen05.ld of their 32-lane quarter, bias add, and
//               stores where each warp writes 32 consecutive m (128 B) per
//               column, i.e. coalesced rows of L_base.
#include <cuda.h>
#include <string.h>
#include <mutex>

#include "common.cuh"

namespace domino {

namespace {

constexpr int kBM = 128;          // MMA M (weight rows per tile)
constexpr int kBK = 64;           // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kThreads = 192;
constexpr uint32_t kABytes = kBM * kBK * 2;

struct TcProb {
  CUtensorMap tmA;
  float* out;
  const __nv_bfloat16* bias;
  int64_t ldo;
  int M;
  int m_tiles;
  int tile_begin;
  int evict_first;
};

struct TcParams {
  CUtensorMap tmB;
  TcProb prob[2];
  int nprob;
  int N, K, BN, n_tiles, k_chunks, stages, total_tiles;
  uint32_t tmem_cols;
  Ctl* ctl;
  uint64_t timeout_ns;
};

__device__ __forceinline__ void decode_tile(const TcParams& p, int t, int& pi, int& mt, int& nt) {
  pi = (p.nprob > 1 && t >= p.prob[1].tile_begin) ? 1 : 0;
  const int local = t - p.prob[pi].tile_begin;
  mt = local / p.n_tiles;
  nt = local - mt * p.n_tiles;
}

__global__ void __launch_bounds__(kThreads, 1) gemm_bf16_tc_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int stages = p.stages;
  const uint32_t b_bytes = (uint32_t)p.BN * kBK * 2;
  uint8_t* sA = smem;
  uint8_t* sB = smem + (size_t)stages * kABytes;
  uint64_t* full = (uint64_t*)(sB + (size_t)stages * b_bytes);
  uint64_t* empty = full + stages;
  uint64_t* tfull = empty + stages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = (uint32_t*)(drain + 1);
  volatile int* s_abort = (volatile int*)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *s_abort = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&p.tmB);
    for (int i = 0; i < p.nprob; ++i) tma_prefetch_desc(&p.prob[i].tmA);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, p.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_first = l2_policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      long issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x) {
        int pi, mt, nt;
        decode_tile(p, t, pi, mt, nt);
        const TcProb& pr = p.prob[pi];
        for (int kc = 0; kc < p.k_chunks; ++kc) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, s_abort, p.ctl, p.timeout_ns)) { ok = false; break; }
          mbar_expect_tx(&full[stage], kABytes + b_bytes);
          if (pr.evict_first)
            tma_load_2d_hint(sA + (size_t)stage * kABytes, &pr.tmA, kc * kBK, mt * kBM, &full[stage], pol_first);
          else
            tma_load_2d(sA + (size_t)stage * kABytes, &pr.tmA, kc * kBK, mt * kBM, &full[stage]);
          tma_load_2d(sB + (size_t)stage * b_bytes, &p.tmB, kc * kBK, nt * p.BN, &full[stage]);
          ++issued;
          if (++stage == stages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        // Give up, but first let the copies already in flight land.
        for (long j = issued - 1; j >= 0 && j >= issued - stages; --j)
          mbar_wait(&full[j % stages], (uint32_t)((j / stages) & 1), nullptr, p.ctl, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kBM, p.BN);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.total_tiles && ok; t += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (uint32_t)((local >> 1) & 1);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, s_abort, p.ctl, p.timeout_ns)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * p.BN);
        for (int kc = 0; kc < p.k_chunks; ++kc) {
          if (!mbar_wait(&full[stage], phase, s_abort, p.ctl, p.timeout_ns)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = sdesc_k_sw128(smem_u32(sA + (size_t)stage * kABytes));
          const uint64_t bd = sdesc_k_sw128(smem_u32(sB + (size_t)stage * b_bytes));
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            umma_bf16(d_tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc,
                      (kc > 0 || k > 0) ? 1u : 0u);
          umma_commit(&empty[stage]);
          if (++stage == stages) { stage = 0; phase ^= 1u; }
        }
        if (ok) umma_commit(&tfull[acc]);
      }
      // Wait until every MMA issued above has finished before TMEM is freed.
      umma_commit(drain);
      mbar_wait(drain, 0, nullptr, p.ctl, p.timeout_ns);
    }
  } else {
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    int local = 0;
    for (int t = blockIdx.x; t < p.total_tiles; t += gridDim.x, ++local) {
      int pi, mt, nt;
      decode_tile(p, t, pi, mt, nt);
      const TcProb& pr = p.prob[pi];
      const int acc = local & 1;
      const uint32_t acc_phase = (uint32_t)((local >> 1) & 1);
      if (!mbar_wait(&tfull[acc], acc_phase, s_abort, p.ctl, p.timeout_ns)) break;
      tc_fence_after();
      const int m = mt * kBM + row;
      const int n0 = nt * p.BN;
      const float bias = (pr.bias != nullptr && m < pr.M) ? __bfloat162float(pr.bias[m]) : 0.0f;
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * p.BN);
      for (int c0 = 0; c0 < p.BN; c0 += 16) {
        if (n0 + c0 >= p.N) break;  // warp-uniform
        float v[16];
        tmem_ld16(tb + (uint32_t)c0, v);
        if (m < pr.M) {
          float* o = pr.out + (int64_t)(n0 + c0) * pr.ldo + m;
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (n0 + c0 + j < p.N) o[(int64_t)j * pr.ldo] = v[j] + bias;
        }
      }
      tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(&tempty[acc]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

// ---------------------------------------------------------------------------
// Tensor maps (driver entry point fetched through the runtime, so the library
// links no driver library and loads on machines without a GPU).
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)ptr;
  });
  return fn;
}

// bf16 matrix [rows, K] with row stride `ld` elements, boxes of box_rows x 64.
bool make_tmap_bf16(CUtensorMap* tm, const void* base, int rows, int K, int64_t ld, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * 2)};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

cudaError_t gemm_bf16_tc(const GemmA* probs, int nprob, const void* B, int64_t ldb, int N, int K,
                         Ctl* ctl, cudaStream_t stream) {
  if (nprob < 1 || nprob > 2 || N <= 0 || K <= 0) return cudaErrorInvalidValue;
  TcParams p;
  memset(&p, 0, sizeof(p));
  // N tiling: BN <= 256, multiple of 16, tiles as even as possible.
  const int n_tiles = (N + 255) / 256;
  int bn = (N + n_tiles - 1) / n_tiles;
  bn = (bn + 15) / 16 * 16;
  p.N = N;
  p.K = K;
  p.BN = bn;
  p.n_tiles = (N + bn - 1) / bn;
  p.k_chunks = (K + kBK - 1) / kBK;
  p.nprob = nprob;
  if (!make_tmap_bf16(&p.tmB, B, N, K, ldb, bn)) return cudaErrorInvalidValue;
  int tiles = 0;
  for (int i = 0; i < nprob; ++i) {
    TcProb& pr = p.prob[i];
    if (!make_tmap_bf16(&pr.tmA, probs[i].A, probs[i].M, K, probs[i].lda, kBM)) return cudaErrorInvalidValue;
    pr.out = probs[i].out;
    pr.bias = (const __nv_bfloat16*)probs[i].bias;
    pr.ldo = probs[i].ldo;
    pr.M = probs[i].M;
    pr.m_tiles = (probs[i].M + kBM - 1) / kBM;
    pr.tile_begin = tiles;
    pr.evict_first = (p.n_tiles == 1) ? 1 : 0;  // weight read exactly once
    tiles += pr.m_tiles * p.n_tiles;
  }
  p.total_tiles = tiles;
  uint32_t cols = 32;
  while (cols < (uint32_t)(2 * bn)) cols <<= 1;
  p.tmem_cols = cols;
  p.ctl = ctl;
  p.timeout_ns = wait_timeout_ns();

  const uint32_t stage_bytes = kABytes + (uint32_t)bn * kBK * 2;
  const uint32_t budget = 220 * 1024;
  int stages = (int)((budget - 2048) / stage_bytes);
  if (stages > 12) stages = 12;
  if (stages < 2) return cudaErrorInvalidValue;
  p.stages = stages;
  const size_t smem = 1024 + (size_t)stages * stage_bytes + 8 * (2 * stages + 5) + 16;

  cudaError_t e = cudaFuncSetAttribute(gemm_bf16_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       227 * 1024);
  if (e != cudaSuccess) return e;
  int grid = num_sms();
  if (grid > tiles) grid = tiles;
  gemm_bf16_tc_kernel<<<grid, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// fp32 operands: classic 64x64 shared-memory tiled SIMT GEMM.
// ---------------------------------------------------------------------------
namespace {
__global__ void __launch_bounds__(256) gemm_f32_kernel(const float* __restrict__ A, int64_t lda, int M,
                                                       const float* __restrict__ B, int64_t ldb, int N,
                                                       int K, float* __restrict__ out, int64_t ldo,
                                                       const float* __restrict__ bias) {
  __shared__ float As[16][65];
  __shared__ float Bs[16][65];
  const int m0 = blockIdx.x * 64, n0 = blockIdx.y * 64;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += 16) {
    for (int i = threadIdx.x; i < 1024; i += 256) {
      const int r = i >> 4, kk = i & 15;
      As[kk][r] = (m0 + r < M && k0 + kk < K) ? A[(int64_t)(m0 + r) * lda + k0 + kk] : 0.0f;
      Bs[kk][r] = (n0 + r < N && k0 + kk < K) ? B[(int64_t)(n0 + r) * ldb + k0 + kk] : 0.0f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
    const float bi = bias ? bias[m] : 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < N) out[(int64_t)n * ldo + m] = acc[i][j] + bi;
    }
  }
}
}  // namespace

cudaError_t gemm_f32_simt(const GemmA* probs, int nprob, const void* B, int64_t ldb, int N, int K,
                          cudaStream_t stream) {
  for (int i = 0; i < nprob; ++i) {
    dim3 grid((probs[i].M + 63) / 64, (N + 63) / 64);
    gemm_f32_kernel<<<grid, 256, 0, stream>>>((const float*)probs[i].A, probs[i].lda, probs[i].M,
                                              (const float*)B, ldb, N, K, probs[i].out, probs[i].ldo,
                                              (const float*)probs[i].bias);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace domino
