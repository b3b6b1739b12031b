// Small-batch Domino head chain (bf16 weights, rank 256, batch <= 4): the
// low-concurrency serving case, one persistent CTA per SM.
//
// Same arithmetic as the general chain kernel (chain.cu); what differs is where
// W2 lives across the P dependent steps:
//  - Each CTA owns ~1000 vocabulary rows of W2 (512 bytes each). The first 512
//    stay in tensor memory (TMEM, 256 KB per SM), one whole row per TMEM lane
//    and 128-column block. The next rows stay in shared memory (bank-swizzled
//    so that 32 lanes read 32 rows without conflicts), all loaded once per
//    chain with coalesced row reads (the TMEM rows pass through the
//    shared-memory buffer on their way). The remainder goes to registers: at batch 1 up to 10 rows per warp
//    stay there for the whole chain; larger batches reload 6 rows per warp
//    every step, in flight across the step's first wait. Rows beyond those are
//    read from L2 each step.
//  - Resident rows: one row per lane, so a dot product needs no cross-lane
//    reduction; u is read from shared memory as broadcasts. Register rows: the
//    32 lanes of a warp split a row's 256 columns (coalesced loads) and eight
//    rows are reduced together with a transposing butterfly.
//  - The dot products run on the CUDA cores with packed fp32x2 FMAs. (On this
//    GPU one tcgen05.mma of M = 128, K = 16 costs ~116 cycles whatever N is, so
//    at N <= 16 the tensor core covers a 128 x 256 tile slower than 16 warps of
//    FMAs; the batched kernel uses it where N is large.)
//  - The hidden-side GRU sums W_hh S_i of the CTA's units run while the
//    step's argmax keys are exchanged, so the next step starts with gate
//    math only. S_i travels in 64-bit words that carry the step number next
//    to the value: a reader polls the tag and needs no fence.
//  - The gate-table values of the CTA's hidden units and the L_base (and
//    noise) segment are prefetched into shared memory off the critical path
//    (the segment by bulk copy).
//  - No grid barrier: each step's two all-to-all exchanges carry their own
//    completion. Every CTA adds (W1_s S partial in 2^-32 fixed point) << 16
//    plus one into each 64-bit bottleneck accumulator, so its low 16 bits
//    count the contributions; the accumulators are never cleared, and a
//    reader polls until the count reaches n_contrib (i + 1) and takes the
//    exact difference from the previous step's value. For the argmax, every
//    CTA folds its best (value, id) key into the step's key with an atomic
//    max and then, with release semantics, increments a counter in the same
//    16 bytes; one thread per CTA polls both with one 16-byte load until all
//    CTAs have arrived, starts the next gate gather from that key, and
//    confirms it with an acquire of the count and a fresh read of the key
//    while the gather runs. All waits are bounded; on
//    timeout the kernel records the error, raises the abort flag and leaves.
// Per step: GRU gates -> counted fixed-point W1_s S partials -> wait for the
// counts, u = SiLU(.) -> W2 GEMV + L_base (+ noise) -> publish best key ->
// wait for all keys (meanwhile W_hh S_i): token and next gate values.
#include "common.cuh"

namespace domino {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kR = 256;               // rank (row = 256 bf16 = 512 bytes)
constexpr int kTmemRows = 512;        // 16 warps x 32 rows
constexpr int kUaccPad = 16;
constexpr float kInvFix = 1.0f / 4294967296.0f;  // exact power of two

struct SmallP {
  int bs, P, d, g, V, nu_max, rows_max, smem_rows;
  int seg;   // floats per request in the staged L_base / noise segments
  int bulk;  // 1: segments and P_h rows arrive by bulk copy (16-byte aligned rows)
  const float* gate_table;
  const __nv_bfloat16* w_hh;
  const __nv_bfloat16* b_hh;
  const __nv_bfloat16* w1;
  const __nv_bfloat16* w2;
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
  unsigned long long* keys;  // per (step, request): {max key, arrival count} in 16 bytes
  unsigned long long* S;     // [2][bs][g] words: value bits | (step + 1) << 32
  long long* uacc;
  int n_contrib;             // CTAs that own hidden units (add to every accumulator)
  float part_limit;          // largest |partial| that keeps every accumulator in range
  uint64_t timeout_ns;
};

__device__ __forceinline__ long long ld_relaxed_s64(const long long* p) {
  long long v;
  asm volatile("ld.relaxed.gpu.global.s64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void ld_relaxed_v2_u64(const unsigned long long* p, unsigned long long& a,
                                                  unsigned long long& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void cp_async4(void* smem_dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 columns of this thread's lane (one 128-byte quarter of a W2 row).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// Issue a 16-column TMEM load; the registers are valid only after
// tmem_wait16() on the same array (which also orders their uses after it).
__device__ __forceinline__ void tmem_issue16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// u packed as fp32 pairs: p[i] = {u[2i], u[2i+1]}.
struct U8 {
  unsigned long long p[4];
};

__device__ __forceinline__ unsigned long long pack2(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}

// Dot of 8 bf16 (one 16-byte slice of a W2 row) with 8 fp32 of u, using
// packed fp32x2 FMAs: each 32-bit word holds elements 2i (low half) and
// 2i + 1 (high half); both become exact fp32 with one shift / one mask.
__device__ __forceinline__ float dot8(const uint4& v, const U8& u) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  unsigned long long acc = 0ull;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const unsigned long long x = pack2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(x), "l"(u.p[i]));
  }
  float a, b;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(acc));
  return a + b;
}

// One lane, one W2 row: accumulate 32 elements (16 words, element 2i in the
// low half of word i) times u[0..31] of every request into two packed
// fp32x2 accumulators per request. u_s rows are fp32 pairs read as 16-byte
// broadcasts.
template <int BS>
__device__ __forceinline__ void dot32_lane(const uint32_t (&w)[16], const float* u_s, int ustride,
                                           unsigned long long (&acc)[BS][2]) {
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    unsigned long long x[4];
#pragma unroll
    for (int t = 0; t < 4; ++t)
      x[t] = pack2(__uint_as_float(w[4 * e + t] << 16), __uint_as_float(w[4 * e + t] & 0xFFFF0000u));
#pragma unroll
    for (int b = 0; b < BS; ++b) {
      const ulonglong2 ua = *(const ulonglong2*)(u_s + b * ustride + e * 8);
      const ulonglong2 ub = *(const ulonglong2*)(u_s + b * ustride + e * 8 + 4);
      unsigned long long& a = acc[b][e & 1];
      asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(x[0]), "l"(ua.x));
      asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(x[1]), "l"(ua.y));
      asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(x[2]), "l"(ub.x));
      asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(a) : "l"(x[3]), "l"(ub.y));
    }
  }
}

__device__ __forceinline__ float fold2(unsigned long long a0, unsigned long long a1) {
  float p, q, r, t;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(p), "=f"(q) : "l"(a0));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r), "=f"(t) : "l"(a1));
  return (p + q) + (r + t);
}

// Shared-memory copy of the resident W2 rows: four 128-byte column quarters
// [kc][row], the 16-byte chunks of a row permuted by (chunk ^ (row & 7)) so
// that 32 lanes reading 32 consecutive rows hit every bank once per 8 lanes.
__device__ __forceinline__ int w2s_index(int kc, int rr, int c, int rows_s) {
  return (kc * rows_s + rr) * 8 + (c ^ (rr & 7));
}

__device__ __forceinline__ float dot8_f(const uint4& v, const float (&u)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    s = fmaf(__uint_as_float(w[i] << 16), u[2 * i], s);
    s = fmaf(__uint_as_float(w[i] & 0xFFFF0000u), u[2 * i + 1], s);
  }
  return s;
}

// Reduce 8 per-lane partial dots (one per row) across the warp with a
// transposing butterfly; afterwards lanes with (lane & 3) == 0 hold the full
// dot of row ((lane>>4)&1)*4 + ((lane>>3)&1)*2 + ((lane>>2)&1).
__device__ __forceinline__ float reduce8(float (&pr)[8], int lane) {
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
  return pr[0];
}

__device__ __forceinline__ int row_of_lane(int lane) {
  return ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
}

template <int BS>
__global__ void __launch_bounds__(kThreads, 1) chain_small_kernel(const __grid_constant__ SmallP p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int G = gridDim.x, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = p.g, V = p.V, P = p.P, nu_max = p.nu_max;
  const int j0 = (int)((int64_t)g * c / G), j1 = (int)((int64_t)g * (c + 1) / G), nu = j1 - j0;
  const int v0 = (int)((int64_t)V * c / G), v1 = (int)((int64_t)V * (c + 1) / G);
  const int nrows = v1 - v0;
  const int rows_t = min(kTmemRows, nrows);
  const int rows_s = min(p.smem_rows, nrows - rows_t);
  const int rows_g = nrows - rows_t - rows_s;
  const int gbase = rows_t + rows_s;
  // Remainder rows past TMEM and shared memory: round robin over all warps.
  constexpr int kSW = kWarps;
  // Batch 1 keeps up to GR remainder rows per warp in registers for the whole
  // chain; larger batches need those registers and reload them every step.
  constexpr bool kRegResident = (BS == 1);
  constexpr int GR = kRegResident ? 10 : 6;

  // ---- shared memory carve-up
  size_t off = 0;
  auto take = [&](size_t bytes) { uint8_t* q = smem + off; off = (off + bytes + 15) & ~(size_t)15; return q; };
  __nv_bfloat16* whh_s = (__nv_bfloat16*)take((size_t)3 * nu_max * g * 2);  // [3*nu][g]
  float* w1s_s = (float*)take((size_t)kR * nu_max * 4);                     // [256][nu]
  float* bhh_s = (float*)take((size_t)3 * nu_max * 4);
  float* sprev_s = (float*)take((size_t)BS * g * 4);                        // S_i (all units)
  float* gi_s = (float*)take((size_t)BS * 3 * nu_max * 4);                  // gate-table values
  float* gh_s = (float*)take((size_t)BS * 3 * nu_max * 4);                  // W_hh S_{i-1}, owned rows
  float* lb_s = (float*)take((size_t)BS * p.seg * 4);                       // L_base segment
  float* gm_s = (float*)take((size_t)(p.temperature > 0.f ? BS : 0) * p.seg * 4);
  float* u_s = (float*)take((size_t)BS * kR * 4);
  float* ph_s = (float*)take((size_t)BS * kR * 4);                        // P_h[i]
  float* snew_s = (float*)take((size_t)BS * nu_max * 4);
  long long* uprev_s = (long long*)take((size_t)BS * kR * 8);               // accumulators at step i-1
  int* tok_s = (int*)take(BS * 4);
  int* fail_s = (int*)take(16);
  int* redo_s = (int*)take(16);
  unsigned long long* spec_s = (unsigned long long*)take((size_t)BS * 8);
  unsigned long long* red_s = (unsigned long long*)take((size_t)kWarps * BS * 8);
  uint32_t* tmem_slot = (uint32_t*)take(16);
  uint64_t* seg_bar = (uint64_t*)take(16);
  uint4* w2s = (uint4*)take((size_t)p.smem_rows * 512);                    // resident rows

  // ---- one-time residency: W_hh rows of the owned units, W1_s columns, W2 rows.
  for (int idx = threadIdx.x; idx < 3 * nu * (g / 8); idx += kThreads) {
    const int row = idx / (g / 8), k8 = idx - row * (g / 8);
    const int q = row / nu, jj = row - q * nu;
    ((uint4*)(whh_s + (size_t)(q * nu + jj) * g))[k8] =
        ld_nc_v4(p.w_hh + (size_t)(q * g + j0 + jj) * g + k8 * 8);
  }
  // W2 rows [row0, row0 + nr) of the CTA's slice into the swizzled row
  // buffer with quarter stride R: one warp instruction reads one whole row.
  // (Unrolling this loop to keep more loads in flight measured slower: all
  // SMs load at once and HBM is the limit.)
  auto stage_rows = [&](int row0, int nr, int R) {
    for (int idx = threadIdx.x; idx < nr * 32; idx += kThreads) {
      const int rr = idx >> 5, l = idx & 31;
      w2s[w2s_index(l >> 3, rr, l & 7, R)] = ld_nc_v4(p.w2 + (size_t)(v0 + row0 + rr) * kR + l * 8);
    }
  };
  {
    // W1_s columns: strided 2-byte reads, so keep four in flight per thread.
    constexpr int kU = 4;
    for (int base = threadIdx.x; base < kR * nu; base += kU * kThreads) {
      __nv_bfloat16 v[kU];
#pragma unroll
      for (int t = 0; t < kU; ++t) {
        const int idx = base + t * kThreads;
        const int k = idx / nu, jj = idx - k * nu;
        v[t] = idx < kR * nu ? p.w1[(size_t)k * (p.d + g) + p.d + j0 + jj] : __float2bfloat16(0.0f);
      }
#pragma unroll
      for (int t = 0; t < kU; ++t) {
        const int idx = base + t * kThreads;
        if (idx < kR * nu) w1s_s[idx] = __bfloat162float(v[t]);
      }
    }
  }
  for (int idx = threadIdx.x; idx < 3 * nu; idx += kThreads) {
    const int q = idx / nu, jj = idx - q * nu;
    bhh_s[idx] = __bfloat162float(p.b_hh[q * g + j0 + jj]);
  }
  // S_{-1} = 0: no hidden-side sums and no previous own state at step 0.
  for (int idx = threadIdx.x; idx < BS * 3 * nu_max; idx += kThreads) gh_s[idx] = 0.0f;
  for (int idx = threadIdx.x; idx < BS * nu_max; idx += kThreads) snew_s[idx] = 0.0f;
  for (int idx = threadIdx.x; idx < BS * kR; idx += kThreads) uprev_s[idx] = 0;
  if (threadIdx.x == 0) {
    *fail_s = 0;
    *redo_s = 0;
    mbar_init(seg_bar, 1);
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // TMEM lane L, columns [128 cb, 128 cb + 128) hold row 128 cb + L of the
  // CTA's first 512 rows: warp w (lane quarter w % 4, column block w / 4)
  // owns rows 128 (w / 4) + 32 (w % 4) + lane, one whole row per lane, i.e.
  // the 32-row group w.
  const uint32_t tw = tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)((warp >> 2) * 128);
  const int t_row0 = (warp >> 2) * 128 + (warp & 3) * 32;
  // TMEM rows pass through the shared-memory row buffer: whole 32-row groups
  // per pass, read from HBM with coalesced 512-byte row loads into the
  // swizzled layout, then each lane takes its own row (conflict-free) to
  // TMEM. Reading one row per lane straight from HBM is about four times
  // slower.
  {
    const int ngroups = (rows_t + 31) / 32;
    const int gpp = p.smem_rows / 32;  // groups per pass (at least 1: checked at launch)
    for (int g0 = 0; g0 < ngroups; g0 += gpp) {
      const int g1 = min(ngroups, g0 + gpp);
      const int r0 = g0 * 32, nr = min(rows_t, g1 * 32) - r0, R = (g1 - g0) * 32;
      stage_rows(r0, nr, R);
      __syncthreads();
      if (t_row0 < rows_t && warp >= g0 && warp < g1) {  // warp-uniform
        const int lr = min(t_row0 + lane, rows_t - 1) - r0;
#pragma unroll 1
        for (int kc = 0; kc < 4; ++kc) {
          uint32_t r[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint4 v = w2s[w2s_index(kc, lr, q, R)];
            r[4 * q] = v.x; r[4 * q + 1] = v.y; r[4 * q + 2] = v.z; r[4 * q + 3] = v.w;
          }
          tmem_st32(tw + (uint32_t)(kc * 32), r);
        }
      }
      __syncthreads();
    }
  }
  tmem_wait_st();
  // The shared-memory rows, loaded once.
  stage_rows(rows_t, rows_s, rows_s);

  // Initial GRU input: the anchors' gate values.
  for (int b = threadIdx.x; b < BS; b += kThreads) {
    int a = p.anchor[b];
    if (a < 0 || a >= V) { dev_error(p.ctl, DEV_ERR_DATA); a = 0; }
    tok_s[b] = a;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < BS * 3 * nu; idx += kThreads) {
    const int b = idx / (3 * nu), rem = idx - b * 3 * nu, q = rem / nu, jj = rem - q * nu;
    gi_s[b * 3 * nu_max + rem] = __ldg(p.gate_table + (size_t)tok_s[b] * 3 * g + q * g + j0 + jj);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int bsr = BS * kR;
  const int lo = p.bulk ? (v0 & 3) : 0;  // segment index of row v0
  int seg_issued = -1;                   // last step whose bulk copies were issued (thread 32)
  bool ok = true;
  const int sw = warp;
  const int ng = rows_g > sw ? (rows_g - sw + kSW - 1) / kSW : 0;
  // The first GR of a warp's remaining rows go to its registers (lane l holds
  // columns [8 l, 8 l + 8)); rows beyond those are read from L2 each step.
  uint4 gw[GR];
  auto load_gw = [&]() {
#pragma unroll
    for (int t = 0; t < GR; ++t)
      gw[t] = (t < ng) ? ld_nc_v4(p.w2 + (size_t)(v0 + gbase + sw + t * kSW) * kR + lane * 8)
                       : make_uint4(0u, 0u, 0u, 0u);
  };
  if (kRegResident) load_gw();

  for (int i = 0; i < P && ok; ++i) {
    // ---------------- A: GRU gates, bottleneck partial adds; then the L_base /
    // noise segment and P_h row go in flight (bulk copies are issued after the
    // adds, off the exchange's critical path).
    if (!p.bulk) {
      for (int idx = (int)threadIdx.x - 32; idx >= 0 && idx < BS * nrows; idx += kThreads - 32) {
        const int b = idx / nrows, rr = idx - b * nrows;
        cp_async4(lb_s + b * p.seg + rr, p.L_base + ((size_t)b * P + i) * V + v0 + rr);
        if (p.temperature > 0.f)
          cp_async4(gm_s + b * p.seg + rr, p.gumbel + (int64_t)b * p.gumbel_bstride + (int64_t)i * V + v0 + rr);
      }
      for (int idx = (int)threadIdx.x - 32; idx >= 0 && idx < bsr; idx += kThreads - 32)
        cp_async4(ph_s + idx, p.P_h + ((size_t)(idx / kR) * P + i) * kR + (idx % kR));
      cp_async_commit();
    }
    {
      // Gates of the owned units; W_hh S_{i-1} was summed during the previous
      // step's key exchange. S_i goes out tagged with step + 1 in each word.
      unsigned long long* Sw = p.S + (size_t)(i & 1) * BS * g;
      const unsigned long long tag = (unsigned long long)(unsigned)(i + 1) << 32;
      for (int idx = threadIdx.x; idx < BS * nu; idx += kThreads) {
        const int b = idx / nu, jj = idx - b * nu;
        const float* gi = gi_s + b * 3 * nu_max;
        const float* gh = gh_s + b * 3 * nu_max;
        const float rg = sigmoidf_(gi[jj] + gh[jj] + bhh_s[jj]);
        const float zg = sigmoidf_(gi[nu + jj] + gh[nu + jj] + bhh_s[nu + jj]);
        const float ng_ = tanhf(gi[2 * nu + jj] + rg * (gh[2 * nu + jj] + bhh_s[2 * nu + jj]));
        const float hn = (1.0f - zg) * ng_ + zg * snew_s[b * nu_max + jj];
        st_relaxed_u64(Sw + (size_t)b * g + j0 + jj, tag | __float_as_uint(hn));
        snew_s[b * nu_max + jj] = hn;
      }
    }
    __syncthreads();
    if (nu > 0) {
      for (int idx = (int)threadIdx.x - 32; idx >= 0 && idx < bsr; idx += kThreads - 32) {
        const int b = idx / kR, k = idx - b * kR;
        float part = 0.0f;
        for (int jj = 0; jj < nu; ++jj) part = fmaf(w1s_s[k * nu + jj], snew_s[b * nu_max + jj], part);
        atomicAdd((unsigned long long*)(p.uacc + (size_t)idx * kUaccPad),
                  ((unsigned long long)fix32_checked(part, p.part_limit, p.ctl) << 16) + 1ull);
      }
    }
    if (p.bulk) {
      // Whole 16-byte units covering [v0, v1) per request, one bulk copy each.
      if (threadIdx.x == 32) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const int a0 = v0 & ~3, a1 = (v1 + 3) & ~3;
        const uint32_t sb = (uint32_t)(a1 - a0) * 4u;
        mbar_expect_tx(seg_bar, (uint32_t)BS * (sb * (p.temperature > 0.f ? 2u : 1u) + (uint32_t)kR * 4u));
#pragma unroll
        for (int b = 0; b < BS; ++b) {
          bulk_copy_g2s(lb_s + b * p.seg, p.L_base + ((size_t)b * P + i) * V + a0, sb, seg_bar);
          if (p.temperature > 0.f)
            bulk_copy_g2s(gm_s + b * p.seg, p.gumbel + (int64_t)b * p.gumbel_bstride + (int64_t)i * V + a0, sb,
                          seg_bar);
          bulk_copy_g2s(ph_s + b * kR, p.P_h + ((size_t)b * P + i) * kR, (uint32_t)kR * 4u, seg_bar);
        }
        seg_issued = i;
      }
    }
    // Per-step register rows: in flight across the wait below.
    if (!kRegResident) load_gw();
    // ---------------- B: wait until every accumulator holds all contributions; u_i.
    if (p.bulk) {
      if (!mbar_wait(seg_bar, (uint32_t)(i & 1), nullptr, p.ctl, p.timeout_ns)) *fail_s = 1;
    } else {
      cp_async_wait_all();
    }
    __syncthreads();
    {
      // The accumulators are never cleared: after step i each holds the sum
      // of steps 0..i and a count of n_contrib (i + 1); this step's sum is
      // the exact difference from the value read at the previous step. No
      // CTA adds step i + 1 before every CTA has published its step-i key,
      // which it does after this wait.
      const int want = (p.n_contrib * (i + 1)) & 0xFFFF;
      for (int idx = threadIdx.x; idx < bsr; idx += kThreads) {
        const long long* src = p.uacc + (size_t)idx * kUaccPad;
        long long v = ld_relaxed_s64(src);
        if ((int)(v & 0xFFFF) != want) {
          const uint64_t t0 = globaltimer_ns();
          unsigned spins = 0;
          while ((int)((v = ld_relaxed_s64(src)) & 0xFFFF) != want) {
            if ((++spins & 63u) == 0) {
              if (ld_volatile_u32(&p.ctl->abort)) { *fail_s = 1; break; }
              if (globaltimer_ns() - t0 > p.timeout_ns) { dev_abort(p.ctl, DEV_ERR_TIMEOUT); *fail_s = 1; break; }
            }
          }
        }
        const long long d = (long long)((unsigned long long)v - (unsigned long long)uprev_s[idx]);
        uprev_s[idx] = v;
        u_s[idx] = siluf_(ph_s[idx] + __ll2float_rn(d >> 16) * kInvFix);  // one rounding, exact scaling
      }
    }
    __syncthreads();
    if (*fail_s) { ok = false; break; }

    // ---------------- C: L = L_base + W2 u (+ noise), best key per request.
    {
      U8 up[BS];
#pragma unroll
      for (int b = 0; b < BS; ++b)
#pragma unroll
        for (int t = 0; t < 4; ++t)
          up[b].p[t] = pack2(u_s[b * kR + lane * 8 + 2 * t], u_s[b * kR + lane * 8 + 2 * t + 1]);
      unsigned long long best[BS];
#pragma unroll
      for (int b = 0; b < BS; ++b) best[b] = 0ull;
      const int rq = row_of_lane(lane);
      auto consider = [&](int b, int lr, float s) {
        const int v = v0 + lr;
        const float logit = lb_s[b * p.seg + lo + lr] + s;
        if (p.logits_out) p.logits_out[((size_t)b * P + i) * V + v] = logit;
        const float dec = p.temperature > 0.f ? logit * p.inv_temperature + gm_s[b * p.seg + lo + lr] : logit;
        const unsigned long long key = value_id_key(dec, (uint32_t)v);
        best[b] = key > best[b] ? key : best[b];
      };
      // Register rows first: warp w holds rows w, w + 16, ...
      // of the remainder in gw[]; any beyond are loaded 8 at a time.
#pragma unroll
      for (int t0 = 0; t0 < GR; t0 += 8) {
        if (t0 < ng) {
#pragma unroll
          for (int b = 0; b < BS; ++b) {
            float pr[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) pr[q] = (t0 + q < GR) ? dot8(gw[(t0 + q < GR) ? t0 + q : 0], up[b]) : 0.f;
            const float s = reduce8(pr, lane);
            const int t = t0 + rq;
            if ((lane & 3) == 0 && t < ng && t < GR) consider(b, gbase + sw + t * kSW, s);
          }
        }
      }
#pragma unroll 1
      for (int t0 = GR; t0 < ng; t0 += 8) {
        uint4 wv[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int t = min(t0 + q, ng - 1);
          wv[q] = ld_nc_v4(p.w2 + (size_t)(v0 + gbase + sw + t * kSW) * kR + lane * 8);
        }
#pragma unroll
        for (int b = 0; b < BS; ++b) {
          float pr[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) pr[q] = dot8(wv[q], up[b]);
          const float s = reduce8(pr, lane);
          const int t = t0 + rq;
          if ((lane & 3) == 0 && t < ng) consider(b, gbase + sw + t * kSW, s);
        }
      }
      // Resident rows, one row per lane: the lane's dot needs no cross-lane
      // reduction. TMEM rows first (each warp one group of 32), then the
      // shared-memory rows in groups of 32, round robin over warps.
      auto consider_lane = [&](int lr, const unsigned long long (&acc)[BS][2]) {
#pragma unroll
        for (int b = 0; b < BS; ++b) consider(b, lr, fold2(acc[b][0], acc[b][1]));
      };
      if (t_row0 < rows_t) {  // warp-uniform
        unsigned long long acc[BS][2];
#pragma unroll
        for (int b = 0; b < BS; ++b) acc[b][0] = acc[b][1] = 0ull;
#pragma unroll 1
        for (int kh = 0; kh < 8; ++kh) {
          uint32_t wv[16];
          tmem_issue16(tw + (uint32_t)(kh * 16), wv);
          tmem_wait16(wv);
          dot32_lane<BS>(wv, u_s + kh * 32, kR, acc);
        }
        if (t_row0 + lane < rows_t) consider_lane(t_row0 + lane, acc);
      }
#pragma unroll 1
      for (int sg = warp; sg * 32 < rows_s; sg += kWarps) {
        const int rr = sg * 32 + lane;
        const int rc = min(rr, rows_s - 1);
        unsigned long long acc[BS][2];
#pragma unroll
        for (int b = 0; b < BS; ++b) acc[b][0] = acc[b][1] = 0ull;
#pragma unroll 1
        for (int kh = 0; kh < 8; ++kh) {
          uint32_t wv[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 v = w2s[w2s_index(kh >> 1, rc, (kh & 1) * 4 + q, rows_s)];
            wv[4 * q] = v.x; wv[4 * q + 1] = v.y; wv[4 * q + 2] = v.z; wv[4 * q + 3] = v.w;
          }
          dot32_lane<BS>(wv, u_s + kh * 32, kR, acc);
        }
        if (rr < rows_s) consider_lane(rows_t + rr, acc);
      }
#pragma unroll
      for (int b = 0; b < BS; ++b) {
        const unsigned long long m = warp_max_u64(best[b]);
        if (lane == 0) red_s[warp * BS + b] = m;
      }
    }
    __syncthreads();
    if (threadIdx.x < BS) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kWarps; ++w) {
        const unsigned long long x = red_s[w * BS + threadIdx.x];
        m = x > m ? x : m;
      }
      unsigned long long* e = p.keys + ((size_t)i * BS + threadIdx.x) * 2;
      if (m) atomicMax(e, m);
      asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"((unsigned*)(e + 1)) : "memory");
    }

    // ---------------- D: wait for every CTA's key (threads < BS) while warps
    // 1.. sum W_hh S_i; token of position i; gate values.
    if (threadIdx.x < BS) {
      const int b = threadIdx.x;
      const unsigned long long* e = p.keys + ((size_t)i * BS + b) * 2;
      unsigned long long m, cnt;
      asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(m), "=l"(cnt) : "l"(e) : "memory");
      if ((int)(unsigned)cnt != G) {
        const uint64_t t0 = globaltimer_ns();
        unsigned spins = 0;
        // While waiting, pull the gate values of the running argmax into L2:
        // the final token is usually known before the last CTA arrives.
        uint32_t spec = 0xFFFFFFFFu;
        const bool gather = i + 1 < P && nu > 0 && !p.force;
        do {
          asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(m), "=l"(cnt) : "l"(e) : "memory");
          if (gather && m != 0ull && key_id(m) != spec) {
            spec = key_id(m);
            if (spec < (uint32_t)V) {
#pragma unroll
              for (int q = 0; q < 3; ++q) {
                const float* a = p.gate_table + (size_t)spec * 3 * g + q * g + j0;
                prefetch_l2(a);
                if ((((uintptr_t)a ^ (uintptr_t)(a + nu - 1)) >> 7) != 0) prefetch_l2(a + nu - 1);
              }
            }
          }
          if ((++spins & 63u) == 0) {
            if (ld_volatile_u32(&p.ctl->abort)) { *fail_s = 1; break; }
            if (globaltimer_ns() - t0 > p.timeout_ns) { dev_abort(p.ctl, DEV_ERR_TIMEOUT); *fail_s = 1; break; }
          }
        } while ((int)(unsigned)cnt != G);
      }
      // The key came from the same vector load that saw the full count, but
      // the memory model orders no element of a vector access after another:
      // it is only a guess. The next step's gate gather starts from it, and
      // the key is confirmed after an acquire of the count below.
      spec_s[b] = m;
      const int tok = m ? (int)key_id(m) : 0;
      int nxt = (p.force && i + 1 < P) ? p.force[(size_t)b * P + i] : tok;
      if (nxt < 0 || nxt >= V) nxt = 0;
      tok_s[b] = nxt;
    } else if (warp > 0 && nu > 0 && i + 1 < P) {
      // While the keys travel: S_i from every CTA (each word carries its step
      // tag, so no fence orders it), then W_hh S_i for the owned units.
      const unsigned long long* Sr = p.S + (size_t)(i & 1) * BS * g;
      const unsigned tag = (unsigned)(i + 1);
      for (int idx = (int)threadIdx.x - 32; idx < BS * g / 2; idx += kThreads - 32) {
        unsigned long long x, y;
        ld_relaxed_v2_u64(Sr + 2 * idx, x, y);
        if ((unsigned)(x >> 32) != tag || (unsigned)(y >> 32) != tag) {
          const uint64_t t0 = globaltimer_ns();
          unsigned spins = 0;
          do {
            ld_relaxed_v2_u64(Sr + 2 * idx, x, y);
            if ((++spins & 63u) == 0) {
              if (ld_volatile_u32(&p.ctl->abort)) { *fail_s = 1; break; }
              if (globaltimer_ns() - t0 > p.timeout_ns) { dev_abort(p.ctl, DEV_ERR_TIMEOUT); *fail_s = 1; break; }
            }
          } while ((unsigned)(x >> 32) != tag || (unsigned)(y >> 32) != tag);
        }
        ((float2*)sprev_s)[idx] = make_float2(__uint_as_float((unsigned)x), __uint_as_float((unsigned)y));
      }
      asm volatile("bar.sync 1, %0;" ::"n"(kThreads - 32) : "memory");
      for (int item = warp - 1; item < BS * nu; item += kWarps - 1) {
        const int b = item / nu, jj = item - b * nu;
        const float* sp = sprev_s + (size_t)b * g;
        const __nv_bfloat16* w0 = whh_s + (size_t)(0 * nu + jj) * g;
        const __nv_bfloat16* w1r = whh_s + (size_t)(1 * nu + jj) * g;
        const __nv_bfloat16* w2r = whh_s + (size_t)(2 * nu + jj) * g;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f;
        for (int k8 = lane; k8 < g / 8; k8 += 32) {
          float sv[8];
          const float4 s0 = ((const float4*)sp)[2 * k8], s1 = ((const float4*)sp)[2 * k8 + 1];
          sv[0] = s0.x; sv[1] = s0.y; sv[2] = s0.z; sv[3] = s0.w;
          sv[4] = s1.x; sv[5] = s1.y; sv[6] = s1.z; sv[7] = s1.w;
          a0 += dot8_f(((const uint4*)w0)[k8], sv);
          a1 += dot8_f(((const uint4*)w1r)[k8], sv);
          a2 += dot8_f(((const uint4*)w2r)[k8], sv);
        }
        a0 = warp_sum(a0);
        a1 = warp_sum(a1);
        a2 = warp_sum(a2);
        if (lane == 0) {
          float* gh = gh_s + b * 3 * nu_max;
          gh[jj] = a0;
          gh[nu + jj] = a1;
          gh[2 * nu + jj] = a2;
        }
      }
    }
    __syncthreads();
    if (*fail_s) { ok = false; break; }
    // Gate values of the next GRU input (warps 1..) while warp 0 confirms the
    // step's keys: an acquire load of the count that was seen complete orders
    // every CTA's atomic maximum (released before its increment) before the
    // key is read again. A key that differs from the guess (never seen so
    // far) replaces the token, and the gather is redone below.
    auto gather_gates = [&](int first) {
      for (int idx = (int)threadIdx.x - first; idx >= 0 && idx < BS * 3 * nu; idx += kThreads - first) {
        const int b = idx / (3 * nu), rem = idx - b * 3 * nu, q = rem / nu, jj = rem - q * nu;
        gi_s[b * 3 * nu_max + rem] = __ldg(p.gate_table + (size_t)tok_s[b] * 3 * g + q * g + j0 + jj);
      }
    };
    if (threadIdx.x < BS) {
      const int b = threadIdx.x;
      const unsigned long long* e = p.keys + ((size_t)i * BS + b) * 2;
      (void)ld_acquire_u32((const unsigned*)(e + 1));
      const unsigned long long m = ld_relaxed_u64(e);
      int tok = 0;
      if (m == 0ull) dev_error(p.ctl, DEV_ERR_DATA);
      else tok = (int)key_id(m);
      if (c == 0) p.tokens[(size_t)b * P + i] = tok;
      int nxt = (p.force && i + 1 < P) ? p.force[(size_t)b * P + i] : tok;
      if (nxt < 0 || nxt >= V) { dev_error(p.ctl, DEV_ERR_DATA); nxt = 0; }
      if (m != spec_s[b] && nxt != tok_s[b]) {
        tok_s[b] = nxt;
        *redo_s = 1;
      }
    } else if (i + 1 < P) {
      gather_gates(32);
    }
    __syncthreads();
    if (*redo_s) {  // block-uniform
      if (i + 1 < P) gather_gates(0);
      __syncthreads();
      if (threadIdx.x == 0) *redo_s = 0;
    }
  }

  if (!ok) {
    cp_async_wait_all();
    if (threadIdx.x == 32 && seg_issued >= 0) mbar_wait(seg_bar, (uint32_t)(seg_issued & 1), nullptr, p.ctl, p.timeout_ns);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// Staged segment: [v0 & ~3, (v1 + 3) & ~3) per request, a multiple of 4 floats.
int small_seg(int rows_max) { return ((rows_max + 3) & ~3) + 4; }

size_t small_fixed_smem(int bs, int g, int nu_max, int rows_max, bool noise) {
  auto a16 = [](size_t x) { return (x + 15) & ~(size_t)15; };
  const int seg = small_seg(rows_max);
  return a16((size_t)3 * nu_max * g * 2) + a16((size_t)kR * nu_max * 4) + a16((size_t)3 * nu_max * 4) +
         a16((size_t)bs * g * 4) + 2 * a16((size_t)bs * 3 * nu_max * 4) + a16((size_t)bs * seg * 4) +
         a16((size_t)(noise ? bs : 0) * seg * 4) + 2 * a16((size_t)bs * kR * 4) +
         a16((size_t)bs * nu_max * 4) + a16((size_t)bs * kR * 8) + a16((size_t)bs * 4) + 16 + 16 +
         a16((size_t)bs * 8) + a16((size_t)kWarps * bs * 8) + 16 + 16;
}

template <int BS>
cudaError_t launch_small_t(const ChainArgs& a, cudaStream_t stream) {
  const int G = num_sms();
  SmallP p;
  p.bs = BS; p.P = a.P; p.d = a.d; p.g = a.g; p.V = a.V;
  p.nu_max = (a.g + G - 1) / G;
  p.rows_max = (a.V + G - 1) / G;
  p.seg = small_seg(p.rows_max);
  const bool noise = a.temperature > 0.0f;
  p.bulk = (a.V % 4) == 0 && ((uintptr_t)a.L_base & 15u) == 0 && ((uintptr_t)a.P_h & 15u) == 0 &&
           (!noise || (((uintptr_t)a.gumbel & 15u) == 0 && (a.gumbel_bstride % 4) == 0));
  const size_t fixed = small_fixed_smem(BS, a.g, p.nu_max, p.rows_max, a.temperature > 0.0f);
  const size_t budget = 227 * 1024;
  if (fixed > budget) return cudaErrorInvalidConfiguration;
  int srows = (int)((budget - fixed) / 512);
  const int rest = p.rows_max - kTmemRows;
  if (srows > rest) srows = rest > 0 ? rest : 0;
  if (srows < 32) srows = 32;  // the row buffer also stages the TMEM rows, 32 at a time
  if (fixed + (size_t)srows * 512 > budget) return cudaErrorInvalidConfiguration;
  p.smem_rows = srows;
  p.gate_table = a.gate_table;
  p.w_hh = (const __nv_bfloat16*)a.w_hh; p.b_hh = (const __nv_bfloat16*)a.b_hh;
  p.w1 = (const __nv_bfloat16*)a.w1; p.w2 = (const __nv_bfloat16*)a.w2;
  p.L_base = a.L_base; p.P_h = a.P_h; p.anchor = a.anchor;
  p.temperature = a.temperature;
  p.inv_temperature = a.temperature > 0.0f ? 1.0f / a.temperature : 0.0f;
  p.gumbel = a.gumbel; p.gumbel_bstride = a.gumbel_bstride;
  p.force = a.force; p.tokens = a.tokens; p.logits_out = a.logits_out;
  p.ctl = a.ctl; p.keys = a.keys; p.S = (unsigned long long*)a.S; p.uacc = a.uacc;
  p.n_contrib = a.g < G ? a.g : G;
  // An accumulator keeps the sum of all P steps' partials (times 2^32, shifted
  // left 16 bits) in a signed 64-bit word: in range while the total stays
  // below 2^15 in magnitude. Bounding each of its n_contrib * P partials by
  // 2^14 / (n_contrib * P) keeps a factor-two margin.
  p.part_limit = (float)(16384.0 / ((double)p.n_contrib * a.P));
  p.timeout_ns = wait_timeout_ns();
  const size_t smem = fixed + (size_t)srows * 512;
  cudaError_t e = cudaFuncSetAttribute(chain_small_kernel<BS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void* args[] = {(void*)&p};
  return cudaLaunchCooperativeKernel((const void*)chain_small_kernel<BS>, dim3(G), dim3(kThreads), args, smem,
                                     stream);
}

}  // namespace

bool chain_small_applies(const ChainArgs& a) {
  if (a.dtype != DOMINO_BF16 || a.r != kR || a.bs < 1 || a.bs > 4 || (a.g % 8) != 0) return false;
  const int G = num_sms();
  // The accumulators' running count has 16 bits.
  if ((int64_t)(a.g < G ? a.g : G) * a.P > 0xFFFF) return false;
  const int nu_max = (a.g + G - 1) / G;
  const int rows_max = (a.V + G - 1) / G;
  // The row buffer holds at least one 32-row group (it stages the TMEM rows).
  return small_fixed_smem(a.bs, a.g, nu_max, rows_max, a.temperature > 0.0f) + 32 * 512 <= 227 * 1024;
}

cudaError_t launch_chain_small(const ChainArgs& a, cudaStream_t stream) {
  switch (a.bs) {
    case 1: return launch_small_t<1>(a, stream);
    case 2: return launch_small_t<2>(a, stream);
    case 3: return launch_small_t<3>(a, stream);
    default: return launch_small_t<4>(a, stream);
  }
}

}  // namespace domino
