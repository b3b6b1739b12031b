// Small-batch Domino head chain (bf16 weights, rank 256, batch <= 4): the
// low-concurrency serving case, one persistent CTA per SM.
//
// Same arithmetic as the general chain kernel (chain.cu); what differs is where
// W2 lives across the P dependent steps and how W2 u is formed:
//  - Each CTA owns ~1000 vocabulary rows of W2 (512 bytes each) in 16-row
//    tiles. The first 32 tiles stay in tensor memory (TMEM, 256 KB per SM),
//    the next ones in shared memory (bank-swizzled), one more per warp in
//    registers, all loaded once per chain with coalesced row reads (the TMEM
//    tiles pass through the shared-memory buffer on their way). Rows past
//    those (none for the Qwen3 shapes at batch 1) are read from L2 each step.
//  - W2 u runs on the tensor core as warp-level bf16 MMAs (m16n8k16, fp32
//    accumulation): A is a 16 x 16 block of W2, B holds u as two bf16 columns
//    per request, hi = bf16(u) and lo = bf16(u - hi) (about 16 mantissa
//    bits), so up to four requests fill the MMA's eight columns. Measured on
//    this GPU: 1024 multiply-adds per cycle per SM this way, against about 58
//    with packed fp32x2 FMAs on unpacked bf16 pairs (two integer operations
//    per pair), and the same MMA count at batch 1 and 4. The TMEM tiles are
//    stored in the MMA's A-fragment order (each thread's lane holds its own
//    fragment words), the shared-memory tiles are read with ldmatrix, the
//    register tile is kept in fragment order. (The single-CTA tcgen05.mma
//    costs ~116 cycles per M = 128, K = 16 step at any N <= 128 here: at
//    N = 8 it would be ten times slower than these MMAs.)
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
//    CTA stores its best (value, id) key in its own slot of the step (one
//    relaxed 64-bit store; the nonzero word is its own completion flag, so
//    neither side needs a fence), and the 32 lanes of warp 0 in every CTA
//    poll all slots and reduce them. All waits are bounded; on
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
constexpr int kTmemTiles = 32;        // 16-row tiles in tensor memory: 16 warps x 2
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
  unsigned long long* keys;  // [P][bs][G] each CTA's best (value, id) key per step and request, zeroed per call
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

// One wait for two outstanding 16-column TMEM loads.
__device__ __forceinline__ void tmem_wait16x2(uint32_t (&r)[16], uint32_t (&s)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
                 "+r"(s[0]), "+r"(s[1]), "+r"(s[2]), "+r"(s[3]), "+r"(s[4]), "+r"(s[5]), "+r"(s[6]), "+r"(s[7]),
                 "+r"(s[8]), "+r"(s[9]), "+r"(s[10]), "+r"(s[11]), "+r"(s[12]), "+r"(s[13]), "+r"(s[14]), "+r"(s[15])
               :
               : "memory");
}

// D += A . B on the tensor core, bf16 operands, fp32 accumulators: one
// m16n8k16 MMA of a warp (A: 16 rows x 16 columns in four registers per
// thread, B: 16 x 8 in two, D: 16 x 8 in four).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               const uint2& b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b.x), "r"(b.y));
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
  // The CTA's rows in 16-row tiles (the MMA's M): the first kTmemTiles in
  // tensor memory (warp w: tiles 2w, 2w + 1), the next ts in shared memory,
  // then kRR rows per warp in registers (warps 0 .. tr - 1), and any rows
  // past those are read from L2 every step (round robin over the warps).
  // Batch 1 keeps a whole tile per warp in registers; larger batches need
  // those registers elsewhere (a half tile there already spills) and keep none.
  constexpr int kRR = BS == 1 ? 16 : 0;
  const int nt = (nrows + 15) >> 4;
  const int tt = min(kTmemTiles, nt);
  const int ts = min(p.smem_rows >> 4, nt - tt);
  const int rbase = 16 * (tt + ts);
  const int tr = kRR ? min(kWarps, max(0, (nrows - rbase + kRR - 1) / max(kRR, 1))) : 0;
  const int rows_t = min(16 * tt, nrows);
  const int rows_s = min(16 * ts, nrows - rows_t);
  const int gbase = rbase + kRR * tr;
  const int rows_g = max(0, nrows - gbase);
  constexpr int kSW = kWarps;

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
  unsigned long long* red_s = (unsigned long long*)take((size_t)kWarps * BS * 8);
  uint32_t* tmem_slot = (uint32_t*)take(16);
  uint64_t* seg_bar = (uint64_t*)take(16);
  uint2* bfrag_s = (uint2*)take((size_t)16 * 32 * 8);  // [kk][lane] B fragments of u (bf16 hi / lo columns)
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
  for (int idx = threadIdx.x; idx < 16 * 32; idx += kThreads) bfrag_s[idx] = make_uint2(0u, 0u);
  if (threadIdx.x == 0) {
    *fail_s = 0;
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
  // Warp w's tensor memory (lane quarter w % 4, columns [128 (w / 4), +128))
  // holds its two tiles 2w, 2w + 1 (CTA rows [32 w, 32 w + 32)) in the MMA's
  // A-fragment order: thread L's lane, column 64 j + 4 kk + q, holds A
  // register q of 16-column chunk kk of tile j, i.e. the bf16 pair
  // (row g + 8 (q & 1), columns 16 kk + 2 t + 8 (q >> 1) + {0, 1}) with
  // g = L / 4, t = L % 4. A 32x32b load of 16 columns then returns four
  // chunks' fragments, one per thread, with no shuffling.
  const int g4 = lane >> 2, t4 = lane & 3;
  const uint32_t tw = tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)((warp >> 2) * 128);
  // The rows pass through the shared-memory row buffer: whole 32-row groups
  // (one warp's two tiles) per pass, read from HBM with coalesced 512-byte
  // row loads into the swizzled layout; each thread then picks its fragment
  // words (conflict-free: the 8 rows of a quarter warp sit in 8 different
  // 16-byte slots) and stores them to its lane.
  {
    const int ngroups = (rows_t + 31) / 32;
    const int gpp = p.smem_rows / 32;  // groups per pass (at least 1: checked at launch)
    for (int g0 = 0; g0 < ngroups; g0 += gpp) {
      const int g1 = min(ngroups, g0 + gpp);
      const int r0 = g0 * 32, nr = min(rows_t, g1 * 32) - r0, R = (g1 - g0) * 32;
      stage_rows(r0, nr, R);
      __syncthreads();
      if (32 * warp < rows_t && warp >= g0 && warp < g1) {  // warp-uniform
#pragma unroll 1
        for (int j = 0; j < 2; ++j) {
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {  // 8 chunks (32 columns) per store
            uint32_t r[32];
#pragma unroll
            for (int m = 0; m < 8; ++m) {
              const int kk = 8 * h + m;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int row = 32 * warp + 16 * j + g4 + 8 * (q & 1);
                const int word = 8 * kk + t4 + 4 * (q >> 1);  // bf16 pair index in the row
                const int lr = min(row, rows_t - 1) - r0;
                r[4 * m + q] = row < rows_t && DCHECK(p.ctl, lr >= 0 && lr < R)
                                   ? ((const uint32_t*)&w2s[w2s_index(word >> 5, lr, (word >> 2) & 7, R)])[word & 3]
                                   : 0u;
              }
            }
            tmem_st32(tw + (uint32_t)(64 * j + 32 * h), r);
          }
        }
      }
      __syncthreads();
    }
  }
  tmem_wait_st();
  // The shared-memory tiles, loaded once; rows of a last partial tile are zero.
  stage_rows(rows_t, rows_s, p.smem_rows);
  for (int idx = threadIdx.x; idx < (16 * ts - rows_s) * 32; idx += kThreads) {
    const int rr = rows_s + (idx >> 5), l = idx & 31;
    w2s[w2s_index(l >> 3, rr, l & 7, p.smem_rows)] = make_uint4(0u, 0u, 0u, 0u);
  }

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
  // The register tile of warp w < tr (rows rbase + 16 w ..), in A-fragment
  // order: rt[kk][q] as in tensor memory above. Loaded once per chain.
  uint32_t rt[16][4];
  if (kRR == 16) {
    const int row0 = rbase + 16 * warp;
#pragma unroll
    for (int kk = 0; kk < 16; ++kk)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int row = row0 + g4 + 8 * (q & 1);
        const int word = 8 * kk + t4 + 4 * (q >> 1);
        rt[kk][q] = (warp < tr && row < nrows) ? __ldg((const uint32_t*)(p.w2 + (size_t)(v0 + row) * kR) + word)
                                               : 0u;
      }
  }
  // Shared-memory tiles per warp (at most two): first to the warps without
  // register rows, then round robin.
  int sidx0 = -1, sidx1 = -1;
  for (int s2 = 0; s2 < ts; ++s2) {
    const int owner = s2 < kWarps - tr ? tr + s2 : (s2 - (kWarps - tr)) % kWarps;
    if (owner == warp) {
      if (sidx0 < 0) sidx0 = s2;
      else if (sidx1 < 0) sidx1 = s2;
    }
  }

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
        if (DCHECK(p.ctl, b < BS && j0 + jj < g)) st_relaxed_u64(Sw + (size_t)b * g + j0 + jj, tag | __float_as_uint(hn));
        snew_s[b * nu_max + jj] = hn;
      }
    }
    __syncthreads();
    if (nu > 0) {
      for (int idx = (int)threadIdx.x - 32; idx >= 0 && idx < bsr; idx += kThreads - 32) {
        const int b = idx / kR, k = idx - b * kR;
        float part = 0.0f;
        for (int jj = 0; jj < nu; ++jj) part = fmaf(w1s_s[k * nu + jj], snew_s[b * nu_max + jj], part);
        if (DCHECK(p.ctl, idx < bsr)) atomicAdd((unsigned long long*)(p.uacc + (size_t)idx * kUaccPad),
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
        const float u = siluf_(ph_s[idx] + __ll2float_rn(d >> 16) * kInvFix);  // one rounding, exact scaling
        u_s[idx] = u;
        // u as two bf16 columns of the MMA's B operand: hi = bf16(u) and
        // lo = bf16(u - hi) (u - hi is exact in fp32), so hi + lo keeps about
        // 16 mantissa bits. Column 2b + part of request b; thread L of a
        // fragment holds column L / 4, rows 2 (L % 4) + {0, 1} (register 0)
        // and 8 + 2 (L % 4) + {0, 1} (register 1) of each 16-row chunk kk.
        const int b = idx / kR, k = idx - b * kR;
        const int kk = k >> 4, kr = k & 15, reg = kr >> 3, t = (kr & 7) >> 1, half = kr & 1;
        const __nv_bfloat16 hi = __float2bfloat16_rn(u);
        const __nv_bfloat16 lo = __float2bfloat16_rn(u - __bfloat162float(hi));
        unsigned short* bh = (unsigned short*)bfrag_s;
        bh[((kk * 32 + (2 * b) * 4 + t) * 2 + reg) * 2 + half] = __bfloat16_as_ushort(hi);
        bh[((kk * 32 + (2 * b + 1) * 4 + t) * 2 + reg) * 2 + half] = __bfloat16_as_ushort(lo);
      }
    }
    __syncthreads();
    if (*fail_s) { ok = false; break; }

    // ---------------- C: L = L_base + W2 u (+ noise), best key per request.
    {
      unsigned long long best[BS];
#pragma unroll
      for (int b = 0; b < BS; ++b) best[b] = 0ull;
      auto consider = [&](int b, int lr, float s) {
        const int v = v0 + lr;
        if (!DCHECK(p.ctl, lr >= 0 && lo + lr < p.seg && v < V)) return;
        const float logit = lb_s[b * p.seg + lo + lr] + s;
        if (p.logits_out) p.logits_out[((size_t)b * P + i) * V + v] = logit;
        const float dec = p.temperature > 0.f ? logit * p.inv_temperature + gm_s[b * p.seg + lo + lr] : logit;
        const unsigned long long key = value_id_key(dec, (uint32_t)v);
        best[b] = key > best[b] ? key : best[b];
      };
      // W2 u for the warp's tiles on the tensor core: D[16 rows x 8 columns]
      // += A[16 x 16 of W2] . B[16 x 8 of u], columns 2b / 2b + 1 the hi / lo
      // parts of request b, rank quarter by rank quarter (each quarter's B
      // fragments loaded once for all the warp's tiles). Independent MMA
      // chains (one per tile) alternate in program order so one warp keeps
      // several in flight. Thread L ends with rows g, g + 8 of columns 2 t,
      // 2 t + 1 (g = L / 4, t = L % 4): the two parts of request t.
      const int nT = 32 * warp < rows_t ? 2 : 0;  // the warp's tensor-memory tiles (both, or none)
      const bool has_r = warp < tr;
      // Epilogue of one tile: thread L (t = L % 4 < BS) owns request t's
      // rows g and g + 8; the batch index stays a compile-time constant.
      auto epi = [&](int row0, const float (&cc)[4]) {
#pragma unroll
        for (int b = 0; b < BS; ++b) {
          if (t4 == b) {
            const int r = row0 + g4;
            const float s0 = cc[0] + cc[1], s1 = cc[2] + cc[3];
            if (r < nrows) consider(b, r, s0);
            if (r + 8 < nrows) consider(b, r + 8, s1);
          }
        }
      };
      auto tmem_pass = [&]() {
        if (nT) {  // warp-uniform: the two tensor-memory tiles, one load round per quarter
          float c0[4], c1[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) c0[q] = c1[q] = 0.0f;
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            uint32_t a[16], e[16];
            tmem_issue16(tw + (uint32_t)(16 * qq), a);
            tmem_issue16(tw + (uint32_t)(64 + 16 * qq), e);
            uint2 bq[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) bq[m] = bfrag_s[(4 * qq + m) * 32 + lane];
            tmem_wait16x2(a, e);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              mma_bf16_16816(c0, a[4 * m], a[4 * m + 1], a[4 * m + 2], a[4 * m + 3], bq[m]);
              mma_bf16_16816(c1, e[4 * m], e[4 * m + 1], e[4 * m + 2], e[4 * m + 3], bq[m]);
            }
          }
          epi(32 * warp, c0);
          epi(32 * warp + 16, c1);
        }
      };
      auto smem_pass = [&]() {  // the shared-memory tiles and the register tile
        float cS0[4], cS1[4], cR[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) cS0[q] = cS1[q] = cR[q] = 0.0f;
        // ldmatrix row addresses: lane L reads row (L & 7) + 8 ((L >> 3) & 1)
        // of the tile, 16-byte chunk 2 kk + (L >> 4).
        const uint32_t w2s_a = smem_u32(w2s);
        const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1), lhalf = lane >> 4;
        const int rr0 = 16 * max(sidx0, 0) + lrow, rr1 = 16 * max(sidx1, 0) + lrow;
        auto ldsm = [&](int rr, int kk, uint32_t (&a)[4]) {
          const int c16 = 2 * kk + lhalf;  // 16-byte chunk of the row
          const uint32_t addr =
              w2s_a + (uint32_t)(w2s_index(c16 >> 3, DCHECK(p.ctl, rr >= 0 && rr < p.smem_rows) ? rr : 0, c16 & 7,
                                           p.smem_rows) *
                                 16);
          asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                       : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                       : "r"(addr));
        };
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const uint2 bk = bfrag_s[kk * 32 + lane];
          uint32_t a[4], e[4];
          if (sidx0 >= 0) ldsm(rr0, kk, a);  // warp-uniform
          if (sidx1 >= 0) ldsm(rr1, kk, e);
          if (kRR == 16 && has_r) mma_bf16_16816(cR, rt[kk][0], rt[kk][1], rt[kk][2], rt[kk][3], bk);
          if (sidx0 >= 0) mma_bf16_16816(cS0, a[0], a[1], a[2], a[3], bk);
          if (sidx1 >= 0) mma_bf16_16816(cS1, e[0], e[1], e[2], e[3], bk);
        }
        if (sidx0 >= 0) epi(rows_t + 16 * sidx0, cS0);
        if (sidx1 >= 0) epi(rows_t + 16 * sidx1, cS1);
        if (kRR == 16 && has_r) epi(rbase + 16 * warp, cR);
      };
      tmem_pass();
      smem_pass();
      // Rows past the resident tiles (none for the Qwen3 shapes at batch 1):
      // warp w takes rows gbase + w, + 16, ...; 32 lanes split a row's 256
      // columns and eight rows are reduced together (packed fp32x2 FMAs).
      if (ng > 0) {
        const int rq = row_of_lane(lane);
#pragma unroll 1
        for (int t0 = 0; t0 < ng; t0 += 8) {
          uint4 wv[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int t = min(t0 + q, ng - 1);
            wv[q] = ld_nc_v4(p.w2 + (size_t)(v0 + gbase + sw + t * kSW) * kR + lane * 8);
          }
#pragma unroll
          for (int b = 0; b < BS; ++b) {
            U8 ub;
#pragma unroll
            for (int t = 0; t < 4; ++t)
              ub.p[t] = pack2(u_s[b * kR + lane * 8 + 2 * t], u_s[b * kR + lane * 8 + 2 * t + 1]);
            float pr[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) pr[q] = dot8(wv[q], ub);
            const float s = reduce8(pr, lane);
            const int t = t0 + rq;
            if ((lane & 3) == 0 && t < ng) consider(b, gbase + sw + t * kSW, s);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < BS; ++b) {
        const unsigned long long m = warp_max_u64(best[b]);
        if (lane == 0) red_s[warp * BS + b] = m;
      }
    }
    __syncthreads();
    // The CTA's best key per request goes to its own slot of the step: one
    // relaxed 64-bit store. The word is its own completion flag (slots are
    // zero before the chain, and every stored key is nonzero: a CTA without
    // rows stores 1, below every real key), so it needs no fence or counter.
    if (threadIdx.x < BS) {
      unsigned long long m = 0ull;
      for (int w = 0; w < kWarps; ++w) {
        const unsigned long long x = red_s[w * BS + threadIdx.x];
        m = x > m ? x : m;
      }
      if (DCHECK(p.ctl, i < P && c < G)) st_relaxed_u64(p.keys + ((size_t)i * BS + threadIdx.x) * G + c, m ? m : 1ull);
    }

    // ---------------- D: warp 0 collects every CTA's keys (each lane polls
    // slots lane, lane + 32, ...; a nonzero word is complete) and reduces
    // them, while warps 1.. sum W_hh S_i; then the token of position i.
    if (warp == 0) {
      constexpr int kSlots = 8;  // slots per lane and request: G <= 256
      const unsigned long long* row0 = p.keys + (size_t)i * BS * G;
      unsigned long long mine[BS];
      unsigned pend = 0u;  // bit b * kSlots + k: slot lane + 32 k of request b not seen yet
#pragma unroll
      for (int b = 0; b < BS; ++b) {
        mine[b] = 0ull;
#pragma unroll
        for (int k = 0; k < kSlots; ++k)
          if (lane + 32 * k < G) pend |= 1u << (b * kSlots + k);
      }
      const uint64_t t0 = globaltimer_ns();
      unsigned spins = 0;
      // While waiting (batch 1, free-running), pull the gate values of the
      // running argmax into L2: the token is usually known before the last
      // CTA's key arrives.
      uint32_t spec = 0xFFFFFFFFu;
      const bool gather = BS == 1 && i + 1 < P && nu > 0 && !p.force;
      while (true) {
        unsigned long long x[BS][kSlots];
#pragma unroll
        for (int b = 0; b < BS; ++b)
#pragma unroll
          for (int k = 0; k < kSlots; ++k)
            x[b][k] = (pend >> (b * kSlots + k)) & 1u ? ld_relaxed_u64(row0 + (size_t)b * G + lane + 32 * k) : 0ull;
#pragma unroll
        for (int b = 0; b < BS; ++b)
#pragma unroll
          for (int k = 0; k < kSlots; ++k)
            if (x[b][k]) {
              mine[b] = x[b][k] > mine[b] ? x[b][k] : mine[b];
              pend &= ~(1u << (b * kSlots + k));
            }
        if (!__any_sync(0xffffffffu, pend != 0u)) break;
        if (gather) {
          const unsigned long long m = warp_max_u64(mine[0]);
          if (lane == 0 && m > 1ull && key_id(m) != spec) {
            spec = key_id(m);
            if (spec < (uint32_t)V) {
#pragma unroll
              for (int q = 0; q < 3; ++q) {
                const float* ga = p.gate_table + (size_t)spec * 3 * g + q * g + j0;
                prefetch_l2(ga);
                if ((((uintptr_t)ga ^ (uintptr_t)(ga + nu - 1)) >> 7) != 0) prefetch_l2(ga + nu - 1);
              }
            }
          }
        }
        if ((++spins & 15u) == 0) {
          int stop = 0;
          if (lane == 0) {
            if (ld_volatile_u32(&p.ctl->abort)) stop = 1;
            else if (globaltimer_ns() - t0 > p.timeout_ns) { dev_abort(p.ctl, DEV_ERR_TIMEOUT); stop = 1; }
          }
          if (__shfl_sync(0xffffffffu, stop, 0)) { if (lane == 0) *fail_s = 1; break; }
        }
      }
      // The tokens, then (warp 0 alone, while warps 1.. still sum W_hh S_i)
      // the gate-table values of the next GRU inputs.
#pragma unroll
      for (int b = 0; b < BS; ++b) {
        const unsigned long long m = warp_max_u64(mine[b]);  // every lane holds the maximum
        int tok = 0;
        if (m <= 1ull) {
          if (lane == 0) dev_error(p.ctl, DEV_ERR_DATA);
        } else {
          tok = (int)key_id(m);
        }
        if (lane == 0 && c == 0) p.tokens[(size_t)b * P + i] = tok;
        int nxt = (p.force && i + 1 < P) ? p.force[(size_t)b * P + i] : tok;
        if (nxt < 0 || nxt >= V) {
          if (lane == 0) dev_error(p.ctl, DEV_ERR_DATA);
          nxt = 0;
        }
        if (i + 1 < P) {
          for (int idx = lane; idx < 3 * nu; idx += 32) {
            const int q = idx / nu, jj = idx - q * nu;
            if (DCHECK(p.ctl, nxt >= 0 && nxt < V && j0 + jj < g && idx < 3 * nu_max))
              gi_s[b * 3 * nu_max + idx] = __ldg(p.gate_table + (size_t)nxt * 3 * g + q * g + j0 + jj);
          }
        }
      }
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
         a16((size_t)bs * nu_max * 4) + a16((size_t)bs * kR * 8) + a16((size_t)bs * 4) + 16 +
         a16((size_t)kWarps * bs * 8) + 16 + 16 + 16 * 32 * 8;
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
  // Shared-memory rows in whole 16-row tiles; the buffer also stages the
  // tensor-memory rows, 32 (one warp's two tiles) at a time.
  int srows = (int)((budget - fixed) / 512) & ~15;
  const int rest = (p.rows_max - 16 * kTmemTiles + 15) & ~15;
  if (srows > rest) srows = rest > 0 ? rest : 0;
  if (srows < 32) srows = 32;
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
  if (G > 256) return false;  // warp 0 polls at most 8 key slots per lane and request
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
