// Batched Domino head chain (bf16 weights, rank 256, 5 <= batch <= 64): the
// high-concurrency case, one persistent CTA per SM, tensor cores for every
// product.
//
// Per step i (requests b = 0..batch-1; S_i = the chain's state after the
// anchor and tokens 0..i-1):
//   S pass   D_s = S16_i [128 x g] . B_s^T, one tcgen05.mma chain (M = 128,
//            K = g) per CTA. S16 holds S_i in bf16 as a high row (2b) and a
//            low row (2b + 1); hi + lo keeps ~16 mantissa bits of S. B_s stacks
//            the CTA's slice of W1[:, d:] rows (bottleneck units k) and the
//            W_hh rows (gates r, z, n) of the hidden units it owns, resident in
//            shared memory. D_s gives u_pre_i for the CTA's k-slice and the
//            hidden-side gate sums W_hh S_i of the next GRU step.
//            u_i = SiLU(P_h[i] + u_pre_i) goes to U16 (bf16 hi / lo rows).
//   W pass   once every CTA's u slice is published: D_w = U16 . W2 tile^T per
//            128-row tile of the CTA's vocabulary range (TMEM lane = a U16
//            row, i.e. one request's high or low part; column = a vocabulary
//            row), W2 tiles streamed by TMA through a shared ring (kept in L2
//            across steps by an evict-last hint), accumulators double-buffered
//            in TMEM. The epilogue adds L_base (and Gumbel noise at T > 0),
//            which the same TMA producer stages into shared memory ahead of
//            use (3-D boxes of 16 requests x 128 vocabulary ids); each lane
//            keeps its request's best (value, id) over its columns, so no
//            per-tile cross-lane reduction is needed; one atomicMax per
//            request and CTA, each request's key on its own 128-byte line.
//            With the draft statistics wanted, each lane also folds its
//            logits into a running log-sum-exp of L_i / T (merged across CTAs
//            once the chain is done), and the S pass writes u_i: what a
//            sampled verification needs instead of the full logits.
//            When the corrected
//            logits are wanted, each full tile's values overwrite the staged
//            L_base box in place and leave by TMA store from there. B_s's shared region
//            doubles as that staging ring: B_s is copied back each step from
//            a per-CTA image in global memory (one bulk copy, overlapped with
//            the wait for S16).
//   GRU      once every CTA's keys are in: token i, the input-side gates from
//            the prepared table, S_{i+1} for the CTA's units (fp32 kept on chip,
//            bf16 hi / lo written to S16).
// The three all-to-all points (u slices, keys, S16) are counted arrivals: a
// release increment per CTA, one thread per CTA polls until all have arrived
// and then acquires (bounded; on timeout the error is recorded, the abort flag
// raised and every CTA leaves).
#include <cuda.h>
#include <string.h>

#include "common.cuh"

namespace domino {

namespace {

constexpr int kThreads = 384;  // warp 0: TMA + polling, warp 1: MMA, warp 2: staging TMA, warps 4-11: TMEM epilogue
constexpr int kKeyGroups = 8;  // the per-request argmax merges in 8 groups of CTAs
constexpr int kR = 256;
constexpr int kStages = 4;
constexpr uint32_t kChunk = 128 * 64 * 2;  // a 128-row x 64-column bf16 chunk (16 KB)
constexpr int kMaxB = 64;

struct BatP {
  CUtensorMap tm_w2;   // W2 [V, 256], box 64 x 128
  CUtensorMap tm_s16;  // S16 [128, g], box 64 x 128
  CUtensorMap tm_u16;  // U16 [NB, 256], box 64 x NB
  CUtensorMap tm_lb;   // L_base viewed [bs][P][V] fp32, box lg_pitch / 4 x 1 x 16
  CUtensorMap tm_gm;   // noise viewed [bs][P][V] fp32 (batch stride as given), box lg_pitch / 4 x 1 x 16
  CUtensorMap tm_lo;   // logits_out viewed [bs][P][V] fp32, box 128 x 1 x 16 (when lo_tma)
  int bs, P, d, g, V, NB, NBs, nu_max, box_z;
  int lo_tma;          // 1: full tiles' logits leave by TMA store from the staging slot
  // Bytes per request row of a staged box: 512 (128 columns) when logits go
  // out (the slot doubles as the store's source), else 528: four columns
  // more, so that the 16 request rows an epilogue warp reads at once start
  // in different bank groups (a 512-byte pitch puts them all in one).
  int lg_pitch;
  uint32_t reg_bytes;  // shared region: B_s in the S pass, L_base / noise staging in the W pass
  const float* gate_table;
  const __nv_bfloat16* w_hh;
  const __nv_bfloat16* b_hh;
  const __nv_bfloat16* w1;
  const float* L_base;
  const float* P_h;
  const int32_t* anchor;
  float temperature, inv_temperature;
  const float* gumbel;
  int64_t gumbel_bstride;
  const int32_t* force;
  int32_t* tokens;
  float* logits_out;
  float* u_out;              // [bs][P][256] u_i, or null
  float* lse_out;            // [bs][P] logsumexp_v L_i[v] / T', or null
  float2* lse_part;          // [P][bs][G] per-CTA (max, sum) partials in log2 units (with lse_out)
  float lse_c;               // log2(e) / T' (T' = T, or 1 at T = 0)
  Ctl* ctl;
  __nv_bfloat16* s16;        // [128][g]
  __nv_bfloat16* u16;        // [NB][256]
  unsigned long long* keys;  // [P][bs][kKeyGroups], 16 words (128 bytes) apart
  unsigned int* ctr;         // [3][P + 1], 8 words apart
  uint8_t* bimg;             // [G][kch][NBs][128 B] B_s images (shared-memory layout)
  uint64_t timeout_ns;
};

__device__ __forceinline__ int vocab_begin(int V, int c, int G) {
  return c >= G ? V : (int)(((int64_t)V * c / G) & ~(int64_t)3);  // 4-aligned (16-byte TMA x)
}

__device__ __forceinline__ void tma_load_3d_hint(void* smem_dst, const void* tmap, int x, int y, int z, uint64_t* bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(smem_dst)),
      "l"((uint64_t)tmap), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Written once and not read here again: evict-first, so W2 keeps its L2 lines.
__device__ __forceinline__ void tma_store_3d(const void* tmap, uint32_t smem_src, int x, int y, int z,
                                             uint64_t policy) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3, %4}], [%1], %5;" ::
                   "l"((uint64_t)tmap), "r"(smem_src), "r"(x), "r"(y), "r"(z), "l"(policy)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void sts_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float4 lds_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ void red_release_add(unsigned int* p) {
  asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p) : "memory");
}
__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// 2^x by the hardware approximation (PTX ex2.approx.ftz: relative error near
// 2^-22, results below 2^-126 flushed to zero).
// The larger of a and b, NaN if either is NaN.
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float y;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Log-sum-exp pairs in base 2: (m, s) stands for m + log2(s); an empty pair
// is (-inf, 0).
__device__ __forceinline__ void lse2_fold(float& m, float& s, float m2, float s2) {
  const float mx = fmaxf(m, m2);
  s = mx == -INFINITY ? 0.0f : s * exp2f(m - mx) + s2 * exp2f(m2 - mx);
  m = mx;
}

// Byte offset of K-major element (row, k) in a 128-byte-swizzled operand made
// of 64-column chunks of `rows` rows each (the layout TMA writes with SWIZZLE_128B).
__device__ __forceinline__ uint32_t sw128_off(int row, int k, int rows) {
  const int kc = k >> 6, kk = k & 63;
  return (uint32_t)(kc * rows * 128 + row * 128 + ((((kk >> 3) ^ (row & 7)) & 7) << 4) + (kk & 7) * 2);
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
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

// One thread: wait until *ctr >= target, then acquire. Bounded.
__device__ bool wait_count(const unsigned* ctr, unsigned target, Ctl* ctl, uint64_t timeout_ns) {
  if (ld_relaxed_u32(ctr) < target) {
    const uint64_t t0 = globaltimer_ns();
    unsigned spins = 0;
    while (ld_relaxed_u32(ctr) < target) {
      if ((++spins & 63u) == 0) {
        if (ld_volatile_u32(&ctl->abort)) return false;
        if (globaltimer_ns() - t0 > timeout_ns) { dev_abort(ctl, DEV_ERR_TIMEOUT); return false; }
      }
    }
  }
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  return true;
}

// kLogits: the corrected logits go out (p.logits_out set); the other
// instance carries none of that code in its epilogue loop.
template <bool kLogits>
__global__ void __launch_bounds__(kThreads, 1) chain_batched_kernel(const __grid_constant__ BatP p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int G = gridDim.x, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bs = p.bs, g = p.g, V = p.V, P = p.P, NB = p.NB, NBs = p.NBs, nu_max = p.nu_max;
  const int j0 = (int)((int64_t)g * c / G), j1 = (int)((int64_t)g * (c + 1) / G), nu = j1 - j0;
  const int k0 = (int)((int64_t)kR * c / G), k1 = (int)((int64_t)kR * (c + 1) / G), ku = k1 - k0;
  const int v0 = vocab_begin(V, c, G), v1 = vocab_begin(V, c + 1, G);
  const int nrows = v1 - v0;
  const int ntiles = (nrows + 127) / 128;
  // The W pass visits its tiles forward on even steps and backward on odd
  // ones: the W2 tiles a step reads last are the first the next step needs,
  // while they are most likely still in L2.
  auto tile_at = [&](int step, int t) { return (step & 1) ? ntiles - 1 - t : t; };
  const int kch = g / 64;  // K chunks of the S pass
  const uint32_t bs_bytes = (uint32_t)kch * NBs * 128;
  const uint32_t lg_slot = 16u * (uint32_t)p.lg_pitch;              // room for one staged box
  const uint32_t lg_bytes = (uint32_t)p.box_z * (uint32_t)p.lg_pitch;  // bytes one box carries
  // Staging slots: an L_base box, then at T > 0 its noise box.
  const uint32_t lg_stride = p.temperature > 0.f ? 2 * lg_slot : lg_slot;
  const int nchunks = (bs + 15) / 16;  // epilogue request chunks of 16
  // Staging slots: at most eight, and a multiple of nchunks, so that every
  // slot only ever holds boxes of one request chunk and is waited on by that
  // chunk's epilogue warps alone. (Shared by chunks, a slot's phase parity
  // would let a warp running ahead take an older fill for its own.)
  const int n_lg_room = (int)(p.reg_bytes / lg_stride) < 8 ? (int)(p.reg_bytes / lg_stride) : 8;
  const int n_lg = n_lg_room - n_lg_room % nchunks;
  // W-pass accumulator rows: U16 rows 0 .. NB of a quadrant group; at batch
  // <= 32 (NB <= 64) they are loaded twice, at rows 0 and 64, so all four
  // TMEM lane quadrants hold requests and each warp takes half the columns.
  const int nq = (NB + 31) / 32;          // quadrants with distinct requests
  const int reps = nq <= 2 ? 2 : 1;       // copies of them
  const int cw = 64 / reps;               // vocabulary columns per epilogue warp and tile

  // ---- shared memory (MMA operands first, 1024-byte aligned)
  uint8_t* ring = smem;                                   // kStages x 16 KB
  uint8_t* bs_op = ring + kStages * kChunk;               // B_s: kch chunks of NBs rows x 128 B
  size_t off = (size_t)(bs_op - smem) + p.reg_bytes;
  auto take = [&](size_t bytes) { uint8_t* q = smem + off; off = (off + bytes + 15) & ~(size_t)15; return q; };
  uint64_t* full = (uint64_t*)take(8 * kStages);
  uint64_t* empty = (uint64_t*)take(8 * kStages);
  uint64_t* s_done = (uint64_t*)take(8);
  uint64_t* u_ready = (uint64_t*)take(8);
  uint64_t* u_copied = (uint64_t*)take(8);  // U16 is in tensor memory: the region may take boxes
  uint64_t* t_full = (uint64_t*)take(16);
  uint64_t* t_empty = (uint64_t*)take(16);
  uint64_t* lg_full = (uint64_t*)take(8 * 8);
  uint64_t* lg_empty = (uint64_t*)take(8 * 8);
  uint64_t* b_ready = (uint64_t*)take(8);
  uint32_t* tmem_slot = (uint32_t*)take(16);
  volatile int* s_abort = (volatile int*)take(16);
  int* fail_s = (int*)take(16);
  float* gh_s = (float*)take((size_t)kMaxB * 3 * nu_max * 4);    // W_hh S + b_hh  [b][3 nu]
  float* sown_s = (float*)take((size_t)kMaxB * nu_max * 4);      // S of own units [b][nu]
  float* gi_s = (float*)take((size_t)kMaxB * 3 * nu_max * 4);    // W_ih x + b_ih  [b][3 nu]
  float* bhh_s = (float*)take((size_t)3 * nu_max * 4);
  int* tok_s = (int*)take(kMaxB * 4);
  unsigned long long* best_s = (unsigned long long*)take((size_t)4 * kMaxB * 8);  // [team][b]
  float2* lsep_s = (float2*)take((size_t)4 * kMaxB * 8);                           // [team][b]

  // ---- one-time set-up
  for (int idx = threadIdx.x; idx < 4 * kMaxB; idx += kThreads) best_s[idx] = 0ull;
  // B_s image (rows [0, ku) = W1 rows k0.. on S, [ku, ku + 3 nu) = W_hh rows
  // q*g + j0 + jj, the rest zero), laid out as the swizzled operand, in this
  // CTA's global slot; copied into shared memory at the start of every step.
  uint8_t* bimg = p.bimg + (size_t)c * bs_bytes;
  for (int idx = threadIdx.x; idx < NBs * (g / 8); idx += kThreads) {
    const int row = idx / (g / 8), k8 = idx - row * (g / 8);
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row < ku) {
      v = *(const uint4*)(p.w1 + (size_t)(k0 + row) * (p.d + g) + p.d + k8 * 8);
    } else if (row < ku + 3 * nu) {
      const int rr = row - ku, q = rr / nu, jj = rr - q * nu;
      v = *(const uint4*)(p.w_hh + (size_t)(q * g + j0 + jj) * g + k8 * 8);
    }
    *(uint4*)(bimg + sw128_off(row, k8 * 8, NBs)) = v;
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  for (int idx = threadIdx.x; idx < 3 * nu; idx += kThreads) {
    const int q = idx / nu, jj = idx - q * nu;
    bhh_s[idx] = __bfloat162float(p.b_hh[q * g + j0 + jj]);
  }
  for (int idx = threadIdx.x; idx < kMaxB * nu_max; idx += kThreads) sown_s[idx] = 0.0f;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    mbar_init(s_done, 1);
    mbar_init(u_ready, 1);
    mbar_init(u_copied, 1);
    mbar_init(b_ready, 1);
    for (int s2 = 0; s2 < 8; ++s2) { mbar_init(&lg_full[s2], 1); mbar_init(&lg_empty[s2], 2 * reps); }
    for (int a = 0; a < 2; ++a) { mbar_init(&t_full[a], 1); mbar_init(&t_empty[a], 8); }
    *s_abort = 0;
    *fail_s = 0;
    mbar_fence_init();
    tma_prefetch_desc(&p.tm_w2);
    tma_prefetch_desc(&p.tm_s16);
    tma_prefetch_desc(&p.tm_u16);
    tma_prefetch_desc(&p.tm_lb);
    tma_prefetch_desc(&p.tm_gm);
    if (kLogits && p.lo_tma) tma_prefetch_desc(&p.tm_lo);
  }
  if (warp == 1) { tmem_alloc(tmem_slot, 512); tmem_relinquish(); }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t d_s = tmem_base;        // S pass: NBs (<= 128) columns at 0
  const uint32_t a_u = tmem_base + 128;  // W pass A operand: U16, 128 lanes x 128 columns (NBs <= 128)
  const uint32_t d_w = tmem_base + 256;  // W pass: 2 x 128 columns at 256

  // GRU update for the tokens in tok_s: input-side gates from the table, then
  // S for the own units; the fp32 state stays here, bf16 hi / lo rows go to S16.
  auto gru_update = [&](bool zero_state) {
    // Gate-table values of the new tokens (rows mostly not in L2): four
    // loads in flight per thread before any is stored.
    constexpr int kGU = 4;
    const int ngi = bs * 3 * nu;
    for (int base = threadIdx.x; base < ngi; base += kGU * kThreads) {
      float v[kGU];
#pragma unroll
      for (int u = 0; u < kGU; ++u) {
        const int idx = base + u * kThreads;
        v[u] = 0.0f;
        if (idx < ngi) {
          const int b = idx / (3 * nu), rem = idx - b * 3 * nu, q = rem / nu, jj = rem - q * nu;
          v[u] = __ldg(p.gate_table + (size_t)tok_s[b] * 3 * g + q * g + j0 + jj);
        }
      }
#pragma unroll
      for (int u = 0; u < kGU; ++u) {
        const int idx = base + u * kThreads;
        if (idx < ngi) {
          const int b = idx / (3 * nu), rem = idx - b * 3 * nu;
          gi_s[b * 3 * nu_max + rem] = v[u];
        }
      }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < bs * nu; idx += kThreads) {
      const int b = idx / nu, jj = idx - b * nu;
      const float* gi = gi_s + b * 3 * nu_max;
      const float* gh = gh_s + b * 3 * nu_max;
      const float ghr = zero_state ? bhh_s[jj] : gh[jj];
      const float ghz = zero_state ? bhh_s[nu + jj] : gh[nu + jj];
      const float ghn = zero_state ? bhh_s[2 * nu + jj] : gh[2 * nu + jj];
      const float rg = sigmoidf_(gi[jj] + ghr);
      const float zg = sigmoidf_(gi[nu + jj] + ghz);
      const float ng = tanhf(gi[2 * nu + jj] + rg * ghn);
      const float h = zero_state ? 0.0f : sown_s[b * nu_max + jj];
      const float hn = (1.0f - zg) * ng + zg * h;
      sown_s[b * nu_max + jj] = hn;
      const __nv_bfloat16 hi = __float2bfloat16_rn(hn);
      const __nv_bfloat16 lo = __float2bfloat16_rn(hn - __bfloat162float(hi));
      p.s16[(size_t)(2 * b) * g + j0 + jj] = hi;
      p.s16[(size_t)(2 * b + 1) * g + j0 + jj] = lo;
    }
    __syncthreads();
  };

  // Step -1 -> 0: S_0 = GRU(emb[anchor], 0); hidden-side gates are b_hh alone.
  for (int idx = threadIdx.x; idx < bs; idx += kThreads) {
    int a = p.anchor[idx];
    if (a < 0 || a >= V) { dev_error(p.ctl, DEV_ERR_DATA); a = 0; }
    tok_s[idx] = a;
  }
  __syncthreads();
  gru_update(true);
  if (threadIdx.x == 0) red_release_add(p.ctr + (0 * (P + 1) + 0) * 8);

  const uint32_t idesc_s = idesc_bf16_f32(128, NBs);
  const uint32_t idesc_w = idesc_bf16_f32(128, 128);  // M = U16 rows (128, rows >= NB ignored), N = W2 tile rows
  const uint32_t u_bytes = (uint32_t)(reps * NB) * kR * 2;
  // Ring positions: the producer (warp 0, lane 0) and the MMA issuer (warp 1,
  // lane 0) each keep their own, advancing through the same chunk sequence.
  uint32_t r_stage = 0, r_phase = 0;
  int wt = 0;  // W-pass tiles done so far (accumulator ring)
  bool ok = true;

  for (int i = 0; i < P && ok; ++i) {
    // ================= S pass (waits for S16_i from every CTA).
    if (threadIdx.x == 0) {
      mbar_expect_tx(b_ready, bs_bytes);
      bulk_copy_g2s(bs_op, bimg, bs_bytes, b_ready);
      if (!wait_count(p.ctr + (0 * (P + 1) + i) * 8, (unsigned)G, p.ctl, p.timeout_ns)) *fail_s = 1;
    }
    __syncthreads();
    if (*fail_s) { ok = false; break; }
    if (warp == 0 && lane == 0) {
      for (int kc = 0; kc < kch; ++kc) {
        if (!mbar_wait(&empty[r_stage], r_phase ^ 1u, s_abort, p.ctl, p.timeout_ns)) { *fail_s = 1; break; }
        mbar_expect_tx(&full[r_stage], kChunk);
        tma_load_2d(ring + r_stage * kChunk, &p.tm_s16, kc * 64, 0, &full[r_stage]);
        if (++r_stage == kStages) { r_stage = 0; r_phase ^= 1u; }
      }
    } else if (warp == 1 && lane == 0) {
      if (!mbar_wait(b_ready, (uint32_t)(i & 1), s_abort, p.ctl, p.timeout_ns)) *fail_s = 1;
      tc_fence_after();
      for (int kc = 0; kc < kch && !*fail_s; ++kc) {
        if (!mbar_wait(&full[r_stage], r_phase, s_abort, p.ctl, p.timeout_ns)) { *fail_s = 1; break; }
        tc_fence_after();
        const uint64_t ad = sdesc_k_sw128(smem_u32(ring + r_stage * kChunk));
        const uint64_t bd = sdesc_k_sw128(smem_u32(bs_op + (size_t)kc * NBs * 128));
#pragma unroll
        for (int k = 0; k < 4; ++k) umma_bf16(d_s, ad + 2 * k, bd + 2 * k, idesc_s, (kc | k) ? 1u : 0u);
        umma_commit(&empty[r_stage]);
        if (++r_stage == kStages) { r_stage = 0; r_phase ^= 1u; }
      }
      umma_commit(s_done);
    } else if (warp >= 4) {
      // Epilogue: TMEM lane = S16 row (2b + hi/lo); columns = B_s rows.
      const int q4 = warp & 3, team = (warp - 4) >> 2;
      const int row = q4 * 32 + lane;
      const int b = row >> 1;
      // This lane's P_h entries (the CTA's k-slice, at most kPhMax), loaded
      // while the MMAs run.
      constexpr int kPhMax = 4;
      float ph[kPhMax];
#pragma unroll
      for (int q = 0; q < kPhMax; ++q) {
        const int col = team * 32 + q;  // the slice's columns sit at the start of B_s
        ph[q] = ((row & 1) == 0 && b < bs && col < ku) ? __ldg(p.P_h + ((size_t)b * P + i) * kR + k0 + col) : 0.0f;
      }
      if (!mbar_wait(s_done, (uint32_t)(i & 1), s_abort, p.ctl, p.timeout_ns)) *fail_s = 1;
      tc_fence_after();
      for (int c0 = team * 32; c0 < NBs; c0 += 64) {
        float v[32];
        tmem_ld32(d_s + ((uint32_t)(q4 * 32) << 16) + (uint32_t)c0, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j], 1);  // hi + lo rows
        if ((row & 1) == 0 && b < bs) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int col = c0 + j;
            if (col < ku && DCHECK(p.ctl, k0 + col < kR && b < p.bs)) {
              const int k = k0 + col;
              const float phk = j < kPhMax && c0 < 32 ? ph[j < kPhMax ? j : 0] : __ldg(p.P_h + ((size_t)b * P + i) * kR + k);
              const float u = siluf_(phk + v[j]);
              if (p.u_out) p.u_out[((size_t)b * P + i) * kR + k] = u;
              const __nv_bfloat16 hi = __float2bfloat16_rn(u);
              const __nv_bfloat16 lo = __float2bfloat16_rn(u - __bfloat162float(hi));
              p.u16[(size_t)(2 * b) * kR + k] = hi;
              p.u16[(size_t)(2 * b + 1) * kR + k] = lo;
            } else if (col < ku + 3 * nu) {
              const int rr = col - ku;
              gh_s[b * 3 * nu_max + rr] = v[j] + bhh_s[rr];
            }
          }
        }
      }
      tc_fence_before();
    }
    __syncthreads();
    if (*fail_s) { ok = false; break; }
    if (threadIdx.x == 0) red_release_add(p.ctr + (1 * (P + 1) + i) * 8);  // u slice published

    // ================= W pass (waits for every CTA's u slice).
    if (threadIdx.x == 0 && !wait_count(p.ctr + (1 * (P + 1) + i) * 8, (unsigned)G, p.ctl, p.timeout_ns)) *fail_s = 1;
    __syncthreads();
    if (*fail_s) { ok = false; break; }
    if (warp == 0 && lane == 0) {
      mbar_expect_tx(u_ready, u_bytes);
      // U16 lands in the staging region (free between the S pass and the
      // first staged box), is copied into tensor memory, and the MMAs read it there.
      for (int r = 0; r < reps; ++r)
        for (int kc = 0; kc < 4; ++kc)
          tma_load_2d(bs_op + (size_t)kc * 128 * 128 + (size_t)r * 32 * nq * 128, &p.tm_u16, kc * 64, 0, u_ready);
      const uint64_t pol = l2_policy_evict_last();
      bool go = true;
      for (int t = 0; t < ntiles && go; ++t) {
        for (int kc = 0; kc < 4; ++kc) {
          if (!mbar_wait(&empty[r_stage], r_phase ^ 1u, s_abort, p.ctl, p.timeout_ns)) { *fail_s = 1; go = false; break; }
          mbar_expect_tx(&full[r_stage], kChunk);
          tma_load_2d_hint(ring + r_stage * kChunk, &p.tm_w2, kc * 64, v0 + tile_at(i, t) * 128, &full[r_stage], pol);
          if (++r_stage == kStages) { r_stage = 0; r_phase ^= 1u; }
        }
      }
    } else if (warp == 2 && lane == 0) {
      // L_base / noise boxes for the epilogue, as far ahead as the ring allows.
      const bool noise = p.temperature > 0.f;
      const int nseq = ntiles * nchunks;
      const uint64_t pol = l2_policy_evict_first();  // read once: keep W2 in L2 instead
      // With logits out, the epilogue leaves each full tile's logits in the
      // slot in place of L_base; they go out by TMA store when the slot is
      // next needed, and the step's last boxes before the step ends (the
      // region holds B_s during the next S pass).
      const int ntf = nrows / 128;  // full tiles
      auto store_box = [&](int lqs) {
        const int is = lqs / nseq, sqs = lqs - is * nseq, chs = sqs % nchunks;
        const int ts = tile_at(is, sqs / nchunks);
        if (ts < ntf) {
          tma_store_3d(&p.tm_lo, smem_u32(bs_op + (size_t)(lqs % n_lg) * lg_stride), v0 + ts * 128, is, chs * 16,
                       pol);
          bulk_wait_read_all();  // the slot may be refilled once the store has read it
        }
      };
      if (!mbar_wait(u_copied, (uint32_t)(i & 1), s_abort, p.ctl, p.timeout_ns)) *fail_s = 1;
      for (int sq = 0; sq < nseq && !*fail_s; ++sq) {
        const int lq = i * nseq + sq;  // staged boxes issued so far (all steps)
        const int ch = sq % nchunks, t = tile_at(i, sq / nchunks);
        const int sl = lq % n_lg;
        if (!mbar_wait(&lg_empty[sl], (uint32_t)(((lq / n_lg) & 1) ^ 1), s_abort, p.ctl, p.timeout_ns)) { *fail_s = 1; break; }
        if (kLogits && p.lo_tma && lq - n_lg >= i * nseq) store_box(lq - n_lg);
        uint8_t* dst = bs_op + (size_t)sl * lg_stride;
        mbar_expect_tx(&lg_full[sl], noise ? 2 * lg_bytes : lg_bytes);
        tma_load_3d_hint(dst, &p.tm_lb, v0 + t * 128, i, ch * 16, &lg_full[sl], pol);
        if (noise) tma_load_3d_hint(dst + lg_slot, &p.tm_gm, v0 + t * 128, i, ch * 16, &lg_full[sl], pol);
      }
      if (kLogits && p.lo_tma && !*fail_s) {
        // The step's last boxes: wait until the epilogue has released each
        // (the phase a refill of the slot would wait for), then store.
        const int end = (i + 1) * nseq;
        for (int lq = end - n_lg > i * nseq ? end - n_lg : i * nseq; lq < end; ++lq) {
          if (!mbar_wait(&lg_empty[lq % n_lg], (uint32_t)((lq / n_lg) & 1), s_abort, p.ctl, p.timeout_ns)) {
            *fail_s = 1;
            break;
          }
          store_box(lq);
        }
      }
    } else if (warp == 1 && lane == 0) {
      bool go = mbar_wait(u_ready, (uint32_t)(i & 1), s_abort, p.ctl, p.timeout_ns);
      if (!go) *fail_s = 1;
      tc_fence_after();
      if (go) {
#pragma unroll
        for (int kc = 0; kc < 4; ++kc) {
          const uint64_t ud = sdesc_k_sw128(smem_u32(bs_op + (size_t)kc * 128 * 128));
#pragma unroll
          for (int k = 0; k < 4; ++k) tmem_cp_128x256b(a_u + (uint32_t)(8 * (4 * kc + k)), ud + 2 * k);
        }
      }
      umma_commit(u_copied);  // the staging producer may overwrite the region once this arrives
      for (int t = 0; t < ntiles && go; ++t) {
        const int wtt = wt + t, acc = wtt & 1;
        if (!mbar_wait(&t_empty[acc], (uint32_t)(((wtt >> 1) & 1) ^ 1), s_abort, p.ctl, p.timeout_ns)) { *fail_s = 1; break; }
        tc_fence_after();
        for (int kc = 0; kc < 4; ++kc) {
          if (!mbar_wait(&full[r_stage], r_phase, s_abort, p.ctl, p.timeout_ns)) { *fail_s = 1; go = false; break; }
          tc_fence_after();
          const uint64_t bd = sdesc_k_sw128(smem_u32(ring + r_stage * kChunk));
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16_ts(d_w + (uint32_t)(acc * 128), a_u + (uint32_t)(8 * (4 * kc + k)), bd + 2 * k, idesc_w,
                         (kc | k) ? 1u : 0u);
          umma_commit(&empty[r_stage]);
          if (++r_stage == kStages) { r_stage = 0; r_phase ^= 1u; }
        }
        if (go) umma_commit(&t_full[acc]);
      }
    } else if (warp >= 4) {
      // Epilogue. TMEM lane 32 q + l of the accumulator is U16 row 32 (q % nq)
      // + l: request b = 16 (q % nq) + l / 2, high part for even l, low for odd; the
      // columns are the tile's 128 vocabulary rows. Quadrant q holds the 16
      // requests of chunk q % nq (copy q / nq); warp (quadrant q, team k)
      // takes columns [cw (k + 2 copy), + cw) of every tile for them, whose
      // L_base (and noise) rows are the staged box of that chunk. The two
      // lanes of a request swap halves of every 32 columns, so
      // each holds hi + lo for 16 of them. Per lane, over its columns of all
      // tiles: the best (decision value, id) key, and, with the draft
      // statistics wanted, a log-sum-exp pair (reference, sum) of
      // y = L / T' in base 2 whose reference only moves up (rescaling the sum).
      const int q4 = warp & 3, team = (warp - 4) >> 2;
      const int nseq = ntiles * nchunks;
      const bool noise = p.temperature > 0.f;
      const bool want_lse = p.lse_out != nullptr;
      const int grp = q4 % nq, rep = q4 / nq;  // the quadrant's requests and copy
      const int b = 16 * grp + (lane >> 1), part = lane & 1;
      const bool live = q4 < nq * reps && grp < nchunks;  // warp-uniform: the quadrant holds requests
      const int slot_id = team + 2 * rep;  // this warp's column range and merge slot
      const bool breq = b < bs;
      uint32_t bk = 0u;  // best decision key and its id over the exactly ranked groups
      int bv = 0;
      // Whole groups of 16 rows without a NaN are ranked by their largest
      // decision value alone; the lane keeps the values of its best such
      // group (the lower rows on equal maxima) and ranks inside it once,
      // after the last tile. Partial groups and groups with a NaN are ranked
      // key by key as they come.
      float gbest = 0.0f, gvals[16];
      int glr = -1;  // first row of the best whole group (-1: none yet)
#pragma unroll
      for (int j = 0; j < 16; ++j) gvals[j] = 0.0f;
      float lref = -INFINITY, lsum = 0.0f;
      for (int t = 0; t < ntiles; ++t) {
        const int wtt = wt + t, acc = wtt & 1;
        if (!mbar_wait(&t_full[acc], (uint32_t)((wtt >> 1) & 1), s_abort, p.ctl, p.timeout_ns)) { *fail_s = 1; break; }
        tc_fence_after();
        bool go = true;
        if (live) {
          const int gq = i * nseq + t * nchunks + grp;  // staged boxes so far (all steps)
          const int sl = gq % n_lg;
          if (!mbar_wait(&lg_full[sl], (uint32_t)((gq / n_lg) & 1), s_abort, p.ctl, p.timeout_ns)) {
            *fail_s = 1;
            go = false;
          } else {
            // This request's row of the box: 128 L_base values (then noise).
            const uint32_t row = smem_u32(bs_op + (size_t)sl * lg_stride) + (uint32_t)(b & 15) * (uint32_t)p.lg_pitch;
            const int tv = tile_at(i, t);  // the tile's place in the CTA's rows
            const bool in_slot = kLogits && p.lo_tma && tv < nrows / 128;
#pragma unroll
            for (int hh = 0; hh < cw / 32; ++hh) {
              const int c0 = cw * slot_id + 32 * hh;
              float dv[32];
              tmem_ld32(d_w + (uint32_t)(acc * 128) + ((uint32_t)(q4 * 32) << 16) + (uint32_t)c0, dv);
              // Even lane keeps columns [c0, c0 + 16), odd lane [c0 + 16, c0 + 32).
              float d[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float send = part ? dv[j] : dv[16 + j];
                const float keep = part ? dv[16 + j] : dv[j];
                d[j] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
              }
              const int cb = c0 + 16 * part;  // the lane's first column
              float lb[16], gm[16];
#pragma unroll
              for (int qq = 0; qq < 4; ++qq) {
                const float4 x = lds_f32x4(row + (uint32_t)(cb + 4 * qq) * 4u);
                lb[4 * qq] = x.x; lb[4 * qq + 1] = x.y; lb[4 * qq + 2] = x.z; lb[4 * qq + 3] = x.w;
                if (noise) {
                  const float4 y = lds_f32x4(row + (uint32_t)lg_slot + (uint32_t)(cb + 4 * qq) * 4u);
                  gm[4 * qq] = y.x; gm[4 * qq + 1] = y.y; gm[4 * qq + 2] = y.z; gm[4 * qq + 3] = y.w;
                } else {
                  gm[4 * qq] = gm[4 * qq + 1] = gm[4 * qq + 2] = gm[4 * qq + 3] = 0.0f;
                }
              }
              const int lr0 = tv * 128 + cb;  // the lane's first row within the CTA's range
              float logit[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) logit[j] = lb[j] + d[j];
              if (kLogits && breq) {
                if (in_slot) {  // in place, stored by TMA from the slot
#pragma unroll
                  for (int j = 0; j < 16; ++j) sts_f32(row + (uint32_t)(cb + j) * 4u, logit[j]);
                } else {
#pragma unroll
                  for (int j = 0; j < 16; ++j)
                    if (lr0 + j < nrows && DCHECK(p.ctl, v0 + lr0 + j < V))
                      p.logits_out[((size_t)b * P + i) * V + v0 + lr0 + j] = logit[j];
                }
              }
              if (breq) {
                // (The logits-out instance ranks every group key by key: there
                // the group maximum measured slower.)
                const bool full = !kLogits && lr0 + 16 <= nrows;
                float dec[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) dec[j] = noise ? logit[j] * p.inv_temperature + gm[j] : logit[j];
                bool exact = !full;
                if (full) {
                  // NaN-propagating maximum: a NaN sends the group to the exact ranking.
                  float mx[8];
#pragma unroll
                  for (int j = 0; j < 8; ++j) mx[j] = fmax_nan(dec[j], dec[j + 8]);
#pragma unroll
                  for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
                    for (int j = 0; j < w; ++j) mx[j] = fmax_nan(mx[j], mx[j + w]);
                  if (mx[0] != mx[0]) {
                    exact = true;
                  } else if (glr < 0 || mx[0] > gbest || (mx[0] == gbest && lr0 < glr)) {
                    // (+0 and -0 compare equal, as their keys do; the lower rows win ties)
                    gbest = mx[0];
                    glr = lr0;
#pragma unroll
                    for (int j = 0; j < 16; ++j) gvals[j] = dec[j];
                  }
                }
                if (exact) {
                  // Two interleaved chains (even / odd columns), then the
                  // group's best against the running one (earlier ids win ties).
                  uint32_t ka = 0u, kb = 0u;
                  int ja = 0, jb = 1;
#pragma unroll
                  for (int j = 0; j < 16; ++j) {
                    const uint32_t k = lr0 + j < nrows ? float_order_key(dec[j]) : 0u;
                    if (j & 1) {
                      if (k > kb) { kb = k; jb = j; }
                    } else {
                      if (k > ka) { ka = k; ja = j; }
                    }
                  }
                  const bool tb = kb > ka || (kb == ka && jb < ja);
                  const uint32_t kg = tb ? kb : ka;
                  const int id = v0 + lr0 + (tb ? jb : ja);
                  if (kg > bk || (kg == bk && id < bv)) {  // tiles may come in either order
                    bk = kg;
                    bv = id;
                  }
                }
                if (want_lse) {
                  bool rescale = !full || lref == -INFINITY;
                  if (!rescale) {
                    const float nref = -lref;
                    float e[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) e[j] = ex2_approx(fmaf(logit[j], p.lse_c, nref));
#pragma unroll
                    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                      for (int j = 0; j < w; ++j) e[j] += e[j + w];
                    if (e[0] <= 0x1p64f) lsum += e[0];  // false for inf and NaN
                    else rescale = true;
                  }
                  if (rescale) {
                    float y[16], mj[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                      y[j] = lr0 + j < nrows ? logit[j] * p.lse_c : -INFINITY;
                      mj[j] = y[j];
                    }
#pragma unroll
                    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                      for (int j = 0; j < w; ++j) mj[j] = fmaxf(mj[j], mj[j + w]);
                    if (mj[0] > lref) {
                      lsum = lref == -INFINITY ? 0.0f : lsum * ex2_approx(lref - mj[0]);
                      lref = mj[0];
                    }
                    float e[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) e[j] = y[j] == -INFINITY ? 0.0f : ex2_approx(y[j] - lref);
#pragma unroll
                    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
                      for (int j = 0; j < w; ++j) e[j] += e[j + w];
                    lsum += e[0];
                  }
                }
              }
            }
            if (in_slot) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // for the TMA store
            __syncwarp();
            if (lane == 0) mbar_arrive(&lg_empty[sl]);  // one arrival per team
          }
        }
        if (!go) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&t_empty[acc]);
      }
      if (glr >= 0) {
        // The best whole group: its first largest key, then against the
        // exactly ranked groups (higher key, else lower id).
        uint32_t kg = 0u;
        int jg = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t k = float_order_key(gvals[j]);
          if (k > kg) { kg = k; jg = j; }
        }
        const int id = v0 + glr + jg;
        if (kg > bk || (kg == bk && id < bv)) { bk = kg; bv = id; }
      }
      // Per request: the two lanes, then (through shared memory) the two teams.
      unsigned long long key = bk ? (((unsigned long long)bk << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)bv))
                                  : 0ull;
      const unsigned long long okey = __shfl_xor_sync(0xffffffffu, key, 1);
      key = okey > key ? okey : key;
      float om = __shfl_xor_sync(0xffffffffu, lref, 1), os = __shfl_xor_sync(0xffffffffu, lsum, 1);
      if (part == 0) lse2_fold(om, os, lref, lsum);  // the even lane's pair, in one order
      if (live && part == 0 && breq) {
        best_s[slot_id * kMaxB + b] = key;
        if (want_lse) lsep_s[slot_id * kMaxB + b] = make_float2(om, os);
      }
    }
    __syncthreads();
    wt += ntiles;
    if (*fail_s) { ok = false; break; }
    // Merge the epilogue warps' bests: one atomicMax per request; arrive.
    for (int b = threadIdx.x; b < bs; b += kThreads) {
      unsigned long long m = 0ull;
      for (int q = 0; q < 2 * reps; ++q) {
        const unsigned long long x = best_s[q * kMaxB + b];
        m = x > m ? x : m;
        best_s[q * kMaxB + b] = 0ull;
      }
      if (m && DCHECK(p.ctl, i < P && b < bs)) atomicMax(p.keys + (((size_t)i * bs + b) * kKeyGroups + (c % kKeyGroups)) * 16, m);
      if (p.lse_out) {
        float pm = -INFINITY, ps = 0.0f;
        for (int q = 0; q < 2 * reps; ++q) {
          const float2 x = lsep_s[q * kMaxB + b];
          lse2_fold(pm, ps, x.x, x.y);
        }
        p.lse_part[((size_t)i * bs + b) * G + c] = make_float2(pm, ps);
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) red_release_add(p.ctr + (2 * (P + 1) + i) * 8);

    // ================= GRU (waits for every CTA's keys): token i, S_{i+1}.
    if (threadIdx.x == 0 && !wait_count(p.ctr + (2 * (P + 1) + i) * 8, (unsigned)G, p.ctl, p.timeout_ns)) *fail_s = 1;
    __syncthreads();
    if (*fail_s) { ok = false; break; }
    for (int b = threadIdx.x; b < bs; b += kThreads) {
      unsigned long long key = 0ull;
      for (int q = 0; q < kKeyGroups; ++q) {
        const unsigned long long x = __ldcg(p.keys + (((size_t)i * bs + b) * kKeyGroups + q) * 16);
        key = x > key ? x : key;
      }
      int tok = 0;
      if (key == 0ull) dev_error(p.ctl, DEV_ERR_DATA);
      else tok = (int)key_id(key);
      if (c == 0) p.tokens[(size_t)b * P + i] = tok;
      int nxt = (p.force && i + 1 < P) ? p.force[(size_t)b * P + i] : tok;
      if (nxt < 0 || nxt >= V) { dev_error(p.ctl, DEV_ERR_DATA); nxt = 0; }
      tok_s[b] = nxt;
    }
    __syncthreads();
    if (i + 1 < P) {
      gru_update(false);
      if (threadIdx.x == 0) red_release_add(p.ctr + (0 * (P + 1) + i + 1) * 8);
    }
  }

  // Draft log-partitions: every CTA's partials of every step were released
  // before its arrival at that step's key count, which this CTA has seen.
  // One warp per (request, step) row, rows spread over the grid.
  if (ok && p.lse_out) {
    for (int row = c * (kThreads / 32) + warp; row < bs * P; row += G * (kThreads / 32)) {
      const int b = row / P, i = row - b * P;
      const float2* part = p.lse_part + ((size_t)i * bs + b) * G;
      float m = -INFINITY, s = 0.0f;
      for (int k = lane; k < G; k += 32) {
        const float2 x = __ldcg(part + k);
        lse2_fold(m, s, x.x, x.y);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, o), os = __shfl_xor_sync(0xffffffffu, s, o);
        lse2_fold(m, s, om, os);
      }
      if (lane == 0) p.lse_out[(size_t)b * P + i] = (m + log2f(s)) * 0.6931471805599453f;
    }
  }

  if (kLogits && p.lo_tma && warp == 2 && lane == 0) bulk_wait_all();  // the logits stores' writes
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool tmap_bf16(CUtensorMap* tm, const void* base, int rows, int cols, int box_rows) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
      return false;
    fn = (EncodeTiledFn)ptr;
  }
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int round16(int x) { return (x + 15) / 16 * 16; }

// fp32 [bs][P][V] view with a given batch stride (elements), box box_w x 1 x box_z.
bool tmap_f32_3d(CUtensorMap* tm, const void* base, int V, int P, int bs, int64_t bstride, int box_z, int box_w) {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess || q != cudaDriverEntryPointSuccess)
      return false;
    fn = (EncodeTiledFn)ptr;
  }
  cuuint64_t dims[3] = {(cuuint64_t)V, (cuuint64_t)P, (cuuint64_t)bs};
  cuuint64_t strides[2] = {(cuuint64_t)V * 4, (cuuint64_t)bstride * 4};
  cuuint32_t box[3] = {(cuuint32_t)box_w, 1, (cuuint32_t)box_z};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

uint32_t region_bytes(int g, int NBs) {
  // B_s in the S pass; in the W pass U16 (64 KB), then eight staged pairs of
  // L_base and noise boxes (16 rows of 528 bytes each): two tiles ahead at
  // batch 64.
  const uint32_t b = (uint32_t)(g / 64) * NBs * 128;
  const uint32_t boxes = 8u * 2u * 16u * 528u;
  return b > boxes ? b : boxes;
}

size_t batched_smem(int g, int NB, int NBs, int nu_max) {
  size_t s = 1024 + (size_t)kStages * kChunk + region_bytes(g, NBs);
  s += 8 * kStages * 2 + 8 + 8 + 8 + 16 + 16 + 16 + 16 + 16 + 16 * 12 + 64 + 64 + 16;
  s += (size_t)kMaxB * 3 * nu_max * 4 * 2 + (size_t)kMaxB * nu_max * 4 + (size_t)3 * nu_max * 4 + kMaxB * 4 +
       (size_t)4 * kMaxB * 8 + (size_t)4 * kMaxB * 8 + 128;
  return s;
}

}  // namespace

// A bf16 [rows, cols] matrix (W2 [V, 256]) as a 2D tensor map: boxes of 64
// columns x box_rows rows, 128-byte swizzle. Shared with the residual draw.
bool tmap_bf16_rows(CUtensorMap* tm, const void* base, int rows, int cols, int box_rows) {
  return tmap_bf16(tm, base, rows, cols, box_rows);
}

size_t batched_ws_bytes(int g) {
  // S16 [128][g] bf16, U16 [128][256] bf16, counters [3][P + 1] x 32 B (P <= 255),
  // then the per-CTA B_s images.
  const int G = num_sms();
  const int NBs = round16((kR + G - 1) / G + 3 * ((g + G - 1) / G));
  return (size_t)128 * g * 2 + (size_t)128 * kR * 2 + (size_t)3 * 256 * 32 + (size_t)G * (g / 64) * NBs * 128;
}

bool chain_batched_applies(const ChainArgs& a) {
  if (!chain_batched_shape_ok(a.dtype, a.bs, a.P, a.g, a.r, a.V)) return false;
  if (!a.s16 || !a.u16 || !a.ctr || !a.bimg) return false;
  // L_base / noise are staged by TMA: 16-byte aligned rows and bases.
  if (((uintptr_t)a.L_base & 15u)) return false;
  if (a.temperature > 0.0f && (((uintptr_t)a.gumbel & 15u) || (a.gumbel_bstride % 4) != 0)) return false;
  return true;
}

bool chain_batched_shape_ok(int dtype, int bs, int P, int g, int r, int V) {
  // Any batch up to 64 works; below 5 the dispatcher prefers the small-batch
  // kernel, except for the draft statistics, which only this kernel computes.
  if (dtype != DOMINO_BF16 || r != kR || bs < 1 || bs > kMaxB || (g % 64) != 0 || P > 255) return false;
  if ((V % 4) != 0) return false;
  const int G = num_sms();
  if (G < kKeyGroups * 16) return false;  // the keys region holds P x bs x num_sms words
  if ((int64_t)V / G + 5 > 256 * 128) return false;  // a lane's tile index fits in a byte
  const int nu_max = (g + G - 1) / G, ku_max = (kR + G - 1) / G;
  const int NBs = round16(ku_max + 3 * nu_max);
  if (NBs > 128) return false;  // tensor memory: S-pass accumulator in columns [0, 128)
  const int NB = round16(2 * bs);
  return batched_smem(g, NB, NBs, nu_max) <= 227 * 1024;
}

cudaError_t launch_chain_batched(const ChainArgs& a, cudaStream_t stream) {
  const int G = num_sms();
  BatP p;
  memset(&p, 0, sizeof(p));
  p.bs = a.bs; p.P = a.P; p.d = a.d; p.g = a.g; p.V = a.V;
  p.nu_max = (a.g + G - 1) / G;
  const int ku_max = (kR + G - 1) / G;
  p.NBs = round16(ku_max + 3 * p.nu_max);
  p.NB = round16(2 * a.bs);
  p.box_z = a.bs < 16 ? a.bs : 16;
  p.lg_pitch = a.logits_out != nullptr ? 512 : 528;
  p.reg_bytes = region_bytes(a.g, p.NBs);
  if (!tmap_bf16(&p.tm_w2, a.w2, a.V, kR, 128) || !tmap_bf16(&p.tm_s16, a.s16, 128, a.g, 128) ||
      !tmap_bf16(&p.tm_u16, a.u16, p.NB, kR, p.NB) ||
      !tmap_f32_3d(&p.tm_lb, a.L_base, a.V, a.P, a.bs, (int64_t)a.P * a.V, p.box_z, p.lg_pitch / 4))
    return cudaErrorInvalidValue;
  if (a.temperature > 0.0f) {
    if (!tmap_f32_3d(&p.tm_gm, a.gumbel, a.V, a.P, a.bs, a.gumbel_bstride, p.box_z, p.lg_pitch / 4))
      return cudaErrorInvalidValue;
  } else {
    p.tm_gm = p.tm_lb;  // never loaded
  }
  p.lo_tma = 0;
  p.tm_lo = p.tm_lb;  // never stored through unless lo_tma
  if (a.logits_out != nullptr && ((uintptr_t)a.logits_out & 15u) == 0 &&
      tmap_f32_3d(&p.tm_lo, a.logits_out, a.V, a.P, a.bs, (int64_t)a.P * a.V, p.box_z, 128))
    p.lo_tma = 1;
  p.gate_table = a.gate_table;
  p.w_hh = (const __nv_bfloat16*)a.w_hh; p.b_hh = (const __nv_bfloat16*)a.b_hh;
  p.w1 = (const __nv_bfloat16*)a.w1;
  p.L_base = a.L_base; p.P_h = a.P_h; p.anchor = a.anchor;
  p.temperature = a.temperature;
  p.inv_temperature = a.temperature > 0.0f ? 1.0f / a.temperature : 0.0f;
  p.gumbel = a.gumbel; p.gumbel_bstride = a.gumbel_bstride;
  p.force = a.force; p.tokens = a.tokens; p.logits_out = a.logits_out;
  p.u_out = a.u_out; p.lse_out = a.lse_out; p.lse_part = a.lse_part;
  p.lse_c = 1.4426950408889634f / (a.temperature > 0.0f ? a.temperature : 1.0f);
  p.ctl = a.ctl; p.s16 = a.s16; p.u16 = a.u16; p.keys = a.keys; p.ctr = a.ctr; p.bimg = a.bimg;
  p.timeout_ns = wait_timeout_ns();
  const size_t smem = batched_smem(a.g, p.NB, p.NBs, p.nu_max);
  const void* fn = a.logits_out != nullptr ? (const void*)chain_batched_kernel<true> : (const void*)chain_batched_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void* args[] = {(void*)&p};
  return cudaLaunchCooperativeKernel(fn, dim3(G), dim3(kThreads), args, smem, stream);
}

}  // namespace domino
