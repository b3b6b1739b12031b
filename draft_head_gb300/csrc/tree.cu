// DominoTree on sm_103a ("DominoTree: Conditional Tree-Structured Drafting with
// Domino for Speculative Decoding", "核心组件").
//
// 1. Top-M candidate select ("候选限制（Top-M）"): per row of L_base, the M best
//    (value desc, id asc). Each (value, id) pair becomes one distinct 64-bit
//    key, so the selection is an exact k-th-largest search: an 8-bit radix
//    select from the top byte down, where after each byte only the keys that
//    share the k-th key's digit go on (so the first pass, on registers, does
//    nearly all the work). Three passes per row: a threshold key from a
//    histogram of a sample of evenly spaced runs (about 2M of the row's keys
//    expected above it); one
//    streaming pass over the row that keeps the keys at or above it; the exact
//    select among those, sorted (bitonic). A row whose threshold kept fewer
//    than M keys, or more than the list holds, is selected from scratch by a
//    single CTA streaming it behind a running threshold, so the result is exact
//    for any input.
//
// 2. Best-first build ("条件评分的最佳优先堆"), one persistent kernel, all
//    requests in lockstep, no grid barrier. Node ids are assigned in pop
//    order and node t is expanded right after it is popped, so iteration t of
//    every request expands its node t. CTA b < bs owns request b; the other
//    CTAs (workers) form Q groups (4, 2 or 1, the most that fit in shared
//    memory), group q serving requests [q bs / Q, (q + 1) bs / Q) with the
//    GRU's hidden units split among its workers.
//      G  each worker runs the GRU step of node t for its units and its
//         group's requests: input-side gates from the prepared table,
//         hidden-side sums W_hh S_parent made when the parent's state was.
//         It adds its units' share of the bottleneck, W1_s[k, units]
//         S_t[units] for every entry k, into node t's accumulators: 64-bit
//         words holding (sum in 2^-32 fixed point) << 16 plus a count of
//         contributions, so the sum is exact and order-free and the count
//         says when it is complete. It stores S_t in words that are nonzero
//         once written, and then, in the shadow of the owners' expansion,
//         reads S_t of the group's requests back from every worker and forms
//         W_hh S_t for its units: the sums node t's children will need.
//      E  the owner of request b polls the r accumulators until their counts
//         are full, u = SiLU(P_h[depth] + .), scores its M candidates
//         l_c = L_base[depth, c] + W2[c] u, takes the log-softmax over the
//         slice and keeps the children, sorted by (score desc, token asc),
//         as node t's sibling group. The best-first heap is the set of group
//         heads: the pop takes the best head under (score desc, parent asc),
//         the same order a binary heap over all pushed children gives. The
//         popped node goes out in its own slot with a release flag that the
//         group's workers wait on before iteration t + 1.
#include "common.cuh"

namespace domino {

namespace {

constexpr int kSelThreads = 512;
constexpr int kTile = 4 * kSelThreads;  // range_topk tile: 4 consecutive values per thread
constexpr int kAhead = 4;               // range_topk tiles in flight per thread
constexpr int kCap = 4096;              // range_topk kept-key buffer; 8 per thread
constexpr int kSample = 4096;           // threshold sample per row; 8 per thread
constexpr int kListCap = 4096;          // candidates per row at or above the threshold
constexpr int kFilterThreads = 256;
constexpr int kFilterSeg = 16384;       // values per filter CTA
constexpr int kFilterAhead = 4;         // 16-byte loads in flight per filter thread
constexpr int kFilterStage = 2048;      // survivors staged per filter CTA before one global append

// Histogram increment; digit 256 means "no key".
__device__ __forceinline__ void hist_add(unsigned* hist, unsigned digit) {
  if (digit < 256u) atomicAdd(&hist[digit], 1u);
}

// Append `key` (when `want`) to list[*count]: one atomic per warp. Called by
// all 32 lanes.
__device__ __forceinline__ void warp_append(bool want, unsigned long long key, unsigned long long* list,
                                            unsigned* count) {
  const unsigned m = __ballot_sync(0xffffffffu, want);
  if (!m) return;
  const int lane = threadIdx.x & 31, leader = __ffs(m) - 1;
  unsigned at = 0u;
  if (lane == leader) at = atomicAdd(count, (unsigned)__popc(m));
  at = __shfl_sync(0xffffffffu, at, leader);
  if (want) list[at + __popc(m & ((1u << lane) - 1u))] = key;
}

// Warp 0: the digit holding the `need`-th largest key of the histogram.
// misc[0] = digit, misc[1] = how many keys of that digit are still needed,
// misc[3] = keys with that digit.
__device__ __forceinline__ void find_digit(const unsigned* hist, unsigned need, unsigned* misc) {
  const int lane = threadIdx.x & 31;
  unsigned local[8];
  unsigned s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    local[j] = hist[lane * 8 + j];
    s += local[j];
  }
  unsigned suf = s;  // keys in the bins of lanes >= lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += t;
  }
  const unsigned above = suf - s;
  if (above < need && need <= suf) {
    unsigned cum = above;
    for (int j = 7; j >= 0; --j) {
      if (cum + local[j] >= need) {
        misc[0] = (unsigned)(lane * 8 + j);
        misc[1] = need - cum;
        misc[3] = local[j];
        break;
      }
      cum += local[j];
    }
  }
}

// The k largest of the distinct nonzero keys held KPT per thread (zero = no
// key; at least k keys exist) -> out[0..k), unordered. Radix select on the
// key bytes from the top; after each byte the keys above the k-th key's
// digit are final, and only the keys sharing its digit go on to the next
// byte (compacted into a shared-memory list), so later passes touch few keys.
template <int KPT>
__device__ void select_topk(const unsigned long long (&rk)[KPT], unsigned k, unsigned long long* out,
                            unsigned long long* bufA, unsigned long long* bufB, unsigned* hist, unsigned* misc) {
  const int tid = threadIdx.x, nt = blockDim.x;
  for (int i = tid; i < 256; i += nt) hist[i] = 0u;
  if (tid == 0) { misc[2] = 0u; misc[4] = 0u; }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < KPT; ++j) hist_add(hist, rk[j] ? (unsigned)(rk[j] >> 56) : 256u);
  __syncthreads();
  if ((tid >> 5) == 0) find_digit(hist, k, misc);
  __syncthreads();
  unsigned dd = misc[0], need = misc[1], cnt = misc[3];
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const unsigned d = rk[j] ? (unsigned)(rk[j] >> 56) : 0u;
    warp_append(rk[j] && d > dd, rk[j], out, &misc[2]);
    warp_append(rk[j] && d == dd, rk[j], bufA, &misc[4]);
  }
  __syncthreads();
  unsigned long long* list = bufA;
  unsigned long long* other = bufB;
  for (int shift = 48; shift >= 0 && cnt > need; shift -= 8) {
    for (int i = tid; i < 256; i += nt) hist[i] = 0u;
    __syncthreads();
    for (unsigned i0 = 0; i0 < cnt; i0 += nt) {  // uniform trip count: full warps call hist_add
      const unsigned i = i0 + tid;
      hist_add(hist, i < cnt ? (unsigned)(list[i] >> shift) & 255u : 256u);
    }
    __syncthreads();
    if ((tid >> 5) == 0) find_digit(hist, need, misc);
    if (tid == 0) misc[4] = 0u;
    __syncthreads();
    dd = misc[0];
    for (unsigned i0 = 0; i0 < cnt; i0 += nt) {  // uniform trip count: full warps append
      const unsigned i = i0 + tid;
      const unsigned long long key = i < cnt ? list[i] : 0ull;
      const unsigned d = (unsigned)(key >> shift) & 255u;
      warp_append(i < cnt && d > dd, key, out, &misc[2]);
      warp_append(i < cnt && d == dd, key, other, &misc[4]);
    }
    __syncthreads();
    need = misc[1];
    cnt = misc[3];
    unsigned long long* t = list; list = other; other = t;
  }
  // The remaining keys sharing every byte with the k-th key are all in.
  const unsigned base = misc[2];
  for (unsigned i = tid; i < cnt && i < need; i += nt) out[base + i] = list[i];
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

// Four consecutive values of a row, from offset o (a multiple of 4): one
// 16-byte load when rows are 16-byte aligned, else four 4-byte loads.
__device__ __forceinline__ float4 load4(const float* src, int o, int len, bool vec) {
  if (vec && o + 3 < len) return __ldcs((const float4*)(src + o));
  float4 v;
  v.x = o < len ? __ldcs(src + o) : 0.0f;
  v.y = o + 1 < len ? __ldcs(src + o + 1) : 0.0f;
  v.z = o + 2 < len ? __ldcs(src + o + 2) : 0.0f;
  v.w = o + 3 < len ? __ldcs(src + o + 3) : 0.0f;
  return v;
}

// Top k keys of one row range [begin, begin + len) (values at src), exact, by
// one CTA: streams the range once, keeping in shared memory only keys above
// a running threshold tau, the k-th best key among those kept so far (no key
// below it can be in the top k). The first tile sets tau through an exact
// select on registers; later tiles arrive kAhead at a time and almost every
// value fails the threshold test, which a warp checks with one vote. When the
// buffer fills, an exact select shrinks it to the top k and raises tau.
// Leaves the top k keys (unordered) in buf[0..k).
__device__ void range_topk(const float* src, int len, int begin, unsigned k, bool vec, unsigned long long* buf,
                           unsigned long long* bufB, unsigned long long* outk, unsigned* hist, unsigned* misc,
                           unsigned* nbuf, unsigned long long* tau_s) {
  unsigned long long tau = 0ull;
  float tau_v = -INFINITY;
  if (threadIdx.x == 0) *nbuf = 0u;
  // Keep the top k of rk; tau = the k-th.
  auto reduce_to_k = [&](const unsigned long long (&rk)[kCap / kSelThreads]) {
    select_topk(rk, k, outk, buf, bufB, hist, misc);
    if (threadIdx.x < 32) {
      unsigned long long m = ~0ull;
      for (unsigned i = threadIdx.x; i < k; i += 32) m = outk[i] < m ? outk[i] : m;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long x = __shfl_xor_sync(0xffffffffu, m, o);
        m = x < m ? x : m;
      }
      if (threadIdx.x == 0) { *tau_s = m; *nbuf = k; }
    }
    for (unsigned i = threadIdx.x; i < k; i += kSelThreads) buf[i] = outk[i];
    __syncthreads();
    tau = *tau_s;
    tau_v = key_value(tau);
  };
  auto shrink = [&]() {
    const unsigned cnt = *nbuf;
    unsigned long long rk[kCap / kSelThreads];
#pragma unroll
    for (int j = 0; j < kCap / kSelThreads; ++j) {
      const unsigned i = threadIdx.x + (unsigned)j * kSelThreads;
      rk[j] = i < cnt ? buf[i] : 0ull;
    }
    reduce_to_k(rk);
  };
  const int ntiles = (len + kTile - 1) / kTile;
  float4 pf[kAhead];  // tiles 1 .. kAhead in flight while tile 0 sets tau
#pragma unroll
  for (int d = 0; d < kAhead; ++d) pf[d] = load4(src, (1 + d) * kTile + 4 * (int)threadIdx.x, len, vec);
  {
    const float4 v = load4(src, 4 * (int)threadIdx.x, len, vec);
    const float vv[4] = {v.x, v.y, v.z, v.w};
    unsigned long long rk[kCap / kSelThreads];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = 4 * (int)threadIdx.x + q;
      rk[q] = i < len ? value_id_key(vv[q], (uint32_t)(begin + i)) : 0ull;
    }
#pragma unroll
    for (int q = 4; q < kCap / kSelThreads; ++q) rk[q] = 0ull;
    __syncthreads();
    reduce_to_k(rk);
  }
  for (int t = 1; t < ntiles; t += kAhead) {
#pragma unroll
    for (int d = 0; d < kAhead; ++d) {
      const int tt = t + d;
      if (tt < ntiles) {  // uniform over the CTA
        const float4 v = pf[d];
        pf[d] = load4(src, (tt + kAhead) * kTile + 4 * (int)threadIdx.x, len, vec);
        const float vv[4] = {v.x, v.y, v.z, v.w};
        const int i0 = tt * kTile + 4 * (int)threadIdx.x;
        bool any = false;
#pragma unroll
        for (int q = 0; q < 4; ++q) any |= (i0 + q < len) && vv[q] >= tau_v;
        if (__any_sync(0xffffffffu, any)) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int i = i0 + q;
            unsigned long long key = 0ull;
            if (i < len && vv[q] >= tau_v) key = value_id_key(vv[q], (uint32_t)(begin + i));
            warp_append(key > tau, key, buf, nbuf);
          }
        }
        __syncthreads();
        if (*nbuf > (unsigned)(kCap - kTile)) shrink();
      }
    }
  }
  if (*nbuf > k) shrink();
}

// Pass 1, one CTA per row: a threshold key from a sample of S = min(n, 4096)
// values: 128 runs of 32 consecutive values (one 128-byte line each), evenly
// spaced over the row, so the pass reads 16 KB of the row rather than a
// sector of every line. The sample's keys go into a histogram of their top
// 12 bits; the threshold is the lower edge of the bin that holds the q-th best
// sample key, q chosen so that about 2k of the row's keys are expected at or
// above it (q = k when the sample is the whole row). Any threshold at or below
// the row's k-th key is correct; a higher one only costs a fallback in pass 3.
__global__ void __launch_bounds__(kSelThreads) topm_sample(const float* __restrict__ values, int n, int M,
                                                           unsigned long long* __restrict__ tau_out) {
  __shared__ unsigned hist[4096];
  __shared__ unsigned wsum[kSelThreads / 32];
  const int row = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int S = min(n, kSample);
  const unsigned k = (unsigned)min(M, n);
  const unsigned q = S == n ? k : min((unsigned)S, (unsigned)(((int64_t)2 * k * S + n - 1) / n) + 3u);
  const float* src = values + (size_t)row * n;
  for (int i = tid; i < 4096; i += kSelThreads) hist[i] = 0u;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kSample / kSelThreads; ++j) {
    const int sidx = tid + j * kSelThreads;
    if (sidx < S) {
      int i = sidx;
      if (S < n) {
        const int run = sidx >> 5, nruns = S >> 5;
        i = (int)(((int64_t)run * (n - 32) / (nruns - 1)) & ~(int64_t)31) + (sidx & 31);
      }
      atomicAdd(&hist[value_id_key(__ldg(src + i), (uint32_t)i) >> 52], 1u);
    }
  }
  __syncthreads();
  // Thread t owns bins [8t, 8t + 8); counts above a bin are suffix sums.
  unsigned b8[8], my = 0u;
#pragma unroll
  for (int j = 0; j < 8; ++j) { b8[j] = hist[8 * tid + j]; my += b8[j]; }
  unsigned suf = my;  // over lanes >= lane of this warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned t = __shfl_down_sync(0xffffffffu, suf, o);
    if (lane + o < 32) suf += t;
  }
  if (lane == 0) wsum[warp] = suf;
  __syncthreads();
  unsigned above = suf - my;
  for (int w = warp + 1; w < kSelThreads / 32; ++w) above += wsum[w];
  if (above < q && q <= above + my) {
    unsigned cum = above;
    for (int j = 7; j >= 0; --j) {
      if (cum + b8[j] >= q) {
        tau_out[row] = (unsigned long long)(8 * tid + j) << 52;
        break;
      }
      cum += b8[j];
    }
  }
}

// Pass 2, one CTA per (row, segment): every key at or above the row's
// threshold goes to the row's candidate list. Survivors are staged in shared
// memory (one shared atomic per warp) and appended with one global atomic per
// CTA; the count keeps running past the list's capacity (and a CTA whose
// stage overflows adds more than the capacity), which pass 3 detects.
__global__ void __launch_bounds__(kFilterThreads) topm_filter(const float* __restrict__ values, int n,
                                                              const unsigned long long* __restrict__ tau_in,
                                                              unsigned long long* __restrict__ lists,
                                                              unsigned* __restrict__ counts) {
  __shared__ unsigned long long stage[kFilterStage];
  __shared__ unsigned nstage, base_s;
  const int row = blockIdx.y, seg = blockIdx.x;
  const int begin = seg * kFilterSeg;
  const int len = min(kFilterSeg, n - begin);
  const float* src = values + (size_t)row * n + begin;
  const bool vec = (n & 3) == 0 && (((uintptr_t)values) & 15u) == 0;
  const unsigned long long tau = tau_in[row];
  const float tau_v = key_value(tau);
  if (threadIdx.x == 0) nstage = 0u;
  __syncthreads();
  constexpr int kStep = 4 * kFilterThreads;
  for (int t0 = 0; t0 < len; t0 += kFilterAhead * kStep) {
    float4 v[kFilterAhead];
#pragma unroll
    for (int d = 0; d < kFilterAhead; ++d) v[d] = load4(src, t0 + d * kStep + 4 * (int)threadIdx.x, len, vec);
#pragma unroll
    for (int d = 0; d < kFilterAhead; ++d) {
      const float vv[4] = {v[d].x, v[d].y, v[d].z, v[d].w};
      const int i0 = t0 + d * kStep + 4 * (int)threadIdx.x;
      bool any = false;
#pragma unroll
      for (int q = 0; q < 4; ++q) any |= (i0 + q < len) && vv[q] >= tau_v;
      if (__any_sync(0xffffffffu, any)) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i = i0 + q;
          unsigned long long key = 0ull;
          if (i < len && vv[q] >= tau_v) key = value_id_key(vv[q], (uint32_t)(begin + i));
          const bool keep = key >= tau && key != 0ull;
          const unsigned m = __ballot_sync(0xffffffffu, keep);
          if (m) {
            const int lane = threadIdx.x & 31, leader = __ffs(m) - 1;
            unsigned at = 0u;
            if (lane == leader) at = atomicAdd(&nstage, (unsigned)__popc(m));
            at = __shfl_sync(0xffffffffu, at, leader);
            const unsigned pos = at + __popc(m & ((1u << lane) - 1u));
            if (keep && pos < (unsigned)kFilterStage) stage[pos] = key;
          }
        }
      }
    }
  }
  __syncthreads();
  const unsigned ns = nstage;
  if (ns == 0u) return;
  // An overflowed stage pushes the row's count past the list capacity.
  if (threadIdx.x == 0) base_s = atomicAdd(counts + row, ns <= (unsigned)kFilterStage ? ns : (unsigned)kListCap + 1u);
  __syncthreads();
  const unsigned base = base_s;
  if (ns > (unsigned)kFilterStage) return;
  unsigned long long* list = lists + (size_t)row * kListCap;
  for (unsigned i = threadIdx.x; i < ns; i += kFilterThreads)
    if (base + i < (unsigned)kListCap) list[base + i] = stage[i];
}

// Pass 3, one CTA per row: the exact top M of the row's candidates, sorted
// (value desc, id asc). When the sample's threshold left fewer than M
// candidates or more than the list holds, the row is selected from scratch
// (range_topk over the whole row), so the result is exact for any input.
// Leaves the row's count at zero for the next call.
__global__ void __launch_bounds__(kSelThreads) topm_final(const float* __restrict__ values, int n, int M,
                                                          const unsigned long long* __restrict__ lists,
                                                          unsigned* __restrict__ counts,
                                                          int32_t* __restrict__ ids, float* __restrict__ vals) {
  extern __shared__ unsigned long long shf[];
  __shared__ unsigned hist[256];
  __shared__ unsigned misc[8];
  __shared__ unsigned nbuf;
  __shared__ unsigned long long tau_s;
  const int row = blockIdx.x;
  int np = 1;
  while (np < M) np <<= 1;
  unsigned long long* buf = shf;                // [kCap]
  unsigned long long* bufB = shf + kCap;        // [kCap]
  unsigned long long* outk = shf + 2 * kCap;    // [256]
  const unsigned cnt = counts[row];
  const unsigned k = (unsigned)M;
  for (int i = threadIdx.x; i < np; i += kSelThreads) outk[i] = 0ull;
  __syncthreads();
  if (cnt >= k && cnt <= (unsigned)kListCap) {
    const unsigned long long* list = lists + (size_t)row * kListCap;
    unsigned long long rk[kListCap / kSelThreads];
#pragma unroll
    for (int j = 0; j < kListCap / kSelThreads; ++j) {
      const unsigned i = threadIdx.x + (unsigned)j * kSelThreads;
      rk[j] = i < cnt ? list[i] : 0ull;
    }
    select_topk(rk, k, outk, buf, bufB, hist, misc);
  } else {
    const bool vec = (n & 3) == 0 && (((uintptr_t)values) & 15u) == 0;
    range_topk(values + (size_t)row * n, n, 0, k, vec, buf, bufB, outk, hist, misc, &nbuf, &tau_s);
    for (unsigned i = threadIdx.x; i < k; i += kSelThreads) outk[i] = buf[i];
    __syncthreads();
  }
  block_bitonic_desc(outk, np);
  for (int i = threadIdx.x; i < M; i += kSelThreads) {
    const unsigned long long key = outk[i];
    ids[(size_t)row * M + i] = (int32_t)key_id(key);
    if (vals) vals[(size_t)row * M + i] = key_value(key);
  }
  if (threadIdx.x == 0) counts[row] = 0u;
}

// ---------------------------------------------------------------------------
// Best-first build.
// ---------------------------------------------------------------------------
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kStageAhead = 8;  // tagged 16-byte loads in flight per thread while staging S_t
constexpr float kInvFix = 1.0f / 4294967296.0f;  // bottleneck sums in 2^-32 fixed point (exact power of two)
__device__ __forceinline__ int ld_relaxed_s32(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_s32(int* p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Wait (bounded) until *tag == want, then acquire.
__device__ bool wait_tag(const int* tag, int want, Ctl* ctl, uint64_t timeout_ns) {
  if (ld_relaxed_s32(tag) != want) {
    const uint64_t t0 = globaltimer_ns();
    unsigned spins = 0;
    while (ld_relaxed_s32(tag) != want) {
      if ((++spins & 63u) == 0) {
        if (ld_volatile_u32(&ctl->abort)) return false;
        if (globaltimer_ns() - t0 > timeout_ns) { dev_abort(ctl, DEV_ERR_TIMEOUT); return false; }
      }
    }
  }
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  return true;
}

__device__ __forceinline__ void st_relaxed_u32(unsigned* p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint4 ld_relaxed_v4_u32(const unsigned* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}
// The bits of v, with +0 replaced by -0 (same arithmetic), so never zero.
__device__ __forceinline__ unsigned nonzero_bits(float v) {
  const unsigned u = __float_as_uint(v);
  return u ? u : 0x80000000u;
}

// Four consecutive weights as fp32 (one 8- or 16-byte shared-memory load).
__device__ __forceinline__ float4 load4w(const __nv_bfloat16* p) {
  const uint2 v = *(const uint2*)p;
  return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u), __uint_as_float(v.y << 16),
                     __uint_as_float(v.y & 0xFFFF0000u));
}
__device__ __forceinline__ float4 load4w(const float* p) { return *(const float4*)p; }

template <typename WT>
struct TreeP {
  int bs, P, d, g, r, V, N, M, Mp, nu_max;
  int Q;        // worker groups; group q serves requests [q bs / Q, (q + 1) bs / Q)
  int bsq_max;  // requests of the largest group
  int RB;      // requests whose node states are staged in shared memory at a time
  int sp_bytes;  // bytes of the staging buffer (states for workers; candidates' rows for owners)
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
  // Zero before each build. State words are written once, so a nonzero
  // word is this build's value (+0 is stored as -0, which computes the
  // same). Each bottleneck accumulator receives one counted fixed-point
  // partial from every worker with hidden units.
  unsigned* tstates;              // [bs][N][g] S_node
  unsigned long long* uacc;       // [bs][N][r] W1_s S_node: (sum of partials * 2^32) << 16 | count
  int32_t* cur;     // [bs][N + 1][4]: token, parent, expand, ready flag of each published node
  uint64_t timeout_ns;
  float inv_tau;  // 1 / scoring temperature
};

// Stage S_t of requests b0 .. b0 + nb - 1 into sp_s ([nb][g] fp32). 16-byte
// loads (four tagged words), kStageAhead in flight per thread; the groups
// with a word not written yet are loaded again together until none is left
// (bounded). A request that does not expand gets zeros. False on timeout or
// abort.
template <typename WT>
__device__ __forceinline__ bool stage_states(const TreeP<WT>& p, int t, int b0, int nb, const int* cur_s,
                                             float* sp_s) {
  const int g = p.g, N = p.N;
  const int n4 = nb * (g / 4);
  for (int base = threadIdx.x; base < n4; base += kStageAhead * kThreads) {
    uint4 x[kStageAhead];
    unsigned pend = 0u;
#pragma unroll
    for (int u = 0; u < kStageAhead; ++u) {
      const int idx = base + u * kThreads;
      x[u] = make_uint4(0u, 0u, 0u, 0u);
      if (idx < n4) {
        const int bl = idx / (g / 4), k4 = idx - bl * (g / 4);
        if (cur_s[(b0 + bl) * 4 + 2]) {
          x[u] = ld_relaxed_v4_u32(p.tstates + ((size_t)(b0 + bl) * N + t) * g + 4 * k4);
          pend |= 1u << u;
        } else {
          ((float4*)(sp_s + (size_t)bl * g))[k4] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
      }
    }
    const uint64_t t0 = globaltimer_ns();
    for (unsigned round = 0; pend; ++round) {
      unsigned again = 0u;
#pragma unroll
      for (int u = 0; u < kStageAhead; ++u) {
        if (!(pend & (1u << u))) continue;
        const int idx = base + u * kThreads;
        const int bl = idx / (g / 4), k4 = idx - bl * (g / 4);
        if (x[u].x && x[u].y && x[u].z && x[u].w)
          ((float4*)(sp_s + (size_t)bl * g))[k4] = make_float4(
              __uint_as_float(x[u].x), __uint_as_float(x[u].y), __uint_as_float(x[u].z), __uint_as_float(x[u].w));
        else
          again |= 1u << u;
      }
      pend = again;
      if (!pend) break;
      if ((round & 15u) == 15u) {
        if (ld_volatile_u32(&p.ctl->abort)) return false;
        if (globaltimer_ns() - t0 > p.timeout_ns) {
          dev_abort(p.ctl, DEV_ERR_TIMEOUT);
          return false;
        }
      }
#pragma unroll
      for (int u = 0; u < kStageAhead; ++u) {
        if (!(pend & (1u << u))) continue;
        const int idx = base + u * kThreads;
        const int bl = idx / (g / 4), k4 = idx - bl * (g / 4);
        x[u] = ld_relaxed_v4_u32(p.tstates + ((size_t)(b0 + bl) * N + t) * g + 4 * k4);
      }
    }
  }
  return true;
}

// After a bulk copy of node t's states of requests b0 .. b0 + nb - 1 into
// sp_s: the 16-byte groups that arrived with a word another worker had not
// written yet (zero) are loaded again until complete (bounded). False on
// timeout or abort.
template <typename WT>
__device__ __forceinline__ bool complete_states(const TreeP<WT>& p, int t, int b0, int nb, const int* cur_s,
                                                float* sp_s) {
  const int g = p.g, N = p.N;
  for (int idx = threadIdx.x; idx < nb * (g / 4); idx += kThreads) {
    const int bl = idx / (g / 4), k4 = idx - bl * (g / 4);
    if (!cur_s[(b0 + bl) * 4 + 2]) continue;
    uint4* d = (uint4*)(sp_s + (size_t)bl * g) + k4;
    uint4 x = *d;
    if (x.x && x.y && x.z && x.w) continue;
    const unsigned* src = p.tstates + ((size_t)(b0 + bl) * N + t) * g + 4 * k4;
    const uint64_t t0 = globaltimer_ns();
    for (unsigned round = 0;; ++round) {
      x = ld_relaxed_v4_u32(src);
      if (x.x && x.y && x.z && x.w) break;
      if ((round & 15u) == 15u) {
        if (ld_volatile_u32(&p.ctl->abort)) return false;
        if (globaltimer_ns() - t0 > p.timeout_ns) {
          dev_abort(p.ctl, DEV_ERR_TIMEOUT);
          return false;
        }
      }
    }
    *d = x;
  }
  return true;
}

template <typename WT>
__global__ void __launch_bounds__(kThreads, 1) tree_kernel(const __grid_constant__ TreeP<WT> p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int G = gridDim.x, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bs = p.bs, g = p.g, r = p.r, P = p.P, N = p.N, M = p.M;
  // CTAs 0..bs-1 own one request each and no hidden units. The other G - bs
  // CTAs (the workers) form Q groups: group q serves requests
  // [q bs / Q, (q + 1) bs / Q) and its workers split the hidden units, so a
  // worker reads and adds into the states and accumulators of its group's
  // requests only.
  const int nw = G - bs, Q = p.Q;
  const bool owner = c < bs;
  // (32-bit arithmetic: g times the CTA count stays far below 2^31.)
  int qg = 0;
  if (owner) {
    while ((qg + 1) * bs / Q <= c) ++qg;
  } else {
    while ((qg + 1) * nw / Q <= c - bs) ++qg;
  }
  const int bq0 = qg * bs / Q, bq1 = (qg + 1) * bs / Q;
  const int bsq = bq1 - bq0, bsq_max = p.bsq_max;
  const int wq0 = qg * nw / Q, nwq = (qg + 1) * nw / Q - wq0;
  const int cw = owner ? -1 : c - bs - wq0;  // worker index within the group
  const int j0 = cw >= 0 ? g * cw / nwq : 0;
  const int j1 = cw >= 0 ? g * (cw + 1) / nwq : 0;
  const int nu = j1 - j0;
  const int nu_max = p.nu_max;
  const unsigned long long n_contrib = (unsigned long long)min(nwq, g);  // the group's workers with units
  // A node's accumulator holds n_contrib partials (times 2^32, shifted left
  // 16 bits) in a signed 64-bit word: in range while their sum stays below
  // 2^15 in magnitude; 2^14 / n_contrib per partial keeps a factor two.
  const float part_limit = 16384.0f / (float)(n_contrib ? n_contrib : 1ull);

  uint64_t* wbar = (uint64_t*)smem;  // completion of the W_hh bulk copies
  uint64_t* sbar = wbar + 1;         // completion of a node's state rows, copied in bulk
  WT* whh_s = (WT*)(smem + 16);
  size_t off = 16 + (((size_t)3 * nu_max * g * sizeof(WT) + 15) & ~(size_t)15);
  WT* w1c_s = (WT*)(smem + off); off += ((size_t)nu_max * r * sizeof(WT) + 15) & ~(size_t)15;  // [jj][k] W1_s[k, j0 + jj]
  float* bhh_s = (float*)(smem + off); off += (size_t)3 * nu_max * 4;
  off = (off + 15) & ~(size_t)15;  // u_s is read as float4
  float* u_s = (float*)(smem + off); off += (size_t)r * 4;
  float* lg_s = (float*)(smem + off); off += (size_t)p.Mp * 4;

  int* ndep_s = (int*)(smem + off); off += (size_t)(N + 1) * 4;
  float* nsc_s = (float*)(smem + off); off += (size_t)(N + 1) * 4;
  int* misc_s = (int*)(smem + off); off += 16 * 4;
  int* fail_s = misc_s + 8;
  int* cur_s = (int*)(smem + off); off += (size_t)bs * 4 * 4;          // [b]: token, parent, expand
  // Per request of the group (index b - bq0):
  float* gi_s = (float*)(smem + off); off += (size_t)bsq_max * 3 * nu_max * 4;      // [3 nu] gate-table values
  float* ghn_s = (float*)(smem + off); off += (size_t)bsq_max * N * 3 * nu_max * 4;  // [node][3 nu] W_hh S_node
  float* sown_s = (float*)(smem + off); off += (size_t)bsq_max * N * nu_max * 4;     // [node][nu] S_node, owned
  off = (off + 15) & ~(size_t)15;
  float* sp_s = (float*)(smem + off); off += (size_t)p.sp_bytes;        // [RB][g] node t's states (staged)
  off = (off + 7) & ~(size_t)7;
  unsigned long long* hbest_s = (unsigned long long*)(smem + off); off += (size_t)(N + 1) * 8;  // group heads
  unsigned long long* grp_s = (unsigned long long*)(smem + off);  // [N][M] sibling groups

  // Weight slices into shared memory: W_hh rows q g + j0 + jj (gate q,
  // owned unit jj) by bulk copy, first needed at the end of the root's
  // iteration (the root has no parent), and the W1_s columns of the owned
  // units. Rows are 16-byte aligned: the head's pointers are, and g * the
  // weight size is a multiple of 16.
  if (threadIdx.x == 0) {
    mbar_init(wbar, 1);
    mbar_init(sbar, 1);
    mbar_fence_init();
    if (nu > 0) {
      const uint32_t row_bytes = (uint32_t)(g * sizeof(WT));
      mbar_expect_tx(wbar, row_bytes * 3u * (uint32_t)nu);
      for (int row = 0; row < 3 * nu; ++row) {
        const int q = row / nu, jj = row - q * nu;
        bulk_copy_g2s(whh_s + (size_t)row * g, p.w_hh + (size_t)(q * g + j0 + jj) * g, row_bytes, wbar);
      }
    }
  }
  bool whh_ready = false;
  uint32_t sphase = 0u;  // parity of sbar's next phase
  for (int idx = threadIdx.x; idx < nu * r; idx += kThreads) {
    const int jj = idx / r, k = idx - jj * r;
    w1c_s[idx] = p.w1[(size_t)k * (p.d + g) + p.d + j0 + jj];
  }
  for (int idx = threadIdx.x; idx < 3 * nu; idx += kThreads) {
    const int q = idx / nu, jj = idx - q * nu;
    bhh_s[idx] = to_f(p.b_hh[q * g + j0 + jj]);
  }
  if (threadIdx.x == 0) *fail_s = 0;
  // Request state lives with CTA b (b < bs): root = node 0.
  const int b_own = c;
  if (owner) {
    for (int k = threadIdx.x; k <= N; k += kThreads) {
      hbest_s[k] = 0ull;
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

  for (int t = 0; t < N; ++t) {
    // ---------------- G: node t of the requests this CTA serves (an owner:
    // its own). Its token, parent and whether it expands come from the
    // owner's publication after iteration t - 1 (acquired; the root at t = 0).
    const int wb0 = owner ? c : bq0, wb1 = owner ? c + 1 : bq1;
    for (int b = wb0 + (int)threadIdx.x; b < wb1; b += kThreads) {
      int tok, parent, expand;
      if (t == 0) {
        tok = p.anchor[b];
        if (tok < 0 || tok >= p.V) tok = 0;
        parent = -1;
        expand = P > 0;
      } else {
        const int* cb = p.cur + ((size_t)b * (N + 1) + t) * 4;
        if (!wait_tag(cb + 3, 1, p.ctl, p.timeout_ns)) *fail_s = 1;
        tok = ld_relaxed_s32(cb + 0);
        parent = ld_relaxed_s32(cb + 1);
        expand = ld_relaxed_s32(cb + 2);
      }
      cur_s[b * 4 + 0] = tok;
      cur_s[b * 4 + 1] = parent;
      cur_s[b * 4 + 2] = expand;
    }
    __syncthreads();
    if (*fail_s) return;
    if (nu > 0) {
      // ---------------- worker: node t's GRU step for its units. Input side
      // from the prepared table; hidden side W_hh S_parent from the sums made
      // when the parent's state was (zero at the root). S_t goes out in
      // words that carry the node's tag.
      for (int idx = threadIdx.x; idx < bsq * 3 * nu; idx += kThreads) {
        const int bl = idx / (3 * nu), rem = idx - bl * 3 * nu, q = rem / nu, jj = rem - q * nu;
        const int b = bq0 + bl;
        if (cur_s[b * 4 + 2])
          gi_s[bl * 3 * nu_max + rem] = __ldg(p.gate_table + (size_t)cur_s[b * 4 + 0] * 3 * g + q * g + j0 + jj);
      }
      __syncthreads();
      for (int idx = threadIdx.x; idx < bsq * nu; idx += kThreads) {
        const int bl = idx / nu, jj = idx - bl * nu, b = bq0 + bl;
        if (!cur_s[b * 4 + 2]) continue;
        const int par = cur_s[b * 4 + 1];
        float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, h = 0.0f;
        if (par >= 0) {
          const float* gh = ghn_s + ((size_t)bl * N + par) * 3 * nu_max;
          a0 = gh[jj];
          a1 = gh[nu + jj];
          a2 = gh[2 * nu + jj];
          h = sown_s[((size_t)bl * N + par) * nu_max + jj];
        }
        const float* gi = gi_s + bl * 3 * nu_max;
        const float rg = sigmoidf_(gi[jj] + a0 + bhh_s[jj]);
        const float zg = sigmoidf_(gi[nu + jj] + a1 + bhh_s[nu + jj]);
        const float ng = tanhf(gi[2 * nu + jj] + rg * (a2 + bhh_s[2 * nu + jj]));
        const float hn = (1.0f - zg) * ng + zg * h;
        if (DCHECK(p.ctl, b < p.bs && t < N && j0 + jj < g))
          st_relaxed_u32(p.tstates + ((size_t)b * N + t) * g + j0 + jj, nonzero_bits(hn));
        sown_s[((size_t)bl * N + t) * nu_max + jj] = hn;
      }
      __syncthreads();  // node t's owned units are in sown_s
      // When the group's requests fit one staging block, node t's state
      // rows start toward shared memory now, by bulk copy, in the shadow of
      // the partials below; words another worker has not written yet arrive
      // as zero and are loaded again after.
      const bool bulk_stage = p.RB >= bsq;  // CTA-uniform
      if (bulk_stage && threadIdx.x == 0) {
        asm volatile("fence.proxy.async;" ::: "memory");  // this CTA's own words, just written
        uint32_t bytes = 0u;
        for (int bl = 0; bl < bsq; ++bl)
          if (cur_s[(bq0 + bl) * 4 + 2]) bytes += (uint32_t)g * 4u;
        mbar_expect_tx(sbar, bytes);
        for (int bl = 0; bl < bsq; ++bl)
          if (cur_s[(bq0 + bl) * 4 + 2])
            bulk_copy_g2s(sp_s + (size_t)bl * g, p.tstates + ((size_t)(bq0 + bl) * N + t) * g, (uint32_t)g * 4u,
                          sbar);
      }
      // Bottleneck partials of the owned units, sum over jj of
      // W1_s[k, j0 + jj] S_t[b, j0 + jj] for every expanding request b of
      // the group and entry k, added in 2^-32 fixed point, shifted left 16
      // and plus one, to node t's accumulator (fire-and-forget atomics).
      // Integer sums are exact, so the total does not depend on the order
      // the adds land in. A thread takes one entry k for up to four
      // requests: one W1_s load feeds four independent FMA chains, and a
      // group of up to eight requests issues every request's adds in one
      // round (an owner waits for the last of its group's workers).
      for (int idx = threadIdx.x; idx < (bsq + 3) / 4 * r; idx += kThreads) {
        const int rq = idx / r, k = idx - rq * r;
        int bl[4];
        bool ex[4];
        const float* sv[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          bl[q] = min(4 * rq + q, bsq - 1);
          ex[q] = 4 * rq + q < bsq && cur_s[(bq0 + bl[q]) * 4 + 2] != 0;
          sv[q] = sown_s + ((size_t)bl[q] * N + t) * nu_max;
        }
        if (!(ex[0] || ex[1] || ex[2] || ex[3])) continue;
        float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
        for (int jj = 0; jj < nu; ++jj) {
          const float w = to_f(w1c_s[jj * r + k]);
#pragma unroll
          for (int q = 0; q < 4; ++q) part[q] = fmaf(w, sv[q][jj], part[q]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (ex[q])
            atomicAdd(p.uacc + ((size_t)(bq0 + bl[q]) * N + t) * r + k,
                      ((unsigned long long)fix32_checked(part[q], part_limit, p.ctl) << 16) + 1ull);
      }
      // S_t of the group's requests, RB at a time, for W_hh S_t of the
      // owned units: the hidden-side gate sums of node t's future children
      // (in the shadow of the owners' expansion).
      for (int b0 = bq0; b0 < bq1; b0 += p.RB) {
        const int nb = min(p.RB, bq1 - b0);
        __syncthreads();  // sp_s is free (the previous reads are done)
        if (bulk_stage) {
          if (!mbar_wait(sbar, sphase, nullptr, p.ctl, p.timeout_ns)) {
            dev_abort(p.ctl, DEV_ERR_TIMEOUT);
            *fail_s = 1;
          }
          sphase ^= 1u;
          if (!complete_states(p, t, b0, nb, cur_s, sp_s)) *fail_s = 1;
        } else if (!stage_states(p, t, b0, nb, cur_s, sp_s)) {
          *fail_s = 1;
        }
        __syncthreads();
        if (!whh_ready) {  // once: the W_hh rows have landed
          if (!mbar_wait(wbar, 0u, nullptr, p.ctl, p.timeout_ns)) {
            dev_abort(p.ctl, DEV_ERR_TIMEOUT);
            *fail_s = 1;
          }
          whh_ready = true;
        }
        // Warp work item: one owned unit for a block of up to 8 requests, so
        // the unit's three W_hh rows are read once per block; 24 dots per
        // lane, one transposing reduction.
        const int nblk = (nb + 7) / 8;
        for (int wi = warp; wi < nu * nblk; wi += kWarps) {
          const int jj = wi / nblk, rb0 = (wi - jj * nblk) * 8;
          const int nr = min(8, nb - rb0);
          bool pr[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) pr[q] = q < nr && cur_s[(b0 + rb0 + q) * 4 + 2] != 0;
          float acc[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
          const WT* wr0 = whh_s + (size_t)(0 * nu + jj) * g;
          const WT* wr1 = whh_s + (size_t)(1 * nu + jj) * g;
          const WT* wr2 = whh_s + (size_t)(2 * nu + jj) * g;
          bool all8 = true;
#pragma unroll
          for (int q = 0; q < 8; ++q) all8 = all8 && pr[q];
          if (all8) {  // warp-uniform: the common case, no per-request branches
            for (int k = 4 * lane; k < g; k += 128) {
              const float4 x0 = load4w(wr0 + k), x1 = load4w(wr1 + k), x2 = load4w(wr2 + k);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const float4 sv = *(const float4*)(sp_s + (size_t)(rb0 + q) * g + k);
                acc[3 * q + 0] = fmaf(x0.x, sv.x, fmaf(x0.y, sv.y, fmaf(x0.z, sv.z, fmaf(x0.w, sv.w, acc[3 * q + 0]))));
                acc[3 * q + 1] = fmaf(x1.x, sv.x, fmaf(x1.y, sv.y, fmaf(x1.z, sv.z, fmaf(x1.w, sv.w, acc[3 * q + 1]))));
                acc[3 * q + 2] = fmaf(x2.x, sv.x, fmaf(x2.y, sv.y, fmaf(x2.z, sv.z, fmaf(x2.w, sv.w, acc[3 * q + 2]))));
              }
            }
          } else
          for (int k = 4 * lane; k < g; k += 128) {
            const float4 x0 = load4w(wr0 + k), x1 = load4w(wr1 + k), x2 = load4w(wr2 + k);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              if (!pr[q]) continue;  // warp-uniform
              const float4 sv = *(const float4*)(sp_s + (size_t)(rb0 + q) * g + k);
              acc[3 * q + 0] = fmaf(x0.x, sv.x, fmaf(x0.y, sv.y, fmaf(x0.z, sv.z, fmaf(x0.w, sv.w, acc[3 * q + 0]))));
              acc[3 * q + 1] = fmaf(x1.x, sv.x, fmaf(x1.y, sv.y, fmaf(x1.z, sv.z, fmaf(x1.w, sv.w, acc[3 * q + 1]))));
              acc[3 * q + 2] = fmaf(x2.x, sv.x, fmaf(x2.y, sv.y, fmaf(x2.z, sv.z, fmaf(x2.w, sv.w, acc[3 * q + 2]))));
            }
          }
          // Transposing reduction of 32 values: afterwards lane i holds the
          // warp sum of acc[i].
#pragma unroll
          for (int w = 16; w >= 1; w >>= 1) {
            const bool up = lane & w;
#pragma unroll
            for (int i = 0; i < w; ++i) {
              const float send = up ? acc[i] : acc[i + w];
              const float keep = up ? acc[i + w] : acc[i];
              acc[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
            }
          }
          const int ql = lane & 7;
          const float a0 = __shfl_sync(0xffffffffu, acc[0], 3 * ql);
          const float a1 = __shfl_sync(0xffffffffu, acc[0], 3 * ql + 1);
          const float a2 = __shfl_sync(0xffffffffu, acc[0], 3 * ql + 2);
          if (lane < nr) {
            const int b = b0 + rb0 + lane;
            if (cur_s[b * 4 + 2]) {
              float* gh = ghn_s + ((size_t)(b - bq0) * N + t) * 3 * nu_max;
              gh[jj] = a0;
              gh[nu + jj] = a1;
              gh[2 * nu + jj] = a2;
            }
          }
        }
      }
      __syncthreads();
    }

    // ---------------- E: the owner of request b expands node t (once every
    // CTA's contribution is in), pops node t + 1 and publishes it.
    if (owner) {
      const int b = b_own;
      const bool expand = cur_s[b * 4 + 2] != 0;
      const int dep = ndep_s[t];
      if (expand) {
        // While the workers run node t's GRU step, stage what the expansion
        // reads: the candidates' ids, their L_base values, their W2 rows
        // (into the state buffer, which an owner does not use) and P_h.
        const int32_t* C = p.cand + ((size_t)b * P + dep) * M;
        const size_t w2c_bytes = ((size_t)M * r * sizeof(WT) + 15) & ~(size_t)15;
        const bool staged = w2c_bytes + (size_t)M * 4 <= (size_t)p.sp_bytes;  // CTA-uniform
        WT* w2c_s = (WT*)sp_s;
        int32_t* cid_s = (int32_t*)((uint8_t*)sp_s + w2c_bytes);
        for (int k = threadIdx.x; k < r; k += kThreads) u_s[k] = __ldg(p.P_h + ((size_t)b * P + dep) * r + k);
        if (staged) {
          for (int m = threadIdx.x; m < M; m += kThreads) {
            int v = C[m];
            if (v < 0 || v >= p.V) {  // never expected: candidate ids come from the select
              dev_error(p.ctl, DEV_ERR_DATA);
              v = 0;
            }
            cid_s[m] = v;
            lg_s[m] = DCHECK(p.ctl, dep >= 0 && dep < P) ? __ldg(p.L_base + ((size_t)b * P + dep) * p.V + v) : 0.0f;
          }
          __syncthreads();
          const int cpr = (int)(r * sizeof(WT) / 16);  // 16-byte chunks per W2 row
          for (int idx = threadIdx.x; idx < M * cpr; idx += kThreads) {
            const int m = idx / cpr, q = idx - m * cpr;
            ((uint4*)w2c_s)[(size_t)m * cpr + q] = __ldg((const uint4*)(p.w2 + (size_t)cid_s[m] * r) + q);
          }
        }
        // u = SiLU(P_h[b, dep] + W1_s S_t): each entry's accumulator holds
        // the sum once every worker's partial is in (its count).
        for (int k = threadIdx.x; k < r; k += kThreads) {
          const unsigned long long* src = p.uacc + ((size_t)b * N + t) * r + k;
          unsigned long long x = ld_relaxed_u64(src);
          if ((x & 0xFFFFull) != n_contrib) {
            const uint64_t t0 = globaltimer_ns();
            unsigned spins = 0;
            while (((x = ld_relaxed_u64(src)) & 0xFFFFull) != n_contrib) {
              if ((++spins & 63u) == 0) {
                if (ld_volatile_u32(&p.ctl->abort)) { *fail_s = 1; break; }
                if (globaltimer_ns() - t0 > p.timeout_ns) { dev_abort(p.ctl, DEV_ERR_TIMEOUT); *fail_s = 1; break; }
              }
            }
          }
          u_s[k] = siluf_(u_s[k] + __ll2float_rn((long long)x >> 16) * kInvFix);  // one rounding, exact scaling
        }
        __syncthreads();
        if (*fail_s) return;
        // Candidate logits l_c = L_base[b, dep, c] + W2[c] . u.
        if (staged) {
          // All operands in shared memory: a warp's candidates m = warp,
          // warp + kWarps, ... four at a time, each summed by the whole warp
          // in the same order as one at a time (so the sums are unchanged),
          // the four chains and their reductions interleaved.
          for (int m0 = warp; m0 < M; m0 += 4 * kWarps) {
            float sacc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            for (int k = 4 * lane; k < r; k += 128) {
              const float4 uv = *(const float4*)(u_s + k);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const int m = m0 + q * kWarps;
                if (m < M) {  // warp-uniform
                  const float4 x = load4w(w2c_s + (size_t)m * r + k);
                  sacc[q] = fmaf(x.x, uv.x, fmaf(x.y, uv.y, fmaf(x.z, uv.z, fmaf(x.w, uv.w, sacc[q]))));
                }
              }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
              for (int q = 0; q < 4; ++q) sacc[q] += __shfl_xor_sync(0xffffffffu, sacc[q], o);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int m = m0 + q * kWarps;
              if (lane == 0 && m < M) lg_s[m] += sacc[q];
            }
          }
        } else
        // Four candidates per warp at a time, their W2 loads in flight together.
        for (int m0 = warp; m0 < M; m0 += 4 * kWarps) {
          int v[4];
          float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int m = m0 + q * kWarps;
            v[q] = m < M ? C[m] : 0;
            if (v[q] < 0 || v[q] >= p.V) {  // never expected: candidate ids come from the select
              if (lane == 0) dev_error(p.ctl, DEV_ERR_DATA);
              v[q] = 0;
            }
          }
          for (int k = 4 * lane; k < r; k += 128) {
            const float4 uv = *(const float4*)(u_s + k);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 x = load4w(p.w2 + (size_t)v[q] * r + k);
              s[q] = fmaf(x.x, uv.x, fmaf(x.y, uv.y, fmaf(x.z, uv.z, fmaf(x.w, uv.w, s[q]))));
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int m = m0 + q * kWarps;
            const float sq = warp_sum(s[q]);
            if (lane == 0 && m < M) lg_s[m] = __ldg(p.L_base + ((size_t)b * P + dep) * p.V + v[q]) + sq;
          }
        }
        __syncthreads();
        // Warp 0: logsumexp over the M-slice (fp32, max-shifted), the children's
        // (score, token) keys as node t's sibling group, and the group's best.
        if (warp == 0) {
          const float it = p.inv_tau;  // log-softmax of l / tau over the slice
          float mx = -INFINITY;
          for (int m = lane; m < M; m += 32) mx = fmaxf(mx, lg_s[m] * it);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
          float se = 0.0f;
          for (int m = lane; m < M; m += 32) se += expf(lg_s[m] * it - mx);
          se = warp_sum(se);
          const float lse = mx + logf(se);
          const float base = nsc_s[t];
          unsigned long long* grp = grp_s + (size_t)t * M;
          unsigned long long hb = 0ull;
          for (int m = lane; m < M; m += 32) {
            const unsigned long long key = value_id_key(base + (lg_s[m] * it - lse), (uint32_t)C[m]);
            grp[m] = key;
            hb = key > hb ? key : hb;
          }
          hb = warp_max_u64(hb);
          if (lane == 0) hbest_s[t] = hb;
        }
      } else if (threadIdx.x == 0) {
        hbest_s[t] = 0ull;  // no children
      }
      // Pop (warp 0): the best group head under (score desc, parent asc), taken
      // out of its group; publish node t + 1.
      if (warp == 0) {
        __syncwarp();
        // The head keys ranked by (score, lower group) in one 64-bit word,
        // whose low half also names the group.
        unsigned long long best = 0ull;
        if (misc_s[0]) {
          for (int gi = lane; gi <= t; gi += 32) {
            const unsigned long long ck = hbest_s[gi];
            if (ck) {
              const unsigned long long cmp = value_id_key(key_value(ck), (uint32_t)gi);
              best = cmp > best ? cmp : best;
            }
          }
        }
        best = warp_max_u64(best);
        const int bestg = best ? (int)key_id(best) : -1;
        const unsigned long long bestchild = best ? hbest_s[bestg] : 0ull;
        if (lane == 0) {
          const int k = t + 1;
          int tok = 0, nexp = 0, dk = 0;
          float sc = 0.0f;
          if (bestg < 0) {
            misc_s[0] = 0;  // candidate tree exhausted
          } else {
            tok = (int)key_id(bestchild);
            sc = key_value(bestchild);
            dk = ndep_s[bestg] + 1;
            ndep_s[k] = dk;
            nsc_s[k] = sc;
            nexp = (k < N && dk < P) ? 1 : 0;
            // The workers gather this token's gate-table row next: start it
            // towards L2 now (one bulk prefetch of the 3g-float row).
            if (nexp && tok < p.V)
              asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.gate_table + (size_t)tok * 3 * g),
                           "r"((uint32_t)(3 * g * 4))
                           : "memory");
          }
          int* cb = p.cur + ((size_t)b * (N + 1) + k) * 4;  // each node its own slot: never overwritten
          cb[0] = tok;
          cb[1] = bestg;
          cb[2] = nexp;
          st_release_s32(cb + 3, 1);
          // The outputs after the publication: no other CTA reads them here.
          if (bestg >= 0) {
            const size_t o = (size_t)b * (N + 1) + k;
            if (DCHECK(p.ctl, k <= N && bestg < k && dk <= P)) {
              p.node_token[o] = tok;
              p.node_parent[o] = bestg;
              p.node_depth[o] = dk;
              p.node_score[o] = sc;
            }
          }
        }
        if (bestg >= 0) {  // warp-uniform: the group's next best becomes its head (for the next pop)
          unsigned long long* grp = grp_s + (size_t)bestg * M;
          unsigned long long nb = 0ull;
          for (int m = lane; m < M; m += 32) {
            unsigned long long kk = grp[m];
            if (kk == bestchild) { grp[m] = 0ull; kk = 0ull; }
            nb = kk > nb ? kk : nb;
          }
          nb = warp_max_u64(nb);
          if (lane == 0) hbest_s[bestg] = nb;
        }
      }
    }
  }
}

int pow2_at_least(int x) {
  int n = 1;
  while (n < x) n <<= 1;
  return n;
}

// Worker groups: Q groups of the G - bs worker CTAs, group q serving
// requests [q bs / Q, (q + 1) bs / Q). A worker of the smallest group holds
// nu_max hidden units; a group serves at most bsq_max requests.
struct TreePlan {
  int Q = 0, nu_max = 0, bsq_max = 0, RB = 0;
  size_t sp_bytes = 0, smem = 0;
};

template <typename WT>
size_t tree_smem_bytes(int bs, int bsq_max, int g, int r, int N, int M, int Mp, int nu_max, size_t sp_bytes) {
  size_t off = 16 + (((size_t)3 * nu_max * g * sizeof(WT) + 15) & ~(size_t)15);  // mbarrier, W_hh rows
  off += ((size_t)nu_max * r * sizeof(WT) + 15) & ~(size_t)15;             // W1_s columns
  off += (size_t)3 * nu_max * 4 + (size_t)r * 4 +
         (size_t)Mp * 4 + 3 * (size_t)(N + 1) * 4 + 16 * 4 + (size_t)bs * 16 + (size_t)bsq_max * 3 * nu_max * 4 +
         (size_t)bsq_max * N * 4 * nu_max * 4 +
         16;  // alignment of u_s
  off = (off + 15) & ~(size_t)15;
  off += sp_bytes;
  off = (off + 7) & ~(size_t)7;
  return off + (size_t)(N + 1) * 8 + (size_t)N * M * 8;
}

// The most worker groups (4, 2 or 1) whose shared memory fits, with at least
// one request and one worker per group; RB = states staged at a time.
template <typename WT>
bool tree_plan(int bs, int g, int r, int N, int M, TreePlan* out) {
  const int nw = num_sms() - bs, Mp = pow2_at_least(M);
  const size_t budget = 227 * 1024;
  for (int Q : {4, 2, 1}) {
    if (Q > bs || Q > nw) continue;
    TreePlan pl;
    pl.Q = Q;
    pl.nu_max = (g + nw / Q - 1) / (nw / Q);
    pl.bsq_max = (bs + Q - 1) / Q;
    const size_t base = tree_smem_bytes<WT>(bs, pl.bsq_max, g, r, N, M, Mp, pl.nu_max, 0);
    if (base + (size_t)g * 4 > budget) continue;
    const size_t rb = (budget - base) / ((size_t)g * 4);
    pl.RB = (int)(rb < (size_t)pl.bsq_max ? rb : (size_t)pl.bsq_max);
    // The buffer also holds an owner's candidate W2 rows and ids when they fit.
    const size_t states = (size_t)pl.RB * g * 4;
    const size_t cands = (((size_t)M * r * sizeof(WT) + 15) & ~(size_t)15) + (size_t)M * 4;
    pl.sp_bytes = cands > states && tree_smem_bytes<WT>(bs, pl.bsq_max, g, r, N, M, Mp, pl.nu_max, cands) <= budget
                      ? cands
                      : states;
    pl.smem = tree_smem_bytes<WT>(bs, pl.bsq_max, g, r, N, M, Mp, pl.nu_max, pl.sp_bytes);
    if (pl.smem > budget) continue;
    *out = pl;
    return true;
  }
  return false;
}

template <typename WT>
cudaError_t launch_tree_t(const TreeArgs& a, cudaStream_t stream) {
  const int G = num_sms();
  TreeP<WT> p;
  p.bs = a.bs; p.P = a.P; p.d = a.d; p.g = a.g; p.r = a.r; p.V = a.V; p.N = a.N; p.M = a.M;
  p.Mp = pow2_at_least(a.M);
  p.gate_table = a.gate_table;
  p.w_hh = (const WT*)a.w_hh; p.b_hh = (const WT*)a.b_hh; p.w1 = (const WT*)a.w1; p.w2 = (const WT*)a.w2;
  p.L_base = a.L_base; p.P_h = a.P_h; p.anchor = a.anchor;
  p.node_token = a.node_token; p.node_parent = a.node_parent; p.node_depth = a.node_depth;
  p.node_score = a.node_score;
  p.ctl = a.ctl; p.cand = a.cand; p.tstates = (unsigned*)a.states; p.cur = a.cur;
  p.uacc = (unsigned long long*)a.uacc;
  p.timeout_ns = wait_timeout_ns();
  p.inv_tau = a.inv_tau;
  TreePlan pl;
  if (!tree_plan<WT>(a.bs, a.g, a.r, a.N, a.M, &pl)) return cudaErrorInvalidConfiguration;
  p.Q = pl.Q; p.nu_max = pl.nu_max; p.bsq_max = pl.bsq_max; p.RB = pl.RB; p.sp_bytes = (int)pl.sp_bytes;
  const size_t smem = pl.smem;
  cudaError_t e = cudaFuncSetAttribute(tree_kernel<WT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void* args[] = {(void*)&p};
  return cudaLaunchCooperativeKernel((const void*)tree_kernel<WT>, dim3(G), dim3(kThreads), args, smem, stream);
}

}  // namespace

size_t topm_ws_bytes(int rows, int n, int M) {
  (void)n; (void)M;
  // thresholds, counts (zero between calls), candidate lists
  return (size_t)rows * 8 + (((size_t)rows * 4 + 255) & ~(size_t)255) + (size_t)rows * kListCap * 8;
}

cudaError_t launch_topm(const float* values, int rows, int n, int M, int32_t* ids, float* vals,
                        void* scratch, cudaStream_t stream) {
  if (rows > 65535 || M > 256 || M < 1 || M > n) return cudaErrorInvalidValue;
  unsigned long long* tau = (unsigned long long*)scratch;
  unsigned* counts = (unsigned*)((uint8_t*)scratch + (size_t)rows * 8);
  unsigned long long* lists =
      (unsigned long long*)((uint8_t*)counts + (((size_t)rows * 4 + 255) & ~(size_t)255));
  topm_sample<<<rows, kSelThreads, 0, stream>>>(values, n, M, tau);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int nseg = (n + kFilterSeg - 1) / kFilterSeg;
  topm_filter<<<dim3(nseg, rows), kFilterThreads, 0, stream>>>(values, n, tau, lists, counts);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t smem_f = ((size_t)2 * kCap + 256) * 8;
  e = cudaFuncSetAttribute(topm_final, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_f);
  if (e != cudaSuccess) return e;
  topm_final<<<rows, kSelThreads, smem_f, stream>>>(values, n, M, lists, counts, ids, vals);
  return cudaGetLastError();
}

size_t tree_ws_bytes(int bs, int P, int g, int r, int N, int M) {
  auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
  return al((size_t)bs * P * M * 4) + al((size_t)bs * N * g * 4) + al((size_t)bs * (N + 1) * 4 * 4) +
         al((size_t)bs * N * r * 8);
}

bool tree_fits(int dtype, int bs, int g, int r, int N, int M) {
  if (bs >= num_sms()) return false;  // at least one worker CTA beside the request owners
  TreePlan pl;
  return dtype == DOMINO_BF16 ? tree_plan<__nv_bfloat16>(bs, g, r, N, M, &pl) : tree_plan<float>(bs, g, r, N, M, &pl);
}

cudaError_t launch_tree(const TreeArgs& a, cudaStream_t stream) {
  if (a.dtype == DOMINO_BF16) return launch_tree_t<__nv_bfloat16>(a, stream);
  return launch_tree_t<float>(a, stream);
}

}  // namespace domino
