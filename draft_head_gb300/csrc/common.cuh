// Device helpers shared by the Domino kernels: status word, bounded waits,
// grid barrier, ordered (value, id) keys, and thin inline-PTX wrappers for
// mbarrier, TMA and tcgen05 on sm_103a.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"

namespace domino {

// ---------------------------------------------------------------------------
// Workspace control block (first 256 bytes of every workspace).
// ---------------------------------------------------------------------------
struct Ctl {
  unsigned int barrier;      // monotonically increasing grid-barrier counter
  unsigned int abort;        // set when any CTA gives up; others leave too
  unsigned int status;       // sticky DEV_ERR_* bits
  unsigned int pad0;
  unsigned long long never;  // flag nothing writes (wait self-test)
  unsigned int pad[58];
};
static_assert(sizeof(Ctl) == 256, "Ctl must be 256 bytes");

// Device error bits (mapped to domino_status by the host).
enum : unsigned int {
  DEV_ERR_TIMEOUT = 1u,
  DEV_ERR_DATA = 2u,
  DEV_ERR_INDEX = 4u,  // checked build: an index check failed (the access was skipped)
};

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_volatile_u32(const unsigned* p) {
  return *(volatile const unsigned*)p;
}

__device__ __forceinline__ void dev_error(Ctl* ctl, unsigned bits) {
  atomicOr(&ctl->status, bits);
}

__device__ __forceinline__ void dev_abort(Ctl* ctl, unsigned bits) {
  atomicOr(&ctl->status, bits);
  atomicExch(&ctl->abort, 1u);
}

// Index checks of the checked build (compiled with -DDOMINO_CHECKED): a
// failed check records DEV_ERR_INDEX in the status word and the guarded
// access is skipped. In the regular build DCHECK is the constant true and the
// compiler removes it.
__device__ __forceinline__ bool domino_checked(Ctl* ctl, bool ok) {
  if (!ok) atomicOr(&ctl->status, (unsigned)DEV_ERR_INDEX);
  return ok;
}
#ifdef DOMINO_CHECKED
#define DCHECK(ctl, cond) (::domino::domino_checked((ctl), (cond)))
#else
#define DCHECK(ctl, cond) true
#endif

// One partial of a cross-CTA sum in 2^-32 fixed point: round(part * 2^32).
// A partial above `limit` in magnitude (NaN included) could carry the
// accumulator past its integer range once all partials are in; it is
// recorded as DEV_ERR_DATA and contributes zero instead of wrapping silently.
__device__ __forceinline__ long long fix32_checked(float part, float limit, Ctl* ctl) {
  if (!(fabsf(part) <= limit)) {
    dev_error(ctl, DEV_ERR_DATA);
    return 0;
  }
  return __float2ll_rn(part * 4294967296.0f);
}

// Grid-wide barrier for a persistent kernel whose CTAs are all resident
// (cooperative launch). The counter only grows; `epoch` is the caller's local
// count of barriers passed. Returns false (and leaves) if the wait runs past
// `timeout_ns` or another CTA aborted.
__device__ __forceinline__ bool grid_barrier(Ctl* ctl, unsigned& epoch, unsigned nblocks,
                                             uint64_t timeout_ns) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    epoch += 1;
    const unsigned target = epoch * nblocks;
    int ok = 1;
    __threadfence();
    atomicAdd(&ctl->barrier, 1u);
    if (ld_acquire_u32(&ctl->barrier) < target) {
      const uint64_t t0 = globaltimer_ns();
      unsigned spins = 0;
      while (ld_acquire_u32(&ctl->barrier) < target) {
        if ((++spins & 63u) == 0) {
          if (ld_volatile_u32(&ctl->abort)) { ok = 0; break; }
          if (globaltimer_ns() - t0 > timeout_ns) { dev_abort(ctl, DEV_ERR_TIMEOUT); ok = 0; break; }
        }
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// Order-preserving map of a float to uint32 (larger float -> larger key);
// -0 is folded onto +0 so the two tie, as they do arithmetically.
__device__ __forceinline__ uint32_t float_order_key(float f) {
  if (f == 0.0f) f = 0.0f;
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_key_float(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

// (value desc, id asc) as one unsigned 64-bit key: the maximum key is the
// largest value with the lowest id.
__device__ __forceinline__ unsigned long long value_id_key(float v, uint32_t id) {
  return ((unsigned long long)float_order_key(v) << 32) | (unsigned long long)(0xFFFFFFFFu - id);
}
__device__ __forceinline__ uint32_t key_id(unsigned long long k) {
  return 0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull);
}
__device__ __forceinline__ float key_value(unsigned long long k) {
  return order_key_float((uint32_t)(k >> 32));
}

__device__ __forceinline__ float sigmoidf_(float t) { return 1.0f / (1.0f + expf(-t)); }
__device__ __forceinline__ float siluf_(float t) { return t / (1.0f + expf(-t)); }

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    unsigned long long w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// ---------------------------------------------------------------------------
// mbarrier / TMA / tcgen05 (inline PTX, sm_100 family).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase. `s_abort` is a CTA-local flag other
// roles set when they give up. Returns false on timeout/abort.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* s_abort,
                                          Ctl* ctl, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  unsigned spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++spins & 15u) == 0) {
      if (s_abort && *s_abort) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        dev_error(ctl, DEV_ERR_TIMEOUT);
        if (s_abort) *s_abort = 1;
        return false;
      }
    }
  }
  return true;
}

// 2-D tiled TMA load global -> shared, completing on `bar` (complete_tx).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"((uint64_t)tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const void* tmap, int x, int y,
                                                 uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"((uint64_t)tmap), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Contiguous global -> shared copy by the bulk-copy engine, completing on
// `bar` (complete_tx). Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* smem_dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(smem_dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)tmap) : "memory");
}

// Tensor memory.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major, 128-byte swizzle: rows of 128 B
// (64 bf16 of K), 8-row swizzle atoms 1024 B apart (stride byte offset);
// the leading byte offset is unused for this layout. Bits 46-47 = 1 (sm_100
// descriptor version), bits 61-63 = 2 (128-byte swizzle).
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor for kind::f16 with bf16 A/B, fp32 D, both K-major:
// D format at bit 4, A/B formats at bits 7/10, N>>3 at bit 17, M>>4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, issued by one thread: A's M rows in
// tensor-memory lanes, K packed two bf16 per 32-bit column.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Shared memory -> tensor memory: a 128-row x 256-bit matrix (one K16 slice of
// a bf16 operand, described like an MMA operand) into 128 lanes x 8 columns.
// Ordered with the issuing thread's later tcgen05.mma.
__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// Arrive on `bar` once all tcgen05 ops issued so far by this thread complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Warp loads 32 TMEM lanes x 16 fp32 columns; thread t gets lane (base + t).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

}  // namespace domino
