// Longest accepted prefix ("Domino: Decoupling Causal Modeling from
// Autoregressive Drafting in Speculative Decoding Review", section 1-1: the
// target checks the drafted block in one pass; tokens advanced per cycle is the
// accepted prefix plus the target's own next token), and the bounded-wait
// self-test.
#include "common.cuh"

namespace domino {

namespace {

// One warp per request: each lane compares a strided set of positions, the
// first mismatch is the minimum mismatching position over the warp.
__global__ void verify_kernel(const int32_t* __restrict__ draft, const int32_t* __restrict__ target,
                              int bs, int P, int32_t* __restrict__ accept,
                              int32_t* __restrict__ advanced) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= bs) return;
  const int32_t* d = draft + (size_t)warp * P;
  const int32_t* t = target + (size_t)warp * P;
  int first = P;
  for (int k = lane; k < P; k += 32)
    if (d[k] != t[k]) { first = k; break; }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
  if (lane == 0) {
    accept[warp] = first;
    advanced[warp] = first + 1;
  }
}

// Waits on a flag that nothing writes; the bound makes it give up and record
// a timeout in the status word.
__global__ void wait_selftest_kernel(Ctl* ctl, uint64_t timeout_ns) {
  if (threadIdx.x != 0) return;
  const uint64_t t0 = globaltimer_ns();
  while (*(volatile unsigned long long*)&ctl->never == 0ull) {
    if (globaltimer_ns() - t0 > timeout_ns) {
      dev_error(ctl, DEV_ERR_TIMEOUT);
      return;
    }
    __nanosleep(1000);
  }
}

}  // namespace

cudaError_t launch_verify(const int32_t* draft, const int32_t* target, int bs, int P,
                          int32_t* accept, int32_t* advanced, cudaStream_t stream) {
  const int threads = 256;
  const int blocks = (bs * 32 + threads - 1) / threads;
  verify_kernel<<<blocks, threads, 0, stream>>>(draft, target, bs, P, accept, advanced);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(Ctl* ctl, uint64_t timeout_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(ctl, timeout_ns);
  return cudaGetLastError();
}

}  // namespace domino
