// Longest accepted prefix ("Domino: Decoupling Causal Modeling from
// Autoregressive Drafting in Speculative Decoding Review", section 1-1: the
// target checks the drafted block in one pass; tokens advanced per cycle is the
// accepted prefix plus the target's own next token), its tree form, and the
// bounded-wait self-test.
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

// Tree acceptance ("DominoTree…", section 验证: tree attention with an
// ancestor-only causal mask). One warp per request. Mask rows: lane i walks
// node i's parent chain (parents precede their children in node order; a
// parent outside [0, i) ends the walk). The walk from the root: at node n the
// lanes look for the child whose token is the target's next token after n;
// the lowest such node id (siblings carry distinct tokens) is the next node.
__global__ void tree_verify_kernel(const int32_t* __restrict__ tok, const int32_t* __restrict__ par,
                                   const int32_t* __restrict__ tgt, int bs, int n1,
                                   int32_t* __restrict__ accept, int32_t* __restrict__ advanced,
                                   int32_t* __restrict__ path, uint8_t* __restrict__ mask) {
  const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (b >= bs) return;
  const int32_t* T = tok + (size_t)b * n1;
  const int32_t* Pa = par + (size_t)b * n1;
  const int32_t* G = tgt + (size_t)b * n1;
  if (mask) {
    for (int i = lane; i < n1; i += 32) {
      uint8_t* row = mask + ((size_t)b * n1 + i) * n1;
      for (int j = 0; j < n1; ++j) row[j] = 0;
      if (T[i] < 0) continue;
      int j = i;
      for (int steps = 0; steps <= n1; ++steps) {
        row[j] = 1;
        if (j == 0) break;
        const int pj = Pa[j];
        if (pj < 0 || pj >= j) break;
        j = pj;
      }
    }
  }
  int node = 0, depth = 0;
  if (path && lane == 0) path[(size_t)b * n1] = 0;
  while (depth < n1 - 1) {
    const int want = G[node];
    int found = n1;
    for (int c = 1 + lane; c < n1; c += 32)
      if (T[c] >= 0 && Pa[c] == node && T[c] == want) found = min(found, c);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) found = min(found, __shfl_xor_sync(0xffffffffu, found, o));
    if (found >= n1) break;
    node = found;
    ++depth;
    if (path && lane == 0) path[(size_t)b * n1 + depth] = node;
  }
  if (path)
    for (int k = depth + 1 + lane; k < n1; k += 32) path[(size_t)b * n1 + k] = -1;
  if (lane == 0) {
    accept[b] = depth;
    advanced[b] = depth + 1;
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

cudaError_t launch_tree_verify(const int32_t* tok, const int32_t* par, const int32_t* tgt, int bs, int n1,
                               int32_t* accept, int32_t* advanced, int32_t* path, uint8_t* mask,
                               cudaStream_t stream) {
  const int threads = 256;
  const int blocks = (bs * 32 + threads - 1) / threads;
  tree_verify_kernel<<<blocks, threads, 0, stream>>>(tok, par, tgt, bs, n1, accept, advanced, path, mask);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(Ctl* ctl, uint64_t timeout_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(ctl, timeout_ns);
  return cudaGetLastError();
}

}  // namespace domino
