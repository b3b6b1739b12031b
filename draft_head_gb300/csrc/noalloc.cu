// Allocation-free variant of the chain entry point.
//
// Some callers cannot call cudaMalloc at all: a process whose device memory
// is handed out by a framework's own pool (no raw allocations allowed), code
// that must not allocate between a warm-up and a latency-critical serving
// loop, or an embedder that links this library without any allocator. For
// them, domino_draft_chain_noalloc() runs the same chain kernel with its
// scratch (barrier counter, status word, per-step argmax keys, GRU state,
// bottleneck accumulators) in one file-scope device array of fixed size.
//
// The array exists once per GPU that loads the library and stays allocated
// until the process exits. All calls on a device share it, and it keeps the
// contents of the last call, so each call clears what must start at zero.
// Two calls that overlap on the GPU (different streams, or different host
// threads) use the same array and race.
#include <mutex>

#include "common.cuh"

namespace domino {

namespace {

constexpr int kNaMaxBatch = 4;
constexpr int kNaMaxP = 32;
constexpr int kNaMaxSMs = 256;
constexpr int kNaMaxG = 2048;
constexpr int kNaMaxR = 256;

constexpr size_t na_al(size_t x) { return (x + 255) & ~(size_t)255; }
// Pieces, in the order the chain kernel's workspace uses them.
constexpr size_t kNaCtl = 0;
constexpr size_t kNaKeys = 256;
constexpr size_t kNaS = kNaKeys + na_al((size_t)kNaMaxP * kNaMaxBatch * kNaMaxSMs * 8);
constexpr size_t kNaUacc = kNaS + na_al((size_t)2 * kNaMaxBatch * kNaMaxG * 8);
constexpr size_t kNaUglob = kNaUacc + na_al((size_t)2 * kNaMaxBatch * kNaMaxR * 16 * 8);
constexpr size_t kNaBytes = kNaUglob + na_al((size_t)kNaMaxBatch * kNaMaxR * 4);  // 659,712 bytes

// Host code must not use this name as a pointer: on the host it is only a
// stand-in for the device object. Its device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_chain_scratch[kNaBytes];

std::mutex g_na_mutex;
void* g_na_ptr[64] = {nullptr};

// Device address of the scratch on the current device; looked up once per
// device (with that device current) and zeroed then.
cudaError_t na_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  if (!g_na_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_chain_scratch);
    if (e != cudaSuccess) return e;
    e = cudaMemset(p, 0, kNaBytes);
    if (e != cudaSuccess) return e;
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    g_na_ptr[dev] = p;
  }
  *out = g_na_ptr[dev];
  return cudaSuccess;
}

// Copy the device status of the chain just run into the caller's int32 and
// clear it, mapped to domino_status codes.
__global__ void na_export_status(Ctl* ctl, int32_t* out) {
  const unsigned s = ctl->status;
  ctl->status = 0u;
  if (out)
    *out = (s & DEV_ERR_TIMEOUT) ? DOMINO_ERR_TIMEOUT
         : (s & DEV_ERR_INDEX)   ? DOMINO_ERR_INDEX
         : (s & DEV_ERR_DATA)    ? DOMINO_ERR_DEVICE_DATA
                                 : DOMINO_OK;
}

}  // namespace
}  // namespace domino

using namespace domino;

extern "C" domino_status domino_draft_chain_noalloc(
    const domino_head* h, const float* L_base, const float* P_h, const int32_t* anchor, int batch, int P,
    float temperature, const float* gumbel, int64_t gumbel_batch_stride, const int32_t* force_tokens,
    int32_t* tokens, float* logits_out, int32_t* device_status, void* stream) {
  if (!h) return DOMINO_ERR_INVALID_ARG;
  if (h->dtype != DOMINO_F32 && h->dtype != DOMINO_BF16) return DOMINO_ERR_INVALID_ARG;
  if (h->d <= 0 || h->e <= 0 || h->g <= 0 || h->r <= 0 || h->V <= 0) return DOMINO_ERR_INVALID_ARG;
  const void* ptrs[] = {h->w_lm, h->emb, h->w_ih, h->w_hh, h->b_ih, h->b_hh, h->w1, h->w2, h->gate_table};
  for (const void* p : ptrs)
    if (!p || ((uintptr_t)p & 15u)) return DOMINO_ERR_INVALID_ARG;
  if (h->dtype == DOMINO_BF16 && ((h->d | h->e | h->g | h->r) & 7)) return DOMINO_ERR_UNSUPPORTED;
  if (h->dtype == DOMINO_F32 && ((h->d | h->e | h->g | h->r) & 3)) return DOMINO_ERR_UNSUPPORTED;
  if (batch < 0 || P < 0) return DOMINO_ERR_INVALID_ARG;
  if (batch == 0 || P == 0) return DOMINO_OK;
  if (!L_base || !P_h || !anchor || !tokens) return DOMINO_ERR_INVALID_ARG;
  if (!(temperature >= 0.0f) || !(temperature < INFINITY)) return DOMINO_ERR_INVALID_ARG;
  if (temperature > 0.0f && (!gumbel || gumbel_batch_stride < (int64_t)P * h->V)) return DOMINO_ERR_INVALID_ARG;
  // The fixed scratch holds at most these sizes.
  if (batch > kNaMaxBatch || P > kNaMaxP || h->g > kNaMaxG || h->r > kNaMaxR || num_sms() > kNaMaxSMs)
    return DOMINO_ERR_UNSUPPORTED;
  if (!chain_fits(h->dtype, batch, h->g, h->r)) return DOMINO_ERR_UNSUPPORTED;

  void* base = nullptr;
  if (na_scratch(&base) != cudaSuccess) return DOMINO_ERR_CUDA;
  uint8_t* w = (uint8_t*)base;
  cudaStream_t s = (cudaStream_t)stream;
  // Clear what the kernel expects at zero: barrier counter and abort flag,
  // the per-step argmax keys, the first bottleneck accumulator buffer and
  // the step-tagged GRU state words.
  void* zp[4] = {w + kNaCtl, w + kNaKeys, w + kNaUacc, w + kNaS};
  const size_t zb[4] = {8, (size_t)P * batch * num_sms() * 8, (size_t)batch * h->r * 16 * 8,
                        (size_t)2 * batch * h->g * 8};
  cudaError_t e = zero_ranges(zp, zb, 4, s);
  if (e != cudaSuccess) return DOMINO_ERR_CUDA;

  ChainArgs a;
  a.dtype = h->dtype; a.bs = batch; a.P = P; a.d = h->d; a.g = h->g; a.r = h->r; a.V = h->V;
  a.gate_table = h->gate_table; a.w_hh = h->w_hh; a.b_hh = h->b_hh; a.w1 = h->w1; a.w2 = h->w2;
  a.L_base = L_base; a.P_h = P_h; a.anchor = anchor;
  a.temperature = temperature; a.gumbel = temperature > 0.0f ? gumbel : nullptr;
  a.gumbel_bstride = gumbel_batch_stride;
  a.force = force_tokens; a.tokens = tokens; a.logits_out = logits_out;
  a.ctl = (Ctl*)(w + kNaCtl);
  a.keys = (unsigned long long*)(w + kNaKeys);
  a.S = (float*)(w + kNaS);
  a.uacc = (long long*)(w + kNaUacc);
  a.uglob = (float*)(w + kNaUglob);
  a.s16 = nullptr;  // batch <= 4: the small-batch kernel needs none of these
  a.u16 = nullptr;
  a.ctr = nullptr;
  a.bimg = nullptr;
  e = launch_chain(a, s);
  if (e != cudaSuccess) return (e == cudaErrorInvalidConfiguration || e == cudaErrorCooperativeLaunchTooLarge)
                                   ? DOMINO_ERR_UNSUPPORTED : DOMINO_ERR_CUDA;
  na_export_status<<<1, 1, 0, s>>>((Ctl*)(w + kNaCtl), device_status);
  return cudaGetLastError() == cudaSuccess ? DOMINO_OK : DOMINO_ERR_CUDA;
}
