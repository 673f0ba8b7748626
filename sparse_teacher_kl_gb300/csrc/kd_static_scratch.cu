// kd_fused_kl_fwd_static: the fused KL forward pass for callers that cannot
// allocate device memory.
//
// Some callers may not call cudaMalloc at all: plugins inside a host framework
// whose allocator owns every byte of device memory (a stray allocation there
// fragments or overflows a pool sized in advance), and latency-sensitive paths
// that cannot afford the implicit device-wide synchronisation cudaMalloc and
// cudaFree may perform.  They also cannot size and pass the workspace that
// kd_fused_kl_fwd asks for.  This entry point uses a fixed scratch area that
// lives in the library itself instead.
//
// The scratch is a file-scope device array of KD_STATIC_SCRATCH_BYTES; every
// GPU that loads the library holds it until the process exits.  Its device
// address is looked up once per device, on the first call made while that
// device is current (so that first call should come before any stream
// capture), and again if the device's CUDA context has changed since (after a
// device reset).  Every call shares the one array and it keeps the last call's
// contents; the control block is cleared at the start of each call.  Calls
// whose work overlaps on the GPU (other streams, other host threads) race on
// the array and must be serialised by the caller.  Device-side conditions are
// recorded in the array's error word, which kd_get_device_error reads when it
// is given a NULL workspace.
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "kd_internal.h"

namespace kd {

static __device__ __align__(256) uint8_t g_static_scratch[KD_STATIC_SCRATCH_BYTES];

// The array's device address, per device ordinal, with the CUDA context it was looked up
// in: a device reset gives the device a new context (and may move the array), so an
// address cached under another context is looked up again.
struct ScratchAddr {
  CUcontext ctx;
  void* ptr;
};
static ScratchAddr g_static_addr[kMaxDevices] = {};
static std::mutex g_static_mu;

static PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
static std::once_flag g_ctx_once;

// The calling thread's current context (NULL if it has none yet or it cannot be read).
static CUcontext current_context() {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  });
  CUcontext c = nullptr;
  if (g_ctx_current == nullptr || g_ctx_current(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

kd_status static_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_mu);
  CUcontext ctx = current_context();
  ScratchAddr& a = g_static_addr[dev];
  if (a.ptr == nullptr || ctx == nullptr || a.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return KD_ERR_CUDA;
    a.ptr = p;
    a.ctx = current_context();  // the lookup above makes the device's context current
  }
  *out = a.ptr;
  return KD_OK;
}

}  // namespace kd

extern "C" int kd_fused_kl_fwd_static(const void* H_bf16, const void* W_bf16, const int32_t* t_ids,
                                      const float* t_logits, const uint8_t* mask, int64_t N, int64_t d, int64_t V,
                                      int K, int64_t chunk, float tau, float* loss_out, float* lse_out,
                                      float* kl_per_token_out, void* stream) {
  const size_t need = kd_fused_kl_workspace(N, d, V, K, chunk);
  if (need == 0) return KD_ERR_INVALID_ARG;
  if (!H_bf16 || !W_bf16 || !t_ids || !t_logits || !loss_out || !lse_out) return KD_ERR_INVALID_ARG;
  if (!(tau > 0.f) || !(tau < INFINITY)) return KD_ERR_INVALID_ARG;
  if (need > size_t(KD_STATIC_SCRATCH_BYTES)) return KD_ERR_WORKSPACE;
  void* scratch = nullptr;
  kd_status st = kd::static_scratch_address(&scratch);
  if (st != KD_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, sizeof(kd::Ctrl), s) != cudaSuccess) return KD_ERR_CUDA;
  return kd_fused_kl_fwd(H_bf16, W_bf16, t_ids, t_logits, mask, N, d, V, K, chunk, tau, loss_out, lse_out,
                         kl_per_token_out, scratch, size_t(KD_STATIC_SCRATCH_BYTES), stream);
}
