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
// capture).  Every call shares the one array and it keeps the last call's
// contents; the control block is cleared at the start of each call.  Calls
// whose work overlaps on the GPU (other streams, other host threads) race on
// the array and must be serialised by the caller.
#include <math.h>

#include <mutex>

#include "kd_internal.h"

namespace kd {

static __device__ __align__(256) uint8_t g_static_scratch[KD_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
static void* g_static_ptr[kMaxDevices] = {};
static std::mutex g_static_mu;

// Device address of the scratch array on the current device (set up once per device).
static kd_status static_scratch_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KD_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) return KD_ERR_CUDA;
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
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
  kd_status st = kd::static_scratch_ptr(&scratch);
  if (st != KD_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, sizeof(kd::Ctrl), s) != cudaSuccess) return KD_ERR_CUDA;
  return kd_fused_kl_fwd(H_bf16, W_bf16, t_ids, t_logits, mask, N, d, V, K, chunk, tau, loss_out, lse_out,
                         kl_per_token_out, scratch, size_t(KD_STATIC_SCRATCH_BYTES), stream);
}
