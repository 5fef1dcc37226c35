// attn_bwd_noalloc: the attention backward for callers that cannot allocate
// device memory. Its scratch lives in a fixed buffer compiled into this
// library instead of a workspace the caller passes in.
//
// Who needs this: code that runs where allocating device memory is not
// allowed or not possible, for example a plugin loaded into a host
// application that owns all GPU memory and hands the plugin no allocator, or a
// steady-state serving loop whose memory is fixed at start-up (cudaMalloc and
// cudaFree can synchronise the device and fragment memory, so such loops ban
// them after initialisation). These callers can still pass inputs and
// outputs, but they cannot provide attn_bwd's workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "attn.h"

namespace {

constexpr int kMaxDevices = 64;

// The scratch buffer: one per device, reserved for as long as the library is
// loaded. Host code must never pass `g_noalloc_scratch` itself to a kernel (in
// host code it is only a stand-in for the device symbol); the device address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

// Device address of the scratch buffer on the current device, looked up once
// per device (with that device current) and cached. nullptr on failure.
void* scratch_address() {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                int B, int H, int Lq, int Lk, int d, float scale, void* stream) {
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  const size_t need = attn_bwd_workspace_size(B, H, Lq, Lk, d);
  if (need == 0) return ATTN_ERR_INVALID_ARG;
  // Too large for the built-in buffer: refuse before touching CUDA.
  if (need > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_WORKSPACE;
  void* scratch = scratch_address();
  if (!scratch) return ATTN_ERR_CUDA;
  return attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, Lq, Lk, d, scale, scratch,
                  ATTN_NOALLOC_SCRATCH_BYTES, stream);
}
