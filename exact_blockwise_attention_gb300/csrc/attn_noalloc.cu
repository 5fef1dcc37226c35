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

#include "attn.h"
#include "kernels.h"

namespace {

// The scratch buffer: one per device, part of this file's device module. With
// the CUDA runtime's lazy module loading the module, and with it the buffer,
// is loaded onto a device when its address is first looked up there (the
// first call on that device, or a B = 0 call made for that purpose), and stays
// reserved until the process exits. Host code must never pass
// `g_noalloc_scratch` itself to a kernel (in host code it is only a stand-in
// for the device symbol); the device address comes from eba::symbol_address,
// which calls cudaGetSymbolAddress with the device current.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

}  // namespace

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                int B, int H, int Lq, int Lk, int d, float scale, void* stream) {
  if (B == 0) {
    // Set-up only: load the buffer onto the current device and look up its
    // address, so that start-up code can reserve it before memory runs short
    // and before any stream capture.
    return eba::symbol_address(&g_noalloc_scratch, eba::kSymNoallocScratch) ? ATTN_OK
                                                                             : ATTN_ERR_CUDA;
  }
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  const size_t need = attn_bwd_workspace_size(B, H, Lq, Lk, d);
  if (need == 0) return ATTN_ERR_INVALID_ARG;
  // Too large for the built-in buffer: refuse before touching CUDA.
  if (need > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_WORKSPACE;
  void* scratch = eba::symbol_address(&g_noalloc_scratch, eba::kSymNoallocScratch);
  if (!scratch) return ATTN_ERR_CUDA;  // the CUDA error is kept for attn_last_cuda_error
  return attn_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, Lq, Lk, d, scale, scratch,
                  ATTN_NOALLOC_SCRATCH_BYTES, stream);
}
