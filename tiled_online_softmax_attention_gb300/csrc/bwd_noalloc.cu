// bwd_noalloc.cu -- attn_bwd_noalloc: the backward pass for callers that cannot
// allocate device memory.
//
// The backward needs a scratch workspace (here, as for attn_bwd_deterministic: two
// float32 values per row).  Some callers have no way to provide one: a plugin whose
// host framework owns every byte of device memory through its own allocator, an
// engine that fixes its memory budget once at start-up, or a foreign-function caller
// that reaches the GPU only through this C ABI and has no CUDA runtime of its own to
// call cudaMalloc with.  For them this entry point takes its scratch from a
// fixed-size array that lives in the library's own device image: every GPU that
// loads the library holds ATTN_NOALLOC_SCRATCH_BYTES of it until the process
// exits.  The caller still passes every input and output buffer.
#include <cstddef>

#include <cuda_runtime.h>

#include "../../include/attn.h"

namespace {

// The shared scratch.  Host code must not pass this name to a kernel: on the
// host it is only a stand-in for the device symbol, and its device address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_bwd_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

// The array's device address on the current device.  Looked up on every call (a
// lookup in the runtime's module table; it allocates nothing): a cached address would
// go stale when cudaDeviceReset tears the context down and a new one loads the module
// again.
attn_status scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
  *out = p;
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                        const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                                        int H, int N, int d, attn_dtype dt, int causal, float scale,
                                        int* dev_status, void* stream) {
  const size_t need = attn_bwd_deterministic_workspace_bytes(B, H, N, d);
  if (need == 0)  // invalid sizes: let the full entry point report which argument is wrong, before any CUDA call
    return attn_bwd_deterministic(q, k, v, o, dout, lse, dq, dk, dv, nullptr, 0, B, H, N, d, dt, causal, scale,
                                  dev_status, stream);
  if (need > ATTN_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const attn_status st = scratch_address(&scratch);
  if (st != ATTN_OK) return st;
  // The preparation stage overwrites every scratch value the gradient stages read,
  // so nothing left by an earlier call needs clearing.
  return attn_bwd_deterministic(q, k, v, o, dout, lse, dq, dk, dv, scratch, ATTN_NOALLOC_SCRATCH_BYTES, B, H, N, d,
                                dt, causal, scale, dev_status, stream);
}
