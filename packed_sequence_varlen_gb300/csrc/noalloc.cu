// Forward attention for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory at the point where they
// run attention: a plugin executed by a host runtime that owns every device
// allocation and offers no scratch API, or a latency-critical serving loop
// that must not call cudaMalloc because it can synchronise the device and
// stall the other streams.  varlen_attn_fwd_noalloc serves them: it runs the
// ordinary forward (contract check, tile plan, attention kernel) with its
// scratch -- the 256-byte status header, the tile map and the per-segment
// record offsets -- in a fixed, file-scope device array instead of a caller
// workspace.
//
// Properties of the static scratch:
//   * kNoAllocScratchBytes (1 MiB) on every GPU that loads this library, held
//     until the process exits.  A shape fits when the workspace the ordinary
//     forward would ask for, varlen_attn_workspace_size(shape, 0), is at most
//     1 MiB; larger shapes are rejected with VA_ERR_WORKSPACE.
//   * Every call on a device shares it and it keeps the last call's contents.
//     Each call's contract check rewrites the status word and its plan rewrites
//     the record counts, the work counters and every record it later reads, so
//     nothing is cleared between calls.  Calls that overlap on the GPU (other
//     streams, other host threads) race on it and must be serialised by the
//     caller.
//   * In host code the array's name is only a host-side stand-in.  Its device
//     address is looked up with cudaGetSymbolAddress on every call, with the
//     caller's device current, so it is always the current context's copy.
#include <cuda_runtime.h>

#include <cstdio>

#include "varlen_attn.h"

namespace va {
void set_error(const char* msg);
}

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the static scratch in the current device's context.
va_status scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess || !p) {
    char msg[160];
    std::snprintf(msg, sizeof msg, "fwd_noalloc: cudaGetSymbolAddress of the static scratch failed: %s",
                  cudaGetErrorString(e));
    va::set_error(msg);
    return VA_ERR_CUDA;
  }
  *out = p;
  return VA_OK;
}

}  // namespace

extern "C" va_status varlen_attn_fwd_noalloc(const void* q_dev, const void* k_dev, const void* v_dev,
                                             const int32_t* cu_seqlens_dev, const va_shape* shape,
                                             float scale, int32_t causal, void* out_dev, float* lse_dev,
                                             va_stream_t stream) {
  const size_t need = varlen_attn_workspace_size(shape, 0);
  if (need == 0)  // the shape itself is invalid: let the forward report why
    return varlen_attn_fwd(q_dev, k_dev, v_dev, cu_seqlens_dev, shape, scale, causal, out_dev, lse_dev,
                           nullptr, 0, stream);
  if (need > kNoAllocScratchBytes) {
    char msg[256];
    std::snprintf(msg, sizeof msg,
                  "fwd_noalloc: this shape needs %zu bytes of scratch (varlen_attn_workspace_size) but the "
                  "static array holds %zu; use varlen_attn_fwd with a workspace",
                  need, kNoAllocScratchBytes);
    va::set_error(msg);
    return VA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const va_status st = scratch_address(&scratch);
  if (st != VA_OK) return st;
  return varlen_attn_fwd(q_dev, k_dev, v_dev, cu_seqlens_dev, shape, scale, causal, out_dev, lse_dev,
                         scratch, kNoAllocScratchBytes, stream);
}

extern "C" va_status varlen_noalloc_read_status(int32_t* status_host, va_stream_t stream) {
  if (!status_host) {
    va::set_error("noalloc_read_status: null pointer");
    return VA_ERR_INVALID_ARG;
  }
  void* scratch = nullptr;
  const va_status st = scratch_address(&scratch);
  if (st != VA_OK) return st;
  return varlen_read_status(scratch, status_host, stream);
}
