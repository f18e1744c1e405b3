// Forward attention for callers that cannot allocate device memory.
//
// Some callers have no way to obtain scratch memory at the point where they
// run attention: a plugin executed by a host runtime that owns every device
// allocation and offers no scratch API, or a latency-critical serving loop
// that must not call cudaMalloc because it can synchronise the device and
// stall the other streams.  varlen_attn_fwd_noalloc serves them: it runs the
// ordinary forward (contract check, tile plan, attention kernel) with its
// scratch -- the 256-byte status header and the tile map -- in a fixed,
// file-scope device array instead of a caller workspace.
//
// Properties of the static scratch:
//   * kNoAllocScratchBytes (1 MiB) on every GPU that loads this library, held
//     until the process exits; it fits tile maps of up to 65,520 records, i.e.
//     (T/256 rounded down + B) * Hq <= 65,520.  Larger shapes are rejected with
//     VA_ERR_WORKSPACE.
//   * Every call on a device shares it and it keeps the last call's contents.
//     The contract check overwrites the status word and the plan rewrites the
//     record count and the map, so nothing needs clearing between calls.
//     Calls that overlap on the GPU (other streams, other host threads) race on
//     it and must be serialised by the caller.
//   * In host code the array's name is only a host-side stand-in; its device
//     address is fetched with cudaGetSymbolAddress once per device, with that
//     device current, on the first call made on it.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "varlen_attn.h"

namespace va {
void set_error(const char* msg);
}

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_dev[kMaxDevices] = {};

// Device address of the static scratch on the current device (set-up on first use).
va_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    va::set_error("fwd_noalloc: no usable current CUDA device");
    return VA_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      va::set_error("fwd_noalloc: cudaGetSymbolAddress of the static scratch failed");
      return VA_ERR_CUDA;
    }
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
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
                  "fwd_noalloc: this shape needs %zu bytes of scratch but the static array holds "
                  "%zu ((T/256 + B) * Hq tile records must be <= 65520); use varlen_attn_fwd with a "
                  "workspace",
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
