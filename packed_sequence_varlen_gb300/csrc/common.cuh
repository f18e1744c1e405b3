// Device helpers shared by the varlen attention kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "varlen_attn.h"

namespace va {

// Workspace header: the first 256 bytes of every workspace.
//   int32 status      -- 0 ok, else a va_status written by a kernel
//   int32 n_items[4]  -- record counts written by the plan kernels
//   int32 where       -- diagnostic (which wait gave up)
//   int32 counter[4]  -- work counters the attention kernels pull records from
// Forward workspaces: n_items[0] counts all records of the map, n_items[kTokSlot] the
// token records at its end; counter[kTokSlot] is the token kernel's work counter.
// Backward workspaces: n_items[1] / n_items[2] count all records of the kv-block / q-block
// maps, n_items[kKvTokSlot] / n_items[kQTokSlot] the token records at their ends;
// counter[1] / counter[2] are the dK/dV and dQ kernels' work counters.
constexpr int kTokSlot = 3;
constexpr int kKvTokSlot = 0, kQTokSlot = 3;

struct WsHeader {
  int32_t status;
  int32_t n_items[4];
  int32_t where;
  int32_t counter[4];
  int32_t pad[54];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

struct alignas(16) TileItem {  // one scheduler record
  int32_t seg, blk, head, count;
};

// Arguments of one tile-map build (see plan.cu).
struct PlanArgs {
  const int32_t* cu;
  int B;
  int heads;
  int BM, BN;
  int kind;  // 0/2: q-block map, 1: kv-block map
  int causal;
  TileItem* out;
  int capacity;
  int32_t* status;   // may be null: no status to honour or report
  int32_t* n_items;  // out
  int32_t* seg_off;  // scratch [B]: first record of each segment
  int32_t* counter;  // work counter the attention kernel pulls items from; zeroed here
  int short_len;      // causal: segments of at most this many tokens go into token tiles
                      // (records {-1 - f, t0, head, rows}); 0 = off
  int32_t* n_tok;     // may be null: out, the number of token records (the map's last ones)
  int32_t* tok_counter;  // may be null: the token kernel's work counter; zeroed here
  int window = -1;       // causal local window w >= 0 (query i sees keys i-w..i), -1 = none;
                         // window maps have no token records
  const int32_t* cu_k = nullptr;  // cross-attention: the K/V boundaries (cu is Q's); null = cu
};

__device__ __forceinline__ void set_status(WsHeader* h, int code) {
  atomicCAS(&h->status, 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Three-input max (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed fp32x2 fused multiply-add / add: (d0, d1) = (a0*b0 + c0, a1*b1 + c1).
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                      float c0, float c1) {
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Stores 32 rows held one per lane (W 16-byte chunks each, W a multiple of 8) so that
// every 8 lanes write 128 contiguous bytes.  Within each group of 8 lanes an 8 x 8
// transpose of 16-byte chunks (three xor-shuffle stages) leaves lane j with chunk j of
// each of the group's 8 rows; store k then writes row (group base + k).  `row` is this
// lane's row, rows of consecutive lanes are `stride` elements apart, and a row is written
// only when its own lane passed valid = true.  Warp-collective.
template <int W, class T>
__device__ __forceinline__ void store_rows_coalesced(uint4 (&a)[W], T* row, int64_t stride, bool valid) {
  static_assert(W % 8 == 0, "rows must be a multiple of 128 bytes");
  const int lane = threadIdx.x & 31, j = lane & 7;
  const unsigned vmask = __ballot_sync(0xffffffffu, valid);
#pragma unroll
  for (int b = 0; b < W / 8; ++b) {
    uint4* c = a + 8 * b;
#pragma unroll
    for (int d = 4; d >= 1; d >>= 1) {
      const bool hi = (j & d) != 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (i & d) continue;
        const uint4 send = hi ? c[i] : c[i + d];
        uint4 recv;
        recv.x = __shfl_xor_sync(0xffffffffu, send.x, d);
        recv.y = __shfl_xor_sync(0xffffffffu, send.y, d);
        recv.z = __shfl_xor_sync(0xffffffffu, send.z, d);
        recv.w = __shfl_xor_sync(0xffffffffu, send.w, d);
        if (hi) c[i] = recv;
        else c[i + d] = recv;
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if ((vmask >> ((lane & ~7) + k)) & 1u)
        reinterpret_cast<uint4*>(row + static_cast<int64_t>(k - j) * stride)[8 * b + j] = c[k];
    }
  }
}

// Same contract as store_rows_coalesced, with 32-byte stores: within each group of 4 lanes
// a 4 x 4 transpose of 32-byte chunks (two xor-shuffle stages) leaves lane j with chunk j
// of each of the group's 4 rows, and every store instruction writes 128 contiguous bytes
// per group with half the instructions.
template <int W, class T>
__device__ __forceinline__ void store_rows_coalesced32(uint4 (&a)[W], T* row, int64_t stride, bool valid) {
  static_assert(W % 8 == 0, "rows must be a multiple of 128 bytes");
  const int lane = threadIdx.x & 31, j = lane & 3;
  const unsigned vmask = __ballot_sync(0xffffffffu, valid);
#pragma unroll
  for (int b = 0; b < W / 8; ++b) {
    uint4* c = a + 8 * b;  // four 32-byte chunks: (c[0], c[1]), (c[2], c[3]), ...
#pragma unroll
    for (int d = 2; d >= 1; d >>= 1) {
      const bool hi = (j & d) != 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (i & d) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint4 send = hi ? c[2 * i + h] : c[2 * (i + d) + h];
          uint4 recv;
          recv.x = __shfl_xor_sync(0xffffffffu, send.x, d);
          recv.y = __shfl_xor_sync(0xffffffffu, send.y, d);
          recv.z = __shfl_xor_sync(0xffffffffu, send.z, d);
          recv.w = __shfl_xor_sync(0xffffffffu, send.w, d);
          if (hi) c[2 * i + h] = recv;
          else c[2 * (i + d) + h] = recv;
        }
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if ((vmask >> ((lane & ~3) + k)) & 1u) {
        char* dst = reinterpret_cast<char*>(row + static_cast<int64_t>(k - j) * stride) + 128 * b + 32 * j;
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(c[2 * k].x),
                     "r"(c[2 * k].y), "r"(c[2 * k].z), "r"(c[2 * k].w), "r"(c[2 * k + 1].x), "r"(c[2 * k + 1].y),
                     "r"(c[2 * k + 1].z), "r"(c[2 * k + 1].w)
                     : "memory");
      }
    }
  }
}

// store_rows_coalesced32 when every row of the warp starts on a 32-byte boundary (the
// 256-bit stores need it), store_rows_coalesced otherwise.
template <int W, class T>
__device__ __forceinline__ void store_rows_fast(uint4 (&a)[W], T* row, int64_t stride, bool valid) {
  if (__all_sync(0xffffffffu, (reinterpret_cast<uintptr_t>(row) & 31u) == 0))
    store_rows_coalesced32(a, row, stride, valid);
  else
    store_rows_coalesced(a, row, stride, valid);
}

// Programmatic dependent launch.  Every kernel of the library starts with griddep_begin():
// it waits until the grids it depends on have completed and their writes are visible
// (at once when launched without the attribute), then lets the next grid in the stream
// be scheduled.  That next grid's CTAs take SMs only after all of this grid's CTAs have
// started, and wait in their own griddep_begin(), so launch latency and prologues overlap
// the previous kernel without any read or write reordering.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_begin() {
  griddep_wait();
  griddep_launch_dependents();
}

// Launches `kernel` with programmatic stream serialization allowed (see griddep_begin).
template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace va
