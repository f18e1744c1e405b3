// Backward preprocessing: D_i = dO_i . O_i for every (token, q head), fp32 [Hq, T].
// It is the row term of dS_ij = P_ij (dP_ij - D_i) in the analytic gradient of the
// forward ("Packing与 FlashAttention Varlen", section 5 names the training branch).
// HBM-bound: 16-byte loads, several rows in flight per warp.
#include <algorithm>

#include "attn_params.cuh"

namespace va {

// D[h, t] = sum_c dO[t,h,c] * O[t,h,c].  Each thread reads 8 consecutive elements of
// O and dO (16-byte loads); D/8 lanes share a row and reduce with shuffles; each warp
// keeps 4 row groups in flight per iteration.
template <int D>
__global__ void __launch_bounds__(256) bwd_rowsum_kernel(const BwdParams p) {
  constexpr int LPR = D / 8;            // lanes per row
  constexpr int RPW = 32 / LPR;         // rows per warp per group
  constexpr int UNR = 4;                // row groups in flight
  if (p.hdr->status != VA_OK) return;
  const int lane = threadIdx.x & 31, sub = lane % LPR, slot = lane / LPR;
  const int rows = p.T * p.Hq;  // < 2^31 for every shape the library accepts
  const int warp0 = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int nwarps = static_cast<int>((gridDim.x * blockDim.x) >> 5);
  for (int r0 = warp0 * RPW * UNR; r0 < rows; r0 += nwarps * RPW * UNR) {
    uint4 a[UNR], b[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int r = r0 + u * RPW + slot;
      if (r < rows) {
        const int t = r / p.Hq, h = r - t * p.Hq;
        const int64_t off = static_cast<int64_t>(t) * p.o_rs + static_cast<int64_t>(h) * p.o_hs + sub * 8;
        a[u] = __ldg(reinterpret_cast<const uint4*>(p.o + off));
        b[u] = __ldg(reinterpret_cast<const uint4*>(p.dout + off));
      } else {
        a[u] = b[u] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a[u]);
      const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b[u]);
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 fx = __bfloat1622float2(x[j]), fy = __bfloat1622float2(y[j]);
        acc = fmaf(fx.x, fy.x, fmaf(fx.y, fy.y, acc));
      }
#pragma unroll
      for (int s2 = LPR / 2; s2 > 0; s2 >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s2);
      const int r = r0 + u * RPW + slot;
      if (sub == 0 && r < rows) {
        const int t = r / p.Hq, h = r - t * p.Hq;
        p.dsum[static_cast<int64_t>(h) * p.T + t] = acc;
      }
    }
  }
}

cudaError_t launch_bwd_rowsum(const BwdParams& p, int d, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(p.T) * p.Hq;
  const int rpb = (256 / 32) * (32 / (d / 8)) * 4;   // rows per block per iteration
  const int rb = static_cast<int>(std::min<int64_t>(152 * 8, (rows + rpb - 1) / rpb));
  if (rb <= 0) return cudaSuccess;
  if (d == 64) bwd_rowsum_kernel<64><<<rb, 256, 0, st>>>(p);
  else bwd_rowsum_kernel<128><<<rb, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace va
