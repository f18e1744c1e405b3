// Backward preprocessing: D_i = dO_i . O_i for every (token, q head), fp32 [Hq, T].
// It is the row term of dS_ij = P_ij (dP_ij - D_i) in the analytic gradient of the
// forward ("Packing与 FlashAttention Varlen", section 5 names the training branch).
// HBM-bound: one warp per row, bf16x2 loads.
#include <algorithm>

#include "attn_params.cuh"

namespace va {

// D[h, t] = sum_c dO[t,h,c] * O[t,h,c], one warp per (t, h).
template <int D>
__global__ void __launch_bounds__(256) bwd_rowsum_kernel(const BwdParams p) {
  if (p.hdr->status != VA_OK) return;
  const int lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(p.T) * p.Hq;
  for (int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; r < rows;
       r += (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5) {
    const int t = static_cast<int>(r / p.Hq), h = static_cast<int>(r % p.Hq);
    const bf16* o = p.o + static_cast<int64_t>(t) * p.o_rs + static_cast<int64_t>(h) * p.o_hs;
    const bf16* g = p.dout + static_cast<int64_t>(t) * p.o_rs + static_cast<int64_t>(h) * p.o_hs;
    float acc = 0.f;
#pragma unroll
    for (int c = lane * 2; c < D; c += 64) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(o + c));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(g + c));
      acc = fmaf(a.x, b.x, fmaf(a.y, b.y, acc));
    }
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) p.dsum[static_cast<int64_t>(h) * p.T + t] = acc;
  }
}

cudaError_t launch_bwd_rowsum(const BwdParams& p, int d, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(p.T) * p.Hq;
  const int rb = static_cast<int>(std::min<int64_t>(152 * 16, (rows * 32 + 255) / 256));
  if (rb <= 0) return cudaSuccess;
  if (d == 64) bwd_rowsum_kernel<64><<<rb, 256, 0, st>>>(p);
  else bwd_rowsum_kernel<128><<<rb, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace va
