// Backward preparation, one launch: D_i = dO_i . O_i for every (token, q head), fp32
// [Hq, T] -- the row term of dS_ij = P_ij (dP_ij - D_i) in the analytic gradient of the
// forward ("Packing与 FlashAttention Varlen", section 5 names the training branch) --
// while one extra CTA validates cu_seqlens and builds the dK/dV and dQ tile maps
// (plan_body.cuh).  D does not depend on the boundaries, so the two run side by side.
// HBM-bound: 16-byte streaming loads, several rows in flight per warp.
#include <algorithm>

#include "attn_params.cuh"
#include "plan_body.cuh"

namespace va {

// D[h, t] = sum_c dO[t,h,c] * O[t,h,c].  Each thread reads 8 consecutive elements of
// O and dO (16-byte loads); D/8 lanes share a row and reduce with shuffles; each warp
// keeps 4 row groups in flight per iteration.
// Blocks 0..nblk-1 of the D computation.
template <int D>
__device__ __forceinline__ void rowsum_body(const BwdParams& p, int blk, int nblk) {
  constexpr int LPR = D / 8;            // lanes per row
  constexpr int RPW = 32 / LPR;         // rows per warp per group
  constexpr int UNR = 4;                // row groups in flight
  const int lane = threadIdx.x & 31, sub = lane % LPR, slot = lane / LPR;
  const int rows = p.T * p.Hq;  // < 2^31 for every shape the library accepts
  const int warp0 = static_cast<int>((blk * blockDim.x + threadIdx.x) >> 5);
  const int nwarps = static_cast<int>((nblk * blockDim.x) >> 5);
  for (int r0 = warp0 * RPW * UNR; r0 < rows; r0 += nwarps * RPW * UNR) {
    uint4 a[UNR], b[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int r = r0 + u * RPW + slot;
      if (r < rows) {
        const int t = r / p.Hq, h = r - t * p.Hq;
        const int64_t off = static_cast<int64_t>(t) * p.o_rs + static_cast<int64_t>(h) * p.o_hs + sub * 8;
        // streaming loads (evict-first): O and dO are read once here
        a[u] = __ldcs(reinterpret_cast<const uint4*>(p.o + off));
        b[u] = __ldcs(reinterpret_cast<const uint4*>(p.dout + off));
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

constexpr int kPrepThreads = 1024;

// Block 0 validates and plans (the status word it writes gates the attention kernels that
// follow, not this launch); blocks 1.. compute D.
template <int D>
__global__ void __launch_bounds__(kPrepThreads) bwd_prep_kernel(const BwdParams p, const PlanPair pp) {
  __shared__ PlanSmem sh;
  griddep_begin();  // O comes from the forward, and the workspace may be the forward's
  if (blockIdx.x == 0) {
    validate_plan_body(pp, sh);
    return;
  }
  rowsum_body<D>(p, blockIdx.x - 1, gridDim.x - 1);
}

cudaError_t launch_bwd_prep(const BwdParams& p, const PlanArgs* maps, int nmaps, int T, int max_seqlen, int d,
                            cudaStream_t st) {
  PlanPair pp{};
  for (int i = 0; i < nmaps && i < 2; ++i) pp.map[i] = maps[i];
  pp.nmaps = nmaps;
  pp.T = T;
  pp.max_seqlen = max_seqlen;
  const int64_t rows = static_cast<int64_t>(p.T) * p.Hq;
  const int rpb = (kPrepThreads / 32) * (32 / (d / 8)) * 4;   // rows per block per iteration
  const int rb = static_cast<int>(std::min<int64_t>(152 * 4, (rows + rpb - 1) / rpb));
  if (d == 64) return launch_pdl(bwd_prep_kernel<64>, dim3(rb + 1), dim3(kPrepThreads), 0, st, p, pp);
  return launch_pdl(bwd_prep_kernel<128>, dim3(rb + 1), dim3(kPrepThreads), 0, st, p, pp);
}


}  // namespace va
