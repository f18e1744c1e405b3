// Backward preparation, one launch: D_i = dO_i . O_i for every (token, q head), fp32
// [Hq, T] -- the row term of dS_ij = P_ij (dP_ij - D_i) in the analytic gradient of the
// forward ("Packing与 FlashAttention Varlen", section 5 names the training branch) --
// while two extra CTAs validate cu_seqlens and build the dK/dV and the dQ tile map, one map
// each (plan_body.cuh).  D does not depend on the boundaries, so all of them run side by side.
// HBM-bound: 16-byte streaming loads, several rows in flight per warp.
#include <algorithm>

#include "attn_params.cuh"
#include "plan_body.cuh"

namespace va {

// 32-byte read-only load that does not allocate in L1 (O and dO are read once here).
__device__ __forceinline__ void ld_stream32(const void* ptr, uint32_t (&r)[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "l"(ptr));
}
__device__ __forceinline__ void ld_stream16(const void* ptr, uint32_t (&r)[8]) {
  const uint4 x = __ldcs(reinterpret_cast<const uint4*>(ptr));
  r[0] = x.x;
  r[1] = x.y;
  r[2] = x.z;
  r[3] = x.w;
}

// D[h, t] = sum_c dO[t,h,c] * O[t,h,c].  Each lane reads VB bytes (VB/2 values) of O and of
// dO per load (32 when every row start is 32-byte aligned, else 16); D*2/VB lanes share a
// row and reduce with shuffles; each warp keeps UNR row groups in flight.
// Blocks 0..nblk-1 of the D computation.
template <int D, int VB>
__device__ __forceinline__ void rowsum_body(const BwdParams& p, int blk, int nblk) {
  constexpr int EPL = VB / 2;           // values per lane
  constexpr int LPR = D / EPL;          // lanes per row
  constexpr int RPW = 32 / LPR;         // rows per warp per group
  constexpr int UNR = VB == 32 ? 2 : 4; // row groups in flight (same bytes either way)
  const int lane = threadIdx.x & 31, sub = lane % LPR, slot = lane / LPR;
  const int rows = p.T * p.Hq;  // < 2^31 for every shape the library accepts
  const int warp0 = static_cast<int>((blk * blockDim.x + threadIdx.x) >> 5);
  const int nwarps = static_cast<int>((nblk * blockDim.x) >> 5);
  for (int r0 = warp0 * RPW * UNR; r0 < rows; r0 += nwarps * RPW * UNR) {
    uint32_t a[UNR][8], b[UNR][8];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int r = r0 + u * RPW + slot;
      if (r < rows) {
        const int t = r / p.Hq, h = r - t * p.Hq;
        const int64_t off = static_cast<int64_t>(t) * p.o_rs + static_cast<int64_t>(h) * p.o_hs + sub * EPL;
        if (VB == 32) {
          ld_stream32(p.o + off, a[u]);
          ld_stream32(p.dout + off, b[u]);
        } else {
          ld_stream16(p.o + off, a[u]);
          ld_stream16(p.dout + off, b[u]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) a[u][j] = b[u][j] = 0u;
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < EPL / 2; ++j) {
        const float2 fx = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a[u][j]));
        const float2 fy = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&b[u][j]));
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

// Two CTAs of 512 threads per SM: one wave holds the planning CTAs and the D blocks.
constexpr int kPrepThreads = 512;
constexpr int kPrepPerSm = 2;

// The first nplan blocks validate and plan (the status word gates the attention kernels
// that follow, not this launch): with nplan = 2 block i builds map i, so the two maps are
// built side by side; with nplan = 1 block 0 builds both.  The other blocks compute D.
template <int D, int VB>
__global__ void __launch_bounds__(kPrepThreads, kPrepPerSm)
    bwd_prep_kernel(const BwdParams p, const PlanPair pp, int nplan) {
  __shared__ PlanSmem sh;
  griddep_begin();  // O comes from the forward, and the workspace may be the forward's
  if (static_cast<int>(blockIdx.x) < nplan) {
    validate_plan_body(pp, sh, nplan == 1 ? -1 : static_cast<int>(blockIdx.x));
    return;
  }
  rowsum_body<D, VB>(p, blockIdx.x - nplan, gridDim.x - nplan);
}

cudaError_t launch_bwd_prep(const BwdParams& p, const PlanArgs* maps, int nmaps, int T, int max_seqlen, int Tk,
                            int max_seqlen_k, int d, cudaStream_t st) {
  PlanPair pp{};
  for (int i = 0; i < nmaps && i < 2; ++i) pp.map[i] = maps[i];
  pp.nmaps = nmaps;
  pp.T = T;
  pp.max_seqlen = max_seqlen;
  pp.Tk = Tk;
  pp.max_seqlen_k = max_seqlen_k;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // one planning block per map while the per-segment offsets fit in shared memory (beyond
  // that the maps share one global array of them, and one block builds both in turn)
  const int nplan = nmaps == 2 && maps[0].B + 1 <= kSmemSegs ? 2 : 1;
  const int64_t rows = static_cast<int64_t>(p.T) * p.Hq;
  const int rpb = (kPrepThreads / 32) * (32 / (d / 8)) * 4;   // rows per block per pass (16-byte loads)
  const int rb = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(std::max(sms, 1) * kPrepPerSm - nplan,
                                                                        (rows + rpb - 1) / rpb)));
  // 32-byte loads when every row start of O and dO is 32-byte aligned
  const bool a32 = (reinterpret_cast<uintptr_t>(p.o) & 31) == 0 && (reinterpret_cast<uintptr_t>(p.dout) & 31) == 0 &&
                   p.o_rs % 16 == 0 && p.o_hs % 16 == 0;
  const dim3 grid(rb + nplan), block(kPrepThreads);
  if (d == 64)
    return a32 ? launch_pdl(bwd_prep_kernel<64, 32>, grid, block, 0, st, p, pp, nplan)
               : launch_pdl(bwd_prep_kernel<64, 16>, grid, block, 0, st, p, pp, nplan);
  return a32 ? launch_pdl(bwd_prep_kernel<128, 32>, grid, block, 0, st, p, pp, nplan)
             : launch_pdl(bwd_prep_kernel<128, 16>, grid, block, 0, st, p, pp, nplan);
}


}  // namespace va
