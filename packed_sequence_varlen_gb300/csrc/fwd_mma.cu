// Forward varlen attention, warp-level mma.sync path (bf16 in, fp32 accumulate).
//
// "Packing与 FlashAttention Varlen", section 5: a work item (segment b, q block
// m, head h) reads Q/K/V rows at offset cu[b] of the flat token axis with
// extent l_b = cu[b+1]-cu[b]; rows past l_b are never loaded (zero fill) and
// never stored, so no cross-segment value is read or written; the causal mask
// is applied only on key blocks that cross the diagonal.  O is written at Q's
// offsets (same flat order as the input) and lse = ln sum exp(scale q.k).
//
// CTA = 8 warps = 128 query rows (16 per warp), key blocks of 64 rows, K/V
// double buffered with cp.async, online softmax in base 2.
#include "attn_params.cuh"

namespace va {

namespace {
constexpr int kFwdBM = 128;
constexpr int kFwdBN = 64;
constexpr int kFwdThreads = 256;
}  // namespace

template <int D>
__global__ void __launch_bounds__(kFwdThreads, 1) fwd_mma_kernel(const FwdParams p) {
  constexpr int BM = kFwdBM, BN = kFwdBN, NT = kFwdThreads;
  constexpr int CPR = D / 8;  // 16-byte chunks per row
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + BM * D * 2;
  uint8_t* sV = sK + 2 * BN * D * 2;

  if (p.hdr->status != VA_OK) return;
  if (static_cast<int>(blockIdx.x) >= p.hdr->n_items[p.slot]) return;
  const TileItem it = p.items[blockIdx.x];
  const int b = it.seg, m = it.blk, h = it.head, nb = it.count;
  const int s0 = p.cu[b];
  const int l = p.cu[b + 1] - s0;
  const int hk = h / p.g;
  const int row0 = m * BM;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const bf16* qb = p.q + static_cast<int64_t>(s0) * p.q_rs + static_cast<int64_t>(h) * p.q_hs;
  const bf16* kb = p.k + static_cast<int64_t>(s0) * p.k_rs + static_cast<int64_t>(hk) * p.k_hs;
  const bf16* vb = p.v + static_cast<int64_t>(s0) * p.v_rs + static_cast<int64_t>(hk) * p.v_hs;

  for (int c = tid; c < BM * CPR; c += NT) {
    const int r = c / CPR, cc = c % CPR;
    const bool ok = row0 + r < l;
    cp_async16(smem_u32(sQ) + swz<D>(r, cc), qb + static_cast<int64_t>(ok ? row0 + r : 0) * p.q_rs + cc * 8, ok);
  }
  auto load_kv = [&](int n, int buf) {
    const uint32_t dk = smem_u32(sK + buf * BN * D * 2), dv = smem_u32(sV + buf * BN * D * 2);
    for (int c = tid; c < BN * CPR; c += NT) {
      const int r = c / CPR, cc = c % CPR;
      const int kr = n * BN + r;
      const bool ok = kr < l;
      const int64_t rr = ok ? kr : 0;
      cp_async16(dk + swz<D>(r, cc), kb + rr * p.k_rs + cc * 8, ok);
      cp_async16(dv + swz<D>(r, cc), vb + rr * p.v_rs + cc * 8, ok);
    }
  };
  load_kv(0, 0);
  cp_async_commit();

  float oacc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};
  uint32_t qf[D / 16][4];
  const int g8 = lane >> 2, t4 = lane & 3;
  const int wrow0 = row0 + warp * 16;  // first local row of this warp

  for (int n = 0; n < nb; ++n) {
    if (n + 1 < nb) load_kv(n + 1, (n + 1) & 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (n == 0) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int r = warp * 16 + (lane & 15);
        const int cc = kk * 2 + (lane >> 4);
        ldsm_x4(smem_u32(sQ) + swz<D>(r, cc), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    const uint32_t kbuf = smem_u32(sK + (n & 1) * BN * D * 2);
    const uint32_t vbuf = smem_u32(sV + (n & 1) * BN * D * 2);
    float s[BN / 8][4];
#pragma unroll
    for (int t = 0; t < BN / 8; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < BN / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        const int r = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int cc = kk * 2 + ((lane >> 3) & 1);
        ldsm_x4(kbuf + swz<D>(r, cc), b0, b1, b2, b3);
        mma_bf16(s[2 * np], qf[kk], b0, b1);
        mma_bf16(s[2 * np + 1], qf[kk], b2, b3);
      }
    }
    const bool need_mask = p.causal ? (n * BN + BN - 1 > wrow0) : (n * BN + BN > l);
    if (need_mask) {
#pragma unroll
      for (int t = 0; t < BN / 8; ++t) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = n * BN + t * 8 + 2 * t4 + (e & 1);
          const int row = wrow0 + g8 + ((e >> 1) << 3);
          const bool bad = p.causal ? (col > row) : (col >= l);
          if (bad) s[t][e] = -INFINITY;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float mx = -INFINITY;
#pragma unroll
      for (int t = 0; t < BN / 8; ++t) mx = fmaxf(mx, fmaxf(s[t][2 * r], s[t][2 * r + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mnew = fmaxf(mrun[r], mx * p.scale_log2);
      const float muse = mnew == -INFINITY ? 0.f : mnew;
      const float alpha = fast_exp2(mrun[r] - muse);
      mrun[r] = mnew;
      float rs = 0.f;
#pragma unroll
      for (int t = 0; t < BN / 8; ++t) {
        const float p0 = fast_exp2(s[t][2 * r] * p.scale_log2 - muse);
        const float p1 = fast_exp2(s[t][2 * r + 1] * p.scale_log2 - muse);
        s[t][2 * r] = p0;
        s[t][2 * r + 1] = p1;
        rs += p0 + p1;
      }
      lrun[r] = lrun[r] * alpha + rs;
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt) {
        oacc[dt][2 * r] *= alpha;
        oacc[dt][2 * r + 1] *= alpha;
      }
    }
#pragma unroll
    for (int j = 0; j < BN / 16; ++j) {
      uint32_t a[4] = {pack_bf16(s[2 * j][0], s[2 * j][1]), pack_bf16(s[2 * j][2], s[2 * j][3]),
                       pack_bf16(s[2 * j + 1][0], s[2 * j + 1][1]),
                       pack_bf16(s[2 * j + 1][2], s[2 * j + 1][3])};
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t b0, b1, b2, b3;
        const int r = j * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int cc = dp * 2 + (lane >> 4);
        ldsm_x4_t(vbuf + swz<D>(r, cc), b0, b1, b2, b3);
        mma_bf16(oacc[2 * dp], a, b0, b1);
        mma_bf16(oacc[2 * dp + 1], a, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // epilogue: normalise, stage bf16 rows in shared memory, copy rows < l out
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    lrun[r] += __shfl_xor_sync(0xffffffffu, lrun[r], 1);
    lrun[r] += __shfl_xor_sync(0xffffffffu, lrun[r], 2);
  }
  const float inv0 = 1.f / lrun[0], inv1 = 1.f / lrun[1];
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
    const int col = dt * 8 + 2 * t4;
    const int r0 = warp * 16 + g8;
    *reinterpret_cast<uint32_t*>(sQ + swz<D>(r0, dt) + (col & 7) * 2) =
        pack_bf16(oacc[dt][0] * inv0, oacc[dt][1] * inv0);
    *reinterpret_cast<uint32_t*>(sQ + swz<D>(r0 + 8, dt) + (col & 7) * 2) =
        pack_bf16(oacc[dt][2] * inv1, oacc[dt][3] * inv1);
  }
  if (t4 == 0) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = wrow0 + g8 + 8 * r;
      if (row < l) p.lse[static_cast<int64_t>(h) * p.T + s0 + row] = (mrun[r] + __log2f(lrun[r])) * kLn2;
    }
  }
  __syncthreads();
  bf16* ob = p.o + static_cast<int64_t>(s0) * p.o_rs + static_cast<int64_t>(h) * p.o_hs;
  for (int c = tid; c < BM * CPR; c += NT) {
    const int r = c / CPR, cc = c % CPR;
    if (row0 + r < l) {
      const uint4 val = *reinterpret_cast<const uint4*>(sQ + swz<D>(r, cc));
      *reinterpret_cast<uint4*>(ob + static_cast<int64_t>(row0 + r) * p.o_rs + cc * 8) = val;
    }
  }
}

template <int D>
static cudaError_t launch_fwd_mma_d(const FwdParams& p, int grid, cudaStream_t st) {
  const int smem = (kFwdBM + 4 * kFwdBN) * D * 2;
  cudaError_t e = cudaFuncSetAttribute(fwd_mma_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (grid > 0) fwd_mma_kernel<D><<<grid, kFwdThreads, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_mma(const FwdParams& p, int d, int grid, cudaStream_t st) {
  return d == 64 ? launch_fwd_mma_d<64>(p, grid, st) : launch_fwd_mma_d<128>(p, grid, st);
}

void fwd_mma_tiles(int* BM, int* BN) {
  *BM = kFwdBM;
  *BN = kFwdBN;
}

}  // namespace va
