// Backward varlen attention, warp-level mma.sync path.
//
// The gradient of the forward definition, with P recomputed from the forward's
// lse ("Packing与 FlashAttention Varlen", section 5 names the training branch):
//   D_i = dO_i . O_i;  P_ij = exp(scale q_i.k_j - lse_i) on visible (i, j);
//   dV_j = sum_i P_ij dO_i;  dS_ij = P_ij (dO_i . v_j - D_i);
//   dK_j = scale sum_i dS_ij q_i;  dQ_i = scale sum_j dS_ij k_j.
// Three kernels: rowsum D; a kv-block kernel that owns dK/dV rows of one kv head
// (summing its q-head group, no atomics); a q-block kernel that owns dQ rows.
// Every kernel keeps to its segment's rows: loads past the segment end are
// zero-filled and those rows are never stored.
#include <algorithm>

#include "attn_params.cuh"

namespace va {

namespace {
constexpr int kDqBM = 128, kDqBN = 64;     // dQ kernel: q rows per CTA, key rows per step
constexpr int kKvBN = 128, kKvBM = 32;     // dK/dV kernel: kv rows per CTA, q rows per step
constexpr int kThreads = 256;
}  // namespace

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

// dQ for one (segment, q block of 128 rows, q head).
template <int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_dq_kernel(const BwdParams p) {
  constexpr int BM = kDqBM, BN = kDqBN, NT = kThreads, CPR = D / 8;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sQ = smem;
  uint8_t* sdO = sQ + BM * D * 2;
  uint8_t* sK = sdO + BM * D * 2;
  uint8_t* sV = sK + 2 * BN * D * 2;
  if (p.hdr->status != VA_OK) return;
  if (static_cast<int>(blockIdx.x) >= p.hdr->n_items[p.q_slot]) return;
  const TileItem it = p.q_items[blockIdx.x];
  const int b = it.seg, m = it.blk, h = it.head, nb = it.count;
  const int s0 = p.cu[b], l = p.cu[b + 1] - s0, hk = h / p.g, row0 = m * BM;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g8 = lane >> 2, t4 = lane & 3;
  const int wrow0 = row0 + warp * 16;

  const bf16* qb = p.q + static_cast<int64_t>(s0) * p.q_rs + static_cast<int64_t>(h) * p.q_hs;
  const bf16* ob = p.dout + static_cast<int64_t>(s0) * p.o_rs + static_cast<int64_t>(h) * p.o_hs;
  const bf16* kb = p.k + static_cast<int64_t>(s0) * p.k_rs + static_cast<int64_t>(hk) * p.k_hs;
  const bf16* vb = p.v + static_cast<int64_t>(s0) * p.v_rs + static_cast<int64_t>(hk) * p.v_hs;
  for (int c = tid; c < BM * CPR; c += NT) {
    const int r = c / CPR, cc = c % CPR;
    const bool ok = row0 + r < l;
    const int64_t rr = ok ? row0 + r : 0;
    cp_async16(smem_u32(sQ) + swz<D>(r, cc), qb + rr * p.q_rs + cc * 8, ok);
    cp_async16(smem_u32(sdO) + swz<D>(r, cc), ob + rr * p.o_rs + cc * 8, ok);
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

  float lse2[2], dsum[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = wrow0 + g8 + 8 * r;
    const bool ok = row < l;
    lse2[r] = ok ? p.lse[static_cast<int64_t>(h) * p.T + s0 + row] * kLog2e : 0.f;
    dsum[r] = ok ? p.dsum[static_cast<int64_t>(h) * p.T + s0 + row] : 0.f;
  }
  float dq[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) dq[i][0] = dq[i][1] = dq[i][2] = dq[i][3] = 0.f;

  for (int n = 0; n < nb; ++n) {
    if (n + 1 < nb) load_kv(n + 1, (n + 1) & 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint32_t kbuf = smem_u32(sK + (n & 1) * BN * D * 2);
    const uint32_t vbuf = smem_u32(sV + (n & 1) * BN * D * 2);
    float s[BN / 8][4], dp[BN / 8][4];
#pragma unroll
    for (int t = 0; t < BN / 8; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[t][e] = dp[t][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t qa[4], da[4];
      const int r = warp * 16 + (lane & 15), cc = kk * 2 + (lane >> 4);
      ldsm_x4(smem_u32(sQ) + swz<D>(r, cc), qa[0], qa[1], qa[2], qa[3]);
      ldsm_x4(smem_u32(sdO) + swz<D>(r, cc), da[0], da[1], da[2], da[3]);
#pragma unroll
      for (int np = 0; np < BN / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        const int br = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int bc = kk * 2 + ((lane >> 3) & 1);
        ldsm_x4(kbuf + swz<D>(br, bc), b0, b1, b2, b3);
        mma_bf16(s[2 * np], qa, b0, b1);
        mma_bf16(s[2 * np + 1], qa, b2, b3);
        ldsm_x4(vbuf + swz<D>(br, bc), b0, b1, b2, b3);
        mma_bf16(dp[2 * np], da, b0, b1);
        mma_bf16(dp[2 * np + 1], da, b2, b3);
      }
    }
    const bool need_mask = p.causal ? (n * BN + BN - 1 > wrow0) : (n * BN + BN > l);
#pragma unroll
    for (int t = 0; t < BN / 8; ++t) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = e >> 1;
        float pv = fast_exp2(s[t][e] * p.scale_log2 - lse2[r]);
        if (need_mask) {
          const int col = n * BN + t * 8 + 2 * t4 + (e & 1);
          const int row = wrow0 + g8 + 8 * r;
          if (p.causal ? (col > row) : (col >= l)) pv = 0.f;
        }
        s[t][e] = pv * (dp[t][e] - dsum[r]);  // dS
      }
    }
#pragma unroll
    for (int j = 0; j < BN / 16; ++j) {
      uint32_t a[4] = {pack_bf16(s[2 * j][0], s[2 * j][1]), pack_bf16(s[2 * j][2], s[2 * j][3]),
                       pack_bf16(s[2 * j + 1][0], s[2 * j + 1][1]),
                       pack_bf16(s[2 * j + 1][2], s[2 * j + 1][3])};
#pragma unroll
      for (int dpp = 0; dpp < D / 16; ++dpp) {
        uint32_t b0, b1, b2, b3;
        const int r = j * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int cc = dpp * 2 + (lane >> 4);
        ldsm_x4_t(kbuf + swz<D>(r, cc), b0, b1, b2, b3);
        mma_bf16(dq[2 * dpp], a, b0, b1);
        mma_bf16(dq[2 * dpp + 1], a, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  // each warp stages its own rows in sQ (it only ever read its own rows of sQ)
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
    const int col = dt * 8 + 2 * t4, r0 = warp * 16 + g8;
    *reinterpret_cast<uint32_t*>(sQ + swz<D>(r0, dt) + (col & 7) * 2) =
        pack_bf16(dq[dt][0] * p.scale, dq[dt][1] * p.scale);
    *reinterpret_cast<uint32_t*>(sQ + swz<D>(r0 + 8, dt) + (col & 7) * 2) =
        pack_bf16(dq[dt][2] * p.scale, dq[dt][3] * p.scale);
  }
  __syncthreads();
  bf16* out = p.dq + static_cast<int64_t>(s0) * p.o_rs + static_cast<int64_t>(h) * p.o_hs;
  for (int c = tid; c < BM * CPR; c += NT) {
    const int r = c / CPR, cc = c % CPR;
    if (row0 + r < l)
      *reinterpret_cast<uint4*>(out + static_cast<int64_t>(row0 + r) * p.o_rs + cc * 8) =
          *reinterpret_cast<const uint4*>(sQ + swz<D>(r, cc));
  }
}

// dK, dV for one (segment, kv block of 128 rows, kv head), summing the q-head group.
template <int D>
__global__ void __launch_bounds__(kThreads, 1) bwd_dkdv_kernel(const BwdParams p) {
  constexpr int BN = kKvBN, BM = kKvBM, NT = kThreads, CPR = D / 8;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sK = smem;
  uint8_t* sV = sK + BN * D * 2;
  uint8_t* sQ = sV + BN * D * 2;          // [2][BM x D]
  uint8_t* sdO = sQ + 2 * BM * D * 2;     // [2][BM x D]
  float* sL = reinterpret_cast<float*>(sdO + 2 * BM * D * 2);  // [2][BM] lse * log2e
  float* sD = sL + 2 * BM;                                      // [2][BM]
  if (p.hdr->status != VA_OK) return;
  if (static_cast<int>(blockIdx.x) >= p.hdr->n_items[p.kv_slot]) return;
  const TileItem it = p.kv_items[blockIdx.x];
  const int b = it.seg, n = it.blk, hk = it.head, nq = it.count;
  const int s0 = p.cu[b], l = p.cu[b + 1] - s0;
  const int Mq = (l + BM - 1) / BM, m_start = Mq - nq;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g8 = lane >> 2, t4 = lane & 3;
  const int kv0 = n * BN, wkv0 = kv0 + warp * 16;

  const bf16* kb = p.k + static_cast<int64_t>(s0) * p.k_rs + static_cast<int64_t>(hk) * p.k_hs;
  const bf16* vb = p.v + static_cast<int64_t>(s0) * p.v_rs + static_cast<int64_t>(hk) * p.v_hs;
  for (int c = tid; c < BN * CPR; c += NT) {
    const int r = c / CPR, cc = c % CPR;
    const bool ok = kv0 + r < l;
    const int64_t rr = ok ? kv0 + r : 0;
    cp_async16(smem_u32(sK) + swz<D>(r, cc), kb + rr * p.k_rs + cc * 8, ok);
    cp_async16(smem_u32(sV) + swz<D>(r, cc), vb + rr * p.v_rs + cc * 8, ok);
  }
  const int iters = nq * p.g;
  auto load_q = [&](int i, int buf) {
    const int m = m_start + i / p.g, h = hk * p.g + i % p.g, q0 = m * BM;
    const bf16* qb = p.q + static_cast<int64_t>(s0) * p.q_rs + static_cast<int64_t>(h) * p.q_hs;
    const bf16* ob = p.dout + static_cast<int64_t>(s0) * p.o_rs + static_cast<int64_t>(h) * p.o_hs;
    const uint32_t dq = smem_u32(sQ + buf * BM * D * 2), dd = smem_u32(sdO + buf * BM * D * 2);
    for (int c = tid; c < BM * CPR; c += NT) {
      const int r = c / CPR, cc = c % CPR;
      const bool ok = q0 + r < l;
      const int64_t rr = ok ? q0 + r : 0;
      cp_async16(dq + swz<D>(r, cc), qb + rr * p.q_rs + cc * 8, ok);
      cp_async16(dd + swz<D>(r, cc), ob + rr * p.o_rs + cc * 8, ok);
    }
    if (tid < BM) {
      const bool ok = q0 + tid < l;
      const int64_t idx = static_cast<int64_t>(h) * p.T + s0 + q0 + tid;
      sL[buf * BM + tid] = ok ? p.lse[idx] * kLog2e : INFINITY;
      sD[buf * BM + tid] = ok ? p.dsum[idx] : 0.f;
    }
  };
  load_q(0, 0);
  cp_async_commit();

  float dk[D / 8][4], dv[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[i][e] = dv[i][e] = 0.f;

  for (int i = 0; i < iters; ++i) {
    if (i + 1 < iters) load_q(i + 1, (i + 1) & 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int buf = i & 1;
    const int q0 = (m_start + i / p.g) * BM;
    const uint32_t qbuf = smem_u32(sQ + buf * BM * D * 2);
    const uint32_t obuf = smem_u32(sdO + buf * BM * D * 2);
    const float* L = sL + buf * BM;
    const float* Dv = sD + buf * BM;
    float st[BM / 8][4], dpt[BM / 8][4];
#pragma unroll
    for (int t = 0; t < BM / 8; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) st[t][e] = dpt[t][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t ka[4], va[4];
      const int r = warp * 16 + (lane & 15), cc = kk * 2 + (lane >> 4);
      ldsm_x4(smem_u32(sK) + swz<D>(r, cc), ka[0], ka[1], ka[2], ka[3]);
      ldsm_x4(smem_u32(sV) + swz<D>(r, cc), va[0], va[1], va[2], va[3]);
#pragma unroll
      for (int np = 0; np < BM / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        const int br = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int bc = kk * 2 + ((lane >> 3) & 1);
        ldsm_x4(qbuf + swz<D>(br, bc), b0, b1, b2, b3);
        mma_bf16(st[2 * np], ka, b0, b1);
        mma_bf16(st[2 * np + 1], ka, b2, b3);
        ldsm_x4(obuf + swz<D>(br, bc), b0, b1, b2, b3);
        mma_bf16(dpt[2 * np], va, b0, b1);
        mma_bf16(dpt[2 * np + 1], va, b2, b3);
      }
    }
    // rows of st are kv rows (key j), columns are q rows (query i)
    const bool need_mask = p.causal && (wkv0 + 15 > q0);
#pragma unroll
    for (int t = 0; t < BM / 8; ++t) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ci = t * 8 + 2 * t4 + (e & 1);
        float pv = fast_exp2(st[t][e] * p.scale_log2 - L[ci]);
        if (need_mask) {
          const int j = wkv0 + g8 + ((e >> 1) << 3);
          if (j > q0 + ci) pv = 0.f;
        }
        st[t][e] = pv;                             // P^T
        dpt[t][e] = pv * (dpt[t][e] - Dv[ci]);     // dS^T
      }
    }
#pragma unroll
    for (int j = 0; j < BM / 16; ++j) {
      uint32_t pa[4] = {pack_bf16(st[2 * j][0], st[2 * j][1]), pack_bf16(st[2 * j][2], st[2 * j][3]),
                        pack_bf16(st[2 * j + 1][0], st[2 * j + 1][1]),
                        pack_bf16(st[2 * j + 1][2], st[2 * j + 1][3])};
      uint32_t sa[4] = {pack_bf16(dpt[2 * j][0], dpt[2 * j][1]), pack_bf16(dpt[2 * j][2], dpt[2 * j][3]),
                        pack_bf16(dpt[2 * j + 1][0], dpt[2 * j + 1][1]),
                        pack_bf16(dpt[2 * j + 1][2], dpt[2 * j + 1][3])};
#pragma unroll
      for (int dpp = 0; dpp < D / 16; ++dpp) {
        uint32_t b0, b1, b2, b3;
        const int r = j * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int cc = dpp * 2 + (lane >> 4);
        ldsm_x4_t(obuf + swz<D>(r, cc), b0, b1, b2, b3);
        mma_bf16(dv[2 * dpp], pa, b0, b1);
        mma_bf16(dv[2 * dpp + 1], pa, b2, b3);
        ldsm_x4_t(qbuf + swz<D>(r, cc), b0, b1, b2, b3);
        mma_bf16(dk[2 * dpp], sa, b0, b1);
        mma_bf16(dk[2 * dpp + 1], sa, b2, b3);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  // each warp stages its own kv rows (it only read its own rows of sK / sV)
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
    const int col = dt * 8 + 2 * t4, r0 = warp * 16 + g8;
    *reinterpret_cast<uint32_t*>(sK + swz<D>(r0, dt) + (col & 7) * 2) =
        pack_bf16(dk[dt][0] * p.scale, dk[dt][1] * p.scale);
    *reinterpret_cast<uint32_t*>(sK + swz<D>(r0 + 8, dt) + (col & 7) * 2) =
        pack_bf16(dk[dt][2] * p.scale, dk[dt][3] * p.scale);
    *reinterpret_cast<uint32_t*>(sV + swz<D>(r0, dt) + (col & 7) * 2) = pack_bf16(dv[dt][0], dv[dt][1]);
    *reinterpret_cast<uint32_t*>(sV + swz<D>(r0 + 8, dt) + (col & 7) * 2) = pack_bf16(dv[dt][2], dv[dt][3]);
  }
  __syncthreads();
  bf16* dkb = p.dk + static_cast<int64_t>(s0) * p.k_rs + static_cast<int64_t>(hk) * p.k_hs;
  bf16* dvb = p.dv + static_cast<int64_t>(s0) * p.k_rs + static_cast<int64_t>(hk) * p.k_hs;
  for (int c = tid; c < BN * CPR; c += NT) {
    const int r = c / CPR, cc = c % CPR;
    if (kv0 + r < l) {
      *reinterpret_cast<uint4*>(dkb + static_cast<int64_t>(kv0 + r) * p.k_rs + cc * 8) =
          *reinterpret_cast<const uint4*>(sK + swz<D>(r, cc));
      *reinterpret_cast<uint4*>(dvb + static_cast<int64_t>(kv0 + r) * p.k_rs + cc * 8) =
          *reinterpret_cast<const uint4*>(sV + swz<D>(r, cc));
    }
  }
}

template <int D>
static cudaError_t set_bwd_attrs() {
  const int smem_dq = (2 * kDqBM + 4 * kDqBN) * D * 2;
  const int smem_kv = (2 * kKvBN + 4 * kKvBM) * D * 2 + 4 * kKvBM * 4;
  cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_dq);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(bwd_dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_kv);
}

cudaError_t launch_bwd_rowsum(const BwdParams& p, int d, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(p.T) * p.Hq;
  const int rb = static_cast<int>(std::min<int64_t>(152 * 16, (rows * 32 + 255) / 256));
  if (rb <= 0) return cudaSuccess;
  if (d == 64) bwd_rowsum_kernel<64><<<rb, 256, 0, st>>>(p);
  else bwd_rowsum_kernel<128><<<rb, 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const BwdParams& p, int d, int grid, cudaStream_t st) {
  cudaError_t e = d == 64 ? set_bwd_attrs<64>() : set_bwd_attrs<128>();
  if (e != cudaSuccess || grid <= 0) return e;
  const int smem64 = (2 * kKvBN + 4 * kKvBM) * 64 * 2 + 4 * kKvBM * 4;
  const int smem128 = (2 * kKvBN + 4 * kKvBM) * 128 * 2 + 4 * kKvBM * 4;
  if (d == 64) bwd_dkdv_kernel<64><<<grid, kThreads, smem64, st>>>(p);
  else bwd_dkdv_kernel<128><<<grid, kThreads, smem128, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const BwdParams& p, int d, int grid, cudaStream_t st) {
  cudaError_t e = d == 64 ? set_bwd_attrs<64>() : set_bwd_attrs<128>();
  if (e != cudaSuccess || grid <= 0) return e;
  if (d == 64) bwd_dq_kernel<64><<<grid, kThreads, (2 * kDqBM + 4 * kDqBN) * 64 * 2, st>>>(p);
  else bwd_dq_kernel<128><<<grid, kThreads, (2 * kDqBM + 4 * kDqBN) * 128 * 2, st>>>(p);
  return cudaGetLastError();
}

void bwd_mma_tiles(int* kvBM, int* kvBN, int* qBM, int* qBN) {
  *kvBM = kKvBM;
  *kvBN = kKvBN;
  *qBM = kDqBM;
  *qBN = kDqBN;
}

}  // namespace va
