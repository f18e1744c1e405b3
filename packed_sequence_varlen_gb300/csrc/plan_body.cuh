// Segment-aware tile scheduler, device side: the planning bodies shared by the
// planning kernels and the backward preparation kernel (which plans in one CTA while the
// others compute D = rowsum(dO * O)).
//
// Segment-aware tile scheduler: builds the work list the attention kernels walk.
//
// "Packing与 FlashAttention Varlen", section 5: a q block m of segment b exists only
// while m*BM < l_b, and its key blocks stop at ceil(min(l_b, (m+1)*BM) / BN) under
// causality (ceil(l_b/BN) otherwise).  Instead of launching max_seqlen-shaped grids
// whose CTAs exit early, the list holds only blocks that have work.
//
// Order (this library's reading; the page fixes none): records that read the same
// K/V tiles are adjacent, so the attention kernels -- which pull records in list
// order from an atomic counter -- run them at the same time and share those tiles
// through L2; longer work goes first:
//   key = (-class_b, b, head, -count, block),  class_b = floor(log2(C_b)),
// with C_b the segment's total tile count (key tiles summed over its q blocks for
// the forward/dQ maps, q blocks summed over its kv blocks for the dK/dV map).
//
// One CTA (any multiple of 32 threads): warps take the 32 cost classes in turn, count
// and rank the segments of a class with warp scans (the segment's first record goes to a small scratch
// array), then a warp per segment writes the segment's records.
#pragma once
#include "common.cuh"

namespace va {

namespace plan_detail {

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Blocks of a segment of length l and its total tile count.
__device__ __forceinline__ void seg_cost(const PlanArgs& a, int l, int& nblk, int& cost) {
  if (a.kind != 1) {
    const int M = ceil_div(l, a.BM), Lk = ceil_div(l, a.BN);
    nblk = M;
    cost = a.causal ? (a.BM / a.BN) * (M - 1) * M / 2 + Lk : M * Lk;
  } else {
    const int N = ceil_div(l, a.BN), Mq = ceil_div(l, a.BM);
    nblk = N;
    cost = a.causal ? N * Mq - (a.BN / a.BM) * N * (N - 1) / 2 : N * Mq;
  }
}

// The j-th record of one (segment, head): most tiles first.
__device__ __forceinline__ void seg_record(const PlanArgs& a, int l, int nblk, int j, int& blk,
                                           int& count) {
  if (a.kind != 1) {
    const int Lk = ceil_div(l, a.BN);
    blk = a.causal ? nblk - 1 - j : j;
    count = a.causal ? min(Lk, (a.BM / a.BN) * (blk + 1)) : Lk;
  } else {
    const int Mq = ceil_div(l, a.BM);
    blk = j;
    count = a.causal ? Mq - (j * a.BN) / a.BM : Mq;
  }
}

__device__ __forceinline__ int cost_class(int c) { return 31 - __clz(max(c, 1)); }

}  // namespace plan_detail
using namespace plan_detail;

constexpr int kPlanThreads = 1024;

// Up to this many segments the boundaries and per-segment offsets live in shared memory
// (one coalesced read of cu_seqlens per launch); beyond it they are read from and kept in
// global memory.
constexpr int kSmemSegs = 4096;

struct PlanSmem {
  int count[32];
  int offset[32];
  int overflow;
  int cu[kSmemSegs + 1];
  int off[kSmemSegs];
};

// Builds one map; every thread of the block (a multiple of 32, at most 1024) takes part.
// cu: the boundaries (the shared-memory copy or a.cu); seg_off: where the per-segment
// offsets go.
__device__ __forceinline__ void plan_body(const PlanArgs& a, PlanSmem& sh, const int* cu, int* seg_off) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  // records per class; warp w takes classes 31 - w, 31 - w - nwarps, ...
  for (int k = 31 - warp; k >= 0; k -= nwarps) {
    int total = 0;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
      const int b = b0 + lane;
      int cnt = 0;
      if (b < a.B) {
        int nblk, cost;
        seg_cost(a, cu[b + 1] - cu[b], nblk, cost);
        if (cost_class(cost) == k) cnt = nblk * a.heads;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      total += cnt;
    }
    if (lane == 0) sh.count[k] = total;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int c = 31; c >= 0; --c) {
      sh.offset[c] = run;
      run += sh.count[c];
    }
    sh.overflow = run > a.capacity;
    *a.n_items = sh.overflow ? 0 : run;
    *a.counter = 0;
    if (sh.overflow && a.status) atomicCAS(a.status, VA_OK, VA_ERR_WORKSPACE);
  }
  __syncthreads();
  if (sh.overflow) return;
  // first record of every segment: class offset + earlier segments of the same class
  for (int k = 31 - warp; k >= 0; k -= nwarps) {
    int base = sh.offset[k];
    for (int b0 = 0; b0 < a.B; b0 += 32) {
      const int b = b0 + lane;
      int cnt = 0;
      if (b < a.B) {
        int nblk, cost;
        seg_cost(a, cu[b + 1] - cu[b], nblk, cost);
        if (cost_class(cost) == k) cnt = nblk * a.heads;
      }
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (cnt > 0) seg_off[b] = base + incl - cnt;
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
  // records: a warp per segment, heads outer, blocks inner
  for (int b = warp; b < a.B; b += nwarps) {
    const int l = cu[b + 1] - cu[b];
    int nblk, cost;
    seg_cost(a, l, nblk, cost);
    const int off = seg_off[b];
    for (int r = lane; r < nblk * a.heads; r += 32) {
      const int h = r / nblk, j = r - h * nblk;
      TileItem t;
      seg_record(a, l, nblk, j, t.blk, t.count);
      t.seg = b;
      t.head = h;
      a.out[off + r] = t;
    }
  }
  __syncthreads();
}

struct PlanPair {
  PlanArgs map[2];
  int nmaps;
  int T, max_seqlen;
};

// Copies cu[0..B] into shared memory when it fits; returns the array to read.
__device__ __forceinline__ const int* stage_cu(const int32_t* cu, int B, PlanSmem& sh) {
  if (B + 1 > kSmemSegs) return cu;
  for (int i = threadIdx.x; i <= B; i += blockDim.x) sh.cu[i] = cu[i];
  __syncthreads();
  return sh.cu;
}

// Validates cu_seqlens (writing the status word) and builds every map of pp.
__device__ __forceinline__ void validate_plan_body(const PlanPair& pp, PlanSmem& sh) {
  const PlanArgs& a0 = pp.map[0];
  const int* cu = stage_cu(a0.cu, a0.B, sh);  // every map is built from the same boundaries
  int bad = 0;
  for (int b = threadIdx.x; b < a0.B; b += blockDim.x) {
    const int x = cu[b], y = cu[b + 1];
    if (y <= x || y - x > pp.max_seqlen) bad = 1;
  }
  if (threadIdx.x == 0 && (cu[0] != 0 || cu[a0.B] != pp.T)) bad = 1;
  bad = __syncthreads_or(bad);
  if (bad) {
    if (threadIdx.x == 0) {
      *a0.status = VA_ERR_BAD_SEQLENS;
      for (int i = 0; i < pp.nmaps; ++i) *pp.map[i].n_items = 0;
    }
    return;
  }
  if (threadIdx.x == 0) *a0.status = VA_OK;
  for (int i = 0; i < pp.nmaps; ++i)
    plan_body(pp.map[i], sh, cu, a0.B + 1 > kSmemSegs ? pp.map[i].seg_off : sh.off);
}

}  // namespace va
