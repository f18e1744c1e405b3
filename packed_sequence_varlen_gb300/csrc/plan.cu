// Segment-aware tile scheduler: builds the work list the attention kernels walk.
//
// "Packing与 FlashAttention Varlen", section 5: the launch bound comes from
// max_seqlen, a q block m of segment b exists only while m*BM < l_b, and its key
// blocks stop at ceil(min(l_b, (m+1)*BM) / BN) under causality (ceil(l_b/BN)
// otherwise).  Instead of launching max_seqlen-shaped grids whose CTAs exit
// early, the list holds only blocks that have work, ordered longest first
// (ties by segment, block, head -- this library's reading).
//
// One CTA of 1024 threads.  A forward segment has at most one q block per key
// when BM is a multiple of BN (causal), and a backward segment at most one kv
// block per key when BN is a multiple of BM, so each key's records are "the
// segments that have this key, in segment order": each warp owns a set of
// keys and ranks the segments with ballots; no global sort is needed.
#include "common.cuh"

namespace va {



// Blocks of one segment (length l) whose key equals k: first block and count.
__device__ __forceinline__ int seg_key_blocks(const PlanArgs& a, int l, int k, int& first) {
  if (a.kind != 1) {
    const int M = (l + a.BM - 1) / a.BM;
    const int Lk = (l + a.BN - 1) / a.BN;
    if (!a.causal) {
      first = 0;
      return k == Lk ? M : 0;
    }
    const int c = a.BM / a.BN;
    if (k == Lk) {
      first = M - 1;
      return 1;
    }
    if (k % c == 0 && k / c - 1 < M - 1) {
      first = k / c - 1;
      return 1;
    }
    return 0;
  } else {
    const int N = (l + a.BN - 1) / a.BN;
    const int Mq = (l + a.BM - 1) / a.BM;
    if (!a.causal) {
      first = 0;
      return k == Mq ? N : 0;
    }
    const int c = a.BN / a.BM;
    const int d = Mq - k;
    if (d < 0 || d % c) return 0;
    const int n = d / c;
    if (n >= N) return 0;
    first = n;
    return 1;
  }
}

constexpr int kPlanThreads = 1024;
constexpr int kMaxKeys = 4096;

struct PlanSmem {
  int count[kMaxKeys + 1];
  int offset[kMaxKeys + 2];
  int overflow;
};

// Builds one map (all 1024 threads of the block take part).
__device__ void plan_body(const PlanArgs& a, PlanSmem& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // pass 1: records per key
  for (int k = a.kmax - warp; k >= 1; k -= 32) {
    int total = 0;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
      const int b = b0 + lane;
      int cnt = 0, first;
      if (b < a.B) cnt = seg_key_blocks(a, a.cu[b + 1] - a.cu[b], k, first);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      total += cnt;
    }
    if (lane == 0) sh.count[k] = total;
  }
  __syncthreads();
  // exclusive scan over keys, longest first
  if (threadIdx.x == 0) {
    int run = 0;
    for (int k = a.kmax; k >= 1; --k) {
      sh.offset[k] = run;
      run += sh.count[k] * a.heads;
    }
    sh.offset[0] = run;
    sh.overflow = run > a.capacity;
    *a.n_items = sh.overflow ? 0 : run;
    if (sh.overflow && a.status) atomicCAS(a.status, VA_OK, VA_ERR_WORKSPACE);
  }
  __syncthreads();
  if (sh.overflow) return;
  // pass 2: place records; rank = earlier segments with the same key
  for (int k = a.kmax - warp; k >= 1; k -= 32) {
    int base = 0;
    for (int b0 = 0; b0 < a.B; b0 += 32) {
      const int b = b0 + lane;
      int cnt = 0, first = 0;
      if (b < a.B) cnt = seg_key_blocks(a, a.cu[b + 1] - a.cu[b], k, first);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int rank = base + incl - cnt;
      for (int j = 0; j < cnt; ++j) {
        TileItem* dst = a.out + sh.offset[k] + (rank + j) * a.heads;
        for (int h = 0; h < a.heads; ++h) {
          TileItem t;
          t.seg = b;
          t.blk = first + j;
          t.head = h;
          t.count = k;
          dst[h] = t;
        }
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
  __shared__ PlanSmem sh;
  if (a.status && *a.status != VA_OK) {
    if (threadIdx.x == 0) *a.n_items = 0;
    return;
  }
  plan_body(a, sh);
}

struct PlanPair {
  PlanArgs map[2];
  int nmaps;
  int T, max_seqlen;
};

// One launch per attention call: checks the cu_seqlens contract (cu[0] == 0,
// cu[B] == T, strictly increasing, every length <= max_seqlen), writes the status
// word (OK or VA_ERR_BAD_SEQLENS), and only if it holds builds the call's maps.
__global__ void __launch_bounds__(kPlanThreads) validate_plan_kernel(PlanPair pp) {
  __shared__ PlanSmem sh;
  const PlanArgs& a0 = pp.map[0];
  int bad = 0;
  for (int b = threadIdx.x; b < a0.B; b += blockDim.x) {
    const int x = a0.cu[b], y = a0.cu[b + 1];
    if (y <= x || y - x > pp.max_seqlen) bad = 1;
  }
  if (threadIdx.x == 0 && (a0.cu[0] != 0 || a0.cu[a0.B] != pp.T)) bad = 1;
  bad = __syncthreads_or(bad);
  if (bad) {
    if (threadIdx.x == 0) {
      *a0.status = VA_ERR_BAD_SEQLENS;
      for (int i = 0; i < pp.nmaps; ++i) *pp.map[i].n_items = 0;
    }
    return;
  }
  if (threadIdx.x == 0) *a0.status = VA_OK;
  for (int i = 0; i < pp.nmaps; ++i) plan_body(pp.map[i], sh);
}

cudaError_t launch_plan(const int32_t* cu, int B, int heads, int BM, int BN, int kind, int causal,
                        int kmax, TileItem* out, int capacity, int32_t* status,
                        int32_t* n_items, cudaStream_t st) {
  PlanArgs a{cu, B, heads, BM, BN, kind, causal, kmax, out, capacity, status, n_items};
  plan_kernel<<<1, kPlanThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_validate_plan(const PlanArgs* maps, int nmaps, int T, int max_seqlen,
                                 cudaStream_t st) {
  PlanPair pp{};
  for (int i = 0; i < nmaps && i < 2; ++i) pp.map[i] = maps[i];
  pp.nmaps = nmaps;
  pp.T = T;
  pp.max_seqlen = max_seqlen;
  validate_plan_kernel<<<1, kPlanThreads, 0, st>>>(pp);
  return cudaGetLastError();
}

int plan_max_keys() { return kMaxKeys; }

}  // namespace va
