// Boundary metadata on the device: lengths -> cu_seqlens, position_ids,
// segment_ids, max_seqlen; and the cu_seqlens contract check.
//
// "Packing与 FlashAttention Varlen", section 3: the cumulative boundary array
// is int32, starts at 0, ends at the total token count and strictly increases;
// max_seqlen = max diff and only bounds launches and tiles.  Section 2
// (packing_row): each sample's positions restart at 0.
#include "common.cuh"

namespace va {

constexpr int kScanThreads = 1024;

// A stream of at most kInlineTokens tokens cut into at most kInlineSegs lengths gets its
// positions and segment ids from the scan's own block, from a shared-memory copy of the
// boundaries: one launch instead of two, and no binary search through global memory.
constexpr int kInlineTokens = 16384;
constexpr int kInlineSegs = 2046;

bool metadata_inline_fill(int n, int T_capacity) {
  return T_capacity > 0 && T_capacity <= kInlineTokens && n <= kInlineSegs;
}

// Segment of token t: b with cu[b] <= t < cu[b + 1], over cu[0..nseg].
__device__ __forceinline__ int find_segment(const int32_t* cu, int nseg, int t) {
  int lo = 0, hi = nseg;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu[mid] <= t) lo = mid; else hi = mid;
  }
  return lo;
}

// Block-wide inclusive scan of one int per thread (1024 threads).
__device__ __forceinline__ int block_inclusive_scan(int x, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  if (warp > 0) x += warp_sums[warp - 1];
  __syncthreads();
  return x;
}

// One block: exclusive scan of the lengths into cu[0..n], tail pad into cu[n+1]; with
// inline_fill (metadata_inline_fill) also position_ids and segment_ids, as the fill kernel
// would write them.  Up to 32 lengths one warp scans them in registers: the launch runs once
// per call on cold instruction caches, and that path is a small fraction of the block scan's.
__global__ void __launch_bounds__(kScanThreads)
    metadata_scan_kernel(const int32_t* __restrict__ lengths, int n, int pad_to,
                         int T_capacity, int32_t* __restrict__ cu, int32_t* __restrict__ max_out,
                         int32_t* __restrict__ status, int inline_fill, int32_t* __restrict__ pos,
                         int32_t* __restrict__ seg) {
  __shared__ int warp_sums[32];
  __shared__ int carry, mx, bad;
  __shared__ int s_cu[kInlineSegs + 2];
  griddep_begin();  // the lengths may come from the kernel just before
  // (one thread) the pad segment, the capacity check and the scalar outputs
  auto finish = [&](int total, int m, int b) {
    int last = total;
    if (pad_to > total) {
      last = pad_to;
      m = max(m, pad_to - total);
    } else if (pad_to > 0 && pad_to < total) {
      b = 1;
    }
    if (last > T_capacity) b = 1;
    cu[n + 1] = last;
    if (inline_fill) s_cu[n + 1] = last;
    *max_out = m;
    *status = b ? VA_ERR_BAD_SEQLENS : VA_OK;
    bad = b;
  };
  if (n <= 32) {  // one warp scans in registers: no block barriers or shared-memory atomics
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      const int L = lane < n ? lengths[lane] : 0;
      int incl = L;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int m = __reduce_max_sync(0xffffffffu, L);
      const int b = __any_sync(0xffffffffu, lane < n && L <= 0) ? 1 : 0;
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      if (lane < n) cu[lane + 1] = s_cu[lane + 1] = incl;
      if (lane == 0) {
        cu[0] = 0;
        s_cu[0] = 0;
        finish(total, m, b);
      }
    }
  } else {
    if (threadIdx.x == 0) {
      carry = 0;
      mx = 0;
      bad = 0;
      cu[0] = 0;
      s_cu[0] = 0;
    }
    __syncthreads();
    for (int base = 0; base < n; base += kScanThreads) {
      const int i = base + threadIdx.x;
      const int L = i < n ? lengths[i] : 0;
      if (i < n && L <= 0) atomicOr(&bad, 1);
      if (i < n) atomicMax(&mx, L);
      const int incl = block_inclusive_scan(L, warp_sums);
      if (i < n) {
        cu[i + 1] = carry + incl;
        if (inline_fill) s_cu[i + 1] = carry + incl;
      }
      __syncthreads();
      if (threadIdx.x == kScanThreads - 1) carry += incl;
      __syncthreads();
    }
    if (threadIdx.x == 0) finish(carry, mx, bad);
  }
  if (!inline_fill) return;
  __syncthreads();
  if (bad) return;
  const int T = s_cu[n + 1];
  const int nseg = (s_cu[n + 1] > s_cu[n]) ? n + 1 : n;
  for (int t = threadIdx.x; t < T && t < T_capacity; t += kScanThreads) {
    const int b = find_segment(s_cu, nseg, t);
    seg[t] = b;
    pos[t] = t - s_cu[b];
  }
}

// Grid over tokens: segment by binary search over cu[0..nseg], position = t - start.
__global__ void metadata_fill_kernel(const int32_t* __restrict__ cu, int n, int T_capacity,
                                     int32_t* __restrict__ pos, int32_t* __restrict__ seg,
                                     const int32_t* __restrict__ status) {
  griddep_begin();  // cu and the status word come from the scan just before
  if (*status != VA_OK) return;
  const int T = cu[n + 1];
  const int nseg = (cu[n + 1] > cu[n]) ? n + 1 : n;
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T && t < T_capacity;
       t += gridDim.x * blockDim.x) {
    const int b = find_segment(cu, nseg, t);
    seg[t] = b;
    pos[t] = t - cu[b];
  }
}

// One block: checks the boundary contract and writes the status word (0 or error).
__global__ void __launch_bounds__(kScanThreads)
    validate_cu_kernel(const int32_t* __restrict__ cu, int B, int T, int max_seqlen,
                       int32_t* __restrict__ status, int overwrite) {
  griddep_begin();
  int bad = 0;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int a = cu[b], c = cu[b + 1];
    if (c <= a || c - a > max_seqlen) bad = 1;
  }
  if (threadIdx.x == 0 && (cu[0] != 0 || cu[B] != T)) bad = 1;
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    if (bad) *status = VA_ERR_BAD_SEQLENS;
    else if (overwrite) *status = VA_OK;
  }
}

cudaError_t launch_metadata_scan(const int32_t* lengths, int n, int pad_to, int T_capacity,
                                 int32_t* cu, int32_t* max_out, int32_t* status, int32_t* pos, int32_t* seg,
                                 cudaStream_t st) {
  const int inl = metadata_inline_fill(n, T_capacity) ? 1 : 0;
  return launch_pdl(metadata_scan_kernel, dim3(1), dim3(kScanThreads), 0, st, lengths, n, pad_to, T_capacity, cu,
                    max_out, status, inl, pos, seg);
}

cudaError_t launch_metadata_fill(const int32_t* cu, int n, int T_capacity, int32_t* pos,
                                 int32_t* seg, const int32_t* status, cudaStream_t st) {
  const int blocks = min(1216, max(1, (T_capacity + 255) / 256));
  return launch_pdl(metadata_fill_kernel, dim3(blocks), dim3(256), 0, st, cu, n, T_capacity, pos, seg, status);
}

cudaError_t launch_validate(const int32_t* cu, int B, int T, int max_seqlen, int32_t* status,
                            int overwrite, cudaStream_t st) {
  return launch_pdl(validate_cu_kernel, dim3(1), dim3(kScanThreads), 0, st, cu, B, T, max_seqlen, status,
                    overwrite);
}

}  // namespace va
