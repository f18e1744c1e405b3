// Boundary compiler on the device: position_ids -> cu_seqlens, B, max_seqlen.
//
// "Packing与 FlashAttention Varlen", section 3: with sample-local positions, every index
// whose position is the reset sentinel starts a sample; the reset indices followed by the
// total token count T form cu_seqlens, and max_seqlen is its largest difference.  The
// sentinel is 0 (the explicit conversion) or the plane's minimum (the generic path, for
// position schemes that do not start at 0).  The result must meet the cumulative
// boundary contract (int32, first 0, last T, strictly increasing); reset indices are
// distinct and below T, so the plane breaks it only when its first token is not a reset.
// With `strict`, positions between resets must also count up by one: a plane that repeats
// coordinates inside a sample (the visual planes of the mRoPE section) cannot carry
// boundaries.
//
// One CTA: each thread takes a contiguous chunk of tokens; block scans give each chunk
// its first output slot (sum of reset counts), the first reset after it (for the last
// length of the chunk) and the minimum / error flags.
#include "plan_body.cuh"

namespace va {

constexpr int kBoundaryThreads = 1024;

__global__ void __launch_bounds__(kBoundaryThreads)
    cu_from_positions_kernel(const int32_t* __restrict__ pos, int T, int reset_at_min, int strict,
                             int32_t* __restrict__ cu, int capacity, int32_t* __restrict__ B_out,
                             int32_t* __restrict__ max_out, int32_t* __restrict__ status) {
  __shared__ int tmp[33];
  griddep_begin();  // the positions may come from the kernel just before
  const int tid = threadIdx.x, nth = blockDim.x;
  const int per = (T + nth - 1) / nth;
  const int lo = min(T, tid * per), hi = min(T, lo + per);
  int dummy;
  int sentinel = 0;
  if (reset_at_min) {
    int m = INT_MAX;
    for (int t = lo; t < hi; ++t) m = min(m, pos[t]);
    block_scan_excl<kScanMin, false>(m, INT_MAX, nth, tmp, &sentinel);
  }
  int cnt = 0, first = T, bad = 0;
  int prev = lo > 0 ? pos[lo - 1] : 0;
  for (int t = lo; t < hi; ++t) {
    const int x = pos[t];
    if (x == sentinel) {
      ++cnt;
      if (first == T) first = t;
    } else if (strict && t > 0 && x != prev + 1) {
      bad = 1;
    }
    prev = x;
  }
  if (tid == 0 && pos[0] != sentinel) bad = 1;  // cu[0] would not be 0
  int nb, any_bad;
  const int slot = block_scan_excl<kScanSum, false>(cnt, 0, nth, tmp, &nb);
  const int next_reset = block_scan_excl<kScanMin, true>(first, T, nth, tmp, &dummy);
  block_scan_excl<kScanMax, false>(bad, 0, nth, tmp, &any_bad);
  const bool overflow = nb + 1 > capacity;  // uniform
  int mx = 0;
  if (!any_bad && !overflow) {
    int k = slot, last = -1;
    for (int t = lo; t < hi; ++t) {
      if (pos[t] != sentinel) continue;
      cu[k++] = t;
      if (last >= 0) mx = max(mx, t - last);
      last = t;
    }
    if (last >= 0) mx = max(mx, next_reset - last);
    if (tid == 0) cu[nb] = T;
  }
  int gmx;
  block_scan_excl<kScanMax, false>(mx, 0, nth, tmp, &gmx);
  if (tid == 0) {
    const bool ok = !any_bad && !overflow;
    *B_out = ok ? nb : 0;
    *max_out = ok ? gmx : 0;
    *status = any_bad ? VA_ERR_BAD_SEQLENS : (overflow ? VA_ERR_WORKSPACE : VA_OK);
  }
}

cudaError_t launch_cu_from_positions(const int32_t* pos, int T, int reset_at_min, int strict, int32_t* cu,
                                     int capacity, int32_t* B_out, int32_t* max_out, int32_t* status,
                                     cudaStream_t st) {
  return launch_pdl(cu_from_positions_kernel, dim3(1), dim3(kBoundaryThreads), 0, st, pos, T, reset_at_min,
                    strict, cu, capacity, B_out, max_out, status);
}

}  // namespace va
