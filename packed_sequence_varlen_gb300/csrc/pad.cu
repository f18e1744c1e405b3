// Padded-batch bridge: a batch padded to [Bp, S] with a 2-D attention mask enters the varlen
// path by dropping its padding, and the packed output is scattered back to the padded shape
// ("Packing与 FlashAttention Varlen", section 4: the padded-batch branch removes the padding,
// the varlen kernel computes, the output is scattered back).
//
// unpad index, three launches:
//   pad_count_kernel   one CTA per batch row: the row's real tokens (mask != 0)
//   pad_scan_kernel    one CTA: cu_seqlens = exclusive scan of the counts, T, max_seqlen; a row
//                      without real tokens sets VA_ERR_BAD_SEQLENS (an empty segment would break
//                      the strictly increasing boundary contract of section 3)
//   pad_index_kernel   one CTA per batch row: a block scan over the row's mask places real
//                      position s at packed index cu[r] + (real tokens before s), and padding
//                      position s at index T + (padding cells before row r) + (padding before s):
//                      indices[] lists the real tokens' flat positions, then -1 for every
//                      padding cell; inverse[] maps each flat position to its packed index or -1
// gather_rows_kernel: dst row i = src row map[i], or a zero row where map[i] < 0 (unpad with the
// indices, pad with the inverse map); 16-byte copies, one CTA per row at a time.
#include <algorithm>

#include "common.cuh"

namespace va {

namespace {
constexpr int kPadThreads = 256;

// Exclusive block scan of one int per thread (kPadThreads threads); *total gets the sum.
__device__ __forceinline__ int block_excl_scan(int x, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  __syncthreads();  // tmp may still be read by the previous round
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kPadThreads / 32; ++w) {
    const int v = tmp[w];
    if (w < warp) base += v;
    tot += v;
  }
  *total = tot;
  return base + incl - x;
}
}  // namespace

__global__ void __launch_bounds__(kPadThreads) pad_count_kernel(const int32_t* mask, int S, int32_t* cu) {
  griddep_begin();
  const int r = blockIdx.x;
  int n = 0;
  for (int s = threadIdx.x; s < S; s += kPadThreads) n += __ldg(mask + static_cast<int64_t>(r) * S + s) != 0;
  n = __reduce_add_sync(0xffffffffu, n);
  __shared__ int part[kPadThreads / 32];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = n;
  __syncthreads();
  if (threadIdx.x == 0) {
    int t = 0;
    for (int w = 0; w < kPadThreads / 32; ++w) t += part[w];
    cu[r + 1] = t;  // the row's count; the scan turns it into the boundary
  }
}

__global__ void __launch_bounds__(1024) pad_scan_kernel(int Bp, int32_t* cu, int32_t* T_out, int32_t* max_out,
                                                        int32_t* status) {
  griddep_begin();
  __shared__ int32_t s_run, s_max, s_bad;
  if (threadIdx.x == 0) {
    s_run = 0;
    s_max = 0;
    s_bad = 0;
  }
  __syncthreads();
  __shared__ int tmp[32];
  for (int r0 = 0; r0 < Bp; r0 += 1024) {
    const int r = r0 + threadIdx.x;
    const int n = r < Bp ? cu[r + 1] : 0;
    // exclusive scan over 1024 threads
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) tmp[warp] = incl;
    __syncthreads();
    int base = 0, tot = 0;
    for (int w = 0; w < 32; ++w) {
      const int v = tmp[w];
      if (w < warp) base += v;
      tot += v;
    }
    const int run = s_run;
    if (r < Bp) {
      cu[r + 1] = run + base + incl;
      if (n == 0) atomicOr(&s_bad, 1);
      atomicMax(&s_max, n);
    }
    __syncthreads();  // every thread has read s_run and tmp
    if (threadIdx.x == 0) s_run = run + tot;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    cu[0] = 0;
    *T_out = s_run;
    *max_out = s_max;
    *status = s_bad ? VA_ERR_BAD_SEQLENS : VA_OK;
  }
}

__global__ void __launch_bounds__(kPadThreads) pad_index_kernel(const int32_t* mask, int S, const int32_t* cu,
                                                                const int32_t* T_in, int32_t* indices,
                                                                int32_t* inverse) {
  griddep_begin();
  __shared__ int tmp[kPadThreads / 32];
  const int r = blockIdx.x, T = *T_in;
  const int64_t row0 = static_cast<int64_t>(r) * S;
  int real_run = cu[r];                                    // packed index of the next real token
  int64_t pad_run = T + (row0 - cu[r]);                    // index of the next padding slot
  for (int s0 = 0; s0 < S; s0 += kPadThreads) {
    const int s = s0 + threadIdx.x;
    const int real = s < S && __ldg(mask + row0 + s) != 0;
    int tot;
    const int before = block_excl_scan(real, tmp, &tot);   // real tokens before s in this round
    if (s < S) {
      const int64_t flat = row0 + s;
      if (real) {
        const int at = real_run + before;
        indices[at] = static_cast<int32_t>(flat);
        inverse[flat] = at;
      } else {
        const int64_t at = pad_run + (threadIdx.x - before);  // padding cells before s in the round
        indices[at] = -1;
        inverse[flat] = -1;
      }
    }
    real_run += tot;
    pad_run += min(kPadThreads, S - s0) - tot;
  }
}

__global__ void __launch_bounds__(kPadThreads) gather_rows_kernel(const uint8_t* src, int64_t src_stride,
                                                                  const int32_t* map, int n_rows, int64_t row_bytes,
                                                                  uint8_t* dst, int64_t dst_stride) {
  griddep_begin();
  const int64_t n16 = row_bytes / 16;
  for (int i = blockIdx.x; i < n_rows; i += gridDim.x) {
    const int r = __ldg(map + i);
    uint4* d = reinterpret_cast<uint4*>(dst + static_cast<int64_t>(i) * dst_stride);
    if (r < 0) {
      for (int64_t c = threadIdx.x; c < n16; c += kPadThreads) __stcs(d + c, make_uint4(0, 0, 0, 0));
    } else {
      const uint4* sp = reinterpret_cast<const uint4*>(src + static_cast<int64_t>(r) * src_stride);
      for (int64_t c = threadIdx.x; c < n16; c += kPadThreads) __stcs(d + c, __ldcs(sp + c));
    }
  }
}

// ---------------------------------------------------------------- host side

cudaError_t launch_unpad_index(int stage, const int32_t* mask, int Bp, int S, int32_t* indices, int32_t* inverse,
                               int32_t* cu, int32_t* T_out, int32_t* max_out, int32_t* status, cudaStream_t st) {
  if (stage == 0) return launch_pdl(pad_count_kernel, dim3(Bp), dim3(kPadThreads), 0, st, mask, S, cu);
  if (stage == 1) return launch_pdl(pad_scan_kernel, dim3(1), dim3(1024), 0, st, Bp, cu, T_out, max_out, status);
  return launch_pdl(pad_index_kernel, dim3(Bp), dim3(kPadThreads), 0, st, mask, S, static_cast<const int32_t*>(cu),
                    static_cast<const int32_t*>(T_out), indices, inverse);
}

cudaError_t launch_gather_rows(const void* src, int64_t src_stride, const int32_t* map, int n_rows, int64_t row_bytes,
                               void* dst, int64_t dst_stride, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = std::min(n_rows, std::max(sms, 1) * 8);
  return launch_pdl(gather_rows_kernel, dim3(grid), dim3(kPadThreads), 0, st, static_cast<const uint8_t*>(src),
                    src_stride, map, n_rows, row_bytes, static_cast<uint8_t*>(dst), dst_stride);
}

}  // namespace va
