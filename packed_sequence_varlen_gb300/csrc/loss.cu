// Packed next-token loss on the device: targets formed inside each segment, and the
// token-weighted cross entropy over the packed stream with its logit gradient.
//
// "Pack sequences without joining their contexts":
//   "Form pairs inside each source range" -- position t of segment [s, e) predicts token
//     t + 1 only while t + 1 < e; the last position of a segment has no target, so packing
//     creates no pair across a boundary (the same layout as sample-local -100 labels shifted
//     by one, "Packing与 FlashAttention Varlen", section 2);
//   "Keep the same nine-target objective" -- the loss is the raw sum of the negative log
//     likelihoods of the eligible targets divided once by their count N, and
//     d(mean)/d(z_ic) = (p_ic - [c == y_i]) / N; cells that are not eligible are skipped
//     before any arithmetic (their logits are never read, their gradient rows are zero).
//
// Kernels (one stream, programmatic dependent launches):
//   loss_targets_kernel   one thread per position: the segment by binary search over cu
//   ce_count_kernel       one CTA: N and the target range check -> count, status word
//   ce_rows_kernel        persistent CTAs (4 per SM), one row at a time, four 16-byte chunks
//                         per thread in flight: pass 1 streams the row once
//                         (chunk max, rescaled sum of exp2, base-2 lse), pass 2 re-reads it
//                         (from L2: the CTA just read it) and writes the gradient row; the
//                         row's NLL goes to a per-row buffer
//   ce_reduce_kernel      one CTA: sum of the per-row NLL in float64, in a fixed order
//                         (deterministic), and the mean
// Rows are streamed with 16-byte loads and stores when every row of logits (and gradient)
// starts on a 16-byte boundary, else element by element.
#include <algorithm>

#include "common.cuh"

namespace va {

namespace {

constexpr int kCeThreads = 256;
constexpr int kCeWarps = kCeThreads / 32;
constexpr int kCountThreads = 1024;
constexpr int kU = 4;             // 16-byte chunks a thread has in flight per pass
constexpr int kCeCtasPerSm = 4;  // resident at once (launch bounds)

struct CeParams {
  const void* logits;
  int64_t l_rs;  // logits row stride (elements)
  const int32_t* targets;
  int T, V, ignore;
  void* grad;    // may be null
  int64_t g_rs;
  float* nll;    // [T] per-row negative log likelihood (0 on rows without a target)
  int32_t* count;
  int32_t* status;
  double* loss;  // {sum, mean}
  int vec;       // rows can be streamed with 16-byte accesses
};

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <class T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// W = elements per 16 bytes
template <class T> struct Vec { static constexpr int W = 16 / sizeof(T); };

// LAST: the row's second and last read (evict first); the first read keeps it in L2 for it
template <bool LAST, class T>
__device__ __forceinline__ uint4 load_raw(const T* p) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  return LAST ? __ldcs(q) : __ldg(q);
}

template <class T>
__device__ __forceinline__ void unpack(const uint4& u, float (&x)[Vec<T>::W]) {
  const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
  for (int i = 0; i < Vec<T>::W; ++i) x[i] = to_f(e[i]);
}

template <class T>
__device__ __forceinline__ void store_vec(T* p, const float (&x)[Vec<T>::W]) {
  uint4 u;
  T* e = reinterpret_cast<T*>(&u);
#pragma unroll
  for (int i = 0; i < Vec<T>::W; ++i) e[i] = from_f<T>(x[i]);
  __stcs(reinterpret_cast<uint4*>(p), u);
}

// Merges running (max, sum of exp2(x - max)) pairs.
__device__ __forceinline__ void ms_merge(float& m, float& s, float m2, float s2) {
  const float mx = fmaxf(m, m2);
  if (mx == -INFINITY) return;  // both empty
  s = s * fast_exp2(m - mx) + s2 * fast_exp2(m2 - mx);
  m = mx;
}

}  // namespace

__global__ void __launch_bounds__(256) loss_targets_kernel(const int32_t* ids, const int32_t* cu, int B, int T,
                                                           int ignore, int32_t* targets) {
  griddep_begin();
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  int lo = 0, hi = B;  // the segment b with cu[b] <= t < cu[b + 1]: last b in [0, B) with cu[b] <= t
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid;
    else hi = mid;
  }
  const int end = __ldg(cu + lo + 1);
  targets[t] = (t + 1 < end && t + 1 < T) ? __ldg(ids + t + 1) : ignore;
}

__global__ void __launch_bounds__(kCountThreads) ce_count_kernel(CeParams p) {
  griddep_begin();
  int n = 0, bad = 0;
  for (int t = threadIdx.x; t < p.T; t += kCountThreads) {
    const int y = __ldg(p.targets + t);
    if (y != p.ignore) {
      ++n;
      bad |= (y < 0 || y >= p.V);
    }
  }
  __shared__ int tot[kCountThreads / 32];
  n = __reduce_add_sync(0xffffffffu, n);
  bad = __reduce_or_sync(0xffffffffu, bad);
  if ((threadIdx.x & 31) == 0) tot[threadIdx.x >> 5] = n | (bad << 30);
  __syncthreads();
  if (threadIdx.x == 0) {
    int N = 0, b = 0;
    for (int w = 0; w < kCountThreads / 32; ++w) {
      N += tot[w] & ((1 << 30) - 1);
      b |= tot[w] >> 30;
    }
    *p.count = N;
    *p.status = (b || N == 0) ? VA_ERR_BAD_TARGETS : VA_OK;
  }
}

template <class T>
__global__ void __launch_bounds__(kCeThreads, 4) ce_rows_kernel(CeParams p) {
  griddep_begin();
  if (*p.status != VA_OK) return;
  constexpr int W = Vec<T>::W;
  const float invN = 1.f / static_cast<float>(*p.count);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ float sm_m[kCeWarps], sm_s[kCeWarps];
  __shared__ float row_lse2;
  const T* logits = static_cast<const T*>(p.logits);
  T* grad = static_cast<T*>(p.grad);
  const int Vv = p.vec ? p.V / W * W : 0;  // vectorised part of a row; the rest element-wise
  for (int row = blockIdx.x; row < p.T; row += gridDim.x) {
    const int y = __ldg(p.targets + row);
    T* g = grad ? grad + static_cast<int64_t>(row) * p.g_rs : nullptr;
    if (y == p.ignore) {  // not eligible: no arithmetic on its logits, a zero gradient row
      if (tid == 0) p.nll[row] = 0.f;
      if (g) {
        float zero[W];
#pragma unroll
        for (int i = 0; i < W; ++i) zero[i] = 0.f;
        for (int c = tid * W; c < Vv; c += kCeThreads * W) store_vec(g + c, zero);
        for (int c = Vv + tid; c < p.V; c += kCeThreads) g[c] = from_f<T>(0.f);
      }
      continue;
    }
    const T* z = logits + static_cast<int64_t>(row) * p.l_rs;
    // pass 1: base-2 log-sum-exp of z * log2(e); kU chunks per thread in flight
    float m = -INFINITY, s = 0.f;
    for (int c0 = tid * W; c0 < Vv; c0 += kU * kCeThreads * W) {
      uint4 raw[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (c0 + u * kCeThreads * W < Vv) raw[u] = load_raw<false>(z + c0 + u * kCeThreads * W);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if (c0 + u * kCeThreads * W >= Vv) continue;
        float x[W];
        unpack<T>(raw[u], x);
        float cm = x[0];
#pragma unroll
        for (int i = 1; i < W; ++i) cm = fmaxf(cm, x[i]);
        if (cm == -INFINITY) continue;  // nothing to add (and -inf - -inf would be NaN)
        cm *= kLog2e;
        float cs = 0.f;
#pragma unroll
        for (int i = 0; i < W; ++i) cs += fast_exp2(fmaf(x[i], kLog2e, -cm));
        ms_merge(m, s, cm, cs);
      }
    }
    for (int c = Vv + tid; c < p.V; c += kCeThreads) {
      const float x = to_f(z[c]) * kLog2e;
      ms_merge(m, s, x, 1.f);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
      ms_merge(m, s, m2, s2);
    }
    if (lane == 0) {
      sm_m[warp] = m;
      sm_s[warp] = s;
    }
    __syncthreads();
    if (tid == 0) {
      float M = sm_m[0], S = sm_s[0];
      for (int w = 1; w < kCeWarps; ++w) ms_merge(M, S, sm_m[w], sm_s[w]);
      const float lse2 = M + __log2f(S);
      row_lse2 = lse2;
      p.nll[row] = (lse2 - to_f(z[y]) * kLog2e) * kLn2;
    }
    __syncthreads();
    const float lse2 = row_lse2;
    // pass 2: gradient (p - onehot) / N
    if (g) {
      for (int c0 = tid * W; c0 < Vv; c0 += kU * kCeThreads * W) {
        uint4 raw[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u)
          if (c0 + u * kCeThreads * W < Vv) raw[u] = load_raw<true>(z + c0 + u * kCeThreads * W);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int c = c0 + u * kCeThreads * W;
          if (c >= Vv) continue;
          float x[W];
          unpack<T>(raw[u], x);
#pragma unroll
          for (int i = 0; i < W; ++i) x[i] = fast_exp2(fmaf(x[i], kLog2e, -lse2)) * invN - (c + i == y ? invN : 0.f);
          store_vec(g + c, x);
        }
      }
      for (int c = Vv + tid; c < p.V; c += kCeThreads) {
        const float x = fast_exp2(fmaf(to_f(z[c]), kLog2e, -lse2)) * invN - (c == y ? invN : 0.f);
        g[c] = from_f<T>(x);
      }
    }
    __syncthreads();  // sm_m / sm_s / row_lse2 are reused by the next row
  }
}

__global__ void __launch_bounds__(kCountThreads) ce_reduce_kernel(CeParams p) {
  griddep_begin();
  __shared__ double part[kCountThreads / 32];
  double acc = 0.0;  // fixed assignment of rows to threads and a fixed reduction order
  for (int t = threadIdx.x; t < p.T; t += kCountThreads) acc += static_cast<double>(p.nll[t]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double sum = 0.0;
    for (int w = 0; w < kCountThreads / 32; ++w) sum += part[w];
    const bool ok = *p.status == VA_OK;
    p.loss[0] = ok ? sum : NAN;
    p.loss[1] = ok ? sum / static_cast<double>(*p.count) : NAN;
  }
}

// ---------------------------------------------------------------- host side

cudaError_t launch_loss_targets(const int32_t* ids, const int32_t* cu, int B, int T, int ignore, int32_t* targets,
                                cudaStream_t st) {
  if (T <= 0) return cudaSuccess;
  return launch_pdl(loss_targets_kernel, dim3((T + 255) / 256), dim3(256), 0, st, ids, cu, B, T, ignore, targets);
}

namespace {
CeParams ce_params(const void* logits, int bf16, int64_t l_rs, const int32_t* targets, int T, int V, int ignore,
                   void* grad, int64_t g_rs, float* nll, int32_t* count, int32_t* status, double* loss) {
  CeParams p{logits, l_rs, targets, T, V, ignore, grad, g_rs, nll, count, status, loss, 0};
  const size_t es = bf16 ? 2 : 4;
  const auto al16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  p.vec = al16(logits) && (l_rs * es) % 16 == 0 && (!grad || (al16(grad) && (g_rs * es) % 16 == 0));
  return p;
}
}  // namespace

// The three launches of varlen_token_ce, in this order on one stream (stage 0: N and the
// target check, 1: the rows, 2: the sum).
cudaError_t launch_token_ce(int stage, const void* logits, int bf16, int64_t l_rs, const int32_t* targets, int T,
                            int V, int ignore, void* grad, int64_t g_rs, float* nll, int32_t* count,
                            int32_t* status, double* loss, cudaStream_t st) {
  const CeParams p = ce_params(logits, bf16, l_rs, targets, T, V, ignore, grad, g_rs, nll, count, status, loss);
  if (stage == 0) return launch_pdl(ce_count_kernel, dim3(1), dim3(kCountThreads), 0, st, p);
  if (stage == 2) return launch_pdl(ce_reduce_kernel, dim3(1), dim3(kCountThreads), 0, st, p);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = static_cast<int>(std::min<int64_t>(T, static_cast<int64_t>(std::max(sms, 1)) * kCeCtasPerSm));
  if (grid <= 0) return cudaSuccess;
  return bf16 ? launch_pdl(ce_rows_kernel<__nv_bfloat16>, dim3(grid), dim3(kCeThreads), 0, st, p)
              : launch_pdl(ce_rows_kernel<float>, dim3(grid), dim3(kCeThreads), 0, st, p);
}

}  // namespace va
