// Segment-aware tile scheduler: the planning kernels.  The planning itself (order,
// per-class ranking, record layout) is in plan_body.cuh.
#include "plan_body.cuh"

namespace va {

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs a) {
  __shared__ PlanSmem sh;
  if (a.status && *a.status != VA_OK) {
    if (threadIdx.x == 0) *a.n_items = 0;
    return;
  }
  const int* cu = stage_cu(a.cu, a.B, sh);
  plan_body(a, sh, cu, a.B + 1 > kSmemSegs ? a.seg_off : sh.off);
}


// One launch per attention call: checks the cu_seqlens contract (cu[0] == 0,
// cu[B] == T, strictly increasing, every length <= max_seqlen), writes the status
// word (OK or VA_ERR_BAD_SEQLENS), and only if it holds builds the call's maps.
// Packs of at most 32 segments (the planner's short path) get 512 threads: on ~10 segments
// the launch took 0.7 us less than with 1024 (fewer warps at each block barrier) and as
// little as with 256, which writes larger maps in more passes.  Larger packs keep 1024, so
// the general path ranks them in as few rounds as it can.
constexpr int kSmallPlanThreads = 512;

__global__ void __launch_bounds__(kPlanThreads) validate_plan_kernel(PlanPair pp) {
  __shared__ PlanSmem sh;
  griddep_begin();  // cu_seqlens may come from the metadata kernels just before
  validate_plan_body(pp, sh);
}

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t st) {
  plan_kernel<<<1, kPlanThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_validate_plan(const PlanArgs* maps, int nmaps, int T, int max_seqlen, int Tk, int max_seqlen_k,
                                 cudaStream_t st) {
  PlanPair pp{};
  for (int i = 0; i < nmaps && i < 2; ++i) pp.map[i] = maps[i];
  pp.nmaps = nmaps;
  pp.T = T;
  pp.max_seqlen = max_seqlen;
  pp.Tk = Tk;
  pp.max_seqlen_k = max_seqlen_k;
  const int threads = nmaps >= 1 && maps[0].B <= 32 ? kSmallPlanThreads : kPlanThreads;
  return launch_pdl(validate_plan_kernel, dim3(1), dim3(threads), 0, st, pp);
}

}  // namespace va
