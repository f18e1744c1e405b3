// Dynamic work distribution inside a persistent CTA.
//
// The TMA producer thread pulls record indices from the map's global counter
// (atomicAdd, so CTAs take records in list order as they free up), decodes the
// record and publishes it through a two-slot shared-memory queue; the MMA thread
// and the softmax threads take the records in the same order.  Slot k & 1 holds
// the k-th record of this CTA; `full` completes when it is written, `empty` when
// every consumer has read it.
#pragma once
#include "sm100_ptx.cuh"

namespace va {
namespace sm100 {

// Publishes this CTA's k-th record.  Returns false when the list is exhausted
// (an invalid record is published so the consumers stop) or on abort (ok=false).
template <class It, class Decode>
__device__ __forceinline__ bool queue_publish(int k, It* slots, uint32_t full0, uint32_t empty0,
                                              int32_t* counter, int n_items, Decode decode,
                                              It& out, volatile int* abort_flag, WsHeader* hdr,
                                              bool& ok) {
  const int s = k & 1;
  ok = mbar_wait(empty0 + 8u * s, ((k >> 1) & 1) ^ 1, abort_flag, hdr, 40);
  if (!ok) return false;
  const int idx = atomicAdd(counter, 1);
  if (idx < n_items) {
    out = decode(idx);
    out.valid = 1;
  } else {
    out = It{};
    out.valid = 0;
  }
  slots[s] = out;
  mbar_arrive(full0 + 8u * s);  // release: the slot's contents become visible
  return out.valid != 0;
}

// queue_publish for a whole warp: lane 0 pulls the index and writes the slot, every lane
// returns the same record and the same flags (the warp stays converged).
template <class It, class Decode>
__device__ __forceinline__ bool queue_publish_w(int k, It* slots, uint32_t full0, uint32_t empty0,
                                                int32_t* counter, int n_items, Decode decode, It& out,
                                                volatile int* abort_flag, WsHeader* hdr, bool& ok) {
  const int s = k & 1;
  ok = wwait(empty0 + 8u * s, ((k >> 1) & 1) ^ 1, abort_flag, hdr, 40);
  if (!ok) return false;
  int idx = 0;
  if ((threadIdx.x & 31) == 0) idx = atomicAdd(counter, 1);
  idx = __shfl_sync(0xffffffffu, idx, 0);
  if (idx < n_items) {
    out = decode(idx);
    out.valid = 1;
  } else {
    out = It{};
    out.valid = 0;
  }
  if ((threadIdx.x & 31) == 0) {
    slots[s] = out;
    mbar_arrive(full0 + 8u * s);  // release: the slot's contents become visible
  }
  __syncwarp();
  return out.valid != 0;
}

// Takes this CTA's k-th record.  Returns false at the end of the list or on abort.
template <class It>
__device__ __forceinline__ bool queue_take(int k, const It* slots, uint32_t full0, uint32_t empty0,
                                           It& out, volatile int* abort_flag, WsHeader* hdr,
                                           bool& ok) {
  const int s = k & 1;
  ok = mbar_wait(full0 + 8u * s, (k >> 1) & 1, abort_flag, hdr, 41);
  if (!ok) return false;
  out = slots[s];
  mbar_arrive(empty0 + 8u * s);
  return out.valid != 0;
}

}  // namespace sm100
}  // namespace va
