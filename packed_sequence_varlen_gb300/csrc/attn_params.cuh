// Kernel parameter blocks for the attention kernels.
#pragma once
#include "common.cuh"

namespace va {

using bf16 = __nv_bfloat16;

struct FwdParams {
  const bf16* q;
  const bf16* k;
  const bf16* v;
  bf16* o;
  float* lse;  // [Hq, T]
  const int32_t* cu;
  const TileItem* items;
  int B;  // segments (cu has B + 1 entries)
  WsHeader* hdr;
  int slot;
  int32_t* counter;  // work counter (records are pulled in list order)
  int T, Hq, Hkv, g;
  int64_t q_rs, q_hs, k_rs, k_hs, v_rs, v_hs, o_rs, o_hs;
  float scale_log2;  // scale * log2(e)
  int causal;
  int window = -1;   // causal local window: query i sees keys i-w..i; -1 = none
  const int32_t* cu_k = nullptr;  // cross-attention: K/V boundaries (cu is Q's); null = cu
  int Tk = 0;                     // cross-attention: rows of K and V
  // Test hook of the failure path (varlen_test_stall_next_forward): a wait limit in ns
  // (0 = the default) and stall = 1, which makes each CTA's producer publish its first work
  // item and then load nothing, so the consumers' bounded waits run out.
  uint64_t wait_ns = 0;
  int stall = 0;
};

struct BwdParams {
  const bf16* q;
  const bf16* k;
  const bf16* v;
  const bf16* o;
  const bf16* dout;
  const float* lse;  // [Hq, T], natural log
  float* dsum;       // D = rowsum(dO * O), [Hq, T]
  bf16* dq;
  bf16* dk;
  bf16* dv;
  const int32_t* cu;
  int B;  // segments (cu has B + 1 entries)
  const TileItem* kv_items;  // kv-block map
  const TileItem* q_items;   // q-block map (dQ pass)
  WsHeader* hdr;
  int kv_slot, q_slot;          // n_items[slot]: all records of the map
  int kv_tok_slot, q_tok_slot;  // n_items[slot]: the token records at the map's end
  int32_t* kv_counter;
  int32_t* q_counter;
  int T, Hq, Hkv, g;
  int64_t q_rs, q_hs, k_rs, k_hs, v_rs, v_hs, o_rs, o_hs;
  float scale;
  float scale_log2;
  int causal;
  int window = -1;   // causal local window: query i sees keys i-w..i; -1 = none
  const int32_t* cu_k = nullptr;  // cross-attention: K/V boundaries (cu is Q's); null = cu
  int Tk = 0;                     // cross-attention: rows of K and V
};

}  // namespace va
