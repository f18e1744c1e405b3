// Host side of the C ABI: argument checks, workspace layout, launch sequences.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <string>
#include <vector>

#include "attn_params.cuh"

namespace va {

// kernels (other translation units)
cudaError_t launch_metadata_scan(const int32_t*, int, int, int, int32_t*, int32_t*, int32_t*, int32_t*,
                                 int32_t*, cudaStream_t);
bool metadata_inline_fill(int n, int T_capacity);
cudaError_t launch_metadata_fill(const int32_t*, int, int, int32_t*, int32_t*, const int32_t*,
                                 cudaStream_t);
cudaError_t launch_validate(const int32_t*, int, int, int, int32_t*, int, cudaStream_t);
cudaError_t launch_cu_from_positions(const int32_t*, int, int, int, int32_t*, int, int32_t*, int32_t*,
                                     int32_t*, cudaStream_t);
cudaError_t launch_plan(const PlanArgs&, cudaStream_t);
cudaError_t launch_validate_plan(const PlanArgs*, int, int, int, int, int, cudaStream_t);
cudaError_t launch_fwd_tc(const FwdParams&, int, int, cudaStream_t);
cudaError_t launch_fwd_tok(const FwdParams&, int, int, cudaStream_t);
void fwd_tc_tiles(int*, int*);
int fwd_tc_token_short();
int bwd_tc_token_short();
cudaError_t launch_bwd_prep(const BwdParams&, const PlanArgs*, int, int, int, int, int, int, cudaStream_t);
cudaError_t launch_unpad_index(int, const int32_t*, int, int, int32_t*, int32_t*, int32_t*, int32_t*, int32_t*,
                               int32_t*, cudaStream_t);
cudaError_t launch_gather_rows(const void*, int64_t, const int32_t*, int, int64_t, void*, int64_t, cudaStream_t);
cudaError_t launch_loss_targets(const int32_t*, const int32_t*, int, int, int, int32_t*, cudaStream_t);
cudaError_t launch_token_ce(int, const void*, int, int64_t, const int32_t*, int, int, int, void*, int64_t, float*,
                            int32_t*, int32_t*, double*, cudaStream_t);
cudaError_t launch_bwd_dkdv_tc(const BwdParams&, int, int, bool, cudaStream_t);
cudaError_t launch_bwd_dq_tc(const BwdParams&, int, int, bool, cudaStream_t);
void bwd_tc_tiles(int*, int*, int*, int*);

static thread_local std::string g_error;
// Test hook of the failure path: a wait limit (ns) armed for the next forward call, 0 = none.
static std::atomic<long long> g_stall_next_fwd{0};

void set_error(const char* msg) { g_error = msg; }

// ------------------------------------------------------------ launch accounting
enum KernelId {
  K_VALIDATE = 0, K_META_SCAN, K_META_FILL, K_PLAN, K_FWD, K_BWD_PREP, K_BWD_DKDV, K_BWD_DQ,
  K_VALIDATE_PLAN, K_FWD_TOK, K_CU_FROM_POS, K_LOSS_TARGETS, K_CE_COUNT, K_CE_ROWS, K_CE_REDUCE, K_PAD_COUNT,
  K_PAD_SCAN, K_PAD_INDEX, K_GATHER_ROWS, K_COUNT
};
const char* const kKernelNames[K_COUNT] = {
    "validate_cu_seqlens", "metadata_scan", "metadata_fill", "plan",          "fwd",
    "bwd_prep",            "bwd_dkdv",      "bwd_dq",        "validate_plan", "fwd_tok",
    "cu_from_positions",   "loss_targets",  "ce_count",      "ce_rows",       "ce_reduce",
    "pad_count",           "pad_scan",      "pad_index",     "gather_rows"};

struct Profiler {
  std::vector<cudaEvent_t> start, stop;
  std::vector<int32_t> ids;
  int cap = 0, n = 0;
};
static Profiler g_prof;
static std::atomic<long long> g_launches{0};

// Runs one kernel launch; counts it and, when profiling, brackets it with events.
template <class F>
cudaError_t launch(int id, cudaStream_t st, F&& f) {
  const bool rec = g_prof.cap > 0 && g_prof.n < g_prof.cap;
  if (rec) cudaEventRecord(g_prof.start[g_prof.n], st);
  cudaError_t e = f();
  if (rec) {
    cudaEventRecord(g_prof.stop[g_prof.n], st);
    g_prof.ids[g_prof.n++] = id;
  }
  if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
  return e;
}

namespace {

va_status fail(va_status st, const std::string& msg) {
  g_error = msg;
  return st;
}

va_status cuda_fail(cudaError_t e, const char* where) {
  return fail(VA_ERR_CUDA, std::string(where) + ": " + cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Token tiles (runs of short segments planned as tiles of consecutive tokens) pay off when
// short segments are common; they are used for causal calls whose mean segment length T / B
// is below this many tokens.  Results do not depend on the choice: it only selects which
// records cover the short segments and which kernel forms run.
constexpr int64_t kTokenMeanLen = 256;

bool token_tiles(const va_shape& s, int32_t causal, int32_t window) {
  return causal && window < 0 && static_cast<int64_t>(s.T) < kTokenMeanLen * s.B;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

void tiles(int kind, int* BM, int* BN) {
  if (kind == 0) {
    fwd_tc_tiles(BM, BN);
  } else {
    int a, b, c, d;
    bwd_tc_tiles(&a, &b, &c, &d);
    if (kind == 1) {
      *BM = a;
      *BN = b;
    } else {
      *BM = c;
      *BN = d;
    }
  }
}

// Upper bound on records of a map: blocks per segment <= l/blk + 1.  Tk: rows of K/V
// (cross-attention; -1 = s.T), which the kv-block map is cut from.
int64_t map_capacity(const va_shape& s, int kind, int Tk = -1) {
  int BM, BN;
  tiles(kind, &BM, &BN);
  const int blk = kind == 1 ? BN : BM;
  const int heads = kind == 1 ? s.Hkv : s.Hq;
  const int rows = kind == 1 && Tk >= 0 ? Tk : s.T;
  return (static_cast<int64_t>(rows) / blk + s.B) * heads;
}

// Cross-attention arguments: the K/V stream's rows and longest segment.
va_status check_cross(const va_shape* s, const int32_t* cu_k, int32_t Tk, int32_t max_k, int32_t window) {
  if (!cu_k) return fail(VA_ERR_INVALID_ARG, "cross: cu_seqlens_k is null");
  if (Tk < 1 || max_k < 1 || max_k > Tk) return fail(VA_ERR_INVALID_ARG, "cross: Tk >= 1 and 1 <= max_seqlen_k <= Tk");
  if (static_cast<int64_t>(Tk) * s->Hkv >= (int64_t(1) << 31)) return fail(VA_ERR_UNSUPPORTED, "Tk * Hkv must stay below 2^31");
  if (window != -1) return fail(VA_ERR_UNSUPPORTED, "cross: no local window");
  return VA_OK;
}

va_status check_shape(const va_shape* s) {
  if (!s) return fail(VA_ERR_INVALID_ARG, "shape is null");
  if (s->T < 0 || s->B < 1 || s->Hq < 1 || s->Hkv < 1 || s->max_seqlen < 1)
    return fail(VA_ERR_INVALID_ARG, "shape: T >= 0, B >= 1, heads >= 1, max_seqlen >= 1");
  if (s->d != 64 && s->d != 128) return fail(VA_ERR_UNSUPPORTED, "head dim must be 64 or 128");
  if (s->Hq % s->Hkv) return fail(VA_ERR_UNSUPPORTED, "Hq must be a multiple of Hkv");
  if (s->max_seqlen > std::max(s->T, 1)) return fail(VA_ERR_INVALID_ARG, "max_seqlen > T");
  const int64_t st[8] = {s->q_row_stride, s->q_head_stride, s->k_row_stride, s->k_head_stride,
                         s->v_row_stride, s->v_head_stride, s->o_row_stride, s->o_head_stride};
  for (int64_t x : st)
    if (x <= 0 || x % 8) return fail(VA_ERR_INVALID_ARG, "strides must be positive multiples of 8");
  for (int64_t x : st)
    if (x < s->d) return fail(VA_ERR_INVALID_ARG, "row and head strides must be >= d");
  if (static_cast<int64_t>(s->T) * std::max(s->Hq, s->Hkv) >= (int64_t(1) << 31))
    return fail(VA_ERR_UNSUPPORTED, "T * heads must stay below 2^31");
  return VA_OK;
}

struct FwdLayout {
  size_t map, segoff, total;
  int64_t cap;
};
FwdLayout fwd_layout(const va_shape& s) {
  FwdLayout L;
  L.cap = map_capacity(s, 0);
  L.map = sizeof(WsHeader);
  L.segoff = align256(L.map + static_cast<size_t>(L.cap) * sizeof(TileItem));
  L.total = align256(L.segoff + static_cast<size_t>(s.B) * sizeof(int32_t));
  return L;
}

struct BwdLayout {
  size_t dsum, kvmap, qmap, segoff, total;
  int64_t cap_kv, cap_q;
};
BwdLayout bwd_layout(const va_shape& s, int Tk = -1) {
  BwdLayout L;
  L.cap_kv = map_capacity(s, 1, Tk);
  L.cap_q = map_capacity(s, 2);
  L.dsum = sizeof(WsHeader);
  L.kvmap = align256(L.dsum + static_cast<size_t>(s.Hq) * s.T * sizeof(float));
  L.qmap = align256(L.kvmap + static_cast<size_t>(L.cap_kv) * sizeof(TileItem));
  L.segoff = align256(L.qmap + static_cast<size_t>(L.cap_q) * sizeof(TileItem));
  L.total = align256(L.segoff + static_cast<size_t>(s.B) * sizeof(int32_t));
  return L;
}

}  // namespace
}  // namespace va

using namespace va;

static va_status plan_impl(const va_shape* s, const int32_t* cu_dev, const int32_t* cu_k, int32_t Tk, int32_t kind,
                           int32_t causal, int32_t window, int32_t* map_dev, int32_t capacity, int32_t* n_items_dev,
                           int32_t* scratch_dev, va_stream_t stream);
static va_status fwd_impl(const void* q, const void* k, const void* v, const int32_t* cu, const int32_t* cu_k,
                          int32_t Tk, int32_t max_k, const va_shape* s, float scale, int32_t causal, int32_t window,
                          void* out, float* lse, void* ws, size_t ws_bytes, va_stream_t stream);
static va_status bwd_impl(const void* q, const void* k, const void* v, const void* out, const float* lse,
                          const void* dout, const int32_t* cu, const int32_t* cu_k, int32_t Tk, int32_t max_k,
                          const va_shape* s, float scale, int32_t causal, int32_t window, void* dq, void* dk, void* dv,
                          void* ws, size_t ws_bytes, va_stream_t stream);

extern "C" {

const char* varlen_last_error(void) { return g_error.c_str(); }

const char* varlen_version(void) { return "varlen_attn 0.1 (sm_103a)"; }

void varlen_shape_contiguous(va_shape* s, int32_t T, int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                             int32_t max_seqlen) {
  if (!s) return;
  s->T = T;
  s->B = B;
  s->Hq = Hq;
  s->Hkv = Hkv;
  s->d = d;
  s->max_seqlen = max_seqlen;
  s->q_row_stride = static_cast<int64_t>(Hq) * d;
  s->q_head_stride = d;
  s->k_row_stride = static_cast<int64_t>(Hkv) * d;
  s->k_head_stride = d;
  s->v_row_stride = static_cast<int64_t>(Hkv) * d;
  s->v_head_stride = d;
  s->o_row_stride = static_cast<int64_t>(Hq) * d;
  s->o_head_stride = d;
}

va_status varlen_build_metadata(const int32_t* lengths_dev, int32_t n, int32_t pad_to,
                                int32_t T_capacity, int32_t* cu_dev, int32_t* pos_dev,
                                int32_t* seg_dev, int32_t* max_dev, int32_t* status_dev,
                                va_stream_t stream) {
  if (n < 0 || pad_to < 0 || T_capacity < 0 || !cu_dev || !max_dev || !status_dev ||
      (n > 0 && !lengths_dev) || (T_capacity > 0 && (!pos_dev || !seg_dev)))
    return fail(VA_ERR_INVALID_ARG, "build_metadata: null pointer or negative size");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch(K_META_SCAN, cs, [&] {
    return launch_metadata_scan(lengths_dev, n, pad_to, T_capacity, cu_dev, max_dev, status_dev, pos_dev, seg_dev,
                                cs);
  });
  // short streams get their positions and segment ids from the scan's block
  if (e == cudaSuccess && T_capacity > 0 && !metadata_inline_fill(n, T_capacity))
    e = launch(K_META_FILL, cs, [&] {
      return launch_metadata_fill(cu_dev, n, T_capacity, pos_dev, seg_dev, status_dev, cs);
    });
  return e == cudaSuccess ? VA_OK : cuda_fail(e, "build_metadata");
}

va_status varlen_validate_cu_seqlens(const int32_t* cu_dev, int32_t B, int32_t T, int32_t max_seqlen,
                                     int32_t* status_dev, va_stream_t stream) {
  if (!cu_dev || !status_dev || B < 1 || T < 0 || max_seqlen < 1)
    return fail(VA_ERR_INVALID_ARG, "validate: null pointer or bad size");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch(K_VALIDATE, cs, [&] {
    return launch_validate(cu_dev, B, T, max_seqlen, status_dev, 0, cs);
  });
  return e == cudaSuccess ? VA_OK : cuda_fail(e, "validate");
}

va_status varlen_cu_seqlens_from_positions(const int32_t* position_ids_dev, int32_t T, int32_t reset_at_min,
                                           int32_t strict, int32_t* cu_seqlens_dev, int32_t capacity,
                                           int32_t* B_dev, int32_t* max_seqlen_dev, int32_t* status_dev,
                                           va_stream_t stream) {
  if (!position_ids_dev || !cu_seqlens_dev || !B_dev || !max_seqlen_dev || !status_dev)
    return fail(VA_ERR_INVALID_ARG, "cu_seqlens_from_positions: null pointer");
  if (T < 1 || capacity < 2)
    return fail(VA_ERR_INVALID_ARG, "cu_seqlens_from_positions: T >= 1 and capacity >= 2");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch(K_CU_FROM_POS, cs, [&] {
    return launch_cu_from_positions(position_ids_dev, T, reset_at_min ? 1 : 0, strict ? 1 : 0, cu_seqlens_dev,
                                    capacity, B_dev, max_seqlen_dev, status_dev, cs);
  });
  return e == cudaSuccess ? VA_OK : cuda_fail(e, "cu_seqlens_from_positions");
}

va_status varlen_attn_tile_sizes(int32_t kind, int32_t d, int32_t* BM, int32_t* BN) {
  if (kind < 0 || kind > 2 || !BM || !BN) return fail(VA_ERR_INVALID_ARG, "tile_sizes: bad kind");
  if (d != 64 && d != 128) return fail(VA_ERR_UNSUPPORTED, "tile_sizes: d must be 64 or 128");
  int a, b;
  tiles(kind, &a, &b);
  *BM = a;
  *BN = b;
  return VA_OK;
}

size_t varlen_attn_workspace_size(const va_shape* s, int32_t for_bwd) {
  if (check_shape(s) != VA_OK) return 0;
  return for_bwd ? bwd_layout(*s).total : fwd_layout(*s).total;
}

va_status varlen_attn_plan(const va_shape* s, const int32_t* cu_dev, int32_t kind, int32_t causal,
                           int32_t* map_dev, int32_t capacity, int32_t* n_items_dev,
                           int32_t* scratch_dev, va_stream_t stream) {
  return varlen_attn_plan_window(s, cu_dev, kind, causal, -1, map_dev, capacity, n_items_dev, scratch_dev, stream);
}

va_status varlen_attn_plan_window(const va_shape* s, const int32_t* cu_dev, int32_t kind, int32_t causal,
                                  int32_t window, int32_t* map_dev, int32_t capacity, int32_t* n_items_dev,
                                  int32_t* scratch_dev, va_stream_t stream) {
  return plan_impl(s, cu_dev, nullptr, -1, kind, causal, window, map_dev, capacity, n_items_dev, scratch_dev, stream);
}

va_status varlen_attn_plan_cross(const va_shape* s, const int32_t* cu_q, const int32_t* cu_k, int32_t Tk, int32_t kind,
                                 int32_t causal, int32_t* map_dev, int32_t capacity, int32_t* n_items_dev,
                                 int32_t* scratch_dev, va_stream_t stream) {
  return plan_impl(s, cu_q, cu_k, Tk, kind, causal, -1, map_dev, capacity, n_items_dev, scratch_dev, stream);
}

}  // extern "C"

static va_status plan_impl(const va_shape* s, const int32_t* cu_dev, const int32_t* cu_k, int32_t Tk, int32_t kind,
                           int32_t causal, int32_t window, int32_t* map_dev, int32_t capacity, int32_t* n_items_dev,
                           int32_t* scratch_dev, va_stream_t stream) {
  va_status st = check_shape(s);
  if (st != VA_OK) return st;
  if (cu_k && (st = check_cross(s, cu_k, Tk, std::max(Tk, 1), window)) != VA_OK) return st;
  if (window < -1 || (window >= 0 && !causal)) return fail(VA_ERR_INVALID_ARG, "plan: window needs causal and >= 0 (-1 = none)");
  if (kind < 0 || kind > 2 || !cu_dev || !map_dev || !n_items_dev || !scratch_dev || capacity < 0)
    return fail(VA_ERR_INVALID_ARG, "plan: bad kind or null pointer");
  if (!aligned16(map_dev)) return fail(VA_ERR_INVALID_ARG, "plan: tile map must be 16-byte aligned");
  if (map_capacity(*s, kind, cu_k ? Tk : -1) > capacity)
    return fail(VA_ERR_WORKSPACE, "plan: capacity below the record bound (T/blk + B) * heads");
  int BM, BN;
  tiles(kind, &BM, &BN);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const PlanArgs pa{cu_dev, s->B, kind == 1 ? s->Hkv : s->Hq, BM, BN, kind, causal ? 1 : 0,
                    reinterpret_cast<TileItem*>(map_dev), capacity, nullptr, n_items_dev,
                    scratch_dev + 4, scratch_dev,
                    (cu_k || !token_tiles(*s, causal, window)) ? 0
                    : kind == 0                                ? fwd_tc_token_short()
                                                               : bwd_tc_token_short(),
                    nullptr, nullptr, window, cu_k};
  cudaError_t e = launch(K_PLAN, cs, [&] { return launch_plan(pa, cs); });
  return e == cudaSuccess ? VA_OK : cuda_fail(e, "plan");
}

extern "C" {

va_status varlen_attn_fwd(const void* q, const void* k, const void* v, const int32_t* cu,
                          const va_shape* s, float scale, int32_t causal, void* out, float* lse,
                          void* ws, size_t ws_bytes, va_stream_t stream) {
  return varlen_attn_fwd_window(q, k, v, cu, s, scale, causal, -1, out, lse, ws, ws_bytes, stream);
}

va_status varlen_attn_fwd_window(const void* q, const void* k, const void* v, const int32_t* cu,
                                 const va_shape* s, float scale, int32_t causal, int32_t window, void* out,
                                 float* lse, void* ws, size_t ws_bytes, va_stream_t stream) {
  return fwd_impl(q, k, v, cu, nullptr, -1, 0, s, scale, causal, window, out, lse, ws, ws_bytes, stream);
}

va_status varlen_attn_fwd_cross(const void* q, const void* k, const void* v, const int32_t* cu_q,
                                const int32_t* cu_k, const va_shape* s, int32_t Tk, int32_t max_seqlen_k, float scale,
                                int32_t causal, void* out, float* lse, void* ws, size_t ws_bytes, va_stream_t stream) {
  return fwd_impl(q, k, v, cu_q, cu_k, Tk, max_seqlen_k, s, scale, causal, -1, out, lse, ws, ws_bytes, stream);
}

}  // extern "C"

static va_status fwd_impl(const void* q, const void* k, const void* v, const int32_t* cu, const int32_t* cu_k,
                          int32_t Tk, int32_t max_k, const va_shape* s, float scale, int32_t causal, int32_t window,
                          void* out, float* lse, void* ws, size_t ws_bytes, va_stream_t stream) {
  va_status st = check_shape(s);
  if (st != VA_OK) return st;
  if (cu_k && (st = check_cross(s, cu_k, Tk, max_k, window)) != VA_OK) return st;
  if (window < -1 || (window >= 0 && !causal)) return fail(VA_ERR_INVALID_ARG, "fwd: window needs causal and >= 0 (-1 = none)");
  if (!q || !k || !v || !cu || !out || !lse || !ws)
    return fail(VA_ERR_INVALID_ARG, "fwd: null pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(ws))
    return fail(VA_ERR_INVALID_ARG, "fwd: pointers must be 16-byte aligned");
  if (!(scale > 0.f) || !(scale < INFINITY)) return fail(VA_ERR_INVALID_ARG, "fwd: scale must be finite and > 0");
  const FwdLayout L = fwd_layout(*s);
  if (ws_bytes < L.total) return fail(VA_ERR_WORKSPACE, "fwd: workspace too small");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(w);
  TileItem* map = reinterpret_cast<TileItem*>(w + L.map);
  if (s->T == 0) {  // nothing to compute; still report a contract violation
    cudaError_t e = launch(K_VALIDATE, cs, [&] {
      return launch_validate(cu, s->B, s->T, s->max_seqlen, &hdr->status, 1, cs);
    });
    return e == cudaSuccess ? VA_OK : cuda_fail(e, "fwd validate");
  }
  int BM, BN;
  tiles(0, &BM, &BN);
  const bool tok = !cu_k && token_tiles(*s, causal, window);
  const PlanArgs pa{cu, s->B, s->Hq, BM, BN, 0, causal ? 1 : 0, map, static_cast<int>(L.cap),
                    &hdr->status, &hdr->n_items[0],
                    reinterpret_cast<int32_t*>(w + L.segoff), &hdr->counter[0],
                    tok ? fwd_tc_token_short() : 0, &hdr->n_items[kTokSlot],
                    &hdr->counter[kTokSlot], window, cu_k};
  cudaError_t e = launch(K_VALIDATE_PLAN, cs, [&] {
    return launch_validate_plan(&pa, 1, s->T, s->max_seqlen, cu_k ? Tk : 0, cu_k ? max_k : 0, cs);
  });
  if (e != cudaSuccess) return cuda_fail(e, "fwd plan");
  FwdParams p{};
  p.q = static_cast<const bf16*>(q);
  p.k = static_cast<const bf16*>(k);
  p.v = static_cast<const bf16*>(v);
  p.o = static_cast<bf16*>(out);
  p.lse = lse;
  p.cu = cu;
  p.items = map;
  p.B = s->B;
  p.hdr = hdr;
  p.slot = 0;
  p.counter = &hdr->counter[0];
  p.T = s->T;
  p.Hq = s->Hq;
  p.Hkv = s->Hkv;
  p.g = s->Hq / s->Hkv;
  p.q_rs = s->q_row_stride;
  p.q_hs = s->q_head_stride;
  p.k_rs = s->k_row_stride;
  p.k_hs = s->k_head_stride;
  p.v_rs = s->v_row_stride;
  p.v_hs = s->v_head_stride;
  p.o_rs = s->o_row_stride;
  p.o_hs = s->o_head_stride;
  p.scale_log2 = scale * kLog2e;
  p.causal = causal ? 1 : 0;
  p.window = window;
  p.cu_k = cu_k;
  p.Tk = cu_k ? Tk : 0;
  const long long stall_ns = g_stall_next_fwd.exchange(0);
  if (stall_ns > 0) {  // test hook: the producers load nothing and the waits give up after stall_ns
    p.wait_ns = static_cast<uint64_t>(stall_ns);
    p.stall = 1;
  }
  // segment records, then (as its programmatic dependent, filling its tail) token records
  e = launch(K_FWD, cs, [&] { return launch_fwd_tc(p, s->d, static_cast<int>(L.cap), cs); });
  if (e != cudaSuccess) return cuda_fail(e, "fwd kernel");
  if (!tok) return VA_OK;
  FwdParams pt = p;
  pt.counter = &hdr->counter[kTokSlot];
  e = launch(K_FWD_TOK, cs, [&] { return launch_fwd_tok(pt, s->d, static_cast<int>(L.cap), cs); });
  return e == cudaSuccess ? VA_OK : cuda_fail(e, "fwd token kernel");
}

extern "C" {

va_status varlen_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                          const float* lse, const void* dout, const int32_t* cu, const va_shape* s,
                          float scale, int32_t causal, void* dq, void* dk, void* dv, void* ws,
                          size_t ws_bytes, va_stream_t stream) {
  return varlen_attn_bwd_window(q, k, v, out, lse, dout, cu, s, scale, causal, -1, dq, dk, dv, ws, ws_bytes,
                                stream);
}

va_status varlen_attn_bwd_window(const void* q, const void* k, const void* v, const void* out,
                                 const float* lse, const void* dout, const int32_t* cu, const va_shape* s,
                                 float scale, int32_t causal, int32_t window, void* dq, void* dk, void* dv,
                                 void* ws, size_t ws_bytes, va_stream_t stream) {
  return bwd_impl(q, k, v, out, lse, dout, cu, nullptr, -1, 0, s, scale, causal, window, dq, dk, dv, ws, ws_bytes,
                  stream);
}

va_status varlen_attn_bwd_cross(const void* q, const void* k, const void* v, const void* out, const float* lse,
                                const void* dout, const int32_t* cu_q, const int32_t* cu_k, const va_shape* s,
                                int32_t Tk, int32_t max_seqlen_k, float scale, int32_t causal, void* dq, void* dk,
                                void* dv, void* ws, size_t ws_bytes, va_stream_t stream) {
  return bwd_impl(q, k, v, out, lse, dout, cu_q, cu_k, Tk, max_seqlen_k, s, scale, causal, -1, dq, dk, dv, ws,
                  ws_bytes, stream);
}

size_t varlen_attn_workspace_size_cross(const va_shape* s, int32_t Tk, int32_t for_bwd) {
  if (check_shape(s) != VA_OK || Tk < 1) return 0;
  return for_bwd ? bwd_layout(*s, Tk).total : fwd_layout(*s).total;
}

}  // extern "C"

static va_status bwd_impl(const void* q, const void* k, const void* v, const void* out, const float* lse,
                          const void* dout, const int32_t* cu, const int32_t* cu_k, int32_t Tk, int32_t max_k,
                          const va_shape* s, float scale, int32_t causal, int32_t window, void* dq, void* dk, void* dv,
                          void* ws, size_t ws_bytes, va_stream_t stream) {
  va_status st = check_shape(s);
  if (st != VA_OK) return st;
  if (cu_k && (st = check_cross(s, cu_k, Tk, max_k, window)) != VA_OK) return st;
  if (window < -1 || (window >= 0 && !causal)) return fail(VA_ERR_INVALID_ARG, "bwd: window needs causal and >= 0 (-1 = none)");
  if (!q || !k || !v || !out || !lse || !dout || !cu || !dq || !dk || !dv || !ws)
    return fail(VA_ERR_INVALID_ARG, "bwd: null pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(ws))
    return fail(VA_ERR_INVALID_ARG, "bwd: pointers must be 16-byte aligned");
  if (!(scale > 0.f) || !(scale < INFINITY)) return fail(VA_ERR_INVALID_ARG, "bwd: scale must be finite and > 0");
  const BwdLayout L = bwd_layout(*s, cu_k ? Tk : -1);
  if (ws_bytes < L.total) return fail(VA_ERR_WORKSPACE, "bwd: workspace too small");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(w);
  TileItem* kvmap = reinterpret_cast<TileItem*>(w + L.kvmap);
  TileItem* qmap = reinterpret_cast<TileItem*>(w + L.qmap);
  if (s->T == 0) {
    cudaError_t e = launch(K_VALIDATE, cs, [&] {
      return launch_validate(cu, s->B, s->T, s->max_seqlen, &hdr->status, 1, cs);
    });
    return e == cudaSuccess ? VA_OK : cuda_fail(e, "bwd validate");
  }
  int BM, BN, BM2, BN2;
  tiles(1, &BM, &BN);
  tiles(2, &BM2, &BN2);
  const bool tok = !cu_k && token_tiles(*s, causal, window);
  int32_t* segoff = reinterpret_cast<int32_t*>(w + L.segoff);
  const PlanArgs pa[2] = {
      {cu, s->B, s->Hkv, BM, BN, 1, causal ? 1 : 0, kvmap, static_cast<int>(L.cap_kv), &hdr->status,
       &hdr->n_items[1], segoff, &hdr->counter[1], tok ? bwd_tc_token_short() : 0,
       &hdr->n_items[kKvTokSlot], nullptr, window, cu_k},
      {cu, s->B, s->Hq, BM2, BN2, 2, causal ? 1 : 0, qmap, static_cast<int>(L.cap_q), &hdr->status,
       &hdr->n_items[2], segoff, &hdr->counter[2], tok ? bwd_tc_token_short() : 0,
       &hdr->n_items[kQTokSlot], nullptr, window, cu_k}};
  BwdParams p{};
  p.q = static_cast<const bf16*>(q);
  p.k = static_cast<const bf16*>(k);
  p.v = static_cast<const bf16*>(v);
  p.o = static_cast<const bf16*>(out);
  p.dout = static_cast<const bf16*>(dout);
  p.lse = lse;
  p.dsum = reinterpret_cast<float*>(w + L.dsum);
  p.dq = static_cast<bf16*>(dq);
  p.dk = static_cast<bf16*>(dk);
  p.dv = static_cast<bf16*>(dv);
  p.cu = cu;
  p.B = s->B;
  p.kv_items = kvmap;
  p.q_items = qmap;
  p.hdr = hdr;
  p.kv_slot = 1;
  p.q_slot = 2;
  p.kv_tok_slot = kKvTokSlot;
  p.q_tok_slot = kQTokSlot;
  p.kv_counter = &hdr->counter[1];
  p.q_counter = &hdr->counter[2];
  p.T = s->T;
  p.Hq = s->Hq;
  p.Hkv = s->Hkv;
  p.g = s->Hq / s->Hkv;
  p.q_rs = s->q_row_stride;
  p.q_hs = s->q_head_stride;
  p.k_rs = s->k_row_stride;
  p.k_hs = s->k_head_stride;
  p.v_rs = s->v_row_stride;
  p.v_hs = s->v_head_stride;
  p.o_rs = s->o_row_stride;
  p.o_hs = s->o_head_stride;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.causal = causal ? 1 : 0;
  p.window = window;
  p.cu_k = cu_k;
  p.Tk = cu_k ? Tk : 0;
  // one launch validates, plans both maps and computes D = rowsum(dO * O)
  cudaError_t e = launch(K_BWD_PREP, cs, [&] {
    return launch_bwd_prep(p, pa, 2, s->T, s->max_seqlen, cu_k ? Tk : 0, cu_k ? max_k : 0, s->d, cs);
  });
  if (e == cudaSuccess)
    e = launch(K_BWD_DKDV, cs, [&] { return launch_bwd_dkdv_tc(p, s->d, static_cast<int>(L.cap_kv), tok, cs); });
  if (e == cudaSuccess)
    e = launch(K_BWD_DQ, cs, [&] { return launch_bwd_dq_tc(p, s->d, static_cast<int>(L.cap_q), tok, cs); });
  return e == cudaSuccess ? VA_OK : cuda_fail(e, "bwd kernels");
}

extern "C" {

va_status varlen_unpad_index(const int32_t* mask, int32_t Bp, int32_t S, int32_t* indices, int32_t* inverse,
                             int32_t* cu, int32_t* T_out, int32_t* max_out, int32_t* status, va_stream_t stream) {
  if (!mask || !indices || !inverse || !cu || !T_out || !max_out || !status)
    return fail(VA_ERR_INVALID_ARG, "unpad_index: null pointer");
  if (Bp < 1 || S < 1 || static_cast<int64_t>(Bp) * S >= (int64_t(1) << 31))
    return fail(VA_ERR_INVALID_ARG, "unpad_index: Bp >= 1, S >= 1 and Bp * S < 2^31");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const KernelId ids[3] = {K_PAD_COUNT, K_PAD_SCAN, K_PAD_INDEX};
  cudaError_t e = cudaSuccess;
  for (int stage = 0; stage < 3 && e == cudaSuccess; ++stage)
    e = launch(ids[stage], cs, [&] {
      return launch_unpad_index(stage, mask, Bp, S, indices, inverse, cu, T_out, max_out, status, cs);
    });
  return e == cudaSuccess ? VA_OK : cuda_fail(e, "unpad_index");
}

va_status varlen_gather_rows(const void* src, int64_t src_stride, const int32_t* map, int32_t n_rows, int64_t row_bytes,
                             void* dst, int64_t dst_stride, va_stream_t stream) {
  if (!src || !map || !dst || n_rows < 0) return fail(VA_ERR_INVALID_ARG, "gather_rows: null pointer or n_rows < 0");
  if (row_bytes <= 0 || row_bytes % 16 || src_stride % 16 || dst_stride % 16 || src_stride < row_bytes ||
      dst_stride < row_bytes || !aligned16(src) || !aligned16(dst))
    return fail(VA_ERR_INVALID_ARG, "gather_rows: rows, strides and pointers must be 16-byte multiples");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch(K_GATHER_ROWS, cs, [&] {
    return launch_gather_rows(src, src_stride, map, n_rows, row_bytes, dst, dst_stride, cs);
  });
  return e == cudaSuccess ? VA_OK : cuda_fail(e, "gather_rows");
}

va_status varlen_loss_targets(const int32_t* ids, const int32_t* cu, int32_t B, int32_t T, int32_t ignore_index,
                              int32_t* targets, va_stream_t stream) {
  if (!ids || !cu || !targets || T < 0 || B < 1) return fail(VA_ERR_INVALID_ARG, "loss_targets: null pointer or bad size");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = launch(K_LOSS_TARGETS, cs, [&] { return launch_loss_targets(ids, cu, B, T, ignore_index, targets, cs); });
  return e == cudaSuccess ? VA_OK : cuda_fail(e, "loss_targets");
}

size_t varlen_token_ce_workspace_size(int32_t T) {
  return T < 0 ? 0 : align256(sizeof(WsHeader) + static_cast<size_t>(T) * sizeof(float));
}

va_status varlen_token_ce(const void* logits, int32_t dtype, int64_t l_rs, const int32_t* targets, int32_t T,
                          int32_t V, int32_t ignore_index, double* loss, int32_t* count, void* grad, int64_t g_rs,
                          void* ws, size_t ws_bytes, va_stream_t stream) {
  if (!logits || !targets || !loss || !count || !ws) return fail(VA_ERR_INVALID_ARG, "token_ce: null pointer");
  if (T < 1 || V < 1 || (dtype != 0 && dtype != 1)) return fail(VA_ERR_INVALID_ARG, "token_ce: T, V >= 1, dtype 0 or 1");
  if (l_rs < V || (grad && g_rs < V)) return fail(VA_ERR_INVALID_ARG, "token_ce: row strides must be >= V");
  if (!aligned16(ws)) return fail(VA_ERR_INVALID_ARG, "token_ce: workspace must be 16-byte aligned");
  if (ws_bytes < varlen_token_ce_workspace_size(T)) return fail(VA_ERR_WORKSPACE, "token_ce: workspace too small");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(ws);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(w);
  float* nll = reinterpret_cast<float*>(w + sizeof(WsHeader));
  cudaError_t e = cudaSuccess;
  const KernelId ids[3] = {K_CE_COUNT, K_CE_ROWS, K_CE_REDUCE};
  for (int stage = 0; stage < 3 && e == cudaSuccess; ++stage)
    e = launch(ids[stage], cs, [&] {
      return launch_token_ce(stage, logits, dtype, l_rs, targets, T, V, ignore_index, grad, g_rs, nll, count,
                             &hdr->status, loss, cs);
    });
  return e == cudaSuccess ? VA_OK : cuda_fail(e, "token_ce");
}

va_status varlen_read_status(const void* ws, int32_t* out, va_stream_t stream) {
  if (!ws || !out) return fail(VA_ERR_INVALID_ARG, "read_status: null pointer");
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(out, ws, sizeof(int32_t), cudaMemcpyDeviceToHost, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  return e == cudaSuccess ? VA_OK : cuda_fail(e, "read_status");
}

va_status varlen_clear_status(void* ws, va_stream_t stream) {
  if (!ws) return fail(VA_ERR_INVALID_ARG, "clear_status: null pointer");
  cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? VA_OK : cuda_fail(e, "clear_status");
}

va_status varlen_profile_enable(int32_t capacity) {
  for (cudaEvent_t e : g_prof.start) cudaEventDestroy(e);
  for (cudaEvent_t e : g_prof.stop) cudaEventDestroy(e);
  g_prof = Profiler{};
  if (capacity < 0) return fail(VA_ERR_INVALID_ARG, "profile_enable: negative capacity");
  if (capacity == 0) return VA_OK;
  g_prof.start.resize(capacity);
  g_prof.stop.resize(capacity);
  g_prof.ids.resize(capacity);
  for (int i = 0; i < capacity; ++i) {
    cudaError_t e = cudaEventCreate(&g_prof.start[i]);
    if (e == cudaSuccess) e = cudaEventCreate(&g_prof.stop[i]);
    if (e != cudaSuccess) {
      g_prof.start.resize(i);
      g_prof.stop.resize(i);
      return cuda_fail(e, "profile_enable");
    }
  }
  g_prof.cap = capacity;
  return VA_OK;
}

va_status varlen_profile_read(int32_t* ids, float* ms, int32_t capacity, int32_t* count) {
  if (!count || (capacity > 0 && (!ids || !ms)))
    return fail(VA_ERR_INVALID_ARG, "profile_read: null pointer");
  const int n = std::min(g_prof.n, capacity);
  for (int i = 0; i < n; ++i) {
    cudaError_t e = cudaEventSynchronize(g_prof.stop[i]);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms[i], g_prof.start[i], g_prof.stop[i]);
    if (e != cudaSuccess) return cuda_fail(e, "profile_read");
    ids[i] = g_prof.ids[i];
  }
  *count = n;
  g_prof.n = 0;
  return VA_OK;
}

const char* varlen_kernel_name(int32_t id) {
  return (id >= 0 && id < K_COUNT) ? kKernelNames[id] : "";
}

int64_t varlen_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

va_status varlen_test_stall_next_forward(int64_t wait_limit_ns) {
  if (wait_limit_ns < 1000000 || wait_limit_ns > 2000000000)
    return fail(VA_ERR_INVALID_ARG, "test_stall_next_forward: the limit must be 1 ms .. 2 s");
  g_stall_next_fwd.store(wait_limit_ns);
  return VA_OK;
}

}  // extern "C"
