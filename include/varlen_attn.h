/*
 * varlen_attn.h -- C ABI of the GB300 (sm_103a) packed-sequence attention library.
 *
 * The library computes block-diagonal causal attention over a padding-free
 * packed token stream.  Q, K, V and O share one token axis of length T
 * ([T, H, d], the last dim contiguous) and the int32 boundary array
 * cu_seqlens[B+1] cuts that axis into B independent segments
 * [cu_seqlens[b], cu_seqlens[b+1]); no [T, T] mask is ever built.
 *   Source: "Packing与 FlashAttention Varlen", section 1 (mental model: physical
 *   continuity, logical discontinuity), section 3 (the cumulative-boundary
 *   contract) and section 5 (per-segment address domain and tile bounds);
 *   "Pack sequences without joining their contexts", "Permission depends on
 *   the example" (block-causal permission rule).
 *
 * Conventions shared by every entry point:
 *   - Ownership: the caller owns every buffer.  Apart from the host planner's
 *     own bookkeeping, the library allocates nothing; workspaces are sized with
 *     varlen_attn_workspace_size() and passed in.  Outputs are overwritten.
 *   - Pointers named *_dev are device pointers; the others are host pointers.
 *   - Asynchrony: device calls are enqueued on the caller's stream and return
 *     at once.  The return code covers what the host can check (arguments,
 *     sizes, alignment, launch errors).  What only the device can see (a
 *     cu_seqlens that breaks the contract, a bounded wait that gave up) is
 *     written as a va_status into the int32 status word at byte 0 of the
 *     workspace; read it after synchronising (varlen_read_status()).  Kernels
 *     that find a non-zero status do no work.
 *   - Errors never trap, abort or throw across the ABI.  varlen_last_error()
 *     gives a message for the last failing call on this host thread.
 *   - dtypes: q, k, v, out, dout, dq, dk, dv are bf16; lse is fp32 [Hq, T].
 *   - Alignment: base pointers 16-byte aligned; row and head strides (in
 *     elements) multiples of 8; d in {64, 128}; Hq % Hkv == 0 (q head h reads
 *     kv head h / (Hq / Hkv)).
 */
#ifndef VARLEN_ATTN_H
#define VARLEN_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* va_stream_t; /* a cudaStream_t; NULL is the legacy default stream */

typedef enum {
  VA_OK = 0,
  VA_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad alignment or stride */
  VA_ERR_UNSUPPORTED = 2,  /* d not in {64,128}, Hq % Hkv != 0, ... */
  VA_ERR_WORKSPACE = 3,    /* workspace smaller than varlen_attn_workspace_size() */
  VA_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
  VA_ERR_BAD_SEQLENS = 5,  /* cu_seqlens breaks the contract (device-detected or host) */
  VA_ERR_TIMEOUT = 6,      /* a bounded device wait gave up (device-detected) */
  VA_ERR_CAPACITY = 7,     /* planner: a document longer than the pack capacity */
  VA_ERR_BAD_TARGETS = 8   /* loss: an eligible target outside [0, V), or none eligible (device-detected) */
} va_status;

/* Shape and strides of one packed call.  Strides are in elements.
 * Source: "Packing与 FlashAttention Varlen", section 5 (per-segment views with
 * row stride and head stride over the flat token axis). */
typedef struct {
  int32_t T;          /* tokens in the stream (= cu_seqlens[B]) */
  int32_t B;          /* segments, cu_seqlens has B+1 entries */
  int32_t Hq, Hkv, d; /* query heads, key/value heads, head dim */
  int32_t max_seqlen; /* upper bound of cu_seqlens[b+1]-cu_seqlens[b]; sizes plans */
  int64_t q_row_stride, q_head_stride;
  int64_t k_row_stride, k_head_stride;
  int64_t v_row_stride, v_head_stride;
  int64_t o_row_stride, o_head_stride; /* out, dout, dq use these; dk/dv use k's */
} va_shape;

/* Fills the strides of a contiguous [T, H, d] layout. */
void varlen_shape_contiguous(va_shape* s, int32_t T, int32_t B, int32_t Hq, int32_t Hkv,
                             int32_t d, int32_t max_seqlen);

/* ---------------------------------------------------------------- host planner
 * Order-preserving next-fit.  Source: "Packing与 FlashAttention Varlen",
 * section 2 (the sequential strategy); "Pack sequences without joining their
 * contexts", "Fill only the current row" and "Extend the existing storage and
 * decoder" (a new pack starts when a document does not fit the space left; a
 * document longer than the capacity is an error, never split; an exact fill
 * opens no extra pack).
 *   lengths[n]        host, document lengths (> 0)
 *   order[n]          host out: document indices grouped by pack (pack order,
 *                     then order inside the pack)
 *   pack_offsets[n+1] host out: pack p holds order[pack_offsets[p] .. pack_offsets[p+1])
 *   n_packs           host out
 * Errors: VA_ERR_INVALID_ARG (null, n < 0, capacity <= 0, length <= 0),
 *         VA_ERR_CAPACITY (a length > capacity).  Synchronous, host only. */
va_status varlen_pack_next_fit(const int32_t* lengths, int32_t n, int32_t capacity,
                               int32_t* order, int32_t* pack_offsets, int32_t* n_packs);

/* Best-fit-decreasing.  Source: "Packing与 FlashAttention Varlen", section 2
 * (the default binpack strategy, which maximises fill and may reorder).  The
 * page fixes no tie rule; this library sorts by length descending then index,
 * puts each document in the open pack with the least room that still fits it
 * (ties: the earliest pack), else opens a pack; packs keep their opening order
 * and documents their insertion order.  Arguments and errors as next-fit.
 * O(n log n). */
va_status varlen_pack_best_fit_decreasing(const int32_t* lengths, int32_t n, int32_t capacity,
                                          int32_t* order, int32_t* pack_offsets,
                                          int32_t* n_packs);

/* ---------------------------------------------------------------- metadata kernel
 * Builds the boundary metadata of one pack on the device.  Source:
 * "Packing与 FlashAttention Varlen", section 2 (packing_row: positions restart
 * at 0 per sample) and section 3 (cu_seqlens: int32, first 0, last T, strictly
 * increasing; max_seqlen = max diff); "Pack sequences without joining their
 * contexts", "Fill only the current row" (occurrence segment ids).
 *   lengths_dev[n]        device, segment lengths in stream order (> 0)
 *   pad_to                if > sum(lengths), a tail pad segment of the
 *                         difference is appended (its positions are 0..p-1);
 *                         0 for none.  The host knows sum(lengths) when it
 *                         packs, so it knows B = n (+1 with a pad).
 *   cu_seqlens_dev[n+2]   device out; entry n+1 equals entry n when there is no pad
 *   position_ids_dev[T]   device out, T = max(sum, pad_to)
 *   segment_ids_dev[T]    device out
 *   max_seqlen_dev[1]     device out
 *   status_dev[1]         device out: 0, or VA_ERR_BAD_SEQLENS for a length <= 0
 *                         or pad_to < sum
 *   T_capacity            elements available in position_ids_dev/segment_ids_dev
 * One kernel launch when T_capacity <= 16384 and n <= 2046 (the scan's block also
 * writes positions and segment ids), else two.
 * Errors: VA_ERR_INVALID_ARG, VA_ERR_CUDA.  Asynchronous. */
va_status varlen_build_metadata(const int32_t* lengths_dev, int32_t n, int32_t pad_to,
                                int32_t T_capacity, int32_t* cu_seqlens_dev,
                                int32_t* position_ids_dev, int32_t* segment_ids_dev,
                                int32_t* max_seqlen_dev, int32_t* status_dev, va_stream_t stream);

/* Checks the cumulative-boundary contract on the device ("Packing与
 * FlashAttention Varlen", section 3): cu[0] == 0, cu[B] == T, strictly
 * increasing, every length <= max_seqlen.  Writes VA_ERR_BAD_SEQLENS into
 * *status_dev on a violation (leaves it untouched otherwise).  Asynchronous. */
va_status varlen_validate_cu_seqlens(const int32_t* cu_seqlens_dev, int32_t B, int32_t T,
                                     int32_t max_seqlen, int32_t* status_dev,
                                     va_stream_t stream);

/* Boundary compiler ("Packing与 FlashAttention Varlen", section 3): sample-local
 * position_ids -> cu_seqlens.  Every index whose position equals the reset
 * sentinel starts a sample -- the sentinel is 0, or with reset_at_min the
 * plane's minimum (for position schemes that do not start at 0); the reset
 * indices followed by T form cu_seqlens and max_seqlen is its largest
 * difference.  The first token must be a reset point (the compiled array must
 * start at 0).  With strict, positions between resets must count up by one, so a
 * plane that repeats coordinates inside a sample is rejected.
 *   position_ids_dev  int32 [T] device in, T >= 1
 *   cu_seqlens_dev    int32 [capacity] device out: cu[0..B] (capacity >= B + 1;
 *                     T + 1 always suffices)
 *   B_dev, max_seqlen_dev   int32 [1] device out (0 on error)
 *   status_dev        int32 [1] device out: VA_OK, VA_ERR_BAD_SEQLENS (first token
 *                     not a reset, or a strict violation), VA_ERR_WORKSPACE
 *                     (capacity < B + 1); cu_seqlens is left unwritten on error
 * Host-detected: VA_ERR_INVALID_ARG (null pointer, T < 1, capacity < 2).
 * Asynchronous. */
va_status varlen_cu_seqlens_from_positions(const int32_t* position_ids_dev, int32_t T,
                                           int32_t reset_at_min, int32_t strict,
                                           int32_t* cu_seqlens_dev, int32_t capacity,
                                           int32_t* B_dev, int32_t* max_seqlen_dev,
                                           int32_t* status_dev, va_stream_t stream);

/* ---------------------------------------------------------------- tile scheduler
 * Tile sizes the attention kernels use (BM query rows x BN key rows for
 * kind 0 = forward map; BM x BN for kind 1 = backward kv map; kind 2 = the
 * backward dQ map).  Host only. */
va_status varlen_attn_tile_sizes(int32_t kind, int32_t d, int32_t* BM, int32_t* BN);

/* Bytes of workspace varlen_attn_fwd (for_bwd = 0) or varlen_attn_bwd
 * (for_bwd = 1) needs for this shape.  Depends on T, B, Hq, Hkv, d, max_seqlen. */
size_t varlen_attn_workspace_size(const va_shape* shape, int32_t for_bwd);

/* Builds a tile map on the device.  Source: "Packing与 FlashAttention
 * Varlen", section 5 (a q block exists only while m*BM < l; its key blocks
 * stop at ceil(min(l, (m+1)*BM)/BN) when causal, ceil(l/BN) otherwise).  The
 * order is this library's reading (the page fixes none): records reading the
 * same K/V tiles are adjacent and longer work goes first,
 *     key = (-floor(log2(C_b)), segment b, head, -count, block)
 * with C_b the segment's total tile count.
 *   kind 0: records {segment, q block, q head, n key blocks}
 *   kind 1: records {segment, kv block, kv head, n q blocks} where the q blocks
 *           of a kv block n start at floor(n*BN/BM) (causal)
 *   kind 2: as kind 0 with the dQ kernel's tile sizes
 * Token tiles: for causal calls whose mean segment length T / B is below 256
 * tokens, segments of at most 64 tokens get no segment records.  Each maximal
 * run of such segments [r0, r1) is cut into tiles of R rows t0 = r0, r0 + R, ...
 * (R = BM, q rows, for kinds 0 and 2; R = BN, key rows, for kind 1) with records
 * {-1 - f, t0, head, rows = min(R, r1 - t0)}, f the segment holding row t0; they
 * follow all segment records, ordered by (t0, head).  Query i sees the keys
 * [start of its segment, i], key j the queries [j, end of its segment) ("Pack
 * sequences without joining their contexts", "Permission depends on the
 * example").  The attention calls apply the same rule, so this builds the maps
 * they use; the results do not depend on it.
 *   tile_map_dev    device out, int32 [capacity][4], 16-byte aligned
 *   n_items_dev     device out, int32
 *   scratch_dev     device scratch, int32 [B + 4]
 *   capacity        records available; VA_ERR_WORKSPACE if the bound
 *                   (T/blk + B)*heads exceeds it
 * Asynchronous. */
va_status varlen_attn_plan(const va_shape* shape, const int32_t* cu_seqlens_dev, int32_t kind,
                           int32_t causal, int32_t* tile_map_dev, int32_t capacity,
                           int32_t* n_items_dev, int32_t* scratch_dev, va_stream_t stream);

/* varlen_attn_plan for a causal local window of `window` keys (query i sees the keys
 * i - window .. i of its segment; -1 = no window, as varlen_attn_plan).  Source:
 * "Packing与 FlashAttention Varlen", section 5 (a local window narrows the key blocks a q
 * block may enumerate, n_block_min/max).  q block m's key blocks start at
 * floor(max(0, m*BM - window) / BN), count = blocks up to its diagonal; kv block n's q blocks
 * stop after floor((n*BN + BN - 1 + window) / BM), count from its diagonal.  Window maps have
 * no token records and keep each segment's blocks in block order (q blocks last-first, kv
 * blocks first-first).  Errors as varlen_attn_plan, plus VA_ERR_INVALID_ARG for window < -1
 * or a window without causal. */
va_status varlen_attn_plan_window(const va_shape* shape, const int32_t* cu_seqlens_dev, int32_t kind,
                                  int32_t causal, int32_t window, int32_t* tile_map_dev, int32_t capacity,
                                  int32_t* n_items_dev, int32_t* scratch_dev, va_stream_t stream);

/* ---------------------------------------------------------------- attention
 * Forward.  Source: "Packing与 FlashAttention Varlen", section 5 (each segment
 * b reads Q/K/V at offset cu[b]*row_stride with extent cu[b+1]-cu[b]; the
 * output is written at Q's offsets, so O has the input's flat order) and
 * section 1 (three independent attentions for [0,5,8,12]).  Per segment, q
 * head h, kv head h/(Hq/Hkv):
 *     s_ij = scale * q_i . k_j  (j <= i when causal, j in the segment),
 *     lse_i = ln sum_j exp(s_ij),  o_i = sum_j exp(s_ij - lse_i) v_j.
 *   q_dev [T,Hq,d], k_dev/v_dev [T,Hkv,d]  bf16 in, strides from shape
 *   cu_seqlens_dev [B+1]                   int32 in
 *   scale                                  usually 1/sqrt(d)
 *   out_dev [T,Hq,d] bf16 out;  lse_dev [Hq,T] fp32 out (natural log)
 *   ws_dev / ws_bytes                      workspace (>= workspace_size(shape, 0))
 * Errors: VA_ERR_INVALID_ARG, VA_ERR_UNSUPPORTED, VA_ERR_WORKSPACE, VA_ERR_CUDA;
 * device-detected VA_ERR_BAD_SEQLENS / VA_ERR_TIMEOUT in the status word. */
va_status varlen_attn_fwd(const void* q_dev, const void* k_dev, const void* v_dev,
                          const int32_t* cu_seqlens_dev, const va_shape* shape, float scale,
                          int32_t causal, void* out_dev, float* lse_dev, void* ws_dev,
                          size_t ws_bytes, va_stream_t stream);

/* varlen_attn_fwd with a causal local window: query i sees the keys i - window .. i of its
 * segment (itself and the window keys before it; FlashAttention's left window size, its
 * right size being 0 under causality); window = -1 is varlen_attn_fwd.  Source:
 * "Packing与 FlashAttention Varlen", section 5 (causal or local window narrows the key
 * blocks inside the segment's tile domain).  Workspace as varlen_attn_fwd.  Errors as
 * varlen_attn_fwd, plus VA_ERR_INVALID_ARG for window < -1 or a window without causal. */
va_status varlen_attn_fwd_window(const void* q_dev, const void* k_dev, const void* v_dev,
                                 const int32_t* cu_seqlens_dev, const va_shape* shape, float scale,
                                 int32_t causal, int32_t window, void* out_dev, float* lse_dev, void* ws_dev,
                                 size_t ws_bytes, va_stream_t stream);

/* Backward.  The analytic gradient of the forward definition, with P
 * recomputed from lse ("Packing与 FlashAttention Varlen", section 5 names the
 * training branch; the gradient itself is the plain derivative):
 *     D_i = dO_i . O_i,  dV_j = sum_i P_ij dO_i,  dP_ij = dO_i . v_j,
 *     dS_ij = P_ij (dP_ij - D_i),  dQ_i = scale sum_j dS_ij k_j,
 *     dK_j = scale sum_i dS_ij q_i;  dK, dV sum over a kv head's q heads.
 *   out_dev, lse_dev   the forward's results; dout_dev [T,Hq,d] bf16
 *   dq_dev [T,Hq,d], dk_dev/dv_dev [T,Hkv,d] bf16 out (overwritten)
 *   ws_dev / ws_bytes  workspace (>= workspace_size(shape, 1))
 * Errors as the forward. */
va_status varlen_attn_bwd(const void* q_dev, const void* k_dev, const void* v_dev,
                          const void* out_dev, const float* lse_dev, const void* dout_dev,
                          const int32_t* cu_seqlens_dev, const va_shape* shape, float scale,
                          int32_t causal, void* dq_dev, void* dk_dev, void* dv_dev, void* ws_dev,
                          size_t ws_bytes, va_stream_t stream);

/* varlen_attn_bwd for the causal local window of varlen_attn_fwd_window (the same window
 * as the forward that produced out and lse); window = -1 is varlen_attn_bwd. */
va_status varlen_attn_bwd_window(const void* q_dev, const void* k_dev, const void* v_dev,
                                 const void* out_dev, const float* lse_dev, const void* dout_dev,
                                 const int32_t* cu_seqlens_dev, const va_shape* shape, float scale,
                                 int32_t causal, int32_t window, void* dq_dev, void* dk_dev, void* dv_dev,
                                 void* ws_dev, size_t ws_bytes, va_stream_t stream);

/* Forward without a workspace, for callers that cannot allocate device memory
 * where they run attention (a plugin inside a host runtime that owns all device
 * allocations, or a serving loop that must not call cudaMalloc because it can
 * synchronise the device).  The pages have no counterpart: this is a deployment
 * convenience.  Same arguments, layouts and results as varlen_attn_fwd, without
 * ws_dev/ws_bytes: the scratch (status header, tile map, segment offsets) lives
 * in a 1 MiB static device array that every GPU loading this library holds
 * until exit.
 *   - Limit: the shape fits when varlen_attn_workspace_size(shape, 0) <= 1 MiB,
 *     that is 256 + align256(16 * (floor(T/256) + B) * Hq) + align256(4 * B)
 *     <= 1,048,576 bytes (align256 rounds up to a multiple of 256).  Larger
 *     shapes return VA_ERR_WORKSPACE with a message and launch nothing.
 *   - Every call looks the array's device address up (cudaGetSymbolAddress,
 *     with the caller's device current).  The first call on a device may load
 *     the library's device code there; make it before any stream capture.
 *   - All calls on a device share the array and it keeps the last call's
 *     contents (each call rewrites what it reads).  Calls that overlap on the
 *     GPU race on it: serialise them (one stream, or events between streams).
 *   - Allocates nothing.  A device-detected error (a cu_seqlens that breaks the
 *     contract, a bounded wait that gave up) leaves out/lse unwritten and is
 *     visible only through varlen_noalloc_read_status. */
va_status varlen_attn_fwd_noalloc(const void* q_dev, const void* k_dev, const void* v_dev,
                                  const int32_t* cu_seqlens_dev, const va_shape* shape, float scale,
                                  int32_t causal, void* out_dev, float* lse_dev, va_stream_t stream);

/* The status word of the last varlen_attn_fwd_noalloc call on the current
 * device: synchronises the stream, then copies the 4-byte word to *status_host
 * (VA_OK, VA_ERR_BAD_SEQLENS or VA_ERR_TIMEOUT).  Allocates nothing.
 * Errors: VA_ERR_INVALID_ARG (null pointer), VA_ERR_CUDA. */
va_status varlen_noalloc_read_status(int32_t* status_host, va_stream_t stream);

/* Test hook of the device-detected failure path; the pages have no counterpart.  Arms the
 * next forward call made in this process (varlen_attn_fwd and its variants): in that call
 * every attention CTA publishes its first work item and then loads nothing, and every
 * bounded wait gives up after wait_limit_ns instead of 2 s.  No copy or MMA is in flight
 * when the waits run out; the kernel writes VA_ERR_TIMEOUT into the status word, drains,
 * frees its tensor memory and returns, leaving out/lse unwritten and the context usable.
 * The token-tile kernel is not affected (use a call without token tiles).  One-shot: the
 * call consumes it.  Errors: VA_ERR_INVALID_ARG unless 1 ms <= wait_limit_ns <= 2 s. */
va_status varlen_test_stall_next_forward(int64_t wait_limit_ns);

/* Copies the workspace status word to *status_host after synchronising the
 * stream.  VA_ERR_CUDA if the copy fails. */
va_status varlen_read_status(const void* ws_dev, int32_t* status_host, va_stream_t stream);

/* Clears the workspace status word (asynchronous). */
va_status varlen_clear_status(void* ws_dev, va_stream_t stream);

/* ---------------------------------------------------------------- cross-attention
 * Q [Tq, Hq, d] cut by cu_seqlens_q[B+1] and K/V [Tk, Hkv, d] cut by cu_seqlens_k[B+1]: the
 * b-th Q slice attends to the b-th K/V slice.  Source: "Packing与 FlashAttention Varlen",
 * section 3 (cu_q and cu_k, each with the boundary contract; the b-th Q slice and K/V slice
 * belong to the same sample) and section 5 (the causal bound is aligned bottom-right:
 * (m+1)*BM + seqlen_k - seqlen_q).  Query i of segment b sees key j when j <= i + lk_b - lq_b
 * (causal) or always (non-causal).  Reading taken here: causal calls need lq_b <= lk_b in every
 * segment (every query sees a key); a segment with lq_b > lk_b, or a cu_seqlens_k that breaks
 * the contract (first 0, last Tk, strictly increasing, lengths <= max_seqlen_k), sets
 * VA_ERR_BAD_SEQLENS in the status word.  shape describes the Q side (T = Tq, max_seqlen =
 * longest Q segment) and every stride; Tk and max_seqlen_k the K/V side.  No token tiles, no
 * local window.  Outputs as varlen_attn_fwd / varlen_attn_bwd (dk, dv have K's rows). */
size_t varlen_attn_workspace_size_cross(const va_shape* shape, int32_t Tk, int32_t for_bwd);

va_status varlen_attn_plan_cross(const va_shape* shape, const int32_t* cu_seqlens_q_dev,
                                 const int32_t* cu_seqlens_k_dev, int32_t Tk, int32_t kind, int32_t causal,
                                 int32_t* tile_map_dev, int32_t capacity, int32_t* n_items_dev,
                                 int32_t* scratch_dev, va_stream_t stream);

va_status varlen_attn_fwd_cross(const void* q_dev, const void* k_dev, const void* v_dev,
                                const int32_t* cu_seqlens_q_dev, const int32_t* cu_seqlens_k_dev,
                                const va_shape* shape, int32_t Tk, int32_t max_seqlen_k, float scale,
                                int32_t causal, void* out_dev, float* lse_dev, void* ws_dev, size_t ws_bytes,
                                va_stream_t stream);

va_status varlen_attn_bwd_cross(const void* q_dev, const void* k_dev, const void* v_dev, const void* out_dev,
                                const float* lse_dev, const void* dout_dev, const int32_t* cu_seqlens_q_dev,
                                const int32_t* cu_seqlens_k_dev, const va_shape* shape, int32_t Tk,
                                int32_t max_seqlen_k, float scale, int32_t causal, void* dq_dev, void* dk_dev,
                                void* dv_dev, void* ws_dev, size_t ws_bytes, va_stream_t stream);

/* ---------------------------------------------------------------- padded-batch bridge
 * A batch padded to [Bp, S] with a 2-D attention mask enters the varlen path by dropping its
 * padding, and the packed output goes back to the padded shape.  Source: "Packing与
 * FlashAttention Varlen", section 4 (the padded-batch branch: remove the padding, run the
 * varlen kernel, scatter the output back).  Each row's real tokens, in order, form one
 * segment, so left, right or scattered padding all work.
 *   mask_dev        int32 [Bp, S] in: nonzero marks a real token
 *   indices_dev     int32 [Bp*S] out: the flat positions r*S + s of the T real tokens in
 *                   row-major order, then -1 for every padding cell (gather map of unpad)
 *   inverse_dev     int32 [Bp*S] out: each flat position's packed index, or -1 (pad map)
 *   cu_seqlens_dev  int32 [Bp+1] out; T_dev, max_seqlen_dev int32 [1] out
 *   status_dev      int32 [1] out: VA_OK, or VA_ERR_BAD_SEQLENS when a row has no real
 *                   token (it would be an empty segment)
 * Errors: VA_ERR_INVALID_ARG (null pointer, Bp < 1, S < 1, Bp*S >= 2^31).  Asynchronous. */
va_status varlen_unpad_index(const int32_t* mask_dev, int32_t Bp, int32_t S, int32_t* indices_dev,
                             int32_t* inverse_dev, int32_t* cu_seqlens_dev, int32_t* T_dev,
                             int32_t* max_seqlen_dev, int32_t* status_dev, va_stream_t stream);

/* Row gather: dst row i = src row map[i], or a zero row where map[i] < 0, for i < n_rows.
 * With varlen_unpad_index's indices it unpads ([Bp*S, row] -> [T, row]); with its inverse
 * map it pads the packed output back ([T, row] -> [Bp*S, row], zeros in the padding).
 *   row_bytes, src/dst_row_stride_bytes  positive multiples of 16 (strides >= row_bytes)
 *   src_dev, dst_dev                     16-byte aligned; map_dev int32 [n_rows]
 * Errors: VA_ERR_INVALID_ARG.  Asynchronous. */
va_status varlen_gather_rows(const void* src_dev, int64_t src_row_stride_bytes, const int32_t* map_dev,
                             int32_t n_rows, int64_t row_bytes, void* dst_dev, int64_t dst_row_stride_bytes,
                             va_stream_t stream);

/* ---------------------------------------------------------------- packed loss
 * Next-token targets of a packed stream of whole documents.  Source: "Pack sequences
 * without joining their contexts", "Form pairs inside each source range" (a document of L
 * tokens gives L - 1 pairs, its final input predicts its own last token and never the next
 * document's first) -- the same layout as sample-local -100 labels shifted by one
 * ("Packing与 FlashAttention Varlen", section 2).  Position t of segment
 * [cu[b], cu[b+1]) gets token_ids[t + 1] while t + 1 < cu[b+1], else ignore_index.
 *   token_ids_dev  int32 [T] in;  cu_seqlens_dev int32 [B+1] in (the attention contract)
 *   targets_dev    int32 [T] out
 * Errors: VA_ERR_INVALID_ARG (null pointer, T < 0, B < 1).  Asynchronous. */
va_status varlen_loss_targets(const int32_t* token_ids_dev, const int32_t* cu_seqlens_dev, int32_t B,
                              int32_t T, int32_t ignore_index, int32_t* targets_dev, va_stream_t stream);

/* Bytes of workspace varlen_token_ce needs for T rows: a 256-byte header (status word at
 * byte 0) and one float per row. */
size_t varlen_token_ce_workspace_size(int32_t T);

/* Token-weighted cross entropy over the packed stream and its logit gradient.  Source: "Pack
 * sequences without joining their contexts", "Keep the same nine-target objective": the
 * loss is the raw sum of the negative log likelihoods of the eligible targets divided once by
 * their count N (every eligible target has equal weight, whatever its row or document);
 * d(mean)/d(z_ic) = (p_ic - [c == y_i]) / N on eligible rows; a row whose target is
 * ignore_index is skipped before any arithmetic (its logits are never read, its gradient row
 * is zero), so non-finite values there cannot leak in.
 *   logits_dev   [T, V], row stride logits_row_stride elements; dtype 0 = fp32, 1 = bf16
 *   targets_dev  int32 [T]: a class in [0, V), or ignore_index
 *   loss_dev     double [2] out: {sum of NLL, sum / N}; NaN on a device-detected error
 *   count_dev    int32 [1] out: N
 *   grad_dev     [T, V] out (row stride grad_row_stride elements), the dtype of the logits,
 *                or NULL for no gradient
 *   ws_dev / ws_bytes  workspace (>= varlen_token_ce_workspace_size(T), 16-byte aligned)
 * Arithmetic in fp32 per row (base-2 log-sum-exp), the sum over rows in fp64 in a fixed order
 * (deterministic).  Errors: VA_ERR_INVALID_ARG, VA_ERR_WORKSPACE, VA_ERR_CUDA; the status
 * word gets VA_ERR_BAD_TARGETS when an eligible target is outside [0, V) or no target is
 * eligible (the mean would have no denominator), and then no row is computed.
 * Asynchronous. */
va_status varlen_token_ce(const void* logits_dev, int32_t dtype, int64_t logits_row_stride,
                          const int32_t* targets_dev, int32_t T, int32_t V, int32_t ignore_index,
                          double* loss_dev, int32_t* count_dev, void* grad_dev, int64_t grad_row_stride,
                          void* ws_dev, size_t ws_bytes, va_stream_t stream);

/* ---------------------------------------------------------------- tracing
 * Per-launch timing.  With capacity > 0, the library records a CUDA event pair
 * on the launching stream around each of the next `capacity` kernel launches
 * it makes (any entry point); capacity 0 switches this off and frees the
 * events.  Host-global state: not for concurrent use from several threads.
 * Errors: VA_ERR_INVALID_ARG, VA_ERR_CUDA. */
va_status varlen_profile_enable(int32_t capacity);

/* Waits for the recorded launches, writes up to `capacity` (kernel id, ms)
 * pairs in launch order, sets *count and restarts recording from slot 0. */
va_status varlen_profile_read(int32_t* kernel_ids, float* ms, int32_t capacity, int32_t* count);

/* Name of a kernel id reported by varlen_profile_read ("" if unknown). */
const char* varlen_kernel_name(int32_t kernel_id);

/* Kernel launches this library has made in this process (all threads). */
int64_t varlen_launch_count(void);

/* Message for the last failing call on this host thread ("" if none). */
const char* varlen_last_error(void);

/* Library version string. */
const char* varlen_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VARLEN_ATTN_H */
