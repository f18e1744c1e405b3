// Backward varlen attention for sm_103a: TMA + tcgen05 MMA with TMEM accumulators.
//
// The gradient of the forward definition, P recomputed from the forward's lse
// ("Packing与 FlashAttention Varlen", section 5 names the training branch):
//   P_ij = exp(scale q_i.k_j - lse_i) on visible (i, j);  D_i = dO_i . O_i;
//   dV_j = sum_i P_ij dO_i;  dS_ij = P_ij (dO_i . v_j - D_i);
//   dK_j = scale sum_i dS_ij q_i;  dQ_i = scale sum_j dS_ij k_j.
//
// Two kernels, each owning its output rows (no atomics, deterministic):
//   dkdv_tc_kernel  work item (segment, 128 kv rows, kv head); steps over the
//                   segment's q blocks of 64 rows at or after the diagonal and
//                   the kv head's q-head group.  Per step:
//                     S^T = K Q^T, dP^T = V dO^T          (SS, M=128 kv, N=64 q)
//                     P^T, dS^T -> bf16 in TMEM            (softmax warps)
//                     dV += P^T dO, dK += dS^T Q           (TS, A from TMEM)
//   dq_tc_kernel    work item (segment, 128 q rows, q head); steps over key
//                   blocks of 64 rows up to the diagonal.  Per step:
//                     S = Q K^T, dP = dO V^T               (SS, M=128 q, N=64 k)
//                     dS -> bf16 in TMEM                   (softmax warps)
//                     dQ += dS K                           (TS)
// Layout of both (384 threads, one CTA per SM, persistent over the tile map):
//   warp 0 TMA producer, which also pulls work items from the map's counter and
//   publishes them (sched.cuh); warp 1 MMA issuer (whole warp, one elected lane issues) +
//   TMEM owner; warp 2 (dK/dV only) stages
//   lse and D of each step in shared memory; warps 4-7 and 8-11 two
//   softmax warpgroups that split every step's 64 columns between them (32
//   each), which halves the softmax latency on each step's dependency chain;
//   S/dP are double-buffered by step, so the tensor core computes step i+1
//   while step i is exponentiated.
// TMEM: S_0 | S_1 | dP_0 | dP_1 (64 columns each) | accumulators.
//
// Token records (runs of segments of at most 64 tokens, at the end of both maps) take the
// same pipeline.  A dK/dV token record {-1 - f, t0, kv head, rows} holds the key rows
// [t0, t0 + rows) and the queries [t0, qend), qend the end of the last row's segment (at
// most three 64-row steps); a dQ token record {-1 - f, t0, q head, rows} holds the query rows
// [t0, t0 + rows) and the keys [cu[f], t0 + rows).  Query i sees the keys [start of its
// segment, i], key j the queries [j, end of its segment): the permission rule of "Pack
// sequences without joining their contexts" ("Permission depends on the example") in its
// range form.  The producer decodes a token record into the item fields the producer, MMA
// and lse/D roles already use, plus a per-row table next to the queue (the key row's segment
// end, or the query row's position in its segment); only the softmax warpgroups treat token
// items differently -- every step masked on both sides -- in a loop of their own that they
// enter after their last segment item, so the segment loop is unchanged.
#include "attn_params.cuh"
#include "sched.cuh"
#include "sm100_ptx.cuh"
#include "tmap.cuh"

namespace va {
using namespace sm100;

namespace {

constexpr int kBwdThreads = 384;
// setmaxnreg moves registers within what the CTA was launched with (168 per thread for
// 384 threads); a split above that total would make the increase wait forever.
constexpr int kLaunchRegs = 168;
constexpr int kRegsCtl = 80, kRegsSoftmax = 208;
static_assert(128 * kRegsCtl + 256 * kRegsSoftmax <= kBwdThreads * kLaunchRegs, "register split exceeds the launch");

__device__ __forceinline__ void drain_wait_b(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > 50000000ull) return;
  }
}

// ================================================================= dK / dV
template <int D>
struct KvCfg {
  static constexpr int KB = 128, QB = 64;
  // Two K buffers (items alternate: the next item's K loads a whole item ahead), one V
  // buffer (the next item's V loads once this item's last dP^T MMA is done, about two steps
  // before it is needed) and a Q/dO ring of QST slots (one step each).  At d = 128 the
  // single V buffer is what leaves room for the ring's fourth slot, which lets the producer
  // load the next item's first Q/dO steps before this item ends.
  static constexpr int QST = D == 128 ? 4 : 8;
  static constexpr int TKV = KB * D * 2;         // one K or V tile
  static constexpr int TQ = QB * D * 2;          // one Q or dO tile
  static constexpr int PKV = KB * 128, PQ = QB * 128;  // 64-column panels
  static constexpr int V_OFF = 2 * TKV;          // K buffers at 0 and TKV, then V
  static constexpr int RING_OFF = 3 * TKV;
  static constexpr int LDS = 4;                            // lse/D ring slots (one step each)
  static constexpr int LD_OFF = RING_OFF + QST * 2 * TQ;  // [LDS][-lse*log2e 64 | -D 64] fp32
  static constexpr int BAR_OFF = LD_OFF + LDS * 2 * 64 * 4;
  static constexpr int B_KF = 0, B_KE = 2, B_VF = 4, B_VE = 5, B_QF = 6, B_QE = 6 + QST, B_SF = 6 + 2 * QST,
                       B_PF = B_SF + 2, B_AF = B_PF + 2, B_AE = B_AF + 1, B_DR = B_AE + 1,
                       B_IF = B_DR + 1, B_IE = B_IF + 2, B_LF = B_IE + 2, B_LE = B_LF + LDS,
                       NBAR = B_LE + LDS;
  static constexpr int QUEUE_OFF = BAR_OFF + NBAR * 8;  // two item slots
  static constexpr int ROWS_OFF = QUEUE_OFF + 2 * 48;   // four 128-byte row tables (item k & 3)
  static constexpr int MISC_OFF = ROWS_OFF + 4 * KB;
  static constexpr int SMEM = MISC_OFF + 16;     // the dynamic smem base is 1024-aligned
};
static_assert(KvCfg<128>::SMEM <= 232448 && KvCfg<64>::SMEM <= 232448, "dK/dV shared memory");

// One dK/dV work item: key rows from s0 + 128 n of kv head hk; step i covers the 64 query rows
// from s0 + 64 (m_start + i / g) of q head hk g + i % g; queries at or past s0 + l are outside
// the item.  valid = 1: a segment record, the segment [s0, s0 + l).  valid = 2: a token record
// (n = m_start = 0), key rows [s0, s0 + kvn), key row s0 + r seen only by the queries before
// s0 + table[r].  valid = 0: the end of the list.
struct KvItem {
  int s0, l, n, hk, m_start, steps;
  int valid;
  int kvn;
  int s0k, lk, off;  // cross-attention: the keys' first row and count, the causal offset lk - l
};
static_assert(sizeof(KvItem) <= 48, "queue slots are 48 bytes");

template <bool WIN, bool X>
__device__ __forceinline__ KvItem kv_decode(const BwdParams& p, int idx) {
  const TileItem it = p.kv_items[idx];
  KvItem r;
  r.s0 = p.cu[it.seg];
  r.l = p.cu[it.seg + 1] - r.s0;
  r.n = it.blk;
  r.hk = it.head;
  const int Mq = (r.l + 63) / 64;
  // the q steps start at the diagonal; without a window they run to the segment's end
  r.m_start = WIN ? it.blk * 2 : Mq - it.count;
  if (X) {  // keys from cu_k; the diagonal moves by the offset lk - l (bottom-right alignment)
    r.s0k = p.cu_k[it.seg];
    r.lk = p.cu_k[it.seg + 1] - r.s0k;
    r.off = p.causal ? r.lk - r.l : 0;
  }
  r.steps = it.count * p.g;
  r.kvn = 0;
  return r;
}

// Segments of at most this many tokens are planned as token records: a key then sees at most
// 64 queries, an item's queries span at most three 64-row steps, and a row's segment end
// (relative to the item's first row) fits the row table's byte.
constexpr int kBwdTokenShort = 64;

// Decodes dK/dV token record idx, {-1 - f, t0, kv head, rows} (whole warp, every lane gets the
// same item), and writes its row table: the segment starts inside the rows come from
// cu[f + 1], cu[f + 2], ... (32 per round) as a 128-bit map, and entry r is the next start
// after row r, or, for the rows of the last segment, that segment's end (qend).
__device__ __forceinline__ KvItem kv_token_decode_w(const BwdParams& p, int idx, uint8_t* table) {
  const TileItem it = p.kv_items[idx];
  const int lane = threadIdx.x & 31, f = -1 - it.seg, t0 = it.blk, rows = it.count;
  uint32_t words[4] = {0u, 0u, 0u, 0u};
  int qend = t0 + rows;  // the contract (cu[B] = T >= t0 + rows) always sets it below
  for (int b0 = f + 1; b0 <= p.B; b0 += 32) {
    const int b = b0 + lane;
    const int x = b <= p.B ? p.cu[b] : INT_MAX;
    const int rr = x - t0;  // >= 1: cu[f + 1] is past row t0
#pragma unroll
    for (int w = 0; w < 4; ++w)
      words[w] |= __reduce_or_sync(0xffffffffu, (rr < rows && (rr >> 5) == w) ? 1u << (rr & 31) : 0u);
    const unsigned past = __ballot_sync(0xffffffffu, rr >= rows);  // the first one ends the last row's segment
    if (past) {
      qend = __shfl_sync(0xffffffffu, x, __ffs(past) - 1);
      break;
    }
  }
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int row = w * 32 + lane;
    int e = qend - t0;
    for (int w2 = 3; w2 > w; --w2)  // the nearest later word with a start wins
      if (words[w2]) e = w2 * 32 + __ffs(words[w2]) - 1;
    const uint32_t above = lane == 31 ? 0u : words[w] & (0xffffffffu << (lane + 1));
    if (above) e = w * 32 + __ffs(above) - 1;
    table[row] = static_cast<uint8_t>(row < rows ? e : 0);
  }
  __threadfence_block();
  KvItem r;
  r.s0 = t0;
  r.l = qend - t0;
  r.n = 0;
  r.hk = it.head;
  r.m_start = 0;
  r.steps = (qend - t0 + 63) / 64 * p.g;
  r.kvn = rows;
  return r;
}

}  // namespace

// WIN: causal local window p.window: a kv block's q steps stop at the window of its last key
// row, and steps that cross a key's window edge also mask the queries past key + w.
// X: cross-attention (p.cu_k): the kv block's keys come from their own boundaries; query i
// sees key j when j <= i + lk - lq, so the q steps start at floor(max(0, n*128 - off) / 64).
template <int D, bool TOK, bool WIN, bool X>
__global__ void __launch_bounds__(kBwdThreads, 1)
    dkdv_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                   const BwdParams p) {
  using C = KvCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  uint8_t* sm = smem_raw;
  if (base & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicCAS(&p.hdr->status, 0, VA_ERR_CUDA);
    return;
  }
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::MISC_OFF + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return base + C::BAR_OFF + 8u * i; };

  KvItem* queue = reinterpret_cast<KvItem*>(sm + C::QUEUE_OFF);
  uint8_t* row_tables = sm + C::ROWS_OFF;
  auto dec = [&](int idx) { return kv_decode<WIN, X>(p, idx); };
  // Launched as a programmatic dependent of the preparation kernel: its maps, D and status
  // are read only after the wait.  The dQ kernel, which reads the same products but none
  // of this kernel's, may then start on SMs as this kernel's CTAs finish.
  griddep_begin();
  if (p.hdr->status != VA_OK) return;
  const int n_items = p.hdr->n_items[p.kv_slot];
  const int n_seg = n_items - p.hdr->n_items[p.kv_tok_slot];  // segment records, then token ones
  if (static_cast<int>(blockIdx.x) >= n_items) return;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::B_KF + b), 1);
      mbar_init(bar(C::B_KE + b), 1);
    }
    mbar_init(bar(C::B_VF), 1);
    mbar_init(bar(C::B_VE), 1);
    for (int s = 0; s < C::QST; ++s) {
      mbar_init(bar(C::B_QF + s), 1);
      mbar_init(bar(C::B_QE + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::B_SF + x), 1);
      mbar_init(bar(C::B_PF + x), 256);  // both softmax warpgroups, one half of the step each
    }
    mbar_init(bar(C::B_AF), 1);
    mbar_init(bar(C::B_AE), 256);
    mbar_init(bar(C::B_DR), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::B_IF + b), 1);
      mbar_init(bar(C::B_IE + b), 32 + 256 + 32);  // MMA warp, softmax warpgroups, lse/D warp
    }
    for (int b = 0; b < C::LDS; ++b) {
      mbar_init(bar(C::B_LF + b), 32);
      mbar_init(bar(C::B_LE + b), 256);
    }
    *abort_flag = 0;
    *wait_limit_slot(abort_flag) = kTimeoutNs;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tq);
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
    prefetch_tmap(&tdo);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    regs_dec<kRegsCtl>();
    {  // the whole warp runs the loop; elect.sync picks the issuing lane
      int qit = 0, item_cnt = 0, k_issued = 0, v_issued = 0;  // items whose K / V load went out
      bool ok = true;
      KvItem nxt;
      // Publishes this CTA's k-th item (the next record of the map): lane 0 pulls its index,
      // the warp decodes it (a token record also fills row table k & 3) and lane 0 writes the
      // slot and releases it.  Returns false at the end of the list or on abort (ok_ = false).
      auto publish = [&](int k, KvItem& out, bool& ok_) -> bool {
        const int s = k & 1;
        ok_ = wwait(bar(C::B_IE + s), ((k >> 1) & 1) ^ 1, abort_flag, p.hdr, 40);
        if (!ok_) return false;
        int idx = 0;
        if (lane == 0) idx = atomicAdd(p.kv_counter, 1);
        idx = __shfl_sync(0xffffffffu, idx, 0);
        if (idx < n_seg) {
          out = kv_decode<WIN, X>(p, idx);
          out.valid = 1;
        } else if (idx < n_items) {
          out = kv_token_decode_w(p, idx, row_tables + (k & 3) * C::KB);
          out.valid = 2;
        } else {
          out = KvItem{};
          out.valid = 0;
        }
        __syncwarp();  // every lane's table bytes before the release
        if (lane == 0) {
          queue[s] = out;
          mbar_arrive(bar(C::B_IF + s));
        }
        __syncwarp();
        return out.valid != 0;
      };
      // K of this CTA's j-th item into buffer j & 1, once item j-2's S^T MMAs are done with it
      auto load_k = [&](const KvItem& J, int j) -> bool {
        const int kb = j & 1;
        if (!wwait(bar(C::B_KE + kb), ((j >> 1) & 1) ^ 1, abort_flag, p.hdr, 21)) return false;
        mbar_expect_tx_w(bar(C::B_KF + kb), C::TKV);
        for (int pn = 0; pn < D / 64; ++pn)
          tma_load_3d_w(base + kb * C::TKV + pn * C::PKV, &tk, bar(C::B_KF + kb), pn * 64, J.hk,
                        (X ? J.s0k : J.s0) + J.n * 128);
        k_issued = j + 1;
        return true;
      };
      // V of this CTA's j-th item into the V buffer, once item j-1's dP^T MMAs are done with it
      auto load_v = [&](const KvItem& J, int j) -> bool {
        if (!wwait(bar(C::B_VE), (j & 1) ^ 1, abort_flag, p.hdr, 20)) return false;
        mbar_expect_tx_w(bar(C::B_VF), C::TKV);
        for (int pn = 0; pn < D / 64; ++pn)
          tma_load_3d_w(base + C::V_OFF + pn * C::PKV, &tv, bar(C::B_VF), pn * 64, J.hk,
                        (X ? J.s0k : J.s0) + J.n * 128);
        v_issued = j + 1;
        return true;
      };
      bool more = TOK ? publish(0, nxt, ok)
                      : queue_publish_w(0, queue, bar(C::B_IF), bar(C::B_IE), p.kv_counter, n_items, dec, nxt,
                                        abort_flag, p.hdr, ok);
      if (ok && more) ok = load_k(nxt, 0);
      for (; ok && more; ++item_cnt) {
        const KvItem I = nxt;  // publish the next record first: its decode overlaps this one
        more = TOK ? publish(item_cnt + 1, nxt, ok)
                   : queue_publish_w(item_cnt + 1, queue, bar(C::B_IF), bar(C::B_IE), p.kv_counter, n_items, dec,
                                     nxt, abort_flag, p.hdr, ok);
        if (!ok) break;
        // This item's first two Q/dO steps, then its V (which waits for the previous item's last
        // dP^T MMA), then the next item's K (a whole item ahead of its use) and the remaining
        // steps.
        const int kv_at = I.steps < 2 ? I.steps : 2;
        for (int i = 0; ok && i <= I.steps; ++i) {
          if (i == kv_at) {
            ok = load_v(I, item_cnt) && (!more || load_k(nxt, item_cnt + 1));
            if (!ok) break;
          }
          if (i == I.steps) break;
          const int m = I.m_start + i / p.g, h = I.hk * p.g + i % p.g;
          const int s = qit % C::QST;
          ok = wwait(bar(C::B_QE + s), ((qit / C::QST) & 1) ^ 1, abort_flag, p.hdr, 22);
          if (!ok) break;
          mbar_expect_tx_w(bar(C::B_QF + s), 2 * C::TQ);
          const uint32_t dst = base + C::RING_OFF + s * 2 * C::TQ;
          for (int pn = 0; pn < D / 64; ++pn) {
            tma_load_3d_w(dst + pn * C::PQ, &tq, bar(C::B_QF + s), pn * 64, h, I.s0 + m * 64);
            tma_load_3d_w(dst + C::TQ + pn * C::PQ, &tdo, bar(C::B_QF + s), pn * 64, h, I.s0 + m * 64);
          }
          ++qit;
        }
      }
      if (!ok) {
        // let every copy this thread started land before the CTA exits
        for (int j = k_issued - 1; j >= 0 && j >= k_issued - 2; --j)
          drain_wait_b(bar(C::B_KF + (j & 1)), (j >> 1) & 1);
        if (v_issued > 0) drain_wait_b(bar(C::B_VF), (v_issued - 1) & 1);
        for (int i = qit - 1; i >= 0 && i >= qit - C::QST; --i)
          drain_wait_b(bar(C::B_QF + i % C::QST), (i / C::QST) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    regs_dec<kRegsCtl>();
    {  // the whole warp runs the loop; elect.sync picks the issuing lane
      constexpr uint32_t idS = idesc_bf16(128, 64, false, false);
      constexpr uint32_t idG = idesc_bf16(128, D, false, true);
      int qit = 0, item_cnt = 0;
      uint32_t pf0 = 0, pf1 = 0;  // p_full phases per buffer (scalars: a runtime index would spill)
      bool ok = true;
      int kb = 0;
      const uint32_t kvlo0 = sdesc_lo(base, 16);                 // K/V, K-major A
      const uint32_t ringK0 = sdesc_lo(base + C::RING_OFF, 16);    // Q/dO as K-major B
      const uint32_t ringM0 = sdesc_lo(base + C::RING_OFF, C::PQ); // Q/dO as MN-major B
      // S^T and dP^T of one step into buffer x; the item's first step first waits for its V
      auto issue_SdP = [&](int x, int slot, bool wait_v) -> bool {
        const uint32_t qd = ringK0 + ((slot * 2 * C::TQ) >> 4), dd = qd + (C::TQ >> 4);
        const uint32_t kd = kvlo0 + ((kb * C::TKV) >> 4), vd = kvlo0 + (C::V_OFF >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t okv = ((kk >> 2) * C::PKV + (kk & 3) * 32) >> 4, oq = ((kk >> 2) * C::PQ + (kk & 3) * 32) >> 4;
          mma_ss_w(tmem + x * 64, kd + okv, qd + oq, idS, kk > 0);
        }
        if (wait_v) {
          if (!wwait(bar(C::B_VF), item_cnt & 1, abort_flag, p.hdr, 20)) return false;
          fence_after_sync();
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t okv = ((kk >> 2) * C::PKV + (kk & 3) * 32) >> 4, oq = ((kk >> 2) * C::PQ + (kk & 3) * 32) >> 4;
          mma_ss_w(tmem + 128 + x * 64, vd + okv, dd + oq, idS, kk > 0);
        }
        mma_commit_w(bar(C::B_SF + x));
        return true;
      };
      for (;; ++item_cnt) {
        KvItem I;
        const bool got_ = queue_take(item_cnt, queue, bar(C::B_IF), bar(C::B_IE), I, abort_flag, p.hdr, ok);
        const bool all_ok = __all_sync(0xffffffffu, ok);
        if (!all_ok) ok = false;
        if (!all_ok || !got_) break;
        kb = item_cnt & 1;
        ok = wwait(bar(C::B_KF + kb), (item_cnt >> 1) & 1, abort_flag, p.hdr, 23);
        if (!ok) break;
        for (int j = 0; ok && j < 2 && j < I.steps; ++j) {
          const int s = (qit + j) % C::QST;
          ok = wwait(bar(C::B_QF + s), ((qit + j) / C::QST) & 1, abort_flag, p.hdr, 24);
          if (!ok) break;
          fence_after_sync();
          ok = issue_SdP(j, s, j == 0);
        }
        if (!ok) break;
        if (I.steps <= 2) {  // the item's last S^T / dP^T MMAs: its K and V buffers may be reloaded
          mma_commit_w(bar(C::B_KE + kb));
          mma_commit_w(bar(C::B_VE));
        }
        for (int i = 0; ok && i < I.steps; ++i) {
          const int x = i & 1, s = (qit + i) % C::QST;
          ok = wwait(bar(C::B_PF + x), (x ? pf1 : pf0) & 1, abort_flag, p.hdr, 25);
          if (!ok) break;
          if (x) ++pf1;
          else ++pf0;
          if (i == 0) {  // the accumulators must have been read out by the previous epilogue
            ok = wwait(bar(C::B_AE), (item_cnt & 1) ^ 1, abort_flag, p.hdr, 26);
            if (!ok) break;
          }
          fence_after_sync();
          const uint32_t qm = ringM0 + ((s * 2 * C::TQ) >> 4), dm = qm + (C::TQ >> 4);
#pragma unroll
          for (int kk = 0; kk < C::QB / 16; ++kk)
            mma_ts_w(tmem + 256, tmem + x * 64 + (kk >> 1) * 32 + (kk & 1) * 8, dm + kk * (2048 >> 4), idG,
                     (i > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < C::QB / 16; ++kk)
            mma_ts_w(tmem + 256 + D, tmem + 128 + x * 64 + (kk >> 1) * 32 + (kk & 1) * 8, qm + kk * (2048 >> 4), idG,
                      (i > 0 || kk > 0) ? 1u : 0u);
          mma_commit_w(bar(C::B_QE + s));
          if (i + 2 < I.steps) {
            const int s2 = (qit + i + 2) % C::QST;
            ok = wwait(bar(C::B_QF + s2), ((qit + i + 2) / C::QST) & 1, abort_flag, p.hdr, 27);
            if (!ok) break;
            fence_after_sync();
            issue_SdP(x, s2, false);
            if (i + 2 == I.steps - 1) {
              mma_commit_w(bar(C::B_KE + kb));
              mma_commit_w(bar(C::B_VE));
            }
          }
        }
        if (!ok) break;
        mma_commit_w(bar(C::B_AF));
        qit += I.steps;
      }
      mma_commit_w(bar(C::B_DR));
      drain_wait_b(bar(C::B_DR), 0);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ lse / D loader
    // For every step, in the order the softmax warpgroups take them: -lse * log2(e) and
    // -D of the step's 64 q rows into a shared-memory ring, negated so the softmax only
    // adds them (out-of-segment rows get -inf / 0, so their P is 0).
    regs_dec<kRegsCtl>();
    int g = 0;  // steps of this CTA so far
    bool ok = true;
    for (int item_cnt = 0;; ++item_cnt) {
      KvItem I;
      const bool got = queue_take(item_cnt, queue, bar(C::B_IF), bar(C::B_IE), I, abort_flag, p.hdr, ok);
      if (!__all_sync(0xffffffffu, ok) || !got) break;
      for (int i = 0; i < I.steps; ++i, ++g) {
        const int slot = g % C::LDS;
        ok = mbar_wait(bar(C::B_LE + slot), ((g / C::LDS) & 1) ^ 1, abort_flag, p.hdr, 30);
        if (!__all_sync(0xffffffffu, ok)) break;
        const int m = I.m_start + i / p.g, h = I.hk * p.g + i % p.g;
        float* dst = reinterpret_cast<float*>(sm + C::LD_OFF) + slot * 128;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = lane + 32 * e;
          const int qr = m * 64 + c;
          const int64_t at = static_cast<int64_t>(h) * p.T + I.s0 + qr;
          const bool in = qr < I.l;
          dst[c] = in ? p.lse[at] * -kLog2e : -INFINITY;
          dst[64 + c] = in ? -p.dsum[at] : 0.f;
        }
        mbar_arrive(bar(C::B_LF + slot));  // release: this lane's values are visible
      }
      if (!ok) break;
    }
  } else if (warp < 4) {
    regs_dec<kRegsCtl>();  // warp 3 has no role
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    regs_inc<kRegsSoftmax>();
    // Both warpgroups take every step, warpgroup x its query columns [32 x, 32 x + 32) of the
    // step's S^T / dP^T buffer (step i uses buffer i & 1), writing P^T and dS^T (bf16) over the
    // first 16 columns of that range; epilogue: 0 -> dV, 1 -> dK.
    const int x = (warp - 4) >> 2;
    const int cw = 32 * x;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + cw;
    const uint32_t dp_addr = tmem + lane_off + 128 + cw;
    const uint32_t acc_addr = tmem + lane_off + 256 + x * D;
    const float* ldring = reinterpret_cast<const float*>(sm + C::LD_OFF);  // [slot][-lse2 64 | -D 64]
    const float sl2 = p.scale_log2;
    uint32_t sf0 = 0, sf1 = 0;  // s_full phases per buffer
    int item_cnt = 0;
    bool ok = true;
    int g0 = 0;  // this CTA's steps before the current item (the lse/D ring index)
    // Epilogue: the accumulators are released as soon as they are in registers, and the packed
    // row is held and stored after this warpgroup's first step of the next item, so that the
    // tensor core starts that item while the previous one is written out.
    uint4 held[D / 8];
    bf16* held_out = nullptr;
    bool held_store = false, holding = false;
    auto flush = [&]() {
      store_rows_coalesced(held, held_out, p.k_rs, held_store);
      holding = false;
    };
    auto take_accumulators = [&](int k, bf16* out, bool store) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(bar(C::B_AF), k & 1, abort_flag, p.hdr, 29))) return false;
      fence_after_sync();
      const float mul = x == 0 ? 1.f : p.scale;
      uint32_t o[D];  // the whole accumulator row in one TMEM round trip
#pragma unroll
      for (int c = 0; c < D / 32; ++c) tmem_ld32(acc_addr + c * 32, o + c * 32);
      tmem_wait_ld();
      fence_before_sync();
      mbar_arrive(bar(C::B_AE));
#pragma unroll
      for (int j = 0; j < D / 2; ++j)
        o[j] = pack_bf16(__uint_as_float(o[2 * j]) * mul, __uint_as_float(o[2 * j + 1]) * mul);
#pragma unroll
      for (int j = 0; j < D / 8; ++j) held[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
      held_out = out;
      held_store = store;
      holding = true;
      return true;
    };
    KvItem J{};        // the first token item, once the segment loop has met it
    bool tok = false;
    for (;; ++item_cnt) {
      KvItem I;
      const bool got = queue_take(item_cnt, queue, bar(C::B_IF), bar(C::B_IE), I, abort_flag, p.hdr, ok);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      if (!got) break;
      if constexpr (TOK) {
        if (I.valid == 2) {  // the token records follow: the loop below
          J = I;
          tok = true;
          break;
        }
      }
      const int kvrow = I.n * 128 + r;
      for (int i = 0; i < I.steps; ++i) {
        const int gs = g0 + i, ls = gs % C::LDS, b = i & 1;
        ok = mbar_wait(bar(C::B_LF + ls), (gs / C::LDS) & 1, abort_flag, p.hdr, 19);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        ok = mbar_wait(bar(C::B_SF + b), (b ? sf1 : sf0) & 1, abort_flag, p.hdr, 28);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        if (b) ++sf1;
        else ++sf0;
        fence_after_sync();
        const int q0 = (I.m_start + i / p.g) * 64 + cw;  // this warpgroup's first query column
        const int lim = kvrow - (X ? I.off : 0) - q0;  // query columns c < lim are masked (key after query)
        // (window) query columns c >= hi are masked too: past the key's window
        const int hi = WIN ? kvrow + p.window + 1 - q0 : 0;
        const bool need_mask =
            p.causal && (I.n * 128 + 127 - (X ? I.off : 0) > q0 || (WIN && q0 + 31 > I.n * 128 + p.window));
        const float* L = ldring + ls * 128 + cw;
        const float* Dd = L + 64;
        // one TMEM round trip: this warpgroup's 32 scores and 32 dP values of this kv row
        uint32_t sv[32], dpv[32];
        tmem_ld32(s_addr + b * 64, sv);
        tmem_ld32(dp_addr + b * 64, dpv);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(L + c);
          const float4 d4 = *reinterpret_cast<const float4*>(Dd + c);
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int j = c + e;
            const float la = e ? l4.z : l4.x, lb = e ? l4.w : l4.y;  // -lse * log2(e)
            const float da = e ? d4.z : d4.x, db = e ? d4.w : d4.y;  // -D
            // scalar FMAs: the packed forms measured slower here (operand pairing moves)
            const float x0 = fmaf(__uint_as_float(sv[j]), sl2, la), x1 = fmaf(__uint_as_float(sv[j + 1]), sl2, lb);
            float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
            if (need_mask) {
              if (j < lim || (WIN && j >= hi)) p0 = 0.f;
              if (j + 1 < lim || (WIN && j + 1 >= hi)) p1 = 0.f;
            }
            const float t0 = __uint_as_float(dpv[j]) + da, t1 = __uint_as_float(dpv[j + 1]) + db;
            sv[j >> 1] = pack_bf16(p0, p1);
            dpv[j >> 1] = pack_bf16(p0 * t0, p1 * t1);
          }
        }
        tmem_st16(s_addr + b * 64, sv);
        tmem_st16(dp_addr + b * 64, dpv);
        mbar_arrive(bar(C::B_LE + ls));  // this thread has read the slot's lse/D
        tmem_wait_st();
        fence_before_sync();
        mbar_arrive(bar(C::B_PF + b));
        if (holding) flush();  // the previous item's row, under this item's first MMAs
      }
      if (!ok) break;
      g0 += I.steps;
      // epilogue: warpgroup 0 takes dV, warpgroup 1 scale * dK
      bf16* out = (x == 0 ? p.dv : p.dk) + static_cast<int64_t>((X ? I.s0k : I.s0) + kvrow) * p.k_rs +
                  static_cast<int64_t>(I.hk) * p.k_hs;
      if (!take_accumulators(item_cnt, out, kvrow < (X ? I.lk : I.l))) {
        ok = false;
        break;
      }
    }
    // Token items (runs of short segments; all of them follow the segment items): every step
    // masked on both sides per key row, rows past the item's keys not stored.
    for (KvItem I = J; TOK && ok && tok;) {
      const int kend = I.s0 + row_tables[(item_cnt & 3) * C::KB + r];  // end of this key's segment
      for (int i = 0; i < I.steps; ++i) {
        const int gs = g0 + i, ls = gs % C::LDS, b = i & 1;
        ok = mbar_wait(bar(C::B_LF + ls), (gs / C::LDS) & 1, abort_flag, p.hdr, 19);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        ok = mbar_wait(bar(C::B_SF + b), (b ? sf1 : sf0) & 1, abort_flag, p.hdr, 28);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        if (b) ++sf1;
        else ++sf0;
        fence_after_sync();
        const int q0 = I.s0 + (i / p.g) * 64 + cw;  // this warpgroup's first query column
        // query columns c < lim (before the key) and c >= hi (past its segment) are masked
        const int lim = I.s0 + r - q0, hi = kend - q0;
        const float* L = ldring + ls * 128 + cw;
        const float* Dd = L + 64;
        // one TMEM round trip: this warpgroup's 32 scores and 32 dP values of this kv row
        uint32_t sv[32], dpv[32];
        tmem_ld32(s_addr + b * 64, sv);
        tmem_ld32(dp_addr + b * 64, dpv);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(L + c);
          const float4 d4 = *reinterpret_cast<const float4*>(Dd + c);
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const int j = c + e;
            const float la = e ? l4.z : l4.x, lb = e ? l4.w : l4.y;  // -lse * log2(e)
            const float da = e ? d4.z : d4.x, db = e ? d4.w : d4.y;  // -D
            // scalar FMAs: the packed forms measured slower here (operand pairing moves)
            const float x0 = fmaf(__uint_as_float(sv[j]), sl2, la), x1 = fmaf(__uint_as_float(sv[j + 1]), sl2, lb);
            float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
            if (j < lim || j >= hi) p0 = 0.f;
            if (j + 1 < lim || j + 1 >= hi) p1 = 0.f;
            const float t0 = __uint_as_float(dpv[j]) + da, t1 = __uint_as_float(dpv[j + 1]) + db;
            sv[j >> 1] = pack_bf16(p0, p1);
            dpv[j >> 1] = pack_bf16(p0 * t0, p1 * t1);
          }
        }
        tmem_st16(s_addr + b * 64, sv);
        tmem_st16(dp_addr + b * 64, dpv);
        mbar_arrive(bar(C::B_LE + ls));  // this thread has read the slot's lse/D
        tmem_wait_st();
        fence_before_sync();
        mbar_arrive(bar(C::B_PF + b));
        if (holding) flush();  // the previous item's row, under this item's first MMAs
      }
      if (!ok) break;
      g0 += I.steps;
      // epilogue: warpgroup 0 takes dV, warpgroup 1 scale * dK; rows past the item's keys are not stored
      bf16* out = (x == 0 ? p.dv : p.dk) + static_cast<int64_t>(I.s0 + r) * p.k_rs +
                  static_cast<int64_t>(I.hk) * p.k_hs;
      if (!take_accumulators(item_cnt, out, r < I.kvn)) {
        ok = false;
        break;
      }
      ++item_cnt;
      const bool got = queue_take(item_cnt, queue, bar(C::B_IF), bar(C::B_IE), I, abort_flag, p.hdr, ok);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      if (!got) break;
    }
    if (ok && holding) flush();  // the CTA's last item
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================= dQ
namespace {

template <int D>
struct QCfg {
  static constexpr int QB = 128, KB = 64;
  // Two Q buffers (items alternate: the next item's Q loads a whole item ahead), one dO
  // buffer (the next item's dO loads once this item's last dP MMA is done, about two steps
  // before it is needed) and a K/V ring of KST slots (one step each).  At d = 128 the single
  // dO buffer is what leaves room for the ring's fourth slot.
  static constexpr int KST = D == 128 ? 4 : 8;
  static constexpr int TQ = QB * D * 2, TKV = KB * D * 2;
  static constexpr int PQ = QB * 128, PKV = KB * 128;
  static constexpr int DO_OFF = 2 * TQ;          // Q buffers at 0 and TQ, then dO
  static constexpr int RING_OFF = 3 * TQ;
  static constexpr int BAR_OFF = RING_OFF + KST * 2 * TKV;
  static constexpr int B_QF = 0, B_QE = 2, B_DF = 4, B_DE = 5, B_KF = 6, B_KE = 6 + KST, B_SF = 6 + 2 * KST,
                       B_PF = B_SF + 2, B_AF = B_PF + 2, B_AE = B_AF + 2, B_DR = B_AE + 2,
                       B_IF = B_DR + 1, B_IE = B_IF + 2, NBAR = B_IE + 2;  // AF/AE: per dQ buffer
  static constexpr int QUEUE_OFF = BAR_OFF + NBAR * 8;  // two item slots
  static constexpr int ROWS_OFF = QUEUE_OFF + 2 * 48;   // four 128-byte row tables (item k & 3)
  static constexpr int MISC_OFF = ROWS_OFF + 4 * QB;
  static constexpr int SMEM = MISC_OFF + 16;     // the dynamic smem base is 1024-aligned
};
static_assert(QCfg<128>::SMEM <= 232448 && QCfg<64>::SMEM <= 232448, "dQ shared memory");

// One dQ work item: query rows from s0 + 128 m of q head h (kv head hk), rows at or past
// s0 + l outside it; step n covers the 64 key rows from kb + 64 n (nb steps).  valid = 1: a
// segment record, the segment [s0, s0 + l) (kb = s0).  valid = 2: a token record (m = 0),
// query row s0 + r seeing only the keys from s0 + r - table[r] (the start of its segment).
// valid = 0: the end of the list.
struct QItem {
  int s0, l, m, h, hk, nb;
  int valid;
  int kb;
  int lk, off;  // cross-attention: the keys' count, the causal offset lk - l
};
static_assert(sizeof(QItem) <= 48, "queue slots are 48 bytes");

template <bool WIN, bool X>
__device__ __forceinline__ QItem q_decode(const BwdParams& p, int idx) {
  const TileItem it = p.q_items[idx];
  QItem r;
  r.s0 = p.cu[it.seg];
  r.l = p.cu[it.seg + 1] - r.s0;
  r.m = it.blk;
  r.h = it.head;
  r.hk = it.head / p.g;
  r.nb = it.count;
  // key steps from the segment start, or (window) from the window of the item's first row
  r.kb = WIN ? r.s0 + max(0, it.blk * 128 - p.window) / 64 * 64 : r.s0;
  if (X) {  // keys from cu_k, the causal bound moved by lk - l (bottom-right alignment)
    r.kb = p.cu_k[it.seg];
    r.lk = p.cu_k[it.seg + 1] - r.kb;
    r.off = p.causal ? r.lk - r.l : 0;
  }
  return r;
}

// Decodes dQ token record idx, {-1 - f, t0, q head, rows} (whole warp, every lane gets the
// same item), and writes its row table: the segment starts inside the rows come from
// cu[f + 1], cu[f + 2], ... (32 per round) as a 128-bit map, and entry r is row r's position
// in its segment.  Its keys start at cu[f].
__device__ __forceinline__ QItem q_token_decode_w(const BwdParams& p, int idx, uint8_t* table) {
  const TileItem it = p.q_items[idx];
  const int lane = threadIdx.x & 31, f = -1 - it.seg, t0 = it.blk, rows = it.count;
  const int kb = p.cu[f];
  uint32_t words[4] = {0u, 0u, 0u, 0u};
  for (int b0 = f + 1; b0 <= p.B; b0 += 32) {
    const int b = b0 + lane;
    const int x = b <= p.B ? p.cu[b] : INT_MAX;
    const int rr = x - t0;  // >= 1: cu[f + 1] is past row t0
#pragma unroll
    for (int w = 0; w < 4; ++w)
      words[w] |= __reduce_or_sync(0xffffffffu, (rr < rows && (rr >> 5) == w) ? 1u << (rr & 31) : 0u);
    if (__any_sync(0xffffffffu, rr >= rows)) break;  // a boundary past the rows was read
  }
  int last = kb - t0;  // start of the segment holding the rows before word w (<= 0)
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int row = w * 32 + lane;
    const uint32_t mine = words[w] & (0xffffffffu >> (31 - lane));
    const int st = mine ? w * 32 + 31 - __clz(mine) : last;
    table[row] = static_cast<uint8_t>(row < rows ? row - st : 0);
    if (words[w]) last = w * 32 + 31 - __clz(words[w]);
  }
  __threadfence_block();
  QItem r;
  r.s0 = t0;
  r.l = rows;
  r.m = 0;
  r.h = it.head;
  r.hk = it.head / p.g;
  r.nb = (t0 + rows - kb + 63) / 64;
  r.kb = kb;
  return r;
}

}  // namespace

// WIN: causal local window p.window: an item's key steps start at the window of its first
// row, and steps that cross a query's window edge also mask the keys before query - w.
// X: cross-attention (p.cu_k): the keys come from their own boundaries and query i sees key
// j when j <= i + lk - lq.
template <int D, bool TOK, bool WIN, bool X>
__global__ void __launch_bounds__(kBwdThreads, 1)
    dq_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                 const BwdParams p) {
  // Launched as a programmatic dependent of the dK/dV kernel: it reads none of that kernel's
  // results (its maps, D and status were final before the dK/dV kernel passed its own wait),
  // so it starts without waiting, on SMs as dK/dV CTAs finish.  Every thread waits for the
  // dK/dV grid on its way out, so this grid completes only after that one and the work that
  // follows in the stream sees both.
  struct WaitOnExit {
    __device__ ~WaitOnExit() { griddep_wait(); }
  } const wait_on_exit;
  using C = QCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t base = smem_u32(smem_raw);
  uint8_t* sm = smem_raw;
  if (base & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) atomicCAS(&p.hdr->status, 0, VA_ERR_CUDA);
    return;
  }
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::MISC_OFF + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return base + C::BAR_OFF + 8u * i; };

  QItem* queue = reinterpret_cast<QItem*>(sm + C::QUEUE_OFF);
  uint8_t* row_tables = sm + C::ROWS_OFF;
  auto dec = [&](int idx) { return q_decode<WIN, X>(p, idx); };
  if (p.hdr->status != VA_OK) return;
  const int n_items = p.hdr->n_items[p.q_slot];
  const int n_seg = n_items - p.hdr->n_items[p.q_tok_slot];  // segment records, then token ones
  if (static_cast<int>(blockIdx.x) >= n_items) return;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::B_QF + b), 1);
      mbar_init(bar(C::B_QE + b), 1);
    }
    mbar_init(bar(C::B_DF), 1);
    mbar_init(bar(C::B_DE), 1);
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(bar(C::B_KF + s), 1);
      mbar_init(bar(C::B_KE + s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::B_SF + x), 1);
      mbar_init(bar(C::B_PF + x), 256);  // both softmax warpgroups, one half of the step each
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::B_AF + b), 1);
      mbar_init(bar(C::B_AE + b), 256);
    }
    mbar_init(bar(C::B_DR), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::B_IF + b), 1);
      mbar_init(bar(C::B_IE + b), 32 + 256);  // MMA warp + both softmax warpgroups
    }
    *abort_flag = 0;
    *wait_limit_slot(abort_flag) = kTimeoutNs;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tq);
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
    prefetch_tmap(&tdo);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    regs_dec<kRegsCtl>();
    {  // the whole warp runs the loop; elect.sync picks the issuing lane
      int kit = 0, item_cnt = 0, q_issued = 0, do_issued = 0;  // items whose Q / dO load went out
      bool ok = true;
      QItem nxt;
      // Publishes this CTA's k-th item (the next record of the map): lane 0 pulls its index,
      // the warp decodes it (a token record also fills row table k & 3) and lane 0 writes the
      // slot and releases it.  Returns false at the end of the list or on abort (ok_ = false).
      auto publish = [&](int k, QItem& out, bool& ok_) -> bool {
        const int s = k & 1;
        ok_ = wwait(bar(C::B_IE + s), ((k >> 1) & 1) ^ 1, abort_flag, p.hdr, 40);
        if (!ok_) return false;
        int idx = 0;
        if (lane == 0) idx = atomicAdd(p.q_counter, 1);
        idx = __shfl_sync(0xffffffffu, idx, 0);
        if (idx < n_seg) {
          out = q_decode<WIN, X>(p, idx);
          out.valid = 1;
        } else if (idx < n_items) {
          out = q_token_decode_w(p, idx, row_tables + (k & 3) * C::QB);
          out.valid = 2;
        } else {
          out = QItem{};
          out.valid = 0;
        }
        __syncwarp();  // every lane's table bytes before the release
        if (lane == 0) {
          queue[s] = out;
          mbar_arrive(bar(C::B_IF + s));
        }
        __syncwarp();
        return out.valid != 0;
      };
      // Q of this CTA's j-th item into buffer j & 1, once item j-2's S MMAs are done with it
      auto load_q = [&](const QItem& J, int j) -> bool {
        const int qb = j & 1;
        if (!wwait(bar(C::B_QE + qb), ((j >> 1) & 1) ^ 1, abort_flag, p.hdr, 31)) return false;
        mbar_expect_tx_w(bar(C::B_QF + qb), C::TQ);
        for (int pn = 0; pn < D / 64; ++pn)
          tma_load_3d_w(base + qb * C::TQ + pn * C::PQ, &tq, bar(C::B_QF + qb), pn * 64, J.h, J.s0 + J.m * 128);
        q_issued = j + 1;
        return true;
      };
      // dO of this CTA's j-th item into the dO buffer, once item j-1's dP MMAs are done with it
      auto load_do = [&](const QItem& J, int j) -> bool {
        if (!wwait(bar(C::B_DE), (j & 1) ^ 1, abort_flag, p.hdr, 30)) return false;
        mbar_expect_tx_w(bar(C::B_DF), C::TQ);
        for (int pn = 0; pn < D / 64; ++pn)
          tma_load_3d_w(base + C::DO_OFF + pn * C::PQ, &tdo, bar(C::B_DF), pn * 64, J.h, J.s0 + J.m * 128);
        do_issued = j + 1;
        return true;
      };
      bool more = TOK ? publish(0, nxt, ok)
                      : queue_publish_w(0, queue, bar(C::B_IF), bar(C::B_IE), p.q_counter, n_items, dec, nxt,
                                        abort_flag, p.hdr, ok);
      if (ok && more) ok = load_q(nxt, 0);
      for (; ok && more; ++item_cnt) {
        const QItem I = nxt;  // publish the next record first: its decode overlaps this one
        more = TOK ? publish(item_cnt + 1, nxt, ok)
                   : queue_publish_w(item_cnt + 1, queue, bar(C::B_IF), bar(C::B_IE), p.q_counter, n_items, dec,
                                     nxt, abort_flag, p.hdr, ok);
        if (!ok) break;
        // This item's first two K/V steps, then its dO (which waits for the previous item's last
        // dP MMA), then the next item's Q (a whole item ahead of its use) and the remaining steps.
        const int qd_at = I.nb < 2 ? I.nb : 2;
        for (int n = 0; ok && n <= I.nb; ++n) {
          if (n == qd_at) {
            ok = load_do(I, item_cnt) && (!more || load_q(nxt, item_cnt + 1));
            if (!ok) break;
          }
          if (n == I.nb) break;
          const int s = kit % C::KST;
          ok = wwait(bar(C::B_KE + s), ((kit / C::KST) & 1) ^ 1, abort_flag, p.hdr, 32);
          if (!ok) break;
          mbar_expect_tx_w(bar(C::B_KF + s), 2 * C::TKV);
          const uint32_t dst = base + C::RING_OFF + s * 2 * C::TKV;
          for (int pn = 0; pn < D / 64; ++pn) {
            tma_load_3d_w(dst + pn * C::PKV, &tk, bar(C::B_KF + s), pn * 64, I.hk, I.kb + n * 64);
            tma_load_3d_w(dst + C::TKV + pn * C::PKV, &tv, bar(C::B_KF + s), pn * 64, I.hk, I.kb + n * 64);
          }
          ++kit;
        }
      }
      if (!ok) {
        // let every copy this thread started land before the CTA exits
        for (int j = q_issued - 1; j >= 0 && j >= q_issued - 2; --j)
          drain_wait_b(bar(C::B_QF + (j & 1)), (j >> 1) & 1);
        if (do_issued > 0) drain_wait_b(bar(C::B_DF), (do_issued - 1) & 1);
        for (int i = kit - 1; i >= 0 && i >= kit - C::KST; --i)
          drain_wait_b(bar(C::B_KF + i % C::KST), (i / C::KST) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    regs_dec<kRegsCtl>();
    {  // the whole warp runs the loop; elect.sync picks the issuing lane
      constexpr uint32_t idS = idesc_bf16(128, 64, false, false);
      constexpr uint32_t idG = idesc_bf16(128, D, false, true);
      int kit = 0, item_cnt = 0;
      uint32_t pf0 = 0, pf1 = 0;  // p_full phases per buffer (scalars: a runtime index would spill)
      bool ok = true;
      int qb = 0;
      const uint32_t qlo0 = sdesc_lo(base, 16);                    // Q/dO, K-major A
      const uint32_t ringK0 = sdesc_lo(base + C::RING_OFF, 16);      // K/V as K-major B
      const uint32_t ringM0 = sdesc_lo(base + C::RING_OFF, C::PKV);  // K as MN-major B
      // S and dP of one step into buffer x; the item's first step first waits for its dO
      auto issue_SdP = [&](int x, int slot, bool wait_do) -> bool {
        const uint32_t kd = ringK0 + ((slot * 2 * C::TKV) >> 4), vd = kd + (C::TKV >> 4);
        const uint32_t qd = qlo0 + ((qb * C::TQ) >> 4), dd = qlo0 + (C::DO_OFF >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t oq = ((kk >> 2) * C::PQ + (kk & 3) * 32) >> 4, ok_ = ((kk >> 2) * C::PKV + (kk & 3) * 32) >> 4;
          mma_ss_w(tmem + x * 64, qd + oq, kd + ok_, idS, kk > 0);
        }
        if (wait_do) {
          if (!wwait(bar(C::B_DF), item_cnt & 1, abort_flag, p.hdr, 30)) return false;
          fence_after_sync();
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t oq = ((kk >> 2) * C::PQ + (kk & 3) * 32) >> 4, ok_ = ((kk >> 2) * C::PKV + (kk & 3) * 32) >> 4;
          mma_ss_w(tmem + 128 + x * 64, dd + oq, vd + ok_, idS, kk > 0);
        }
        mma_commit_w(bar(C::B_SF + x));
        return true;
      };
      for (;; ++item_cnt) {
        QItem I;
        const bool got_ = queue_take(item_cnt, queue, bar(C::B_IF), bar(C::B_IE), I, abort_flag, p.hdr, ok);
        const bool all_ok = __all_sync(0xffffffffu, ok);
        if (!all_ok) ok = false;
        if (!all_ok || !got_) break;
        qb = item_cnt & 1;
        ok = wwait(bar(C::B_QF + qb), (item_cnt >> 1) & 1, abort_flag, p.hdr, 33);
        if (!ok) break;
        for (int j = 0; ok && j < 2 && j < I.nb; ++j) {
          const int s = (kit + j) % C::KST;
          ok = wwait(bar(C::B_KF + s), ((kit + j) / C::KST) & 1, abort_flag, p.hdr, 34);
          if (!ok) break;
          fence_after_sync();
          ok = issue_SdP(j, s, j == 0);
        }
        if (!ok) break;
        if (I.nb <= 2) {  // the item's last S / dP MMAs: its Q and dO buffers may be reloaded
          mma_commit_w(bar(C::B_QE + qb));
          mma_commit_w(bar(C::B_DE));
        }
        for (int n = 0; ok && n < I.nb; ++n) {
          const int x = n & 1, s = (kit + n) % C::KST;
          ok = wwait(bar(C::B_PF + x), (x ? pf1 : pf0) & 1, abort_flag, p.hdr, 35);
          if (!ok) break;
          if (x) ++pf1;
          else ++pf0;
          if (n == 0) {  // this item's dQ buffer must have been read out two items ago
            ok = wwait(bar(C::B_AE + (item_cnt & 1)), ((item_cnt >> 1) & 1) ^ 1, abort_flag, p.hdr, 36);
            if (!ok) break;
          }
          fence_after_sync();
          const uint32_t km = ringM0 + ((s * 2 * C::TKV) >> 4);
#pragma unroll
          for (int kk = 0; kk < C::KB / 16; ++kk)
            mma_ts_w(tmem + 256 + (item_cnt & 1) * D, tmem + 128 + x * 64 + (kk >> 1) * 32 + (kk & 1) * 8,
                     km + kk * (2048 >> 4), idG,
                      (n > 0 || kk > 0) ? 1u : 0u);
          mma_commit_w(bar(C::B_KE + s));
          if (n + 2 < I.nb) {
            const int s2 = (kit + n + 2) % C::KST;
            ok = wwait(bar(C::B_KF + s2), ((kit + n + 2) / C::KST) & 1, abort_flag, p.hdr, 37);
            if (!ok) break;
            fence_after_sync();
            issue_SdP(x, s2, false);
            if (n + 2 == I.nb - 1) {
              mma_commit_w(bar(C::B_QE + qb));
              mma_commit_w(bar(C::B_DE));
            }
          }
        }
        if (!ok) break;
        mma_commit_w(bar(C::B_AF + (item_cnt & 1)));
        kit += I.nb;
      }
      mma_commit_w(bar(C::B_DR));
      drain_wait_b(bar(C::B_DR), 0);
    }
  } else if (warp < 4) {
    regs_dec<kRegsCtl>();  // warps 2 and 3 have no role
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    regs_inc<kRegsSoftmax>();
    // Both warpgroups take every step, warpgroup x its key columns [32 x, 32 x + 32) of the
    // step's S / dP buffer (step n uses buffer n & 1), writing dS (bf16) over the first 16
    // columns of that range of dP; epilogue: dQ columns [x D/2, (x+1) D/2).
    const int x = (warp - 4) >> 2;
    const int cw = 32 * x;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + cw;
    const uint32_t dp_addr = tmem + lane_off + 128 + cw;
    const uint32_t acc_addr = tmem + lane_off + 256;
    const float sl2 = p.scale_log2;
    uint32_t sf0 = 0, sf1 = 0;  // s_full phases per buffer
    int item_cnt = 0;
    bool ok = true;
    // The dQ accumulator is double-buffered (item k uses buffer k & 1), so item k's
    // epilogue waits until this warpgroup has handed in its first step of item k + 1:
    // the tensor core starts the next item meanwhile.
    int pend = -1;          // item whose epilogue is pending, or -1
    bf16* pend_out = nullptr;
    bool pend_store = false;
    auto epilogue = [&]() -> bool {
      const int k = pend;
      pend = -1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(C::B_AF + (k & 1)), (k >> 1) & 1, abort_flag, p.hdr, 39)))
        return false;
      fence_after_sync();
      constexpr int HC = D / 2;  // this warpgroup's columns [x HC, (x + 1) HC), one round trip
      uint32_t o[HC];
#pragma unroll
      for (int c = 0; c < HC / 32; ++c) tmem_ld32(acc_addr + (k & 1) * D + x * HC + c * 32, o + c * 32);
      tmem_wait_ld();
      fence_before_sync();
      mbar_arrive(bar(C::B_AE + (k & 1)));  // the buffer is free once its values are in registers
#pragma unroll
      for (int j = 0; j < HC / 2; ++j)
        o[j] = pack_bf16(__uint_as_float(o[2 * j]) * p.scale, __uint_as_float(o[2 * j + 1]) * p.scale);
      if constexpr (HC % 64 == 0) {
        uint4 ov[HC / 8];
#pragma unroll
        for (int j = 0; j < HC / 8; ++j) ov[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
        store_rows_coalesced(ov, pend_out + x * HC, p.o_rs, pend_store);
      } else if (pend_store) {
        uint4* dst = reinterpret_cast<uint4*>(pend_out + x * HC);
#pragma unroll
        for (int j = 0; j < HC / 8; ++j) dst[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
      }
      return true;
    };
    QItem I;
    bool tok = false;  // the item in I is the first token item
    for (;; ++item_cnt) {
      const bool got = queue_take(item_cnt, queue, bar(C::B_IF), bar(C::B_IE), I, abort_flag, p.hdr, ok);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      if (!got) break;
      if constexpr (TOK) {
        if (I.valid == 2) {  // the token records follow: the loop below
          tok = true;
          break;
        }
      }
      const int qrow = I.m * 128 + r;
      const int64_t at = static_cast<int64_t>(I.h) * p.T + I.s0 + qrow;
      // the row's lse and D: loads issued here, first used after the S wait below, so their
      // latency overlaps it
      const bool qin = qrow < I.l;
      float lse_raw = 0.f, dsum = 0.f;
      if (qin) {
        lse_raw = __ldg(p.lse + at);
        dsum = __ldg(p.dsum + at);
      }
      for (int n = 0; n < I.nb; ++n) {
        const int b = n & 1;
        ok = mbar_wait(bar(C::B_SF + b), (b ? sf1 : sf0) & 1, abort_flag, p.hdr, 38);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        if (b) ++sf1;
        else ++sf0;
        fence_after_sync();
        const float lse2 = qin ? lse_raw * kLog2e : INFINITY;
        // key columns c > lim are masked: after the query (causal) or past the segment end;
        // (window) key columns c < lo too: before the query's window
        const int kn = (WIN ? I.kb - I.s0 : 0) + n * 64 + cw;  // this warpgroup's first key, segment-local
        int lim = p.causal ? qrow - kn : I.l - 1 - kn;
        const int lo = WIN ? qrow - p.window - kn : 0;
        bool need_mask = p.causal ? (kn + 31 > I.m * 128 || (WIN && kn < I.m * 128 + 127 - p.window))
                                  : (kn + 32 > I.l);
        if constexpr (X) {
          lim = p.causal ? qrow + I.off - kn : I.lk - 1 - kn;
          need_mask = p.causal ? (kn + 31 > I.m * 128 + I.off) : (kn + 32 > I.lk);
        }
        // one TMEM round trip: this warpgroup's 32 scores and 32 dP values of this q row
        uint32_t sv[32], dpv[32];
        tmem_ld32(s_addr + b * 64, sv);
        tmem_ld32(dp_addr + b * 64, dpv);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float x0, x1;
          ffma2(x0, x1, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), sl2, sl2, -lse2, -lse2);
          float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          if (need_mask) {
            if (c > lim || (WIN && c < lo)) p0 = 0.f;
            if (c + 1 > lim || (WIN && c + 1 < lo)) p1 = 0.f;
          }
          float t0, t1;
          fadd2(t0, t1, __uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1]), -dsum, -dsum);
          dpv[c >> 1] = pack_bf16(p0 * t0, p1 * t1);
        }
        tmem_st16(dp_addr + b * 64, dpv);
        tmem_wait_st();
        fence_before_sync();
        mbar_arrive(bar(C::B_PF + b));
        if (pend >= 0 && !epilogue()) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      if (pend >= 0 && !epilogue()) {  // this warpgroup had no step in the item
        ok = false;
        break;
      }
      pend = item_cnt;
      pend_out = p.dq + static_cast<int64_t>(I.s0 + qrow) * p.o_rs + static_cast<int64_t>(I.h) * p.o_hs;
      pend_store = qrow < I.l;
    }
    // Token items (runs of short segments; all of them follow the segment items): every step
    // masked on both sides per query row.
    while (TOK && ok && tok) {
      const int qrow = r;  // m = 0
      const int klo = I.s0 + r - row_tables[(item_cnt & 3) * C::QB + r];  // its segment's start
      const int64_t at = static_cast<int64_t>(I.h) * p.T + I.s0 + qrow;
      // the row's lse and D: loads issued here, first used after the S wait below, so their
      // latency overlaps it
      const bool qin = qrow < I.l;
      float lse_raw = 0.f, dsum = 0.f;
      if (qin) {
        lse_raw = __ldg(p.lse + at);
        dsum = __ldg(p.dsum + at);
      }
      for (int n = 0; n < I.nb; ++n) {
        const int b = n & 1;
        ok = mbar_wait(bar(C::B_SF + b), (b ? sf1 : sf0) & 1, abort_flag, p.hdr, 38);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        if (b) ++sf1;
        else ++sf0;
        fence_after_sync();
        const float lse2 = qin ? lse_raw * kLog2e : INFINITY;
        // key columns c > lim (after the query) and c < lo (before its segment) are masked
        const int k0 = I.kb + n * 64 + cw;
        const int lim = I.s0 + r - k0, lo = klo - k0;
        // one TMEM round trip: this warpgroup's 32 scores and 32 dP values of this q row
        uint32_t sv[32], dpv[32];
        tmem_ld32(s_addr + b * 64, sv);
        tmem_ld32(dp_addr + b * 64, dpv);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float x0, x1;
          ffma2(x0, x1, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]), sl2, sl2, -lse2, -lse2);
          float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          if (c > lim || c < lo) p0 = 0.f;
          if (c + 1 > lim || c + 1 < lo) p1 = 0.f;
          float t0, t1;
          fadd2(t0, t1, __uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1]), -dsum, -dsum);
          dpv[c >> 1] = pack_bf16(p0 * t0, p1 * t1);
        }
        tmem_st16(dp_addr + b * 64, dpv);
        tmem_wait_st();
        fence_before_sync();
        mbar_arrive(bar(C::B_PF + b));
        if (pend >= 0 && !epilogue()) {
          ok = false;
          break;
        }
      }
      if (!ok) break;
      if (pend >= 0 && !epilogue()) {  // this warpgroup had no step in the item
        ok = false;
        break;
      }
      pend = item_cnt;
      pend_out = p.dq + static_cast<int64_t>(I.s0 + qrow) * p.o_rs + static_cast<int64_t>(I.h) * p.o_hs;
      pend_store = qrow < I.l;
      ++item_cnt;
      const bool got = queue_take(item_cnt, queue, bar(C::B_IF), bar(C::B_IE), I, abort_flag, p.hdr, ok);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      if (!got) break;
    }
    if (ok && pend >= 0) ok = epilogue();
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- host side


template <int D, bool TOK, bool WIN, bool X>
static cudaError_t launch_dkdv_d(const BwdParams& p, int cap, cudaStream_t st) {
  using C = KvCfg<D>;
  CUtensorMap tq, tk, tv, tdo;
  if (!tmap_rows(&tq, p.q, p.T, p.Hq, D, p.q_rs, p.q_hs, 64) ||
      !tmap_rows(&tdo, p.dout, p.T, p.Hq, D, p.o_rs, p.o_hs, 64) ||
      !tmap_rows(&tk, p.k, X ? p.Tk : p.T, p.Hkv, D, p.k_rs, p.k_hs, 128) ||
      !tmap_rows(&tv, p.v, X ? p.Tk : p.T, p.Hkv, D, p.v_rs, p.v_hs, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(dkdv_tc_kernel<D, TOK, WIN, X>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  // the in-kernel register split assumes the full launch budget; refuse rather than wait
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, dkdv_tc_kernel<D, TOK, WIN, X>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = std::min(cap, std::max(sms, 1));
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(dkdv_tc_kernel<D, TOK, WIN, X>, dim3(grid), dim3(kBwdThreads), C::SMEM, st, tq, tk, tv, tdo, p);
}

template <int D, bool TOK, bool WIN, bool X>
static cudaError_t launch_dq_d(const BwdParams& p, int cap, cudaStream_t st) {
  using C = QCfg<D>;
  CUtensorMap tq, tk, tv, tdo;
  if (!tmap_rows(&tq, p.q, p.T, p.Hq, D, p.q_rs, p.q_hs, 128) ||
      !tmap_rows(&tdo, p.dout, p.T, p.Hq, D, p.o_rs, p.o_hs, 128) ||
      !tmap_rows(&tk, p.k, X ? p.Tk : p.T, p.Hkv, D, p.k_rs, p.k_hs, 64) ||
      !tmap_rows(&tv, p.v, X ? p.Tk : p.T, p.Hkv, D, p.v_rs, p.v_hs, 64))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(dq_tc_kernel<D, TOK, WIN, X>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  // the in-kernel register split assumes the full launch budget; refuse rather than wait
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, dq_tc_kernel<D, TOK, WIN, X>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = std::min(cap, std::max(sms, 1));
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(dq_tc_kernel<D, TOK, WIN, X>, dim3(grid), dim3(kBwdThreads), C::SMEM, st, tq, tk, tv, tdo, p);
}

// tok: the maps hold token records.  The two forms are compiled separately so that the
// segment-only kernels keep their own code: the token branch in the softmax item loop
// measured 15% slower on segment records.
cudaError_t launch_bwd_dkdv_tc(const BwdParams& p, int d, int cap, bool tok, cudaStream_t st) {
  if (p.cu_k)  // cross and window calls plan no token records
    return d == 64 ? launch_dkdv_d<64, false, false, true>(p, cap, st) : launch_dkdv_d<128, false, false, true>(p, cap, st);
  if (p.window >= 0)
    return d == 64 ? launch_dkdv_d<64, false, true, false>(p, cap, st) : launch_dkdv_d<128, false, true, false>(p, cap, st);
  if (tok)
    return d == 64 ? launch_dkdv_d<64, true, false, false>(p, cap, st) : launch_dkdv_d<128, true, false, false>(p, cap, st);
  return d == 64 ? launch_dkdv_d<64, false, false, false>(p, cap, st) : launch_dkdv_d<128, false, false, false>(p, cap, st);
}

cudaError_t launch_bwd_dq_tc(const BwdParams& p, int d, int cap, bool tok, cudaStream_t st) {
  if (p.cu_k)
    return d == 64 ? launch_dq_d<64, false, false, true>(p, cap, st) : launch_dq_d<128, false, false, true>(p, cap, st);
  if (p.window >= 0)
    return d == 64 ? launch_dq_d<64, false, true, false>(p, cap, st) : launch_dq_d<128, false, true, false>(p, cap, st);
  if (tok)
    return d == 64 ? launch_dq_d<64, true, false, false>(p, cap, st) : launch_dq_d<128, true, false, false>(p, cap, st);
  return d == 64 ? launch_dq_d<64, false, false, false>(p, cap, st) : launch_dq_d<128, false, false, false>(p, cap, st);
}

int bwd_tc_token_short() { return kBwdTokenShort; }

void bwd_tc_tiles(int* kvBM, int* kvBN, int* qBM, int* qBN) {
  *kvBM = 64;
  *kvBN = 128;
  *qBM = 128;
  *qBN = 64;
}

}  // namespace va
