// Forward varlen attention for sm_103a: TMA + tcgen05 MMA (TMEM accumulators),
// warp-specialised, persistent.
//
// What it computes ("Packing与 FlashAttention Varlen", sections 1 and 5): for a
// work item (segment b, q block m of 256 rows, q head h) the Q/K/V rows are read
// at offset cu[b] of the flat token axis with extent l = cu[b+1]-cu[b]; key
// blocks run to ceil(min(l, (m+1)*256)/128) (causal) and the causal mask is
// applied only on the one key block that crosses each 128-row tile's diagonal.
// O is written at Q's offsets, rows past l are never stored, and
// lse = ln sum_j exp(scale q.k_j).  Runs of short segments are planned as token tiles and
// computed by fwd_tok.cu's kernel, launched right after this one.
//
// CTA layout (384 threads, one CTA per SM, persistent over the tile map):
//   warp 0      TMA producer (whole warp, one elected lane issues): pulls work items from
//               the map's counter and publishes them
//               (sched.cuh); Q tiles once per item, K/V tiles into an NST-slot ring
//   warp 1      MMA issuer (the whole warp runs the loop, one elected lane issues):
//               S_t = Q_t K^T (SS), O_t += P_t V (TS, P in TMEM);
//               also owns the TMEM allocation
//   warps 4-7   softmax + epilogue for q tile 0 (rows 0..127 of the block; thread = row)
//   warps 8-11  softmax + epilogue for q tile 1 (rows 128..255)
// TMEM (512 columns): S0 | S1 | O0 | O1.  P_t (bf16) overwrites the first half of
// S_t; the MMA pipe executes in issue order, so the next S_t cannot overwrite P_t
// before the PV that reads it.  The two q tiles share every K/V tile, halving
// shared-memory fill traffic per FLOP; while one tile's softmax runs, the tensor
// core works on the other tile.  The running max is only raised when it grows by
// more than 2^8, so O in TMEM is rescaled rarely.
#include "attn_params.cuh"
#include "sched.cuh"
#include "sm100_ptx.cuh"
#include "tmap.cuh"

namespace va {
using namespace sm100;

namespace {

constexpr int kTcBM = 256;  // q rows per work item (two 128-row tiles)
constexpr int kTcBN = 128;  // key rows per K/V tile
static_assert((kTcBM & (kTcBM - 1)) == 0 && (kTcBN & (kTcBN - 1)) == 0, "the planner takes powers of two");
constexpr int kTcThreads = 384;
// setmaxnreg moves registers within what the CTA was launched with (168 per thread for
// 384 threads); a split above that total would make the increase wait forever.
constexpr int kLaunchRegs = 168;
constexpr int kRegsCtl = 80, kRegsSoftmax = 208;
static_assert(128 * kRegsCtl + 256 * kRegsSoftmax <= kTcThreads * kLaunchRegs, "register split exceeds the launch");
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct TcCfg {
  static constexpr int NST = D == 128 ? 5 : 12;        // K/V ring slots
  static constexpr int TILE = 128 * D * 2;             // bytes of one 128-row Q, K or V tile
  static constexpr int PANEL = 128 * 128;              // one 64-column (128-byte) panel of a tile
  static constexpr int Q_OFF = 0;                      // Q tiles 0 and 1
  static constexpr int KV_OFF = 2 * TILE;
  static constexpr int BAR_OFF = KV_OFF + NST * TILE;
  // barriers: q_full[tile], q_empty[tile], kv_full[NST], kv_empty[NST], s_full[2], p_full[2],
  // o_full[2], drain, item queue full[2] / empty[2]
  static constexpr int B_QF = 0, B_QE = 2, B_KVF = 4, B_KVE = 4 + NST, B_SF = 4 + 2 * NST,
                       B_PF = B_SF + 2, B_OF = B_PF + 2, B_DR = B_OF + 2, B_IF = B_DR + 1,
                       B_IE = B_IF + 2, NBAR = B_IE + 2;
  static constexpr int QUEUE_OFF = BAR_OFF + NBAR * 8;          // two Item slots
  static constexpr int MISC_OFF = QUEUE_OFF + 2 * 64;
  static constexpr int SMEM = MISC_OFF + 16 + 1024;    // + slack to align the base to 1024
  static constexpr int OCOLS = D;                      // TMEM columns of one O accumulator
};

struct Item {
  int s0, l, h, hk, m, nb, nb0;
  int t1;
  int valid;
  int kb;  // local window: the item's first key tile (its key tiles are kb .. kb + nb - 1)
  int s0k, lk, off;  // cross-attention: the keys' first row and count, the causal offset lk - l
};
static_assert(sizeof(Item) <= 64, "queue slots are 64 bytes");

template <bool WIN, bool X>
__device__ __forceinline__ Item decode(const FwdParams& p, int idx) {
  const TileItem it = p.items[idx];
  Item r;
  r.s0 = p.cu[it.seg];
  r.l = p.cu[it.seg + 1] - r.s0;
  r.h = it.head;
  r.hk = it.head / p.g;
  r.m = it.blk;
  r.nb = it.count;
  r.t1 = r.m * kTcBM + 128 < r.l ? 1 : 0;
  r.nb0 = (p.causal && r.t1) ? r.nb - 1 : r.nb;
  if (WIN) r.kb = max(0, r.m * kTcBM - p.window) / kTcBN;
  if (X) {  // keys from cu_k; q tile 0 may share its diagonal key tile with tile 1
    r.s0k = p.cu_k[it.seg];
    r.lk = p.cu_k[it.seg + 1] - r.s0k;
    r.off = p.causal ? r.lk - r.l : 0;
    if (p.causal && r.t1) r.nb0 = (min(r.lk, r.m * kTcBM + 128 + r.off) + kTcBN - 1) / kTcBN;
  }
  return r;
}

// Masks columns j < lo and j > lim, and returns the row max x sl2 (local window: the left
// edge of the row's window and its diagonal).
__device__ __forceinline__ float row_max2(uint32_t* v, int lo, int lim, float sl2) {
#pragma unroll
  for (int j = 0; j < 128; ++j)
    if (j < lo || j > lim) v[j] = __float_as_uint(-INFINITY);
  float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    m0 = fmax3(m0, __uint_as_float(v[8 * j]), __uint_as_float(v[8 * j + 1]));
    m1 = fmax3(m1, __uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3]));
    m2 = fmax3(m2, __uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5]));
    m3 = fmax3(m3, __uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]));
  }
  return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)) * sl2;
}

// Bounded wait used only while shutting down after an abort: ignores the abort flag.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > 50000000ull) return;
  }
}

// The 128 scores of this thread's row: one TMEM round trip.
__device__ __forceinline__ void row_load(uint32_t s_addr, uint32_t* v) {
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, v + c * 32);
  tmem_wait_ld();
}

// Masks columns j > lim (when MASK) and returns the row max x sl2.
template <bool MASK>
__device__ __forceinline__ float row_max(uint32_t* v, int lim, float sl2) {
  if (MASK) {
#pragma unroll
    for (int j = 0; j < 128; ++j)
      if (j > lim) v[j] = __float_as_uint(-INFINITY);
  }
  float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    m0 = fmax3(m0, __uint_as_float(v[8 * j]), __uint_as_float(v[8 * j + 1]));
    m1 = fmax3(m1, __uint_as_float(v[8 * j + 2]), __uint_as_float(v[8 * j + 3]));
    m2 = fmax3(m2, __uint_as_float(v[8 * j + 4]), __uint_as_float(v[8 * j + 5]));
    m3 = fmax3(m3, __uint_as_float(v[8 * j + 6]), __uint_as_float(v[8 * j + 7]));
  }
  return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)) * sl2;
}

// p = exp2(s * sl2 - mu) packed in place as bf16 pairs into v[0..63]; returns the row sum.
__device__ __forceinline__ float row_exp(uint32_t* v, float sl2, float mu) {
  float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    float x0, x1;
    ffma2(x0, x1, __uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]), sl2, sl2, -mu, -mu);
    const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
    if (j & 1) fadd2(b0, b1, b0, b1, p0, p1);
    else fadd2(a0, a1, a0, a1, p0, p1);
    v[j] = pack_bf16(p0, p1);
  }
  return (a0 + a1) + (b0 + b1);
}

}  // namespace

// WIN: causal local window p.window (query i sees keys i-w..i): an item's key tiles start at
// the window of its first row, and tiles that cross a row's window edge are masked on both
// sides; a row may see nothing in its first tiles (its running max stays -inf and the first
// visible tile takes over with a zero-weight rescale).
// X: cross-attention (p.cu_k): keys from their own boundaries, the causal bound aligned
// bottom-right (key j visible to query i when j <= i + lk - lq), so the masked key tiles are
// the one or two that cross a q tile's diagonal band.
template <int D, bool WIN, bool X>
__global__ void __launch_bounds__(kTcThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const FwdParams p) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::MISC_OFF + 4);
  Item* queue = reinterpret_cast<Item*>(sm + C::QUEUE_OFF);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return base + C::BAR_OFF + 8u * i; };
  auto dec = [&](int idx) { return decode<WIN, X>(p, idx); };

  griddep_begin();  // the tile map and status come from the planning launch just before
  if (p.hdr->status != VA_OK) return;
  // segment records only: the token records at the map's end go to fwd_tok.cu's kernel
  const int n_items = p.hdr->n_items[p.slot] - p.hdr->n_items[kTokSlot];
  if (static_cast<int>(blockIdx.x) >= n_items) return;

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::B_QF + b), 1);
      mbar_init(bar(C::B_QE + b), 1);
    }
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar(C::B_KVF + s), 1);
      mbar_init(bar(C::B_KVE + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::B_SF + t), 1);
      mbar_init(bar(C::B_PF + t), 128);
      mbar_init(bar(C::B_OF + t), 1);
    }
    mbar_init(bar(C::B_DR), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::B_IF + b), 1);
      mbar_init(bar(C::B_IE + b), 32 + 256);  // MMA warp + both softmax warpgroups
    }
    *abort_flag = 0;
    *wait_limit_slot(abort_flag) = p.wait_ns ? p.wait_ns : kTimeoutNs;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tq);
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  // Registers: what the producer/MMA warpgroup (warps 0-3) gives back goes to the two
  // softmax warpgroups, which hold a whole 128-score row.  Every warp sets its budget at
  // the top of its role.
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    regs_dec<kRegsCtl>();
    {  // the whole warp runs the loop; elect.sync picks the issuing lane
      int kv_it = 0, item_cnt = 0, qcnt[2] = {0, 0};
      bool ok = true;
      Item nxt;
      bool more = queue_publish_w(0, queue, bar(C::B_IF), bar(C::B_IE), p.counter, n_items, dec, nxt,
                                abort_flag, p.hdr, ok);
      if (p.stall) more = false;  // test hook: the first item is published and nothing is loaded
      for (; ok && more; ++item_cnt) {
        const Item I = nxt;  // publish the next record first: its decode overlaps this one
        more = queue_publish_w(item_cnt + 1, queue, bar(C::B_IF), bar(C::B_IE), p.counter, n_items,
                             dec, nxt, abort_flag, p.hdr, ok);
        if (!ok) break;
        // Q tile t is released by the item's last S_t MMA (tile 0 one key tile before tile 1)
        for (int t = 0; ok && t < (I.t1 ? 2 : 1); ++t) {
          ok = wwait(bar(C::B_QE + t), (qcnt[t] & 1) ^ 1, abort_flag, p.hdr, 1);
          if (!ok) break;
          mbar_expect_tx_w(bar(C::B_QF + t), C::TILE);
          for (int pn = 0; pn < D / 64; ++pn)
            tma_load_3d_w(base + C::Q_OFF + t * C::TILE + pn * C::PANEL, &tq, bar(C::B_QF + t), pn * 64,
                        I.h, I.s0 + I.m * kTcBM + t * 128);
          ++qcnt[t];
        }
        if (!ok) break;
        for (int n = 0; ok && n < I.nb; ++n) {
          for (int kv = 0; kv < 2; ++kv) {
            const int s = kv_it % C::NST;
            ok = wwait(bar(C::B_KVE + s), ((kv_it / C::NST) & 1) ^ 1, abort_flag, p.hdr, 2);
            if (!ok) break;
            mbar_expect_tx_w(bar(C::B_KVF + s), C::TILE);
            for (int pn = 0; pn < D / 64; ++pn)
              tma_load_3d_w(base + C::KV_OFF + s * C::TILE + pn * C::PANEL, kv ? &tv : &tk,
                          bar(C::B_KVF + s), pn * 64, I.hk, (X ? I.s0k : I.s0) + (WIN ? I.kb + n : n) * kTcBN);
            ++kv_it;
          }
        }
      }
      if (!ok) {
        // let every copy this thread started land before the CTA exits
        for (int t = 0; t < 2; ++t)
          if (qcnt[t] > 0) drain_wait(bar(C::B_QF + t), (qcnt[t] - 1) & 1);
        for (int i = kv_it - 1; i >= 0 && i >= kv_it - C::NST; --i)
          drain_wait(bar(C::B_KVF + i % C::NST), (i / C::NST) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    regs_dec<kRegsCtl>();
    {  // the whole warp runs the loop; elect.sync picks the issuing lane
      constexpr uint32_t idS = idesc_bf16(128, kTcBN, false, false);
      constexpr uint32_t idPV = idesc_bf16(128, D, false, true);
      int kv_it = 0, item_cnt = 0;
      uint32_t pf[2] = {0, 0};
      bool ok = true;
      uint32_t qcnt[2] = {0, 0};
      const uint32_t qlo[2] = {sdesc_lo(base + C::Q_OFF, 16), sdesc_lo(base + C::Q_OFF + C::TILE, 16)};
      const uint32_t klo0 = sdesc_lo(base + C::KV_OFF, 16);
      const uint32_t vlo0 = sdesc_lo(base + C::KV_OFF, C::PANEL);
      auto issue_S = [&](int t, int slot) {
        const uint32_t qd = qlo[t], kd = klo0 + ((slot * C::TILE) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * C::PANEL + (kk & 3) * 32) >> 4;
          mma_ss_w(tmem + t * 128, qd + off, kd + off, idS, kk > 0);
        }
        mma_commit_w(bar(C::B_SF + t));
      };
      auto issue_PV = [&](int t, int slot, bool acc) {
        const uint32_t vd = vlo0 + ((slot * C::TILE) >> 4);
        const uint32_t d_tm = tmem + 256 + t * C::OCOLS, p_tm = tmem + t * 128;
#pragma unroll
        for (int kk = 0; kk < kTcBN / 16; ++kk)
          mma_ts_w(d_tm, p_tm + kk * 8, vd + kk * (2048 >> 4), idPV, (acc || kk > 0) ? 1u : 0u);
        mma_commit_w(bar(C::B_OF + t));
      };
      for (;; ++item_cnt) {
        Item I;
        const bool got_ = queue_take(item_cnt, queue, bar(C::B_IF), bar(C::B_IE), I, abort_flag, p.hdr, ok);
        const bool all_ok = __all_sync(0xffffffffu, ok);
        if (!all_ok) ok = false;
        if (!all_ok || !got_) break;
        ok = wwait(bar(C::B_QF + 0), qcnt[0] & 1, abort_flag, p.hdr, 3);
        if (!ok) break;
        if (I.t1) {
          ok = wwait(bar(C::B_QF + 1), qcnt[1] & 1, abort_flag, p.hdr, 3);
          if (!ok) break;
        }
        int ks = kv_it % C::NST;
        ok = wwait(bar(C::B_KVF + ks), (kv_it / C::NST) & 1, abort_flag, p.hdr, 4);
        if (!ok) break;
        fence_after_sync();
        ++kv_it;
        issue_S(0, ks);
        if (I.nb0 == 1) {
          mma_commit_w(bar(C::B_QE + 0));  // last S_0 of the item: Q tile 0 may be reloaded
          ++qcnt[0];
        }
        if (I.t1) {
          issue_S(1, ks);
          if (I.nb == 1) {
            mma_commit_w(bar(C::B_QE + 1));
            ++qcnt[1];
          }
        }
        mma_commit_w(bar(C::B_KVE + ks));
        for (int n = 0; ok && n < I.nb; ++n) {
          const int vs = kv_it % C::NST;
          ok = wwait(bar(C::B_KVF + vs), (kv_it / C::NST) & 1, abort_flag, p.hdr, 5);
          if (!ok) break;
          ++kv_it;
          if (n < I.nb0) {
            ok = wwait(bar(C::B_PF + 0), pf[0] & 1, abort_flag, p.hdr, 6);
            if (!ok) break;
            ++pf[0];
            fence_after_sync();
            issue_PV(0, vs, n > 0);
          }
          int ks2 = -1;
          if (n + 1 < I.nb) {
            ks2 = kv_it % C::NST;
            ok = wwait(bar(C::B_KVF + ks2), (kv_it / C::NST) & 1, abort_flag, p.hdr, 7);
            if (!ok) break;
            ++kv_it;
            fence_after_sync();
            if (n + 1 < I.nb0) {
              issue_S(0, ks2);
              if (n + 1 == I.nb0 - 1) {
                mma_commit_w(bar(C::B_QE + 0));
                ++qcnt[0];
              }
            }
          }
          if (I.t1) {
            ok = wwait(bar(C::B_PF + 1), pf[1] & 1, abort_flag, p.hdr, 8);
            if (!ok) break;
            ++pf[1];
            fence_after_sync();
            issue_PV(1, vs, n > 0);
          }
          mma_commit_w(bar(C::B_KVE + vs));
          if (ks2 >= 0) {
            if (I.t1) {
              issue_S(1, ks2);
              if (n + 1 == I.nb - 1) {
                mma_commit_w(bar(C::B_QE + 1));
                ++qcnt[1];
              }
            }
            mma_commit_w(bar(C::B_KVE + ks2));
          }
        }
      }
      // every MMA this thread issued must finish before TMEM is released
      mma_commit_w(bar(C::B_DR));
      drain_wait(bar(C::B_DR), 0);
    }
  } else if (warp < 4) {
    regs_dec<kRegsCtl>();  // warps 2 and 3 have no role
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    // warps 4-7 own q tile 0, warps 8-11 q tile 1; a warp reaches TMEM lanes 32*(warp % 4)
    regs_inc<kRegsSoftmax>();
    const int t = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + t * 128;
    const uint32_t o_addr = tmem + lane_off + 256 + t * C::OCOLS;
    const float sl2 = p.scale_log2;
    uint32_t sf = 0, of_base = 0;
    bool ok = true;
    for (int k = 0;; ++k) {
      Item I;
      const bool got = queue_take(k, queue, bar(C::B_IF), bar(C::B_IE), I, abort_flag, p.hdr, ok);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      if (!got) break;
      if (t == 1 && !I.t1) continue;
      const int nbt = t == 0 ? I.nb0 : I.nb;
      const int qrow = I.m * kTcBM + t * 128 + r;
      float m_ref = -INFINITY, lsum = 0.f;
      for (int n = 0; n < nbt; ++n) {
        ok = mbar_wait(bar(C::B_SF + t), sf & 1, abort_flag, p.hdr, 9);
        if (!__all_sync(0xffffffffu, ok)) {  // TMEM loads below are warp-collective
          ok = false;
          break;
        }
        ++sf;
        fence_after_sync();
        // The causal mask touches only the last key tile of each q tile (its diagonal
        // tile); non-causal masks only key columns past the segment end.
        bool need_mask = p.causal ? (n == nbt - 1) : (n * kTcBN + kTcBN > I.l);
        int lim = p.causal ? qrow - (WIN ? I.kb + n : n) * kTcBN : I.l - 1 - n * kTcBN;  // mask j > lim
        if constexpr (X) {  // bottom-right alignment: the diagonal band may span two key tiles
          need_mask = p.causal ? (n * kTcBN + kTcBN - 1 > I.m * kTcBM + t * 128 + I.off) : (n * kTcBN + kTcBN > I.lk);
          lim = p.causal ? qrow + I.off - n * kTcBN : I.lk - 1 - n * kTcBN;
        }
        // One TMEM round trip per tile: the row into registers, its max, then
        // p = exp2(s * sl2 - m_ref) packed in place and stored over the first half of S_t.
        // The reference max m_ref is raised only when the row max grew by more than 2^8
        // (rare); O_t, which holds PV_{n-1}, is then rescaled in TMEM first.
        uint32_t v[128];
        row_load(s_addr, v);
        float mt;
        if constexpr (WIN) {  // keys before qrow - w are outside the window
          const int ka = (I.kb + n) * kTcBN;
          const bool need_w = ka < I.m * kTcBM + t * 128 + 127 - p.window;
          mt = (need_mask || need_w) ? row_max2(v, qrow - p.window - ka, lim, sl2) : row_max<false>(v, lim, sl2);
        } else {
          mt = need_mask ? row_max<true>(v, lim, sl2) : row_max<false>(v, lim, sl2);
        }
        if (n == 0) {
          m_ref = mt;
        } else {
          const bool resc = mt > m_ref + kRescaleThreshold;
          if (__any_sync(0xffffffffu, resc)) {
            const float alpha = resc ? fast_exp2(m_ref - mt) : 1.f;
            if (resc) {
              m_ref = mt;
              lsum *= alpha;
            }
            ok = mbar_wait(bar(C::B_OF + t), (of_base + n - 1) & 1, abort_flag, p.hdr, 10);
            if (!__all_sync(0xffffffffu, ok)) {
              ok = false;
              break;
            }
            fence_after_sync();
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(o_addr + c * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
              tmem_st32(o_addr + c * 32, o);
            }
            tmem_wait_st();
          }
        }
        const float rs = row_exp(v, sl2, m_ref == -INFINITY ? 0.f : m_ref);
        tmem_st32(s_addr, v);  // P over the first 64 columns of S_t
        tmem_st32(s_addr + 32, v + 32);
        lsum += rs;
        tmem_wait_st();
        fence_before_sync();
        mbar_arrive(bar(C::B_PF + t));
      }
      if (!ok) break;
      // epilogue: O / l -> bf16 rows < l; lse
      ok = mbar_wait(bar(C::B_OF + t), (of_base + nbt - 1) & 1, abort_flag, p.hdr, 11);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      of_base += nbt;
      fence_after_sync();
      const float inv = 1.f / lsum;
      const bool store = qrow < I.l;
      bf16* orow = p.o + static_cast<int64_t>(I.s0 + qrow) * p.o_rs + static_cast<int64_t>(I.h) * p.o_hs;
      {
        uint32_t o[D];  // the whole row in one TMEM round trip
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32(o_addr + c * 32, o + c * 32);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < D / 2; ++j)
          o[j] = pack_bf16(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
        uint4 ov[D / 8];
#pragma unroll
        for (int j = 0; j < D / 8; ++j) ov[j] = make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
        store_rows_fast(ov, orow, p.o_rs, store);  // 32-byte stores measured faster here
      }
      if (store)
        p.lse[static_cast<int64_t>(I.h) * p.T + I.s0 + qrow] = (m_ref + __log2f(lsum)) * kLn2;
    }
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------- host side

template <int D, bool WIN, bool X>
static cudaError_t launch_d(const FwdParams& p, int cap, cudaStream_t st) {
  using C = TcCfg<D>;
  CUtensorMap tq, tk, tv;
  if (!tmap_rows(&tq, p.q, p.T, p.Hq, D, p.q_rs, p.q_hs, 128) ||
      !tmap_rows(&tk, p.k, X ? p.Tk : p.T, p.Hkv, D, p.k_rs, p.k_hs, 128) ||
      !tmap_rows(&tv, p.v, X ? p.Tk : p.T, p.Hkv, D, p.v_rs, p.v_hs, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel<D, WIN, X>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  // the in-kernel register split assumes the full launch budget; refuse rather than wait
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, fwd_tc_kernel<D, WIN, X>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = std::min(cap, std::max(sms, 1));
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(fwd_tc_kernel<D, WIN, X>, dim3(grid), dim3(kTcThreads), C::SMEM, st, tq, tk, tv, p);
}

cudaError_t launch_fwd_tc(const FwdParams& p, int d, int cap, cudaStream_t st) {
  if (p.cu_k) return d == 64 ? launch_d<64, false, true>(p, cap, st) : launch_d<128, false, true>(p, cap, st);
  if (p.window >= 0) return d == 64 ? launch_d<64, true, false>(p, cap, st) : launch_d<128, true, false>(p, cap, st);
  return d == 64 ? launch_d<64, false, false>(p, cap, st) : launch_d<128, false, false>(p, cap, st);
}

void fwd_tc_tiles(int* BM, int* BN) {
  *BM = kTcBM;
  *BN = kTcBN;
}

}  // namespace va
