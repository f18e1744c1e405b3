// Forward varlen attention for runs of short segments (token tiles), sm_103a: TMA +
// tcgen05 MMA (TMEM accumulators), warp-specialised, persistent.  Runs after the segment
// kernel (fwd_tc.cu) as its programmatic dependent, so its CTAs take SMs as the segment
// kernel's CTAs run out of work.
//
// What it computes: a run of segments of at most 64 tokens is cut by the planner into
// items of 256 consecutive tokens (q tile 0: rows 0..127, q tile 1: rows 128..255), each
// holding many segments.  Row i sees the keys [start of its segment, i] -- the permission
// rule of "Pack sequences without joining their contexts" ("Permission depends on the
// example": same segment, key not later than the query) in its range form ("What the
// permission symbols mean"); lse_i = ln sum_j exp(scale q_i.k_j) and o_i as in the segment
// kernel.  Key tiles of 128 rows start at the start of the segment holding the item's
// first row, so an item reads at most three.
//
// Layout and pipeline as in the segment kernel (warp 0 TMA producer, warp 1 MMA issuer,
// warps 4-11 softmax + epilogue for the two q tiles; TMEM S0 | S1 | O0 | O1), with three
// differences:
//   * the producer writes, with each record, a table row -> position in its segment
//     (shared memory, one byte per row) from the boundaries cu[f], cu[f+1], ...;
//   * every key tile is masked on both sides, per row;
//   * a row sees at most 64 keys, so a warp's 32 rows see at most 95 consecutive keys:
//     32-column chunks of S that no row of the warp sees are neither masked nor
//     exponentiated, and P = 0 is stored there directly.
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
  static constexpr int ROWS_OFF = QUEUE_OFF + 2 * 48;            // two 256-byte row tables
  static constexpr int MISC_OFF = ROWS_OFF + 2 * kTcBM;
  static constexpr int SMEM = MISC_OFF + 16 + 1024;    // + slack to align the base to 1024
  static constexpr int OCOLS = D;                      // TMEM columns of one O accumulator
};

// Token tiles hold segments of at most this many tokens: a row's position in its
// segment then fits the row table's byte, and an item reads at most three key tiles.
constexpr int kTokenShort = kTcBN / 2;
constexpr uint8_t kRowUnused = 0xff;  // row table entry of rows past the item's end
static_assert(kTokenShort < kRowUnused, "positions must fit a byte");

// One work item as the consumers see it: q rows [q0, q0 + rows) (tile t holds rows
// q0 + 128 t ...), key tiles from row kb, f the segment holding row q0.
struct Item {
  int q0, rows, kb, h, hk, nb, nb0;
  int t1, f, x0;  // x0: this producer lane's cu[f + lane] (fill_rows)
  int pad, valid;
};
static_assert(sizeof(Item) == 48, "queue slots are 48 bytes");

// Token record {-1 - f, t0, head, rows}; lane 0 of the producer warp loads cu[f]
// together with the boundaries after it (fill_rows).
__device__ __forceinline__ Item decode(const FwdParams& p, int idx) {
  const TileItem it = p.items[idx];
  Item r;
  r.h = it.head;
  r.hk = it.head / p.g;
  r.f = -1 - it.seg;
  r.q0 = it.blk;
  r.rows = it.count;
  const int lane = threadIdx.x & 31;
  r.x0 = r.f + lane <= p.B ? p.cu[r.f + lane] : INT_MAX;
  r.kb = __shfl_sync(0xffffffffu, r.x0, 0);
  r.nb = (r.q0 + r.rows - r.kb + kTcBN - 1) / kTcBN;
  r.t1 = r.rows > 128 ? 1 : 0;
  r.nb0 = r.t1 ? (r.q0 + 128 - r.kb + kTcBN - 1) / kTcBN : r.nb;
  r.pad = 0;
  return r;
}

// Row table of a token item (whole warp): entry r = position of row q0 + r in its
// segment, kRowUnused past the item's rows.  Segment starts inside the item are found
// 32 boundaries at a time (cu[f], cu[f + 1], ...; x0 = this lane's cu[f + lane], already
// loaded by decode) and kept as a 256-bit map.
__device__ __forceinline__ void fill_rows(const FwdParams& p, const Item& I, int x0, uint8_t* table) {
  const int lane = threadIdx.x & 31;
  uint32_t words[kTcBM / 32];
#pragma unroll
  for (int w = 0; w < kTcBM / 32; ++w) words[w] = 0;
  for (int b0 = I.f;; b0 += 32) {
    const int b = b0 + lane;
    const int x = b0 == I.f ? x0 : (b <= p.B ? p.cu[b] : INT_MAX);
    const int r = x - I.q0;  // <= 0 only for cu[f], which starts the rows before q0
    const bool in = b <= p.B && r > 0 && r < I.rows;
#pragma unroll
    for (int w = 0; w < kTcBM / 32; ++w)
      words[w] |= __reduce_or_sync(0xffffffffu, (in && (r >> 5) == w) ? 1u << (r & 31) : 0u);
    if (!__shfl_sync(0xffffffffu, b <= p.B && r < I.rows, 31)) break;  // last boundary read is past the item
  }
  int last = I.kb - I.q0;  // start of the segment holding the rows before word w (<= 0)
#pragma unroll
  for (int w = 0; w < kTcBM / 32; ++w) {
    const int row = w * 32 + lane;
    const uint32_t mine = words[w] & (0xffffffffu >> (31 - lane));
    const int st = mine ? w * 32 + 31 - __clz(mine) : last;
    table[row] = row < I.rows ? static_cast<uint8_t>(row - st) : kRowUnused;
    if (words[w]) last = w * 32 + 31 - __clz(words[w]);
  }
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

// Token rows see at most 64 keys, so most 32-column chunks of a key tile are invisible to
// every row of a warp.  Bit c of the result: some lane's visible range [lo, hi] meets
// columns [32c, 32c + 31].  Segment rows use all four chunks.
__device__ __forceinline__ uint32_t chunks_needed(int lo, int hi) {
  uint32_t need = 0;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    if (__any_sync(0xffffffffu, hi >= c * 32 && lo <= c * 32 + 31)) need |= 1u << c;
  return need;
}

// Row max x sl2 over the chunks in `need` (warp-uniform), columns outside [lo, lim] set to
// -inf first.
__device__ __forceinline__ float row_max(uint32_t* v, uint32_t need, int lo, int lim, float sl2) {
  float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (!(need & (1u << c))) continue;
#pragma unroll
    for (int j = c * 32; j < c * 32 + 32; ++j)
      if (j > lim || j < lo) v[j] = __float_as_uint(-INFINITY);
#pragma unroll
    for (int j = c * 32; j < c * 32 + 32; j += 8) {
      m0 = fmax3(m0, __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
      m1 = fmax3(m1, __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
      m2 = fmax3(m2, __uint_as_float(v[j + 4]), __uint_as_float(v[j + 5]));
      m3 = fmax3(m3, __uint_as_float(v[j + 6]), __uint_as_float(v[j + 7]));
    }
  }
  return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3)) * sl2;
}

// p = exp2(s * sl2 - mu) packed in place as bf16 pairs into v[0..63] for the chunks in
// `need` (the others are left as they are: p_store writes zeros there); returns the row
// sum.  Chunks go in ascending order: chunk c's packed words v[16c .. 16c+15] overwrite
// only inputs of chunks <= c, already consumed.
__device__ __forceinline__ float row_exp(uint32_t* v, uint32_t need, float sl2, float mu) {
  float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    if (need & (1u << c)) {
#pragma unroll
      for (int j = c * 16; j < c * 16 + 16; ++j) {
        float x0, x1;
        ffma2(x0, x1, __uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]), sl2, sl2, -mu, -mu);
        const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
        if (j & 1) fadd2(b0, b1, b0, b1, p0, p1);
        else fadd2(a0, a1, a0, a1, p0, p1);
        v[j] = pack_bf16(p0, p1);
      }
    }
  }
  return (a0 + a1) + (b0 + b1);
}

// Stores P (64 packed columns) over the first half of S: the chunks in `need` from v,
// zeros for the others.
__device__ __forceinline__ void p_store(uint32_t s_addr, const uint32_t* v, uint32_t need) {
  if (need == 0xfu) {
    tmem_st32(s_addr, v);
    tmem_st32(s_addr + 32, v + 32);
  } else {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (need & (1u << c)) tmem_st16(s_addr + 16 * c, v + 16 * c);
      else tmem_st16_zero(s_addr + 16 * c);
    }
  }
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    fwd_tok_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const FwdParams p) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* sm = smem_raw + (base - raw);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::MISC_OFF + 4);
  Item* queue = reinterpret_cast<Item*>(sm + C::QUEUE_OFF);
  uint8_t* row_tables = sm + C::ROWS_OFF;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) -> uint32_t { return base + C::BAR_OFF + 8u * i; };
  // Launched as the segment kernel's programmatic dependent: that kernel lets it start
  // only after its own wait on the planning launch, whose results (status, map, counts)
  // are therefore complete, and the two grids write disjoint rows.  Each CTA waits for the
  // segment kernel only before it exits, so that this grid completes after it: the next
  // launch, which waits on this grid alone, then sees both grids' output.
  griddep_launch_dependents();
  const int n_items = p.hdr->status == VA_OK ? p.hdr->n_items[kTokSlot] : 0;  // token records
  const int first = p.hdr->n_items[p.slot] - n_items;                          // follow segment ones
  if (static_cast<int>(blockIdx.x) >= n_items) {
    griddep_wait();
    return;
  }

  // Publishes this CTA's k-th item (whole producer warp): the decoded record and, for a
  // token item, its row table; every lane arrives on the slot's full barrier after its
  // own writes.  Returns false at the end of the list or on abort (ok = false).
  auto publish = [&](int k, Item& out, bool& ok) -> bool {
    const int s = k & 1;
    ok = wwait(bar(C::B_IE + s), ((k >> 1) & 1) ^ 1, abort_flag, p.hdr, 40);
    if (!ok) return false;
    int idx = 0;
    if (lane == 0) idx = atomicAdd(p.counter, 1);
    idx = __shfl_sync(0xffffffffu, idx, 0);
    if (idx < n_items) {
      out = decode(p, first + idx);
      out.valid = 1;
      fill_rows(p, out, out.x0, row_tables + s * kTcBM);
    } else {
      out = Item{};
      out.valid = 0;
    }
    if (lane == 0) queue[s] = out;
    mbar_arrive(bar(C::B_IF + s));
    return out.valid != 0;
  };


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
      mbar_init(bar(C::B_IF + b), 32);        // every producer lane (row tables)
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
      bool more = publish(0, nxt, ok);
      // The next record is published once this item's Q tiles and first K/V tiles are
      // issued: its decode then overlaps this item's first MMAs instead of delaying them.
      constexpr int kPairsBeforePublish = C::NST / 2;
      for (; ok && more; ++item_cnt) {
        const Item I = nxt;
        // Q tile t is released by the item's last S_t MMA (tile 0 one key tile before tile 1)
        for (int t = 0; ok && t < (I.t1 ? 2 : 1); ++t) {
          ok = wwait(bar(C::B_QE + t), (qcnt[t] & 1) ^ 1, abort_flag, p.hdr, 1);
          if (!ok) break;
          mbar_expect_tx_w(bar(C::B_QF + t), C::TILE);
          for (int pn = 0; pn < D / 64; ++pn)
            tma_load_3d_w(base + C::Q_OFF + t * C::TILE + pn * C::PANEL, &tq, bar(C::B_QF + t), pn * 64,
                        I.h, I.q0 + t * 128);
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
                          bar(C::B_KVF + s), pn * 64, I.hk, I.kb + n * kTcBN);
            ++kv_it;
          }
          if (ok && n + 1 == min(I.nb, kPairsBeforePublish)) more = publish(item_cnt + 1, nxt, ok);
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
      int pos = 0;  // token items: this row's position in its segment (kRowUnused: no row)
      {
        const int s = k & 1;
        ok = mbar_wait(bar(C::B_IF + s), (k >> 1) & 1, abort_flag, p.hdr, 41);
        if (ok) {
          I = queue[s];
          pos = row_tables[s * kTcBM + t * 128 + r];
          mbar_arrive(bar(C::B_IE + s));
        }
      }
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      if (!I.valid) break;
      if (t == 1 && !I.t1) continue;
      const int nbt = t == 0 ? I.nb0 : I.nb;
      const int qrow = t * 128 + r;                  // row within the item
      const int qrel = I.q0 + qrow - I.kb;           // row relative to the first key
      // visible keys relative to kb: [lo0, hi0], the row's own segment up to itself
      const int hi0 = qrel;
      const int lo0 = pos == kRowUnused ? INT_MAX / 2 : qrel - pos;
      float m_ref = -INFINITY, lsum = 0.f;
      for (int n = 0; n < nbt; ++n) {
        ok = mbar_wait(bar(C::B_SF + t), sf & 1, abort_flag, p.hdr, 9);
        if (!__all_sync(0xffffffffu, ok)) {  // TMEM loads below are warp-collective
          ok = false;
          break;
        }
        ++sf;
        fence_after_sync();
        const int lim = hi0 - n * kTcBN, lim_lo = lo0 - n * kTcBN;  // keep lim_lo <= j <= lim
        // One TMEM round trip per tile: the row into registers, its max, then
        // p = exp2(s * sl2 - m_ref) packed in place and stored over the first half of S_t.
        // The reference max m_ref is raised only when the row max grew by more than 2^8
        // (rare); O_t, which holds PV_{n-1}, is then rescaled in TMEM first.
        uint32_t v[128];
        float mt;
        row_load(s_addr, v);
        const uint32_t need = chunks_needed(lim_lo, lim);
        mt = row_max(v, need, lim_lo, lim, sl2);
        if (n == 0) {
          m_ref = mt;
        } else {
          // A row with nothing visible so far (a token row whose segment starts in a later
          // key tile) had p = exp2(-inf) = 0 everywhere: its O_t and lsum are exactly zero
          // and take the new max without a rescale.
          const bool fresh = m_ref == -INFINITY;
          if (fresh) m_ref = mt;
          const bool resc = !fresh && mt > m_ref + kRescaleThreshold;
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
        const float mu = m_ref == -INFINITY ? 0.f : m_ref;
        const float rs = row_exp(v, need, sl2, mu);
        p_store(s_addr, v, need);  // P over the first 64 columns of S_t
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
      const bool store = qrow < I.rows;
      bf16* orow = p.o + static_cast<int64_t>(I.q0 + qrow) * p.o_rs + static_cast<int64_t>(I.h) * p.o_hs;
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
        p.lse[static_cast<int64_t>(I.h) * p.T + I.q0 + qrow] = (m_ref + __log2f(lsum)) * kLn2;
    }
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
  griddep_wait();
}

// ---------------------------------------------------------------- host side

template <int D>
static cudaError_t launch_d(const FwdParams& p, int cap, cudaStream_t st) {
  using C = TcCfg<D>;
  CUtensorMap tq, tk, tv;
  if (!tmap_rows(&tq, p.q, p.T, p.Hq, D, p.q_rs, p.q_hs, 128) ||
      !tmap_rows(&tk, p.k, p.T, p.Hkv, D, p.k_rs, p.k_hs, 128) ||
      !tmap_rows(&tv, p.v, p.T, p.Hkv, D, p.v_rs, p.v_hs, 128))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fwd_tok_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  // the in-kernel register split assumes the full launch budget; refuse rather than wait
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, fwd_tok_kernel<D>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs < kLaunchRegs) return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = std::min(cap, std::max(sms, 1));
  if (grid <= 0) return cudaSuccess;
  return launch_pdl(fwd_tok_kernel<D>, dim3(grid), dim3(kTcThreads), C::SMEM, st, tq, tk, tv, p);
}

cudaError_t launch_fwd_tok(const FwdParams& p, int d, int cap, cudaStream_t st) {
  return d == 64 ? launch_d<64>(p, cap, st) : launch_d<128>(p, cap, st);
}

int fwd_tc_token_short() { return kTokenShort; }

}  // namespace va
