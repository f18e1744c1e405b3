// Segment-aware tile scheduler, device side: the planning bodies shared by the
// planning kernels and the backward preparation kernel (which plans in one CTA while the
// others compute D = rowsum(dO * O)).
//
// Segment-aware tile scheduler: builds the work list the attention kernels walk.
//
// "Packing与 FlashAttention Varlen", section 5: a q block m of segment b exists only
// while m*BM < l_b, and its key blocks stop at ceil(min(l_b, (m+1)*BM) / BN) under
// causality (ceil(l_b/BN) otherwise).  Instead of launching max_seqlen-shaped grids
// whose CTAs exit early, the list holds only blocks that have work.
//
// Order (this library's reading; the page fixes none): records that read the same
// K/V tiles are adjacent, so the attention kernels -- which pull records in list
// order from an atomic counter -- run them at the same time and share those tiles
// through L2; longer work goes first:
//   key = (-class_b, b, head, -count, block),  class_b = floor(log2(C_b)),
// with C_b the segment's total tile count (key tiles summed over its q blocks for
// the forward/dQ maps, q blocks summed over its kv blocks for the dK/dV map).
//
// One CTA (any multiple of 32 threads, at most 1024), of which the first
// min(CTA, B rounded up to 32) rank: per-class record totals (warp match + reduce), the
// classes' first records, then rounds of one segment per thread in which a warp-level
// prefix over the warp's segments of the same class and one scan over the warps per class
// place each segment's first record; each thread writes its segment's records (whole warps
// take segments with many).  The depth per round is fixed, so the planner's latency does
// not grow with the number of classes.  Tile sizes are powers of two (block counts are
// shifts).
//
// Token tiles (causal, short_len > 0): segments of at most short_len tokens get no segment
// records.  Each maximal run [r0, r1) of consecutive short segments is cut into tiles of
// R rows starting at r0 (R = BM, q rows, for the forward and dQ maps; R = BN, key rows, for
// the dK/dV map), and each tile gets one record per head,
//   {seg = -1 - f, blk = t0, head, count = rows = min(R, r1 - t0)},
// f being the segment that holds row t0.  Query i of a run sees keys [start of its segment,
// i] -- the permission rule of "Pack sequences without joining their contexts" ("Permission
// depends on the example") in its range form; key j is seen by the queries [j, end of its
// segment).  Token records follow all segment records, ordered by (t0, head).  Runs are found with block-wide scans over contiguous chunks of
// segments per thread: the last long segment before a chunk (max scan), the first long
// segment after it (min scan from the end), then the tile counts (sum scan).
#pragma once
#include "common.cuh"

namespace va {

namespace plan_detail {

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ceil(a / b) and a / b for b a power of two
__device__ __forceinline__ int ceil_p2(int a, int b) { return (a + b - 1) >> (__ffs(b) - 1); }
__device__ __forceinline__ int div_p2(int a, int b) { return a >> (__ffs(b) - 1); }

__device__ __forceinline__ bool token_mode(const PlanArgs& a) { return a.causal && a.short_len > 0; }

// What a map build is, fixed at compile time: the planner's time is mostly fetching its
// own instructions (it runs once per call, on one SM), so each kind of map gets its own
// compact code path.  KV: kv-block map (kind 1), else q-block map (kinds 0 and 2).
// WIN: causal local window a.window (query i sees keys i-w..i): a q block m's key blocks
// start at floor(max(0, m*BM - w) / BN); a kv block n's q blocks stop after
// floor((n*BN + BN - 1 + w) / BM) ("Packing与 FlashAttention Varlen", section 5: the local
// window narrows n_block_min/max).
// X: cross-attention (a.cu_k): a segment has lq queries and lk keys, the causal bound is
// aligned bottom-right (key j visible to query i when j <= i + lk - lq): q block m has
// ceil(min(lk, (m+1)*BM + lk - lq) / BN) key blocks, kv block n its q blocks from
// floor(max(0, n*BN - (lk - lq)) / BM) ("Packing与 FlashAttention Varlen", section 5).
template <bool KV, bool CAUSAL, bool TOKENS, bool WIN = false, bool X = false>
struct MapKind {
  static constexpr bool kv = KV, causal = CAUSAL, tokens = TOKENS, win = WIN, x = X;
};

// Cross-attention record count of q block m (q-block maps) or kv block n (kv-block maps).
template <class M>
__device__ __forceinline__ int x_count(const PlanArgs& a, int lq, int lk, int blk) {
  if (!M::kv) return M::causal ? ceil_p2(min(lk, (blk + 1) * a.BM + lk - lq), a.BN) : ceil_p2(lk, a.BN);
  return ceil_p2(lq, a.BM) - (M::causal ? div_p2(max(0, blk * a.BN - (lk - lq)), a.BM) : 0);
}

// Windowed record count of q block m (q-block maps) or kv block n (kv-block maps).
template <class M>
__device__ __forceinline__ int win_count(const PlanArgs& a, int l, int blk) {
  if (!M::kv) {
    const int nmax = ceil_p2(min(l, (blk + 1) * a.BM), a.BN);
    return nmax - div_p2(max(0, blk * a.BM - a.window), a.BN);
  }
  const int Mq = ceil_p2(l, a.BM);
  return min(Mq, div_p2(blk * a.BN + a.BN - 1 + a.window, a.BM) + 1) - div_p2(blk * a.BN, a.BM);
}

// Blocks of a segment of length l (lk keys under cross-attention) and its total tile count
// (none for token-tiled segments).
template <class M>
__device__ __forceinline__ void seg_cost(const PlanArgs& a, int l, int lk, int& nblk, int& cost) {
  if (M::x) {
    nblk = M::kv ? ceil_p2(lk, a.BN) : ceil_p2(l, a.BM);
    cost = 0;
    for (int b = 0; b < nblk; ++b) cost += x_count<M>(a, l, lk, b);
  } else if (M::tokens && l <= a.short_len) {
    nblk = 0;
    cost = 0;
  } else if (M::win) {  // no closed form worth keeping: sum the blocks (one thread per segment)
    nblk = M::kv ? ceil_p2(l, a.BN) : ceil_p2(l, a.BM);
    cost = 0;
    for (int b = 0; b < nblk; ++b) cost += win_count<M>(a, l, b);
  } else if (!M::kv) {
    const int M_ = ceil_p2(l, a.BM), Lk = ceil_p2(l, a.BN);
    nblk = M_;
    cost = M::causal ? div_p2(a.BM, a.BN) * (M_ - 1) * M_ / 2 + Lk : M_ * Lk;
  } else {
    const int N = ceil_p2(l, a.BN), Mq = ceil_p2(l, a.BM);
    nblk = N;
    cost = M::causal ? N * Mq - div_p2(a.BN, a.BM) * N * (N - 1) / 2 : N * Mq;
  }
}

// The j-th record of one (segment, head): most tiles first.
template <class M>
__device__ __forceinline__ void seg_record(const PlanArgs& a, int l, int lk, int nblk, int j, int& blk, int& count) {
  if (M::x) {  // the no-cross orders: q blocks last-first (causal), kv blocks first-first
    blk = (M::kv || !M::causal) ? j : nblk - 1 - j;
    count = x_count<M>(a, l, lk, blk);
  } else if (M::win) {  // q blocks last-first, kv blocks first-first: the no-window orders
    blk = M::kv ? j : nblk - 1 - j;
    count = win_count<M>(a, l, blk);
  } else if (!M::kv) {
    const int Lk = ceil_p2(l, a.BN);
    blk = M::causal ? nblk - 1 - j : j;
    count = M::causal ? min(Lk, div_p2(a.BM, a.BN) * (blk + 1)) : Lk;
  } else {
    const int Mq = ceil_p2(l, a.BM);
    blk = j;
    count = M::causal ? Mq - div_p2(j * a.BN, a.BM) : Mq;
  }
}

__device__ __forceinline__ int cost_class(int c) { return 31 - __clz(max(c, 1)); }

enum ScanOp { kScanSum, kScanMax, kScanMin };

template <int OP>
__device__ __forceinline__ int scan_op(int x, int y) {
  return OP == kScanSum ? x + y : (OP == kScanMax ? max(x, y) : min(x, y));
}

// Barrier among the first n threads of the block (n a multiple of 32): the planner runs on
// as many warps as there are segments to spread, the others skip it.
__device__ __forceinline__ void plan_sync(int n) { asm volatile("bar.sync 1, %0;" ::"r"(n) : "memory"); }

// Exclusive scan of one value per thread over the first nth threads, in thread order or
// (REV) from the last one down; `ident` is the operator's identity, *total the result
// over all of them.  Each of those threads calls it; tmp is 33 ints of shared memory.
template <int OP, bool REV>
__device__ int block_scan_excl(int x, int ident, int nth, int* tmp, int* total) {
  const int nw = nth >> 5;
  const int lane = REV ? 31 - (threadIdx.x & 31) : (threadIdx.x & 31);
  const int warp = REV ? nw - 1 - static_cast<int>(threadIdx.x >> 5) : static_cast<int>(threadIdx.x >> 5);
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = REV ? __shfl_down_sync(0xffffffffu, incl, o) : __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl = scan_op<OP>(incl, y);
  }
  int excl = REV ? __shfl_down_sync(0xffffffffu, incl, 1) : __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = ident;
  if (nw == 1) {  // one warp: no shared memory, no block barrier
    __syncwarp();   // (but order the lanes' shared-memory accesses around the scan)
    *total = __shfl_sync(0xffffffffu, incl, REV ? 0 : 31);
    return excl;
  }
  plan_sync(nth);  // tmp may still be read by an earlier scan
  if (lane == 31) tmp[warp] = incl;
  plan_sync(nth);
  if (threadIdx.x < 32) {  // scan of the warp totals, in logical warp order
    const int i = threadIdx.x;
    int w = i < nw ? tmp[i] : ident;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (i >= o) w = scan_op<OP>(w, y);
    }
    int we = __shfl_up_sync(0xffffffffu, w, 1);
    if (i == 0) we = ident;
    __syncwarp();
    if (i < nw) tmp[i] = we;
    if (i == 31) tmp[32] = w;
  }
  plan_sync(nth);
  *total = tmp[32];
  return scan_op<OP>(tmp[warp], excl);
}

// Per-thread state of the token-tile pass: the thread's chunk of segments [lo, hi), the
// last long segment before it, the first long segment after it, its tile count and the
// index of its first tile.
struct TokenChunk {
  int lo, hi, ns_before, ns_after, first_tile, n_tiles;
};

__device__ __forceinline__ TokenChunk token_scan(const PlanArgs& a, const int* cu, int tile, int lo, int hi,
                                                 int nth, int* tmp, int* n_tiles_total) {
  TokenChunk c;
  c.lo = lo;
  c.hi = hi;
  int last_ns = -1, first_ns = a.B;
  for (int b = c.lo; b < c.hi; ++b)
    if (cu[b + 1] - cu[b] > a.short_len) {
      if (first_ns == a.B) first_ns = b;
      last_ns = b;
    }
  int dummy;
  c.ns_before = block_scan_excl<kScanMax, false>(last_ns, -1, nth, tmp, &dummy);
  c.ns_after = block_scan_excl<kScanMin, true>(first_ns, a.B, nth, tmp, &dummy);
  int cnt = 0, ns = c.ns_before;
  for (int b = c.lo; b < c.hi; ++b) {
    const int x = cu[b], y = cu[b + 1];
    if (y - x > a.short_len) {
      ns = b;
    } else {
      const int rs = cu[ns + 1];  // start of this segment's run
      cnt += ceil_p2(y - rs, tile) - ceil_p2(x - rs, tile);
    }
  }
  c.n_tiles = cnt;
  c.first_tile = block_scan_excl<kScanSum, false>(cnt, 0, nth, tmp, n_tiles_total);
  return c;
}

// Writes the token records of one chunk, from record index base; tiles of `tile` rows.
__device__ __forceinline__ void token_records(const PlanArgs& a, const int* cu, int tile, const TokenChunk& c,
                                              int base) {
  int ns = c.ns_before, g = c.first_tile;
  for (int b = c.lo; b < c.hi; ++b) {
    const int x = cu[b], y = cu[b + 1];
    if (y - x > a.short_len) {
      ns = b;
      continue;
    }
    const int rs = cu[ns + 1];
    const int k0 = ceil_p2(x - rs, tile), k1 = ceil_p2(y - rs, tile);
    if (k1 <= k0) continue;
    int nx = b + 1;  // first long segment after b: its start ends the run
    while (nx < c.hi && cu[nx + 1] - cu[nx] <= a.short_len) ++nx;
    const int re = cu[nx < c.hi ? nx : c.ns_after];
    for (int k = k0; k < k1; ++k, ++g) {
      const int t0 = rs + k * tile;
      for (int h = 0; h < a.heads; ++h) {
        TileItem t;
        t.seg = -1 - b;
        t.blk = t0;
        t.head = h;
        t.count = min(tile, re - t0);
        const int at = base + g * a.heads + h;
        if (at >= 0 && at < a.capacity) a.out[at] = t;  // boundaries that break the contract
                                                        // must not write outside the map
      }
    }
  }
}

}  // namespace plan_detail
using namespace plan_detail;

constexpr int kPlanThreads = 1024;

// Up to this many segments the boundaries and per-segment offsets live in shared memory
// (one coalesced read of cu_seqlens per launch); beyond it they are read from and kept in
// global memory.
constexpr int kSmemSegs = 4096;

constexpr int kNoClass = 32;  // class of a segment without records

// The small-map path's table: the segments in map order (class descending, then index).
struct SmallPlanTable {
  int seg[32], off[33], nblk[32], len[32];
};

struct PlanSmem {
  SmallPlanTable small;
  int scan[33];
  int overflow;
  int seg_total;
  int cls_total[32];  // records per cost class
  int cls_base[32];   // first record of each class (largest class first)
  int cls_run[32];    // records of the class placed by earlier rounds
  int wtot[32][33];   // per warp and class: records of the round, then the warp's first record
  int cu[kSmemSegs + 1];
  int off[kSmemSegs];
};

// Writes records of segments [g0, g0 + 32) with the whole warp, 32 records per pass: lane i
// of a pass takes record r of the group's concatenated records and finds its segment by a
// binary search over the lanes' inclusive record counts.  k warps share a group; this one
// takes passes s, s + k, ...
template <class M>
__device__ __forceinline__ void write_group(const PlanArgs& a, const int* cu, const int* seg_off, int g0, int s,
                                            int k) {
  const int lane = threadIdx.x & 31, b = g0 + lane;
  int l = 0, lk = 0, nblk = 0, n = 0, off = 0;
  if (b < a.B) {
    int cost;
    l = cu[b + 1] - cu[b];
    lk = M::x ? a.cu_k[b + 1] - a.cu_k[b] : l;
    seg_cost<M>(a, l, lk, nblk, cost);
    n = nblk * a.heads;
    if (n > 0) off = seg_off[b];
  }
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  for (int r0 = s * 32; r0 < total; r0 += k * 32) {
    const int r = r0 + lane;
    int sgi = 0;  // first lane whose inclusive count exceeds r
#pragma unroll
    for (int step = 16; step > 0; step >>= 1)
      if (__shfl_sync(0xffffffffu, incl, sgi + step - 1) <= r) sgi += step;
    const int sl = __shfl_sync(0xffffffffu, l, sgi), snb = __shfl_sync(0xffffffffu, nblk, sgi);
    const int slk = __shfl_sync(0xffffffffu, lk, sgi);
    const int soff = __shfl_sync(0xffffffffu, off, sgi);
    const int sbeg = __shfl_sync(0xffffffffu, incl - n, sgi);
    if (r < total) {
      const int rr = r - sbeg, h = rr / snb, j = rr - h * snb;
      TileItem t;
      seg_record<M>(a, sl, slk, snb, j, t.blk, t.count);
      t.seg = g0 + sgi;
      t.head = h;
      if (soff + rr >= 0 && soff + rr < a.capacity) a.out[soff + rr] = t;  // boundaries that break
                                                                           // the contract must not
                                                                           // write outside the map
    }
  }
}

// Class and record count of segment b (kNoClass / 0 past the end or without records).
template <class M>
__device__ __forceinline__ void seg_class(const PlanArgs& a, const int* cu, int b, int& c, int& n, int& l,
                                          int& nblk) {
  c = kNoClass;
  n = 0;
  l = 0;
  nblk = 0;
  if (b < a.B) {
    int cost;
    l = cu[b + 1] - cu[b];
    seg_cost<M>(a, l, M::x ? a.cu_k[b + 1] - a.cu_k[b] : l, nblk, cost);
    if (nblk > 0) {
      c = cost_class(cost);
      n = nblk * a.heads;
    }
  }
}

// The ranking part of plan_body, on the first nth threads: class totals, class bases, then
// rounds of nth segments (segment b = round * nth + thread, so segment order is kept within
// a class): a warp-level prefix among the warp's segments of the same class and one scan
// over the warps per class present give each segment's first record (seg_off).
template <class M>
__device__ __forceinline__ void rank_and_write(const PlanArgs& a, PlanSmem& sh, const int* cu, int* seg_off,
                                               int nth) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = nth >> 5;
  if (tid < 32) {
    sh.cls_total[tid] = 0;
    sh.cls_run[tid] = 0;
  }
  plan_sync(nth);
  for (int b0 = 0; b0 < a.B; b0 += nth) {  // class totals
    int c, n, l, nblk;
    seg_class<M>(a, cu, b0 + tid, c, n, l, nblk);
    const unsigned peers = __match_any_sync(0xffffffffu, c);
    const int sum = static_cast<int>(__reduce_add_sync(peers, static_cast<unsigned>(n)));
    if (c != kNoClass && lane == __ffs(peers) - 1) atomicAdd(&sh.cls_total[c], sum);
  }
  int n_tiles = 0;
  TokenChunk tc{};
  if (M::tokens) {
    const int per = ceil_div(a.B, nth);
    const int lo = min(a.B, tid * per), hi = min(a.B, lo + per);
    tc = token_scan(a, cu, M::kv ? a.BN : a.BM, lo, hi, nth, sh.scan, &n_tiles);
  }
  plan_sync(nth);
  if (tid < 32) {  // class bases, largest class first
    const int k = 31 - lane, v = sh.cls_total[k];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    sh.cls_base[k] = incl - v;
    if (lane == 31) sh.seg_total = incl;
  }
  plan_sync(nth);
  const int run = sh.seg_total;
  const int total = run + n_tiles * a.heads;  // token records follow the segment records
  const bool overflow = total > a.capacity;   // uniform over the nth threads
  if (tid == 0) {
    *a.n_items = overflow ? 0 : total;
    *a.counter = 0;
    if (a.n_tok) *a.n_tok = overflow ? 0 : n_tiles * a.heads;
    if (a.tok_counter) *a.tok_counter = 0;
    sh.overflow = overflow;
    if (overflow && a.status) atomicCAS(a.status, VA_OK, VA_ERR_WORKSPACE);
  }
  if (overflow) return;
  unsigned present = 0;
  for (int k = 0; k < 32; ++k) present |= sh.cls_total[k] > 0 ? 1u << k : 0u;
  for (int b0 = 0; b0 < a.B; b0 += nth) {
    const int b = b0 + tid;
    int c, n, l, nblk;
    seg_class<M>(a, cu, b, c, n, l, nblk);
    // inclusive prefix of n over the warp's lanes of the same class, one scan per class
    int incl = 0;
    for (unsigned todo = __ballot_sync(0xffffffffu, c != kNoClass); todo;) {
      const int cc = __shfl_sync(0xffffffffu, c, __ffs(todo) - 1);
      int x = c == cc ? n : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (c == cc) incl = x;
      todo &= ~__ballot_sync(0xffffffffu, c == cc);
    }
    if (nw == 1) {  // one warp, one round: the warp's part of a class starts at the class
      if (n > 0) seg_off[b] = sh.cls_base[c] + incl - n;
      continue;
    }
    sh.wtot[warp][lane] = 0;
    __syncwarp();
    const unsigned peers = __match_any_sync(0xffffffffu, c);
    if (c != kNoClass && lane == 31 - __clz(peers)) sh.wtot[warp][c] = incl;  // the class's last lane
    plan_sync(nth);
    for (int k = warp; k < 32; k += nw) {  // first record of each warp's part of class k
      if (!((present >> k) & 1)) continue;
      const int v = lane < nw ? sh.wtot[lane][k] : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const int base = sh.cls_base[k] + sh.cls_run[k];
      __syncwarp();
      if (lane < nw) sh.wtot[lane][k] = base + x - v;
      if (lane == 31) sh.cls_run[k] += x;
      __syncwarp();
    }
    plan_sync(nth);
    if (n > 0) seg_off[b] = sh.wtot[warp][c] + incl - n;
    plan_sync(nth);  // wtot is reused by the next round
  }
  if (M::tokens) token_records(a, cu, M::kv ? a.BN : a.BM, tc, run);
}

// Builds one map.  Every thread of the block (a multiple of 32, at most 1024) calls it.
// The first nth = min(block, B rounded up to 32) threads rank the segments (and write the
// token records); then every warp of the block writes segment records, 32 segments at a
// time.
// cu: the boundaries (the shared-memory copy or a.cu); seg_off: where the per-segment
// offsets go.
template <class M>
__device__ __forceinline__ void plan_body_m(const PlanArgs& a, PlanSmem& sh, const int* cu, int* seg_off) {
  const int nth = min(static_cast<int>(blockDim.x), max(32, (a.B + 31) & ~31));
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  if (static_cast<int>(threadIdx.x) < nth) rank_and_write<M>(a, sh, cu, seg_off, nth);
  __syncthreads();
  if (!sh.overflow) {
    const int ngroups = (a.B + 31) >> 5;
    if (ngroups >= nwarps) {
      for (int g = warp; g < ngroups; g += nwarps) write_group<M>(a, cu, seg_off, g * 32, 0, 1);
    } else {  // fewer groups than warps: k warps per group
      const int k = nwarps / ngroups;
      if (warp < ngroups * k) write_group<M>(a, cu, seg_off, (warp % ngroups) * 32, warp / ngroups, k);
    }
  }
  __syncthreads();  // shared memory is reused by the next map
}

__device__ __forceinline__ void plan_body(const PlanArgs& a, PlanSmem& sh, const int* cu, int* seg_off) {
  if (a.cu_k) {
    if (a.kind == 1) {
      if (a.causal) plan_body_m<MapKind<true, true, false, false, true>>(a, sh, cu, seg_off);
      else plan_body_m<MapKind<true, false, false, false, true>>(a, sh, cu, seg_off);
    } else {
      if (a.causal) plan_body_m<MapKind<false, true, false, false, true>>(a, sh, cu, seg_off);
      else plan_body_m<MapKind<false, false, false, false, true>>(a, sh, cu, seg_off);
    }
    return;
  }
  if (a.causal && a.window >= 0) {
    if (a.kind == 1) plan_body_m<MapKind<true, true, false, true>>(a, sh, cu, seg_off);
    else plan_body_m<MapKind<false, true, false, true>>(a, sh, cu, seg_off);
    return;
  }
  if (a.kind == 1) {
    if (!a.causal) plan_body_m<MapKind<true, false, false>>(a, sh, cu, seg_off);
    else if (token_mode(a)) plan_body_m<MapKind<true, true, true>>(a, sh, cu, seg_off);
    else plan_body_m<MapKind<true, true, false>>(a, sh, cu, seg_off);
  } else if (a.causal) {
    if (token_mode(a)) plan_body_m<MapKind<false, true, true>>(a, sh, cu, seg_off);
    else plan_body_m<MapKind<false, true, false>>(a, sh, cu, seg_off);
  } else {
    plan_body_m<MapKind<false, false, false>>(a, sh, cu, seg_off);
  }
}

struct PlanPair {
  PlanArgs map[2];
  int nmaps;
  int T, max_seqlen;
  int Tk = 0, max_seqlen_k = 0;  // cross-attention (map[0].cu_k set): the K/V stream
};

// Maps of at most 32 segments without token tiles, local window or cross-attention: the
// same records in the same order as plan_body, from a far shorter instruction path.  A
// planning launch runs once per call on cold instruction caches, so its time goes mostly to
// fetching instructions; the general path's ranking (class totals, bases, per-class scans)
// took about 6 us of it on a 10-segment pack.  Here warp 0 checks the boundaries and ranks
// the segments in registers (lane b holds segment b; its key is (31 - class, b), its first
// record the sum of the records of the segments with smaller keys), and the block writes
// the records, one per thread and pass.
__device__ __forceinline__ bool small_plan_ok(const PlanPair& pp, int i0, int i1) {
  if (pp.map[0].B < 1 || pp.map[0].B > 32) return false;
  for (int i = i0; i < i1; ++i) {
    const PlanArgs& a = pp.map[i];
    if (a.cu_k || (a.causal && a.window >= 0) || token_mode(a)) return false;
  }
  return true;
}

template <class M>
__device__ __forceinline__ void small_rank(const PlanArgs& a, int lane, int l, SmallPlanTable& t, int& total) {
  int nblk = 0, cost = 0;
  if (lane < a.B) seg_cost<M>(a, l, l, nblk, cost);
  const int n = nblk * a.heads;
  const unsigned key = lane < a.B ? (static_cast<unsigned>(31 - cost_class(cost)) << 5) | lane : 0xffffffffu;
  int rank = 0, off = 0;
#pragma unroll 4
  for (int j = 0; j < 32; ++j) {
    const unsigned kj = __shfl_sync(0xffffffffu, key, j);
    const int nj = __shfl_sync(0xffffffffu, n, j);
    if (kj < key) {
      ++rank;
      off += nj;
    }
  }
  total = static_cast<int>(__reduce_add_sync(0xffffffffu, static_cast<unsigned>(n)));
  if (lane < a.B) {
    t.seg[rank] = lane;
    t.off[rank] = off;
    t.nblk[rank] = nblk;
    t.len[rank] = l;
  }
  if (lane == 0) t.off[a.B] = total;
}

template <class M>
__device__ __forceinline__ void small_write(const PlanArgs& a, const SmallPlanTable& t, int total) {
  for (int r = threadIdx.x; r < total; r += blockDim.x) {
    int k = 0;  // the segment (in map order) that holds record r
#pragma unroll
    for (int step = 16; step > 0; step >>= 1)
      if (k + step < a.B && t.off[k + step] <= r) k += step;
    const int rr = r - t.off[k], nb = t.nblk[k], h = rr / nb, j = rr - h * nb;
    TileItem it;
    seg_record<M>(a, t.len[k], t.len[k], nb, j, it.blk, it.count);
    it.seg = t.seg[k];
    it.head = h;
    a.out[r] = it;
  }
}

// Every thread of the block calls it.  Shared state: sh.small (the table), sh.overflow (the
// boundary check's verdict) and sh.seg_total (the current map's record count).
__device__ __forceinline__ void small_plan(const PlanPair& pp, PlanSmem& sh, int i0, int i1) {
  const PlanArgs& a0 = pp.map[0];
  const int lane = threadIdx.x & 31;
  int l = 0, bad = 0;
  if (threadIdx.x < 32) {
    int x = 0, y = 0;
    if (lane < a0.B) {
      x = a0.cu[lane];
      y = a0.cu[lane + 1];
      l = y - x;
      if (y <= x || l > pp.max_seqlen) bad = 1;
      if (lane == 0 && x != 0) bad = 1;
      if (lane == a0.B - 1 && y != pp.T) bad = 1;
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) sh.overflow = bad;
  }
  __syncthreads();
  if (sh.overflow) {  // the boundaries break the contract
    if (threadIdx.x == 0) {
      if (i0 == 0) *a0.status = VA_ERR_BAD_SEQLENS;
      for (int i = i0; i < i1; ++i) {
        *pp.map[i].n_items = 0;
        if (pp.map[i].n_tok) *pp.map[i].n_tok = 0;
      }
    }
    return;
  }
  if (threadIdx.x == 0 && i0 == 0) *a0.status = VA_OK;
  for (int i = i0; i < i1; ++i) {
    const PlanArgs& a = pp.map[i];
    __syncthreads();  // the table of the previous map has been read
    if (threadIdx.x < 32) {
      int total = 0;
      if (a.kind == 1) {
        if (a.causal) small_rank<MapKind<true, true, false>>(a, lane, l, sh.small, total);
        else small_rank<MapKind<true, false, false>>(a, lane, l, sh.small, total);
      } else {
        if (a.causal) small_rank<MapKind<false, true, false>>(a, lane, l, sh.small, total);
        else small_rank<MapKind<false, false, false>>(a, lane, l, sh.small, total);
      }
      if (lane == 0) {
        const bool overflow = total > a.capacity;
        *a.n_items = overflow ? 0 : total;
        *a.counter = 0;
        if (a.n_tok) *a.n_tok = 0;
        if (a.tok_counter) *a.tok_counter = 0;
        if (overflow && a.status) atomicCAS(a.status, VA_OK, VA_ERR_WORKSPACE);
        sh.seg_total = overflow ? 0 : total;
      }
    }
    __syncthreads();
    const int total = sh.seg_total;
    if (a.kind == 1) {
      if (a.causal) small_write<MapKind<true, true, false>>(a, sh.small, total);
      else small_write<MapKind<true, false, false>>(a, sh.small, total);
    } else {
      if (a.causal) small_write<MapKind<false, true, false>>(a, sh.small, total);
      else small_write<MapKind<false, false, false>>(a, sh.small, total);
    }
  }
}

// Copies cu[0..B] into shared memory when it fits; returns the array to read.
__device__ __forceinline__ const int* stage_cu(const int32_t* cu, int B, PlanSmem& sh) {
  if (B + 1 > kSmemSegs) return cu;
  for (int i = threadIdx.x; i <= B; i += blockDim.x) sh.cu[i] = cu[i];
  __syncthreads();
  return sh.cu;
}

// Validates cu_seqlens and builds the maps of pp: every map (only < 0), writing the status
// word, or map `only` alone (the CTA that builds map 0 writes the status word).  Two CTAs
// that each build one map share nothing but the boundaries they read.  Neither can overflow:
// the library sizes a map at (rows / tile + B) * heads records, which bounds the records of
// any boundaries that pass the check, so the second CTA's map never writes the status word.
__device__ __forceinline__ void validate_plan_body(const PlanPair& pp, PlanSmem& sh, int only = -1) {
  if (small_plan_ok(pp, only < 0 ? 0 : only, only < 0 ? pp.nmaps : only + 1)) {
    small_plan(pp, sh, only < 0 ? 0 : only, only < 0 ? pp.nmaps : only + 1);
    return;
  }
  const PlanArgs& a0 = pp.map[0];
  const int* cu = stage_cu(a0.cu, a0.B, sh);  // every map is built from the same boundaries
  int bad = 0;
  for (int b = threadIdx.x; b < a0.B; b += blockDim.x) {
    const int x = cu[b], y = cu[b + 1];
    if (y <= x || y - x > pp.max_seqlen) bad = 1;
  }
  if (threadIdx.x == 0 && (cu[0] != 0 || cu[a0.B] != pp.T)) bad = 1;
  if (a0.cu_k) {  // the K/V boundaries obey the same contract; causal needs lq <= lk
    const int32_t* ck = a0.cu_k;
    for (int b = threadIdx.x; b < a0.B; b += blockDim.x) {
      const int x = ck[b], y = ck[b + 1];
      if (y <= x || y - x > pp.max_seqlen_k || (a0.causal && cu[b + 1] - cu[b] > y - x)) bad = 1;
    }
    if (threadIdx.x == 0 && (ck[0] != 0 || ck[a0.B] != pp.Tk)) bad = 1;
  }
  bad = __syncthreads_or(bad);
  const int i0 = only < 0 ? 0 : only, i1 = only < 0 ? pp.nmaps : only + 1;
  if (bad) {
    if (threadIdx.x == 0) {
      if (i0 == 0) *a0.status = VA_ERR_BAD_SEQLENS;
      for (int i = i0; i < i1; ++i) {
        *pp.map[i].n_items = 0;
        if (pp.map[i].n_tok) *pp.map[i].n_tok = 0;
      }
    }
    return;
  }
  if (threadIdx.x == 0 && i0 == 0) *a0.status = VA_OK;
  for (int i = i0; i < i1; ++i)
    plan_body(pp.map[i], sh, cu, a0.B + 1 > kSmemSegs ? pp.map[i].seg_off : sh.off);
}

}  // namespace va
