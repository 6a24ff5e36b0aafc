// Device-side tile scheduler.  Reads cu_seqlens on the device (the host
// never sees their values) and writes work lists sorted by cost, longest
// first, so a persistent kernel that walks the list in order balances ragged
// sequences; the backward's lists A and B instead go by (sequence, head)
// groups, longer sequences first (see `grouped` below).  One block per list:
//   list A: query tiles of 128 rows; cost = number of key tiles of `bn_a`
//           rows the tile needs (the mask window bounds its keys: causal
//           tiles only need keys up to their last row, a left bound cuts
//           keys before the first row);
//   list B: key tiles of 128 rows; cost = number of query tiles of `bq_b`
//           rows that can see the tile; each key tile is emitted once per
//           head, and with split_b = 2 (D = 256) the list has two halves, one
//           pass over every tile each (head field: h * split_b + pass);
//   list F: (plans only) list A again with inner tiles of `bn_f` keys, the
//           forward's, so that one launch schedules a forward and a backward.
// A plan's block 0 also records the sizes the plan was made for.
// Each unit record is two int4: {sequence, tile, head (x split_b), cost} and
// {q offset, q length, k offset, k length}, so a consumer needs one round
// trip to global memory per unit.  Units with cost 0 are kept (their rows
// must be written as zeros) and sort last.  Order inside one cost bucket is
// whatever the atomics give; it only changes timing, never results.  For the
// backward, the list-B block also writes ds_base: the first stored dS block
// of every sequence (an exclusive scan of H * ds_blocks_head over them).
#include <climits>

#include "kernels.h"

namespace hstu {

namespace {

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Sequence b as {q offset, q length, k offset, k length}, from cu_seqlens.
__device__ __forceinline__ int4 seq_global(const SchedArgs& a, int b) {
  const int q0 = __ldg(a.cu_q + b), k0 = __ldg(a.cu_k + b);
  return make_int4(q0, max(0, __ldg(a.cu_q + b + 1) - q0), k0, max(0, __ldg(a.cu_k + b + 1) - k0));
}

// Bits [lo, hi) of a 32-bit word, clamped to [0, 32).
__device__ __forceinline__ uint32_t bits32(int lo, int hi) {
  lo = max(lo, 0);
  hi = min(hi, 32);
  if (hi <= lo) return 0u;
  const uint32_t below_hi = hi == 32 ? 0xffffffffu : (1u << hi) - 1u;
  return below_hi & ~((1u << lo) - 1u);
}

// Arbitrary mask: the live tiles of bn keys (64 or 128) among tiles
// [u0, u1) of 128-row query tile tq, counted from its blocks' bit words (a
// 64-key tile is live when its 128-key tile is).
__device__ __forceinline__ int func_live_tiles(const FuncMask& f, int q0, int b, int tq, int Lq,
                                               int bn, int u0, int u1) {
  const bool two = kBM * tq + 64 < Lq;
  const int64_t r0 = static_cast<int64_t>(qb_slot(q0, b, 2 * tq)) * f.kt_words;
  auto word = [&](int w) {  // the tile's OR of its two blocks (slots are consecutive)
    uint32_t x = __ldg(f.qb_bits + r0 + w);
    if (two) x |= __ldg(f.qb_bits + r0 + f.kt_words + w);
    return x;
  };
  int n = 0;
  if (bn == kBM) {
    for (int w = u0 >> 5; w <= (u1 - 1) >> 5; ++w)
      n += __popc(word(w) & bits32(u0 - 32 * w, u1 - 32 * w));
    return n;
  }
  for (int u = u0; u < u1; ++u) {  // 64-key tiles: tile u / 2 of 128 keys
    const int s = u >> 1;
    n += static_cast<int>((word(s >> 5) >> (s & 31)) & 1u);
  }
  return n;
}

// Cost of query tile t (lists A and F): its inner tiles of 2^lbn keys (the
// window's rule of query_tile_keys, with shifts for the divisions).
__device__ __forceinline__ int cost_a(const SchedArgs& a, int4 sq, int b, int t, int lbn,
                                      bool func) {
  if (func) {  // arbitrary mask: the live tiles of the tile's key hull
    const int bn = 1 << lbn;
    const int2 h = func_tile_keys(a.fm, sq.x, b, t, sq.y);
    if (h.x >= h.y) return 0;
    return func_live_tiles(a.fm, sq.x, b, t, sq.y, bn, h.x / bn, (h.y + bn - 1) / bn);
  }
  const int r0 = kBM * t, r1 = imin(kBM * t + kBM, sq.y);
  const int j0 = a.win.left < 0 ? 0 : imax(0, r0 - a.win.left);
  const int j1 = a.win.right < 0 ? sq.w : imin(sq.w, r1 + a.win.right);
  return (r1 > r0 && j1 > j0) ? ((j1 + (1 << lbn) - 1) >> lbn) - (j0 >> lbn) : 0;
}

// Arbitrary mask, list B, warp-wide: for key tile t = tb + lane (tb a
// multiple of 32, t < nt), the hull {first, count} of the 64-row query blocks
// whose key hull meets the tile, and how many of them have the tile live.
// The warp reads 32 blocks' hulls and bit words at a time and compares them
// with each tile of the group by ballots.  Every lane of the warp calls it.
__device__ void func_key_tiles_warp(const SchedArgs& a, int4 sq, int b, int tb, int nt,
                                    int2& hull, int& live) {
  const int lane = threadIdx.x & 31;
  const int n_qb = ceil_div(sq.y, 64);
  const int w = tb >> 5;  // the group's bit word
  int first = INT_MAX, last = -1, n = 0;
  for (int mb = 0; mb < n_qb; mb += 32) {
    const int m = mb + lane;
    int2 h = make_int2(0, 0);
    uint32_t bits = 0;
    if (m < n_qb) {
      const int slot = qb_slot(sq.x, b, m);
      h = a.fm.qb_range[slot];
      bits = a.fm.qb_bits[static_cast<int64_t>(slot) * a.fm.kt_words + w];
    }
    for (int k = 0; k < 32 && tb + k < nt; ++k) {
      const int c0 = kBM * (tb + k), c1 = min(c0 + kBM, sq.w);
      const bool meets = h.x < h.y && h.x < c1 && h.y > c0;
      const uint32_t bm = __ballot_sync(0xffffffffu, meets);
      const uint32_t bl = __ballot_sync(0xffffffffu, (bits >> k) & 1u);
      if (lane == k && bm != 0u) {
        first = min(first, mb + __ffs(bm) - 1);
        last = max(last, mb + 31 - __clz(bm));
        n += __popc(bl);
      }
    }
  }
  hull = last >= 0 ? make_int2(first, last - first + 1) : make_int2(0, 0);
  live = n;
}

// Cost of key tile s (list B; the arbitrary mask's walk is warp-wide): its
// query blocks of 2^lbq rows (key_tile_queries, with shifts).
__device__ __forceinline__ int cost_b(const SchedArgs& a, int4 sq, int s, int lbq) {
  const int c0 = kBM * s, c1 = imin(kBM * s + kBM, sq.w);
  const int i0 = a.win.right < 0 ? 0 : imax(0, c0 - a.win.right);
  const int i1 = a.win.left < 0 ? sq.y : imin(sq.y, c1 + a.win.left);
  return (c1 > c0 && i1 > i0) ? ((i1 + (1 << lbq) - 1) >> lbq) - (i0 >> lbq) : 0;
}

// Block 0 builds list A, block 1 list B, block 2 (plans) list F.
__device__ __forceinline__ int list_cmax(const SchedArgs& a, int list) {
  return list == 0 ? a.cmax_a : list == 1 ? a.cmax_b : a.cmax_f;
}

// Exclusive prefix sum over 1024 threads; returns this thread's offset and
// writes the block total.
__device__ int block_exclusive_scan(int v, int* total) {
  __shared__ int warp_sums[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncwarp();  // reconverge before the aligned CTA barrier
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncwarp();  // reconverge before the aligned CTA barrier
  __syncthreads();
  int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  *total = warp_sums[31];
  __syncwarp();  // reconverge before the aligned CTA barrier
  __syncthreads();
  return before;
}

}  // namespace

// One list's passes (block 0: list A, 1: B, 2: F).  Every block barrier
// comes before the first global store: a barrier behind outstanding global
// stores measured about a microsecond each, so the header words, the
// readiness counts, the staged list and the dS bases all leave at the end.
__global__ void __launch_bounds__(kSchedThreads) hstu_sched_kernel(const __grid_constant__ SchedArgs a) {
  extern __shared__ int hist[];  // cost buckets | cached sequence records | staged records
  __shared__ int ds_all;         // list B, backward: the dS blocks of the whole batch
  const int list = blockIdx.x;
  const int cmax = list_cmax(a, list);
  int4* seqs = reinterpret_cast<int4*>(hist + sched_hist_ints(cmax));
  int4* stage = seqs + (a.cache_seqs ? a.B : 0);
  const bool list_b = list == 1;
  const int cap = list == 0 ? a.cap_a : list == 1 ? a.cap_b : a.cap_f;
  int4* units = list == 0 ? a.units_a : list == 1 ? a.units_b : a.units_f;
  const int bn = list == 2 ? a.bn_f : a.bn_a;  // query-tile lists
  const int lbn = __ffs(bn) - 1, lbq = __ffs(a.bq_b) - 1;  // tile sizes are powers of two
  const int units_slot = list == 0 ? kHdrUnitsA : list == 1 ? kHdrUnitsB : kHdrUnitsF;
  const int next_slot = list == 0 ? kHdrNextA : list == 1 ? kHdrNextB : kHdrNextF;
  const int overflow_slot = list == 0 ? kHdrOverflow : list == 1 ? kHdrOverflowB : kHdrOverflowF;
  // List B at D = 256 holds two passes over every key tile: the dV passes
  // first, then the dK passes in the same order, each half sorted by cost.
  const int split = list_b ? a.split_b : 1;
  const int per_tile = a.H;  // units of one tile in one half
  const int nb = cmax + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nwarps = blockDim.x >> 5;
  const bool func = a.fm.func != nullptr;
  // The backward's lists A and B are ordered by (sequence, head) groups
  // instead: sequences with more 128-token tiles first, each sequence's units
  // contiguous, head by head (key tiles in order, query tiles last first, so
  // the costly ones of a group lead).  The long units still come first and
  // the short ones last, and a group's units run close together, sharing its
  // Q / dO and K tiles in L2 (measured: long workload 1037 -> 1024 us,
  // skewed 536 -> 531 us, recsys unchanged).  Buckets count units per key.
  const bool grouped = a.ds_base != nullptr && list != 2;
  auto seq_key = [&](int4 sq) { return min((max(sq.y, sq.w) + kBM - 1) / kBM, cmax); };

  for (int i = tid; i < nb; i += blockDim.x) hist[i] = 0;
  // Launched early behind the previous grid of the stream, which may still
  // read this workspace or write cu_seqlens: wait for it first.
  grid_dependency_wait();
  // the attention grid queued behind this one may start its prologue now
  if (tid == 0) grid_launch_dependents();
  // every pass reads the sequences: one coalesced read of cu_seqlens
  if (a.cache_seqs)
    for (int b = tid; b < a.B; b += blockDim.x) seqs[b] = seq_global(a, b);
  auto seq = [&](int b) { return a.cache_seqs ? seqs[b] : seq_global(a, b); };
  __syncwarp();  // reconverge before the aligned CTA barrier
  __syncthreads();

  // pass 1: histogram of costs; a warp per sequence, a lane per tile (grouped
  // lists: of sequence keys, a thread per sequence, weighted by its units)
  const bool func_b = list_b && func;  // the warp-wide list-B walk
  if (grouped) {
    for (int b = tid; b < a.B; b += blockDim.x) {
      const int4 sq = seq(b);
      const int nt = list_b ? (sq.w + kBM - 1) / kBM : (sq.y + kBM - 1) / kBM;
      atomicAdd(&hist[seq_key(sq)], per_tile * nt);
    }
  }
  for (int b = warp; b < a.B && !grouped; b += nwarps) {
    const int4 sq = seq(b);
    const int Lq = sq.y, Lk = sq.w;
    const int nt = list_b ? (Lk + kBM - 1) / kBM : (Lq + kBM - 1) / kBM;
    for (int tb = 0; tb < nt; tb += 32) {
      const int t = tb + lane;
      int cost = 0;
      if (func_b) {
        int2 r;
        func_key_tiles_warp(a, sq, b, tb, nt, r, cost);
      } else if (t < nt) {
        cost = list_b ? cost_b(a, sq, t, lbq) : cost_a(a, sq, b, t, lbn, func);
      }
      if (t < nt) atomicAdd(&hist[min(cost, cmax)], per_tile);
    }
  }
  __syncwarp();  // reconverge before the aligned CTA barrier
  __syncthreads();

  // pass 2: exclusive scan over costs in descending order (rank 0 = cmax)
  const int chunk = (nb + blockDim.x - 1) / blockDim.x;
  const int r0 = min(nb, tid * chunk), r1 = min(nb, r0 + chunk);
  int local = 0;
  for (int r = r0; r < r1; ++r) local += hist[cmax - r];
  int total;
  int run = block_exclusive_scan(local, &total);
  for (int r = r0; r < r1; ++r) {
    int c = cmax - r;
    int h = hist[c];
    hist[c] = run;
    run += h;
  }
  __syncwarp();  // reconverge before the aligned CTA barrier
  __syncthreads();

  // pass 3 (backward, list-B block): first dS block of each sequence, a scan
  // over the sequences (written out at the end)
  const bool ds_pass = list_b && a.ds_base != nullptr;
  const int per = (a.B + blockDim.x - 1) / blockDim.x;
  const int s0 = min(a.B, tid * per), s1 = min(a.B, s0 + per);
  auto blocks = [&](int b) {
    const int4 sq = seq(b);
    return a.H * ds_blocks_head(sq.y, sq.w, a.win);
  };
  int ds_run = 0;
  if (ds_pass) {  // block-uniform: every thread takes the scan's barriers
    int sum = 0;
    for (int b = s0; b < s1; ++b) sum += blocks(b);
    int all;
    ds_run = block_exclusive_scan(sum, &all);
    if (tid == 0) ds_all = all;
  }

  // pass 4: complete unit records at their bucket cursors; into shared
  // memory when the whole list fits there (one coalesced copy follows),
  // else straight to global memory
  const bool staged = split * total <= a.stage_units;
  int overflow = 0;
  for (int b = warp; b < a.B; b += nwarps) {
    const int4 sq = seq(b);
    const int q0 = sq.x, Lq = sq.y, k0 = sq.z, Lk = sq.w;
    const int nt = list_b ? (Lk + kBM - 1) / kBM : (Lq + kBM - 1) / kBM;
    // grouped: this sequence's first unit, taken from its key's bucket
    int gbase = 0;
    if (grouped) {
      if (lane == 0) gbase = atomicAdd(&hist[seq_key(sq)], per_tile * nt);
      gbase = __shfl_sync(0xffffffffu, gbase, 0);
    }
    for (int tb = 0; tb < nt; tb += 32) {
      const int t = tb + lane;
      int cost = 0;
      if (func_b) {  // also record the key tile's query hull
        int2 r;
        func_key_tiles_warp(a, sq, b, tb, nt, r, cost);
        if (t < nt) a.fm.kt_range[kt_slot(k0, b, t)] = r;
      } else if (t < nt) {
        cost = list_b ? cost_b(a, sq, t, lbq) : cost_a(a, sq, b, t, lbn, func);
      }
      if (t >= nt) continue;
      const int pos = grouped ? 0 : atomicAdd(&hist[min(cost, cmax)], per_tile);
      int4* dst = staged ? stage : units;
      for (int p = 0; p < split; ++p) {
        for (int e = 0; e < per_tile; ++e) {
          const int u = p * total + (grouped ? gbase + e * nt + (list_b ? t : nt - 1 - t)
                                             : pos + e);
          if (u < cap) {
            dst[2 * u] = make_int4(b, t, e * split + p, cost);
            dst[2 * u + 1] = make_int4(q0, Lq, k0, Lk);
          } else {
            overflow = 1;
          }
        }
      }
    }
  }
  __syncwarp();  // reconverge before the aligned CTA barrier
  const bool dropped = __syncthreads_or(overflow) != 0;  // units beyond the list's capacity
  if (staged)
    for (int i = tid; i < 2 * min(split * total, cap); i += blockDim.x) units[i] = stage[i];

  // the global words, after the last barrier
  if (ds_pass) {
    for (int b = s0; b < s1; ++b) {
      a.ds_base[b] = ds_run;
      ds_run += blocks(b);
    }
  }
  if (list_b && a.ready != nullptr) {  // the dK/dV -> dQ readiness counts start at zero
    for (int i = tid; i < a.B * a.H; i += blockDim.x) a.ready[i] = 0;
  }
  if (tid == 0) {
    if (list == 0) {
      a.header[kHdrStatus] = 0;
      a.header[kHdrWhere] = 0;
      a.header[kHdrDone] = 0;
      if (gridDim.x == 1) {
        a.header[kHdrOverflowB] = 0;
        a.header[kHdrNextB] = 0;
      }
      if (gridDim.x < 3) {
        a.header[kHdrOverflowF] = 0;
        a.header[kHdrUnitsF] = 0;
      }
      for (int i = 0; i < kPlanKeyInts; ++i) a.header[kHdrKey + i] = a.key[i];
    }
    a.header[next_slot] = 0;
    if (list_b) a.header[kHdrNextB2] = 0;
    a.header[units_slot] = min(split * total, cap);
    if (list_b && a.ready != nullptr) a.header[kHdrEpoch] = 0;
    // sequences longer than the caller's max_seqlen_q: the dS blocks would
    // not fit; the dK/dV units then skip the stores past the end (list B's
    // overflow word reports it)
    const bool ds_over = ds_pass && (ds_all > a.ds_cap || ds_all < 0);
    if (ds_pass) a.ds_base[a.B] = ds_all;
    a.header[overflow_slot] = dropped || ds_over ? 1 : 0;
  }
}

// Bits of the 128-key tiles 32 w .. 32 w + 31 whose keys below Lk all lie in
// [a, c) (c <= Lk): tiles from ceil(a / 128), up to the last one that ends
// by c, or the sequence's last tile when c reaches Lk.
__device__ __forceinline__ uint32_t full_tile_bits(int a, int c, int Lk, int w) {
  if (a >= c) return 0u;
  const int t0 = (a + kBM - 1) / kBM;
  const int t1 = (c >= Lk ? (Lk + kBM - 1) / kBM : c / kBM) - 1;  // last tile, inclusive
  const int u0 = max(t0 - 32 * w, 0), u1 = min(t1 - 32 * w, 31);
  if (u0 > u1) return 0u;
  const uint32_t upto = u1 == 31 ? 0xffffffffu : (2u << u1) - 1u;
  return upto & ~((1u << u0) - 1u);
}

// Bits of the 128-key tiles 32 w .. 32 w + 31 that keys [a, c) touch.
__device__ __forceinline__ uint32_t tile_bits(int a, int c, int w) {
  if (a >= c) return 0u;
  const int t0 = max(a / kBM - 32 * w, 0), t1 = min((c - 1) / kBM - 32 * w, 31);
  if (t0 > t1) return 0u;
  const uint32_t upto = t1 == 31 ? 0xffffffffu : (2u << t1) - 1u;  // bits 0 .. t1
  return upto & ~((1u << t0) - 1u);
}

// Arbitrary mask: one warp per 64-row query block; each lane takes two rows,
// forms each row's key hull from its endpoints (every interval cut to
// [0, Lk)), and the warp reduces the 64 hulls to the block's; the same for
// the block's live-tile bitmap (OR of the tiles every interval touches).
__global__ void __launch_bounds__(256) hstu_func_ranges_kernel(const int32_t* cu_q,
                                                               const int32_t* cu_k, FuncMask fm) {
  const int b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x * 8 + warp;
  // the previous grid of the stream may still read this workspace
  grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int q0 = __ldg(cu_q + b), Lq = __ldg(cu_q + b + 1) - q0;
  const int Lk = __ldg(cu_k + b + 1) - __ldg(cu_k + b);
  if (64 * m >= Lq) return;
  int lo = INT_MAX, hi = INT_MIN;
  for (int rr = 0; rr < 2; ++rr) {
    const int i = 64 * m + 32 * rr + lane;
    if (i >= Lq) continue;
    const int64_t t = static_cast<int64_t>(q0) + i;
    const int f0 = min(__ldg(fm.func + t), Lk);  // [0, F0)
    if (f0 > 0) { lo = 0; hi = max(hi, f0); }
    for (int n = 1; n + 1 < fm.n; n += 2) {
      const int a = max(__ldg(fm.func + n * fm.len + t), 0);
      const int c = min(__ldg(fm.func + (n + 1) * fm.len + t), Lk);
      if (a < c) { lo = min(lo, a); hi = max(hi, c); }
    }
  }
  lo = __reduce_min_sync(0xffffffffu, lo);
  hi = __reduce_max_sync(0xffffffffu, hi);
  if (lane == 0) fm.qb_range[qb_slot(q0, b, m)] = lo < hi ? make_int2(lo, hi) : make_int2(0, 0);
  // the block's live 128-key tiles, 32 per word: the tiles each interval
  // touches; and its full tiles: those inside one interval of every row
  const int64_t slot = static_cast<int64_t>(qb_slot(q0, b, m)) * fm.kt_words;
  for (int w = 0; w < fm.kt_words; ++w) {
    uint32_t word = 0, full = 0xffffffffu;
    for (int rr = 0; rr < 2; ++rr) {
      const int i = 64 * m + 32 * rr + lane;
      if (i >= Lq) continue;
      const int64_t t = static_cast<int64_t>(q0) + i;
      const int f0 = min(__ldg(fm.func + t), Lk);
      word |= tile_bits(0, f0, w);
      uint32_t row_full = full_tile_bits(0, f0, Lk, w);
      for (int n = 1; n + 1 < fm.n; n += 2) {
        const int a = max(__ldg(fm.func + n * fm.len + t), 0);
        const int c = min(__ldg(fm.func + (n + 1) * fm.len + t), Lk);
        word |= tile_bits(a, c, w);
        row_full |= full_tile_bits(a, c, Lk, w);
      }
      full &= row_full;
    }
    word = __reduce_or_sync(0xffffffffu, word);
    full = __reduce_and_sync(0xffffffffu, full);
    if (lane == 0) {
      fm.qb_bits[slot + w] = word;
      fm.qb_full[slot + w] = full & word;
    }
  }
}

cudaError_t launch_func_ranges(const int32_t* cu_q, const int32_t* cu_k, int B, int max_qb,
                               const FuncMask& fm, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>((max_qb + 7) / 8), static_cast<unsigned>(B));
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, hstu_func_ranges_kernel, cu_q, cu_k, fm);
}

cudaError_t launch_sched(int lists, int smem, cudaStream_t st, bool pdl, const SchedArgs& a) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(lists));
  cfg.blockDim = dim3(kSchedThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, hstu_sched_kernel, a);
}

// One thread waits on a barrier that nothing completes; the bounded wait must
// give up after `timeout_ns`, record the timeout in the header and return.
__global__ void hstu_selftest_timeout_kernel(int* header, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int flags[2];
  if (threadIdx.x == 0) {
    header[kHdrStatus] = 0;
    header[kHdrWhere] = 0;
    header[kHdrOverflow] = 0;
    header[kHdrOverflowB] = 0;
    mbar_init(smem_u32(&bar), 1);
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
    const WaitCtl wc{header, flags, timeout_ns};
    wait_bar(smem_u32(&bar), 0, wc, 0x7e5);
  }
}

cudaError_t launch_selftest_timeout(int* header, uint64_t timeout_ns, cudaStream_t st) {
  hstu_selftest_timeout_kernel<<<1, 32, 0, st>>>(header, timeout_ns);
  return cudaGetLastError();
}

}  // namespace hstu
