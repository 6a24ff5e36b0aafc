// Internal interface between the host library and the device kernels:
// tile configurations, argument blocks and launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "common.cuh"

namespace hstu {

constexpr int kSchedThreads = 1024;
// Up to this many sequences the scheduler keeps every sequence's offsets and
// lengths in shared memory (16 bytes each), read from cu_seqlens once.
constexpr int kSchedCacheSeqs = 4096;
// Lists of up to this many units are assembled in shared memory (32 bytes
// each) and written out in one coalesced copy.
constexpr int kSchedStageUnits = 2048;
__host__ __device__ constexpr int sched_hist_ints(int cmax) { return (cmax + 1 + 3) & ~3; }
// Forward kernel: warp 0 TMA, warp 1 issues S = Q K^T, warps 2-9 SiLU row
// work (two per TMEM lane quarter, taking alternate key steps), warps 10-13
// O epilogue (one per lane quarter), warp 14 issues O += P V.
constexpr int kFwdRowWarps = 8;
constexpr int kFwdEpiWarps = 4;
constexpr int kFwdPvWarp = 2 + kFwdRowWarps + kFwdEpiWarps;
constexpr int kAttnThreads = 32 * (kFwdPvWarp + 1);
// Backward kernel, dK/dV phase: warp 0 TMA, warp 1 MMA, warps 2-9 row work (two warps per
// TMEM lane quarter, one per half of the columns), warp 10 issues the
// accumulation MMAs, so the two MMA streams wait on their own barriers
// without stalling each other.  Few row warps per SM sub-partition leave
// the issuing threads more of its issue slots.
constexpr int kDkdvRowWarps = 8;
constexpr int kDkdvThreads = 64 + 32 * kDkdvRowWarps + 32;
// Backward kernel, dQ phase (dQ = dS K from the stored dS blocks): warp 0 TMA, warp 1 MMA,
// warps 2-5 epilogue (one per TMEM lane quarter).
constexpr int kDqEpiWarps = 4;
constexpr int kTmemCols = 512;

// Bytes of shared memory a kernel needs beyond its tiles: barriers, the TMEM
// address slot, the abort flags, and slack to align the tiles to 1024 bytes.
constexpr int kCtlBytes = 1024;
constexpr int kAlignSlack = 1024;
// K/V steps warmed in L2 ahead of the TMA loads (and of the next unit);
// the dK/dV units' 64-query steps run twice as many Q/dO tiles ahead.
constexpr int kPrefetch = 4;
constexpr int kPrefetchQ = 8;

// ---------------------------------------------------------------- mask window
// Token window ("HSTU Attention (Blackwell SM100/SM103)", section "Mask
// support", window_size = (left, right)), -1 meaning no bound on that side:
// key j is valid for query i (both local to the sequence) iff j < Lk,
// j >= i - left when left >= 0, and j <= i + right when right >= 0.
// (-1, 0) is causal, (-1, -1) full.
struct Window {
  int left, right;
};
__host__ __device__ constexpr int imin(int a, int b) { return a < b ? a : b; }
__host__ __device__ constexpr int imax(int a, int b) { return a > b ? a : b; }
__host__ __device__ constexpr bool win_causal(Window w) { return w.left < 0 && w.right == 0; }
__host__ __device__ constexpr bool win_full(Window w) { return w.left < 0 && w.right < 0; }

// Keys a 128-row query tile t needs: inner key tiles of bn keys, the first
// one `first` and `count` of them (0: the tile sees no key; its rows are
// zeros).  Rows past Lq are not counted.
__host__ __device__ inline void query_tile_keys(int t, int Lq, int Lk, Window w, int bn,
                                                int& first, int& count) {
  const int r0 = kBM * t, r1 = imin(kBM * t + kBM, Lq);           // rows [r0, r1)
  const int j0 = w.left < 0 ? 0 : imax(0, r0 - w.left);           // keys [j0, j1)
  const int j1 = w.right < 0 ? Lk : imin(Lk, r1 + w.right);
  first = j0 / bn;
  count = (r1 > r0 && j1 > j0) ? (j1 + bn - 1) / bn - first : 0;
}

// Queries a 128-key tile s is seen by: query blocks of bq rows, the first
// one `first` and `count` of them.  Keys past Lk are not counted.
__host__ __device__ inline void key_tile_queries(int s, int Lq, int Lk, Window w, int bq,
                                                 int& first, int& count) {
  const int c0 = kBM * s, c1 = imin(kBM * s + kBM, Lk);           // keys [c0, c1)
  const int i0 = w.right < 0 ? 0 : imax(0, c0 - w.right);         // queries [i0, i1)
  const int i1 = w.left < 0 ? Lq : imin(Lq, c1 + w.left);
  first = i0 / bq;
  count = (c1 > c0 && i1 > i0) ? (i1 + bq - 1) / bq - first : 0;
}

// ---------------------------------------------------------------- arbitrary mask
// func_tensor ("Mask support"): query token t's valid keys are the union
// [0, F0) U [F1, F2) U ... of its N endpoints F_n = func[n * len + t] (N odd,
// local key indices), cut to j < Lk.  Units iterate the contiguous hull of
// the tiles their rows can see, and the exact predicate is applied inside:
//   qb_range[qb_slot(b, m)]: {kmin, kmax}, the key hull of 64-row query block
//     m of sequence b (kmin >= kmax: no key), written by the range kernel;
//   kt_range[kt_slot(b, s)]: {first query block, count}, the hull of the
//     query blocks whose key hull meets 128-key tile s, written by the
//     scheduler.
// Slots are floor(offset / tile) + b + index, disjoint between sequences
// without a scan (floor((o + L) / n) + 1 >= floor(o / n) + ceil(L / n)).
//   qb_bits[qb_slot(b, m) * kt_words + s / 32], bit s % 32: 128-key tile s
//     is live for query block m (some row of the block sees a key of the
//     tile), written by the range kernel.  Units visit only live tiles (and
//     key tiles only live query blocks) inside their hulls.
struct FuncMask {
  const int32_t* func;  // null: no arbitrary mask (the window decides)
  int n;
  int64_t len;
  int2* qb_range;
  int2* kt_range;
  uint32_t* qb_bits;
  uint32_t* qb_full;    // same layout: every row of the block sees every key (< Lk) of the tile
  int kt_words;         // ceil(ceil(max_seqlen_k / 128) / 32)
};
__host__ __device__ inline int qb_slot(int q0, int b, int m) { return q0 / 64 + b + m; }
__host__ __device__ inline int kt_slot(int k0, int b, int s) { return k0 / kBM + b + s; }
// Key hull of 128-row query tile t from its two blocks' hulls.
__device__ inline int2 func_tile_keys(const FuncMask& f, int q0, int b, int t, int Lq) {
  const int2 a = f.qb_range[qb_slot(q0, b, 2 * t)];
  int2 h = a;
  if (kBM * t + 64 < Lq) {
    const int2 c = f.qb_range[qb_slot(q0, b, 2 * t + 1)];
    if (c.x < c.y) h = a.x < a.y ? make_int2(imin(a.x, c.x), imax(a.y, c.y)) : c;
  }
  return h;
}

// 128-key tile s is live for 64-row query block m of sequence b.
__device__ __forceinline__ bool func_live(const FuncMask& f, int q0, int b, int m, int s) {
  const uint32_t w =
      __ldg(f.qb_bits + static_cast<int64_t>(qb_slot(q0, b, m)) * f.kt_words + (s >> 5));
  return (w >> (s & 31)) & 1u;
}

// Every row of 64-row query block m sees every key of 128-key tile s (the
// keys below Lk): the pair needs no per-element mask and no endpoints.
__device__ __forceinline__ bool func_full(const FuncMask& f, int q0, int b, int m, int s) {
  const uint32_t w =
      __ldg(f.qb_full + static_cast<int64_t>(qb_slot(q0, b, m)) * f.kt_words + (s >> 5));
  return (w >> (s & 31)) & 1u;
}

// Walks, in order, the live tiles (bn = 64 or 128 keys) of 128-row query
// tile tq: those whose 128-key tile is live for block 2 tq or, inside the
// sequence, 2 tq + 1.  It keeps the two blocks' bit words of 32 tiles of 128
// keys and loads the next pair only when the walk leaves them, so a step
// costs no dependent load (one per 32 tiles of 128 keys).
struct TileWalk {
  const uint32_t* row0;  // qb_bits row of block 2 tq
  const uint32_t* row1;  // of block 2 tq + 1 (null: past the sequence end)
  int w;                 // index of the words held (-1: none)
  uint32_t bits0, bits1;
  __device__ __forceinline__ void init(const FuncMask& f, int q0, int b, int tq, int Lq) {
    row0 = f.qb_bits + static_cast<int64_t>(qb_slot(q0, b, 2 * tq)) * f.kt_words;
    row1 = kBM * tq + 64 < Lq ? row0 + f.kt_words : nullptr;  // slots are consecutive
    w = -1;
    bits0 = bits1 = 0u;
  }
  __device__ __forceinline__ void hold(int wi) {
    if (wi == w) return;
    w = wi;
    bits0 = __ldg(row0 + wi);
    bits1 = row1 != nullptr ? __ldg(row1 + wi) : 0u;
  }
  // First live tile t' >= t (in tiles of 2^lbn keys, lbn = 6 or 7); t_end if none.
  __device__ __forceinline__ int next(int t, int t_end, int lbn) {
    while (t < t_end) {
      const int s = t >> (7 - lbn);  // its 128-key tile
      hold(s >> 5);
      const uint32_t rest = (bits0 | bits1) >> (s & 31);
      if (rest == 0u) {  // none left in this word
        t = (32 * (w + 1)) << (7 - lbn);
        continue;
      }
      const int s2 = s + __ffs(rest) - 1;
      return imax(t, s2 << (7 - lbn));
    }
    return t_end;
  }
  // Whether 128-key tile s (in the words held, after next) is live for block
  // 2 tq (second = false) or 2 tq + 1.
  __device__ __forceinline__ bool live(int s, bool second) const {
    return (((second ? bits1 : bits0) >> (s & 31)) & 1u) != 0u;
  }
};

// Walks, in order, the 64-row query blocks for which 128-key tile s is live
// (and tells which of them see the whole tile).  The bits of 32 blocks sit in
// 32 different rows; they are gathered 32 at a time: by the whole warp, one
// load per lane, or by one thread, 32 independent loads.
struct BlockWalk {
  int base;            // first block of the masks held (-1: none)
  uint32_t live, full;  // bit i: block base + i
  __device__ __forceinline__ void init() { base = -1; live = full = 0u; }
  template <bool WARP>
  __device__ __forceinline__ void gather(const FuncMask& f, int q0, int b, int s, int m0, int m_end) {
    base = m0;
    const int64_t col = s >> 5;
    const int sh = s & 31;
    if constexpr (WARP) {
      const int m = m0 + static_cast<int>(threadIdx.x & 31);
      uint32_t lw = 0u, fw = 0u;
      if (m < m_end) {
        const int64_t r = static_cast<int64_t>(qb_slot(q0, b, m0)) * f.kt_words + col +
                          static_cast<int64_t>(m - m0) * f.kt_words;
        lw = __ldg(f.qb_bits + r);
        fw = __ldg(f.qb_full + r);
      }
      live = __ballot_sync(0xffffffffu, (lw >> sh) & 1u);
      full = __ballot_sync(0xffffffffu, (fw >> sh) & 1u);
    } else {
      // predicated, independent loads: one round trip for all 32
      uint32_t lv = 0u, fl = 0u;
      const int64_t r0 = static_cast<int64_t>(qb_slot(q0, b, m0)) * f.kt_words + col;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const bool in = m0 + i < m_end;
        const int64_t r = r0 + static_cast<int64_t>(i) * f.kt_words;  // slots are consecutive
        const uint32_t lw = in ? __ldg(f.qb_bits + r) : 0u;
        const uint32_t fw = in ? __ldg(f.qb_full + r) : 0u;
        lv |= ((lw >> sh) & 1u) << i;
        fl |= ((fw >> sh) & 1u) << i;
      }
      live = lv;
      full = fl;
    }
  }
  // First block m' >= m live for tile s; m_end if none.  WARP: every lane
  // of the warp calls it with the same arguments.
  template <bool WARP>
  __device__ __forceinline__ int next(const FuncMask& f, int q0, int b, int s, int m, int m_end) {
    while (m < m_end) {
      if (base < 0 || m < base || m >= base + 32) gather<WARP>(f, q0, b, s, m, m_end);
      const uint32_t rest = live >> (m - base);
      if (rest == 0u) {
        m = base + 32;
        continue;
      }
      return m + __ffs(rest) - 1;
    }
    return m_end;
  }
  // Block m (returned by next) sees every key of the tile.
  __device__ __forceinline__ bool is_full(int m) const {
    const int d = m - base;
    return d >= 0 && d < 32 && ((full >> d) & 1u) != 0u;
  }
};

// Bits [lo - base, hi - base) of an n-bit word (n = 32 or 64), clamped.
__device__ __forceinline__ uint64_t bit_range64(int lo, int hi, int base) {
  const int e0 = imin(imax(lo - base, 0), 64), e1 = imin(imax(hi - base, 0), 64);
  if (e1 <= e0) return 0;
  const uint64_t below1 = e1 >= 64 ? ~0ull : (1ull << e1) - 1;
  return below1 & ~((1ull << e0) - 1);
}
// Arbitrary mask: valid keys of query token t among keys [base, base + 64),
// cut to j < Lk, as bits (bit e: key base + e).  The caller passes the row's
// first three endpoints (e0 = F0, e1 = F1, e2 = F2, read ahead of use); the
// rest, if any, are read here.
__device__ __forceinline__ uint64_t func_row_bits3(const FuncMask& f, int64_t t, int e0, int e1,
                                                   int e2, int base, int Lk) {
  uint64_t m = bit_range64(0, imin(e0, Lk), base);
  if (f.n >= 3) m |= bit_range64(e1, imin(e2, Lk), base);
  for (int n = 3; n + 1 < f.n; n += 2)
    m |= bit_range64(__ldg(f.func + n * f.len + t), imin(__ldg(f.func + (n + 1) * f.len + t), Lk),
                     base);
  return m;
}

struct SchedArgs {
  const int32_t* cu_q;
  const int32_t* cu_k;
  int B, H;
  Window win;
  FuncMask fm;               // arbitrary mask (fm.func null: none)
  int bn_a, cmax_a, cap_a;   // list A: query tiles, inner tiles of bn_a keys
  int4* units_a;
  int bq_b, split_b, cmax_b, cap_b;  // list B: key tiles, inner tiles of bq_b queries
  int4* units_b;
  int bn_f, cmax_f, cap_f;   // list F (plans): the forward's query tiles, bn_f-key inner tiles
  int4* units_f;
  int* header;
  int* ds_base;              // backward: (B + 1) first dS block of each sequence, or null
  int* ready;                // backward: B x H readiness counts, zeroed here, or null
  int ds_cap;                // backward: dS blocks the workspace holds
  int cache_seqs;            // 1: sequence records cached in shared memory
  int stage_units;           // lists of at most this many units are staged in shared memory
  int key[kPlanKeyInts];     // plans: the sizes recorded in the header
};

// ---------------------------------------------------------------- dS blocks
// The backward stores dS (times 2, in the input dtype) as blocks of 64
// queries x 128 keys, query-major ([query][key], 256 bytes per query row),
// one block per (sequence, head, key tile j, 64-query block m) with m among
// the query blocks that can see key tile j (key_tile_queries).  Sequence b
// owns blocks [ds_base[b], ds_base[b+1]): H runs of ds_blocks_head(...)
// blocks, head-major; inside a head, key tile j's blocks start at
// ds_block_off(j, ...) and hold its query blocks in order.
constexpr int kDsKeys = 128, kDsQueries = 64;
constexpr int kDsBlockBytes = kDsKeys * kDsQueries * 2;

// The backward is one launch: each CTA runs dK/dV units, then dQ units.  Every
// row warp of a dK/dV unit of sequence b and head h (each of its two passes
// at D = 256) adds 1 to ready[b H + h] once its dS stores of the unit are
// fenced, so a call raises the count by ready_target(Lk_b), and the dS
// blocks of (b, h) are complete once it has; a dQ unit of (b, h) waits for
// that before it reads them.  The scheduler zeroes the counts and the epoch
// word; a planned call, which has no scheduling launch of its own, counts
// from epoch x target, and its last CTA advances the epoch.
__host__ __device__ inline int ready_target(int Lk, int split) {
  return kDkdvRowWarps * split * ((Lk + kDsKeys - 1) / kDsKeys);
}

// Stored blocks of key tile j: first query block and count.
__host__ __device__ inline void ds_blocks_of(int j, int Lq, int Lk, Window w, int& m0, int& n) {
  key_tile_queries(j, Lq, Lk, w, kDsQueries, m0, n);
}
// Blocks of key tiles 0 .. j-1 of one head (j at most the sequence's key
// tiles).  Causal and full have closed forms; other windows sum the tiles.
__host__ __device__ inline int ds_block_off(int j, int Lq, int Lk, Window w) {
  const int n_qb = (Lq + kDsQueries - 1) / kDsQueries;
  if (win_full(w)) return j * n_qb;
  if (win_causal(w)) {  // key tile j holds n_qb - 2 j blocks while positive
    const int jj = j < (n_qb + 1) / 2 ? j : (n_qb + 1) / 2;
    return jj * n_qb - jj * (jj - 1);
  }
  int off = 0;
  for (int t = 0; t < j; ++t) {
    int m0, n;
    ds_blocks_of(t, Lq, Lk, w, m0, n);
    off += n;
  }
  return off;
}
// Blocks of one head of a sequence.
__host__ __device__ inline int ds_blocks_head(int Lq, int Lk, Window w) {
  return ds_block_off((Lk + kDsKeys - 1) / kDsKeys, Lq, Lk, w);
}

struct AttnArgs {
  int64_t total_q, total_k;
  int H;
  Window win;
  float alpha;
  float inv_L;          // 1 / L_scale
  int* header;          // workspace header
  const int4* units;    // work list walked by this kernel (two int4 per unit)
  int units_slot;       // header word holding its length
  uint64_t timeout_ns;  // limit of every barrier wait
  int next_slot;        // header word counting units claimed so far
  int pdl_wait;         // 0: none, 1: wait for the previous grid first, 2: only before exit
  void* o0;             // fwd: out, dQ units: dq, dK/dV units: dv
  int64_t o0_st, o0_sh;
  void* o1;             // dkdv kernel: dk
  int64_t o1_st, o1_sh;
  int d_out;            // output columns per head: the kernel's D, or 32 when a
                        // head dimension of 32 runs zero-padded through the D = 64 kernels
  FuncMask fm;              // arbitrary mask (fm.func null: the window decides)
  const int* page_ids;      // forward over a paged K/V cache: page of each 128-key block
  const int* page_indptrs;  //   and each sequence's first entry in page_ids; null: contiguous K/V
  void* ds;             // backward: dS blocks (written by dK/dV, read by dQ)
  const int* ds_base;   // backward: first dS block of each sequence (B + 1)
  int ds_cap;           // backward: dS blocks the workspace holds
  int* ready;           // backward: B x H readiness counts (see ready_target)
  int planned;          // 1: the work list comes from a plan (see below)
  int part;             // list B at D = 256: 0 whole list, 1 its first half (dV pass), 2 its second
  int key[kPlanKeyInts];  // planned: this call's sizes, which must be the plan's
};

// A planned call checks that the plan was made for its sizes (else it
// records HSTU_ERR_INVALID_ARG and does no work) and returns the length of
// its work list.  Call after the grid dependency wait.
__device__ __forceinline__ int work_units(const AttnArgs& a) {
  if (a.planned) {
    // one round trip: the recorded sizes as three 16-byte loads (from L2;
    // an earlier grid wrote them), compared without short-circuiting
    const int4* k4 = reinterpret_cast<const int4*>(a.header + kHdrKey);
    const int4 r0 = __ldcg(k4), r1 = __ldcg(k4 + 1), r2 = __ldcg(k4 + 2);
    const int n = __ldcg(a.header + a.units_slot);
    const int rec[12] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w, r2.x, r2.y, r2.z, r2.w};
    bool same = true;
#pragma unroll
    for (int i = 0; i < kPlanKeyInts; ++i) same &= rec[i] == a.key[i];
    if (!same) {
      if (blockIdx.x == 0 && threadIdx.x == 0) atomicCAS(a.header + kHdrStatus, 0, kStatusBadMeta);
      return 0;
    }
    return n;
  }
  return *reinterpret_cast<volatile int*>(a.header + a.units_slot);
}

// A plan serves any number of calls in stream order, so a planned kernel
// leaves its unit counter at zero: the last CTA to finish resets it (every
// CTA has made its last claim by then).  Call once per CTA, at its end.
__device__ __forceinline__ void release_work(const AttnArgs& a) {
  if (!a.planned || threadIdx.x != 0) return;
  __threadfence();
  if (atomicAdd(a.header + kHdrDone, 1) == static_cast<int>(gridDim.x) - 1) {
    atomicExch(a.header + a.next_slot, 0);
    atomicExch(a.header + kHdrDone, 0);
  }
}

// ------------------------------------------------------------ forward config
// Separate K and V rings: a K stage frees as soon as S = Q K^T completes, a V
// stage only after O += P V, so K runs further ahead.
template <int D>
struct FwdCfg {
  static constexpr int BN = D == 256 ? 64 : 128;     // keys per inner tile
  static constexpr int NQ = D == 256 ? 1 : 2;        // Q buffers
  static constexpr int NK = 3;                       // K stages (one per S buffer)
  static constexpr int NV = D == 64 ? 6 : 2;         // V stages
  static constexpr int Q_BYTES = kBM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int TILE_BYTES = NQ * Q_BYTES + (NK + NV) * KV_BYTES;
  static constexpr int SMEM = TILE_BYTES + kCtlBytes + kAlignSlack;
};

// ------------------------------------------------------------ dQ config
// One stage: the two dS blocks of a 128-query tile against one 128-key tile
// (2 x 16 KB), and that key tile (128 x D).
template <int D>
struct DqCfg {
  static constexpr int NS = D == 64 ? 4 : (D == 128 ? 3 : 2);  // stages
  static constexpr int A_BYTES = 2 * kDsBlockBytes;
  static constexpr int K_BYTES = kDsKeys * D * 2;
  static constexpr int STAGE_BYTES = A_BYTES + K_BYTES;
  static constexpr int TILE_BYTES = NS * STAGE_BYTES;
  static constexpr int SMEM = TILE_BYTES + kCtlBytes + kAlignSlack;
};

// ------------------------------------------------------------ dK/dV config
// 64-query half-steps: S^T and dP^T are double-buffered in TMEM next to the
// accumulators, A^T and dS^T are written in place over them.  Separate Q and
// dO rings.  At D <= 128 one pass accumulates dV and dK together (PASS
// both).  At D = 256 the two fp32 accumulators would fill TMEM, so a key
// tile is visited twice: a dV pass (S^T and dV += A^T dO, no V tile, so its
// shared memory holds more Q / dO stages) and a dK pass (S^T, dP^T and
// dK += dS^T Q, dO released right after dP^T); each keeps a 256-column
// accumulator, and neither recomputes a product of the other's half.
enum : int { kPassBoth = 0, kPassDV = 1, kPassDK = 2 };
template <int D, int PASS>
struct DkdvCfg {
  static constexpr int BQ = 64;                      // queries per inner tile
  static constexpr int DH = D;                       // accumulator columns
  static constexpr int SPLIT = D == 256 ? 2 : 1;     // list-B units per key tile and head
  static constexpr bool LOAD_V = PASS != kPassDV;    // the dV pass needs no V tile
  static constexpr int NKV = PASS == kPassBoth ? 2 : 1;  // stationary (K, V) buffers
  static constexpr int NSQ = D == 64 ? 8 : D == 128 ? 3 : PASS == kPassDV ? 3 : 2;  // Q stages
  static constexpr int NSD = D == 64 ? 8 : D == 128 ? 3 : PASS == kPassDV ? 2 : 1;  // dO stages
  static constexpr int KV_BYTES = kBM * D * 2;
  static constexpr int KV_STRIDE = (LOAD_V ? 2 : 1) * KV_BYTES;  // one (K, V) buffer
  static constexpr int Q_BYTES = BQ * D * 2;
  static constexpr int TILE_BYTES = NKV * KV_STRIDE + (NSQ + NSD) * Q_BYTES;
};
// The backward kernel's tile area: the largest of its phases.
template <int D>
struct BwdCfg {
  static constexpr int T_DKDV = D == 256 ? imax(DkdvCfg<D, kPassDV>::TILE_BYTES,
                                                DkdvCfg<D, kPassDK>::TILE_BYTES)
                                         : DkdvCfg<D, kPassBoth>::TILE_BYTES;
  static constexpr int TILE_BYTES = imax(T_DKDV, DqCfg<D>::TILE_BYTES);
  static constexpr int SMEM = TILE_BYTES + kCtlBytes + kAlignSlack;
  // control block: barriers (at most kBars) | TMEM slot (8 B) | flags (16 B) | unit ring
  static constexpr int kBars = 80;
};

static_assert(FwdCfg<128>::SMEM <= 232448 && BwdCfg<128>::SMEM <= 232448, "smem");
static_assert(FwdCfg<256>::SMEM <= 232448 && BwdCfg<256>::SMEM <= 232448, "smem");
static_assert(FwdCfg<64>::SMEM <= 232448 && BwdCfg<64>::SMEM <= 232448, "smem");

__global__ void hstu_sched_kernel(const __grid_constant__ SchedArgs a);
// Arbitrary mask: key hull of every 64-row query block (grid: blocks of 8
// query blocks x sequences; one warp per query block).
cudaError_t launch_func_ranges(const int32_t* cu_q, const int32_t* cu_k, int B, int max_qb,
                               const FuncMask& fm, cudaStream_t st, bool pdl);
// Scheduler launch: `lists` blocks (1: list A only, 2: lists A and B).
cudaError_t launch_sched(int lists, int smem, cudaStream_t st, bool pdl, const SchedArgs& a);

// Launchers: return cudaErrorInvalidValue for a head_dim outside {64,128,256}.
// Tensor maps: forward (q: 128-row box, k/v: BN-row box); dq (dS blocks:
// 64 x 128 box, k: 128-row box); dkdv (k/v: 128-row box, q/do: BQ-row box,
// dk/dv: 128-row box, written by TMA stores of whole key tiles).
// Launch of a persistent attention kernel.  With `pdl` the grid may start
// while the previous grid in the stream is still running (programmatic
// dependent launch); the kernel orders itself with griddepcontrol.wait as
// AttnArgs::pdl_wait says.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_attn(void (*kern)(KArgs...), int grid, int threads, int smem,
                               cudaStream_t st, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

cudaError_t launch_fwd(int D, bool bf16, int grid, cudaStream_t st, bool pdl, const CUtensorMap& tq,
                       const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a);
// Tensor maps of the backward kernel: K, V (128-row boxes), Q, dO (the
// dK/dV query tile), dK, dV (TMA-stored whole key tiles) and the dS blocks.
struct BwdMaps {
  CUtensorMap k, v, q, dout, dk, dv, ds;
};
// The backward: dK/dV units (list B, `a`; at D = 256 its first half, the dV
// pass, and `a2` its second half, the dK pass), then dQ units (list A, `aq`).
cudaError_t launch_bwd(int D, bool bf16, int grid, cudaStream_t st, bool pdl, const BwdMaps& m,
                       const AttnArgs& a, const AttnArgs& a2, const AttnArgs& aq);
cudaError_t launch_selftest_timeout(int* header, uint64_t timeout_ns, cudaStream_t st);

}  // namespace hstu
