// HSTU attention backward, dQ part: dQ_i = (alpha/L_scale) sum_j dS'_ij k_j
// with dS'_ij = M_ij <dO_i, v_j> SiLU'(alpha q_i.k_j) (chain rule of "HSTU
// Attention (Blackwell SM100/SM103)", Overview equations).
//
// The dK/dV units already form dS' for every (key tile, 64-query block) the
// mask leaves non-empty and stores it (doubled, 16-bit) in the workspace;
// this phase is the remaining contraction dQ = dS' K, a plain tensor-core
// GEMM with no recomputation of S or dP.  It runs in the backward kernel
// after the CTA's dK/dV units (same launch, same shared memory and TMEM), so
// a dQ unit starts as soon as the dK/dV units of its sequence and head have
// stored their dS blocks (the readiness counts), not after the slowest CTA's
// last dK/dV unit and a second launch.  Query-stationary and atomic-free on
// data: each 128-row query tile is owned by one CTA, which streams the tile's
// two dS blocks and the matching key tile per 128-key step and accumulates
// dQ in TMEM, so results do not depend on scheduling.
//   warp 0      TMA: per step the two 64-query dS blocks (16 KB each) and
//               the 128-key K tile into one ring stage; the blocks land as
//               rows 0-63 and 64-127 of one K-major 128 x 128 A tile.
//   warp 1      tcgen05 issuer: dQ (+)= dS K, A = dS K-major, B = K read
//               N-major; two TMEM accumulators, so one unit's epilogue
//               overlaps the next unit's MMAs.
//   warps 2-5   epilogue, one per TMEM lane quarter: dQ * alpha / (2 L_scale)
//               with predicated row stores.
// Rows of a tile past the sequence end (or a second dS block the sequence
// does not have) are computed from stale shared memory but never stored:
// each output row depends only on its own A row.
#pragma once

#include "kernels.h"

namespace hstu {
namespace dq {

// Barrier slots of the dQ phase (NS ring stages, two TMEM accumulators).
template <int D>
struct Bars {
  static constexpr int NS = DqCfg<D>::NS, NACC = 2;
  enum {
    FULL = 0, EMPTY = FULL + NS, ACCFULL = EMPTY + NS, ACCEMPTY = ACCFULL + NACC,
    UFULL = ACCEMPTY + NACC, UEMPTY = UFULL + kUnitRing, DRAIN = UEMPTY + kUnitRing,
    NBARS = DRAIN + 1
  };
};

// Thread 0 initialises the phase's barriers at `bars`.
template <int D>
__device__ __forceinline__ void init_bars(uint64_t* bars) {
  using B = Bars<D>;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  for (int i = 0; i < B::NS; ++i) { mbar_init(bar(B::FULL + i), 1); mbar_init(bar(B::EMPTY + i), 1); }
  for (int i = 0; i < B::NACC; ++i) {
    mbar_init(bar(B::ACCFULL + i), 1);
    mbar_init(bar(B::ACCEMPTY + i), kDqEpiWarps);
  }
  for (int i = 0; i < kUnitRing; ++i) {
    mbar_init(bar(B::UFULL + i), 1);
    mbar_init(bar(B::UEMPTY + i), 1 + kDqEpiWarps);
  }
  mbar_init(bar(B::DRAIN), 1);
  fence_mbar_init();
}

// The dQ phase: warp 0 TMA, warp 1 MMA issuer, warps 2-5 epilogue; other
// warps return at once.  `base` is the 1024-aligned tile area, `bars` the
// barriers set up by init_bars, `ring` the unit ring, `tmem` the CTA's TMEM
// (2 D columns used).  The caller synchronises the block afterwards.
template <int D, bool BF16>
__device__ __forceinline__ void run(const CUtensorMap* tm_ds, const CUtensorMap* tm_k,
                                    const AttnArgs& a, uint32_t base, uint64_t* bars,
                                    volatile int* flags, UnitInfo* ring, uint32_t tmem) {
  using C = DqCfg<D>;
  using B = Bars<D>;
  constexpr int NS = C::NS, KCH = D / 64, NACC = B::NACC;
  constexpr uint32_t IDESC = idesc_f16(BF16, kBM, D, false, true);
  static_assert(NACC * D <= kTmemCols, "TMEM budget");
  enum { FULL = B::FULL, EMPTY = B::EMPTY, ACCFULL = B::ACCFULL, ACCEMPTY = B::ACCEMPTY,
         UFULL = B::UFULL, UEMPTY = B::UEMPTY, DRAIN = B::DRAIN };
  auto stage_a = [&](int s) { return base + s * C::STAGE_BYTES; };
  auto stage_k = [&](int s) { return base + s * C::STAGE_BYTES + C::A_BYTES; };
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const WaitCtl wc{a.header, flags, a.timeout_ns};
  const WaitCtl drain{a.header, flags + 1, a.timeout_ns};
  const int n_units = work_units(a);
  const UnitQueue uq{ring, bar(UFULL), bar(UEMPTY)};
  const int split = D == 256 ? 2 : 1;  // dK/dV units per key tile and head

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t g = 0;
      bool ok = true;
      // planned calls count on from the calls before (see ready_target)
      const uint32_t epoch =
          a.ready != nullptr && a.planned ? static_cast<uint32_t>(__ldcg(a.header + kHdrEpoch)) : 0u;
      // metadata beyond the sizes dropped dK/dV units (the call reports an
      // invalid argument): their counts would never complete, so skip the waits
      const bool counted = a.ready != nullptr && __ldcg(a.header + kHdrOverflowB) == 0;
      // the last read of each dS block: its lines may leave L2 first
      const uint64_t ds_policy = l2_policy_evict_first();
      UnitInfo nx = load_unit_info(a.units, blockIdx.x, n_units);
      for (uint32_t uk = 0; ok; ++uk) {
        const UnitInfo U = nx;
        if (!unit_push(uq, uk, U, wc)) { ok = false; break; }
        if (U.n < 0) break;
        nx = load_unit_info(a.units, gridDim.x + atomicAdd(a.header + a.next_slot, 1), n_units);
        if (U.n <= 0) continue;
        const int h = U.hz, i = U.tile;
        const int n_qb = (U.Lq + kDsQueries - 1) / kDsQueries;
        const int b0 = __ldg(a.ds_base + U.b), b1 = __ldg(a.ds_base + U.b + 1);
        const int head_blk = b0 + h * ((b1 - b0) / a.H);  // this head's first block
        const bool second = 2 * i + 1 < n_qb;            // the tile's upper 64 queries exist
        const uint32_t bytes = (second ? 2 : 1) * kDsBlockBytes + C::K_BYTES;
        // the unit's key tiles: kt0 .. kt0 + U.n - 1, or under an arbitrary
        // mask the U.n live tiles of the hull [kt0, kt_end)
        int kt0, nkt, kt_end = 0;
        const bool func = a.fm.func != nullptr;
        if (func) {
          const int2 hk = func_tile_keys(a.fm, U.q0, U.b, i, U.Lq);
          kt0 = hk.x / kDsKeys;
          kt_end = (hk.y + kDsKeys - 1) / kDsKeys;
        } else {
          query_tile_keys(i, U.Lq, U.Lk, a.win, kDsKeys, kt0, nkt);
        }
        // blocks of the key tiles before (an arbitrary mask keeps n_qb slots per
        // key tile, the full mask's layout)
        int off = ds_block_off(kt0, U.Lq, U.Lk, a.win);
        // the dS blocks of (b, h) are read only once all its dK/dV units stored them
        if (counted) {
          const uint32_t target = static_cast<uint32_t>(ready_target(U.Lk, split));
          if (!wait_count(a.ready + U.b * a.H + h, epoch * target, target, a.header, flags,
                          a.timeout_ns, 0x007)) {
            ok = false;
            break;
          }
        }
        int kt_next = kt0;  // live-tile cursor (arbitrary mask)
        TileWalk tw;  // the unit's live tiles, 32 per bit word
        if (func) tw.init(a.fm, U.q0, U.b, i, U.Lq);
        for (int jj = 0; jj < U.n; ++jj, ++g) {
          const int s = g % NS;
          int j = kt0 + jj;
          if (func) {
            j = tw.next(kt_next, kt_end, 7);
            kt_next = j + 1;
            off = j * n_qb;  // the full mask's layout
          }
          if (!wait_bar(bar(EMPTY + s), ((g / NS) & 1) ^ 1, wc, 0x002)) { ok = false; break; }
          // query blocks 2i and 2i + 1 of key tile j; a block the mask leaves
          // empty was never stored and is read as zeros from an out-of-range
          // block index (the TMA fill; the box still counts in full)
          int m0, cnt;
          bool live0 = true, live1 = true;
          if (func) {
            const int2 r = a.fm.kt_range[kt_slot(U.k0, U.b, j)];
            m0 = r.x;
            cnt = r.y;
            live0 = tw.live(j, false);
            live1 = second && tw.live(j, true);
          } else {
            ds_blocks_of(j, U.Lq, U.Lk, a.win, m0, cnt);
          }
          const int blk0 =
              (live0 && 2 * i >= m0 && 2 * i < m0 + cnt) ? head_blk + off + 2 * i - m0 : -1;
          const int blk1 = (live1 && 2 * i + 1 >= m0 && 2 * i + 1 < m0 + cnt)
                               ? head_blk + off + 2 * i + 1 - m0
                               : -1;
          if (!func) off += cnt;
          mbar_arrive_expect_tx(bar(FULL + s), bytes);
          // A tile: 64-key chunk c of query rows 0-63 (block 2i) and 64-127 (2i + 1)
#pragma unroll
          for (int c = 0; c < kDsKeys / 64; ++c) {
            tma_load_3d_hint(stage_a(s) + c * (kBM * 128), tm_ds, bar(FULL + s), 64 * c, 0, blk0,
                             ds_policy);
            if (second)
              tma_load_3d_hint(stage_a(s) + c * (kBM * 128) + kDsQueries * 128, tm_ds,
                               bar(FULL + s), 64 * c, 0, blk1, ds_policy);
          }
#pragma unroll
          for (int c = 0; c < KCH; ++c)
            tma_load_3d(stage_k(s) + c * (kDsKeys * 128), tm_k, bar(FULL + s), 64 * c, h,
                        U.k0 + kDsKeys * j);
        }
      }
      for (uint32_t i = g > NS ? g - NS : 0; i < g; ++i)
        wait_bar(bar(FULL + i % NS), (i / NS) & 1, drain, 0x0f1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t g = 0, oi = 0;
      bool ok = true;
      for (uint32_t uk = 0; ok; ++uk) {
        UnitInfo U;
        if (!unit_pop(uq, uk, U, wc)) { ok = false; break; }
        if (U.n < 0) break;
        if (U.n <= 0) continue;
        const int ab = oi % NACC;
        const uint32_t tAcc = tmem + ab * D;
        if (!wait_bar(bar(ACCEMPTY + ab), ((oi / NACC) & 1) ^ 1, wc, 0x103)) { ok = false; break; }
        tc_fence_after();
        for (int j = 0; j < U.n; ++j, ++g) {
          const int s = g % NS;
          if (!wait_bar(bar(FULL + s), (g / NS) & 1, wc, 0x106)) { ok = false; break; }
          // A: dS, M = 128 query rows, K = keys in 64-key chunks 16 KB apart;
          // B: K tile, N = D in 64-column chunks, K = keys down the rows.
          const SDesc ad = kdesc(stage_a(s));
          const SDesc kd = mndesc<kDsKeys>(stage_k(s));
#pragma unroll
          for (int kk = 0; kk < kDsKeys / 16; ++kk)
            mma_ss(tAcc, desc_kmajor<kBM>(ad, kk), desc_mnmajor<kDsKeys>(kd, kk, 0), IDESC,
                   (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(EMPTY + s));
        }
        if (!ok) break;
        mma_commit(bar(ACCFULL + ab));
        ++oi;
      }
      mma_commit(bar(DRAIN));
      wait_bar(bar(DRAIN), 0, drain, 0x1ff);
    }
  } else if (warp < 2 + kDqEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const float out_scale = 0.5f * a.alpha * a.inv_L;  // dS is stored doubled
    uint32_t oi = 0;
    bool ok = true;
    for (uint32_t uk = 0; ok; ++uk) {
      UnitInfo U;
      if (!unit_pop_warp(uq, uk, U, wc)) { ok = false; break; }
      if (U.n < 0) break;
      const int i = kBM * U.tile + r;
      const int64_t grow = static_cast<int64_t>(U.q0) + i;
      const bool row_ok = i < U.Lq && grow < a.total_q;
      char* orow = static_cast<char*>(a.o0) +
                   (grow * a.o0_st + static_cast<int64_t>(U.hz) * a.o0_sh) * 2;
      if (U.n <= 0) {
        if (row_ok) {
          if (D == 64 && a.d_out == 32) store_zero_n<32>(orow);  // zero-padded head dim 32
          else store_zero_n<D>(orow);
        }
        continue;
      }
      const int ab = oi % NACC;
      if (!wait_bar_warp(bar(ACCFULL + ab), (oi / NACC) & 1, wc, 0x202)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tAcc = tmem + ab * D + lane_off;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t x[32];
        tmem_ld32(tAcc + 32 * c, x);
        if (c == D / 32 - 1) warp_arrive(bar(ACCEMPTY + ab));  // every column is read
        if (row_ok && 32 * c < a.d_out) store_row_n<32, BF16>(orow + c * 64, x, out_scale);
      }
      ++oi;
    }
  }
}

}  // namespace dq
}  // namespace hstu
