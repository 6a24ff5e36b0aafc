// HSTU attention forward ("HSTU Attention (Blackwell SM100/SM103)",
// Overview): O = (1/L_scale) (M (.) SiLU(alpha Q K^T)) V per sequence and head.
//
// Persistent, warp-specialised kernel; one CTA per SM walks the longest-first
// list of 128-row query tiles written by the scheduler kernel.
//   warp 0      TMA producer: Q tile per unit, K_g ahead of V_{g-2}, one
//               flat stream across units.
//   warp 1      issues S_g = Q K_g^T into TMEM buffer g % 3 as soon as K_g has
//               landed and O += P_{g-3} V_{g-3} has consumed that buffer.
//   warp 14     issues O += P_g V_g as soon as P_g and V_g are ready.
//               The tensor pipe queues only about one instruction ahead, so
//               an issuing thread that stops to wait or to do bookkeeping
//               leaves it idle; two issuers keep it fed while either waits,
//               and S runs up to three steps ahead of P V.
//   warps 2-9   SiLU row work, two warps per TMEM lane quarter: with 128-key
//               steps each takes one 64-key half of every step (warps 2-5
//               the first, 6-9 the second), so a step's SiLU takes half as
//               long and S comes back to the issuer sooner; with 64-key steps
//               (D = 256) they take alternate steps.  tcgen05.ld S, alpha
//               scale, SiLU, mask, round to 16 bits, tcgen05.st P in place
//               over the first half of the warp's S columns.
//   warps 10-13 O epilogue, one per lane quarter: O * (1/L_scale) with
//               predicated row stores; O is released as soon as it is read,
//               so the SiLU warps never stop at a unit boundary.
// No softmax, so no running max or rescale: O simply accumulates in TMEM.
// A unit only visits the key tiles its rows can see under the mask window
// (causal: up to the last row; a left bound starts later); masked entries
// are set to exactly 0, never -inf, since SiLU(-inf) is NaN.  Rows of a tile past the sequence end are computed but not stored;
// keys past it are masked, and past the tensor end TMA fills zeros.
//
// K_g and S_g share ring slot g % 3: S_g completing frees K_g, so the producer
// waits on the S barrier instead of a separate K-empty barrier.
//
// P_g (16-bit, two per column) overwrites the first half of each 64-column
// half of its own S buffer (the whole buffer's first half for 64-key steps),
// which S_{g+3} overwrites again; S_{g+3} is issued only after the commit of
// O += P_g V_g has arrived on that buffer's PV-done barrier.
#include "kernels.h"

namespace hstu {

namespace {

template <int D, bool BF16, bool FUNC>
__global__ void __launch_bounds__(kAttnThreads, 1)
    hstu_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
  using C = FwdCfg<D>;
  constexpr int BN = C::BN, NQ = C::NQ, NK = C::NK, NV = C::NV, KCH = D / 64;
  constexpr int LBN = BN == 64 ? 6 : 7;  // log2 BN
  constexpr int NSB = 3;        // S buffers in TMEM
  constexpr int NCH = BN / 64;  // 64-column chunks of one S tile
  // 128-key steps: the two SiLU warps of a lane quarter split every step's
  // columns (64 each), so a step's SiLU takes half as long; each writes its
  // P over the first half of its own 64 S columns.  64-key steps (D = 256):
  // the two warps take alternate steps and P fills the buffer's first half.
  constexpr bool SPLIT = NCH == 2;
  static_assert(NK == NSB, "K slot g % NSB is freed by the S_g barrier");
  constexpr uint32_t IDESC_S = idesc_f16(BF16, kBM, BN, false, false);
  constexpr uint32_t IDESC_PV = idesc_f16(BF16, kBM, D, false, true);
  // TMEM columns: S0 | S1 | S2 | O.  P_g is packed two per column into the
  // first half of its S buffer.
  constexpr uint32_t COL_S = 0, COL_O = NSB * BN;
  static_assert(COL_O + D <= kTmemCols, "TMEM budget");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sQ = base;
  const uint32_t sK = sQ + NQ * C::Q_BYTES;
  const uint32_t sV = sK + NK * C::KV_BYTES;

  enum {
    QFULL = 0, QEMPTY = QFULL + NQ, KFULL = QEMPTY + NQ,
    VFULL = KFULL + NK, VEMPTY = VFULL + NV, SFULL = VEMPTY + NV, PFULL = SFULL + NSB,
    PVDONE = PFULL + NSB, OFULL = PVDONE + NSB, OEMPTY = OFULL + 1, UFULL = OEMPTY + 1,
    UEMPTY = UFULL + kUnitRing, DRAIN = UEMPTY + kUnitRing, NBARS = DRAIN + 2
  };
  // control block: barriers | TMEM slot (8 B) | flags (16 B) | unit ring
  static_assert(NBARS * 8 + 24 + kUnitRing * sizeof(UnitInfo) <= kCtlBytes, "control block");
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + C::TILE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [0] abort, [1] 0
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NQ; ++i) { mbar_init(bar(QFULL + i), 1); mbar_init(bar(QEMPTY + i), 1); }
    for (int i = 0; i < NK; ++i) mbar_init(bar(KFULL + i), 1);
    for (int i = 0; i < NV; ++i) { mbar_init(bar(VFULL + i), 1); mbar_init(bar(VEMPTY + i), 1); }
    for (int i = 0; i < NSB; ++i) {
      mbar_init(bar(SFULL + i), 1);
      mbar_init(bar(PFULL + i), SPLIT ? kFwdRowWarps : 4);  // every SiLU warp of the step
      mbar_init(bar(PVDONE + i), 1);
    }
    mbar_init(bar(OFULL), 1);
    mbar_init(bar(OEMPTY), kFwdEpiWarps);
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(bar(UFULL + i), 1);
      mbar_init(bar(UEMPTY + i), 2 + kFwdRowWarps + kFwdEpiWarps);
    }
    mbar_init(bar(DRAIN), 1);
    mbar_init(bar(DRAIN + 1), 1);
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q); tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) { tmem_alloc(smem_u32(tmem_slot), kTmemCols); tmem_relinquish(); }
  __syncwarp();  // thread 0's set-up above diverged warp 0
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{a.header, flags, a.timeout_ns};
  const WaitCtl drain{a.header, flags + 1, a.timeout_ns};
  // everything below reads what earlier grids wrote (work list, inputs)
  if (a.pdl_wait == 1) grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();
  const int n_units = work_units(a);
  const UnitQueue uq{reinterpret_cast<UnitInfo*>(const_cast<int*>(flags + 4)), bar(UFULL), bar(UEMPTY)};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // One flat stream over all of this CTA's units: Q of a unit before its
    // first K, and K_g before V_{g-LA} (S runs ahead of P V).  The next
    // unit's Q and first K tiles therefore go out before this unit's last V
    // tiles, so a unit boundary does not wait for a fresh load.
    if (lane == 0) {
      uint32_t qi = 0, ki = 0, vi = 0;
      auto load_kv = [&](const CUtensorMap* map, uint32_t base_s, int nst, uint32_t& cnt,
                         int full, int empty, int row, int h, int where) -> bool {
        const int s = cnt % nst;
        if (!wait_bar(bar(empty + s), ((cnt / nst) & 1) ^ 1, wc, where)) return false;
        mbar_arrive_expect_tx(bar(full + s), C::KV_BYTES);
#pragma unroll
        for (int c = 0; c < KCH; ++c)
          tma_load_3d(base_s + s * C::KV_BYTES + c * (BN * 128), map, bar(full + s), 64 * c, h, row);
        ++cnt;
        return true;
      };
      // V loads not yet issued (at most LA of them): key row and head
      constexpr int LA = 2;
      int v_row0 = 0, v_h0 = 0, v_row1 = 0, v_h1 = 0, nv = 0;
      bool ok = true;
      // units are claimed one ahead: the next claim overlaps this unit's loads
      // the first unit of each CTA is its own index; later ones come from the counter
      UnitInfo nx = load_unit_info(a.units, blockIdx.x, n_units);
      for (uint32_t uk = 0; ok; ++uk) {
        const UnitInfo U = nx;
        if (!unit_push(uq, uk, U, wc)) { ok = false; break; }
        if (U.n < 0) break;
        nx = load_unit_info(a.units, gridDim.x + atomicAdd(a.header + a.next_slot, 1), n_units);
        if (U.n <= 0) continue;
        const int h = U.hz;
        const int q_row0 = U.q0 + kBM * U.tile;
        // the unit's key tiles: kt0 .. kt0 + U.n - 1, or under an arbitrary
        // mask the U.n live tiles of the hull [kt0, kt_end)
        int kt0, nkt, kt_end = 0;
        if constexpr (FUNC) {
          const int2 hk = func_tile_keys(a.fm, U.q0, U.b, U.tile, U.Lq);
          kt0 = hk.x / BN;
          kt_end = (hk.y + BN - 1) / BN;
        } else {
          query_tile_keys(U.tile, U.Lq, U.Lk, a.win, BN, kt0, nkt);
        }
        const int kv_row0 = U.k0 + BN * kt0;
        int kt_next = kt0;  // live-tile cursor
        TileWalk tw;  // arbitrary mask: the unit's live tiles, 32 per bit word
        if constexpr (FUNC) tw.init(a.fm, U.q0, U.b, U.tile, U.Lq);
        // Paged K/V: key tile kt lives in page page_ids[page_indptrs[b] +
        // kt BN / 128], whose K rows start at row 256 p and V rows at
        // 256 p + 128 of the cache's map.  The next tile's page is looked up
        // one tile ahead, so the lookup is off the load path.
        const bool paged = a.page_ids != nullptr;
        int pi0 = 0, pg_next = 0;
        if (paged) {
          pi0 = __ldg(a.page_indptrs + U.b);
          pg_next = __ldg(a.page_ids + pi0 + (kt0 * BN) / 128);
        }
        const int qb = qi % NQ;
        if (!wait_bar(bar(QEMPTY + qb), ((qi / NQ) & 1) ^ 1, wc, 0x001)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(QFULL + qb), C::Q_BYTES);
#pragma unroll
        for (int c = 0; c < KCH; ++c)
          tma_load_3d(sQ + qb * C::Q_BYTES + c * (kBM * 128), &tm_q, bar(QFULL + qb), 64 * c, h,
                      q_row0);
        ++qi;
        // No L2 warm-up here: measured, the extra prefetch requests slowed
        // the forward's own tile loads more than they saved.
        for (int n = 0; n < U.n; ++n) {
          int row = kv_row0 + BN * n, vrow = row;
          if constexpr (FUNC) {
            const int kt = tw.next(kt_next, kt_end, LBN);
            kt_next = kt + 1;
            row = vrow = U.k0 + BN * kt;
          }
          if (paged) {
            const int kt = kt0 + n, pg = pg_next;
            if (n + 1 < U.n) pg_next = __ldg(a.page_ids + pi0 + ((kt + 1) * BN) / 128);
            row = 256 * pg + (kt * BN) % 128;
            vrow = row + 128;
          }
          if (!load_kv(&tm_k, sK, NK, ki, KFULL, SFULL, row, h, 0x002)) { ok = false; break; }
          if (nv == LA) {
            if (!load_kv(&tm_v, sV, NV, vi, VFULL, VEMPTY, v_row0, v_h0, 0x003)) { ok = false; break; }
            v_row0 = v_row1; v_h0 = v_h1;
            v_row1 = vrow; v_h1 = h;
          } else if (nv == 1) {
            v_row1 = vrow; v_h1 = h; nv = 2;
          } else {
            v_row0 = vrow; v_h0 = h; nv = 1;
          }
        }
      }
      if (ok && nv >= 1) ok = load_kv(&tm_v, sV, NV, vi, VFULL, VEMPTY, v_row0, v_h0, 0x003);
      if (ok && nv == 2) ok = load_kv(&tm_v, sV, NV, vi, VFULL, VEMPTY, v_row1, v_h1, 0x003);
      // let the last copies land before the block may exit
      for (uint32_t i = qi > NQ ? qi - NQ : 0; i < qi; ++i)
        wait_bar(bar(QFULL + i % NQ), (i / NQ) & 1, drain, 0x0f1);
      for (uint32_t i = ki > NK ? ki - NK : 0; i < ki; ++i)
        wait_bar(bar(KFULL + i % NK), (i / NK) & 1, drain, 0x0f2);
      for (uint32_t i = vi > NV ? vi - NV : 0; i < vi; ++i)
        wait_bar(bar(VFULL + i % NV), (i / NV) & 1, drain, 0x0f3);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S issuer
    if (lane == 0) {
      uint32_t qi = 0, ki = 0, g = 0;
      bool ok = true;
      for (uint32_t uk = 0; ok; ++uk) {
        UnitInfo U;
        if (!unit_pop(uq, uk, U, wc)) { ok = false; break; }
        if (U.n < 0) break;
        const int un = U.n;
        if (un <= 0) continue;
        const int qb = qi % NQ;
        if (!wait_bar(bar(QFULL + qb), (qi / NQ) & 1, wc, 0x104)) { ok = false; break; }
        const SDesc qd = kdesc(sQ + qb * C::Q_BYTES);
        for (int n = 0; n < un; ++n, ++ki, ++g) {
          const int ks = ki % NK, sb = g % NSB;
          if (!wait_bar(bar(KFULL + ks), (ki / NK) & 1, wc, 0x105)) { ok = false; break; }
          // buffer sb last held P_{g-3}: O += P_{g-3} V_{g-3} must have read it
          if (g >= NSB) {
            if (!wait_bar(bar(PVDONE + sb), ((g / NSB) - 1) & 1, wc, 0x106)) { ok = false; break; }
            tc_fence_after();
          }
          const SDesc kd = kdesc(sK + ks * C::KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + COL_S + sb * BN, desc_kmajor<kBM>(qd, kk), desc_kmajor<BN>(kd, kk),
                   IDESC_S, kk > 0 ? 1u : 0u);
          mma_commit(bar(SFULL + sb));  // also frees K slot ks == sb
          if (n == un - 1) mma_commit(bar(QEMPTY + qb));
        }
        ++qi;
      }
      mma_commit(bar(DRAIN));
      wait_bar(bar(DRAIN), 0, drain, 0x1ff);
    }
  } else if (warp == kFwdPvWarp) {
    // ------------------------------------------------------------ P V issuer
    if (lane == 0) {
      const uint32_t tO = tmem + COL_O;
      uint32_t vi = 0, g = 0, oi = 0;
      bool ok = true;
      for (uint32_t uk = 0; ok; ++uk) {
        UnitInfo U;
        if (!unit_pop(uq, uk, U, wc)) { ok = false; break; }
        if (U.n < 0) break;
        const int un = U.n;
        if (un <= 0) continue;
        for (int n = 0; n < un; ++n, ++vi, ++g) {
          const int vs = vi % NV, sb = g % NSB;
          if (!wait_bar(bar(VFULL + vs), (vi / NV) & 1, wc, 0x101)) { ok = false; break; }
          if (!wait_bar(bar(PFULL + sb), (g / NSB) & 1, wc, 0x102)) { ok = false; break; }
          if (n == 0 && !wait_bar(bar(OEMPTY), (oi & 1) ^ 1, wc, 0x103)) { ok = false; break; }
          tc_fence_after();
          const SDesc vd = mndesc<BN>(sV + vs * C::KV_BYTES);
          const uint32_t tP = tmem + COL_S + sb * BN;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)  // P of keys [16 kk, 16 kk + 16): 8 columns,
            mma_ts(tO, tP + 8 * kk + (SPLIT ? 32 * (kk / 4) : 0),  // at 64 h + .. for key half h
                   desc_mnmajor<BN>(vd, kk, 0), IDESC_PV, (n > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(VEMPTY + vs));
          mma_commit(bar(PVDONE + sb));
          if (n == un - 1) mma_commit(bar(OFULL));
        }
        ++oi;
      }
      mma_commit(bar(DRAIN + 1));
      wait_bar(bar(DRAIN + 1), 0, drain, 0x1fe);
    }
  } else if (warp < 2 + kFwdRowWarps) {
    // ------------------------------------------------------------ SiLU
    // Warp w owns TMEM lane quarter w % 4 (its 32 rows).  With 128-key steps
    // it takes the 64-column half par of every step and writes P over that
    // half's first 32 columns; with 64-key steps it takes the steps of parity
    // par and writes P over the buffer's first half.
    const int wq = warp & 3, par = (warp - 2) >> 2;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + COL_S + lane_off;
    const float half_alpha = 0.5f * a.alpha;
    uint32_t g = 0;
    bool ok = true;
    for (uint32_t uk = 0; ok; ++uk) {
      UnitInfo U;
      if (!unit_pop_warp(uq, uk, U, wc)) { ok = false; break; }
      if (U.n < 0) break;
      const int Lk = U.Lk;
      const int i = kBM * U.tile + r;
      const int i_warp = kBM * U.tile + wq * 32;  // first row of this warp
      int kt0, nkt, kt_end = 0;
      constexpr bool func = FUNC;  // arbitrary mask: a separate instantiation
      if constexpr (func) {
        const int2 hk = func_tile_keys(a.fm, U.q0, U.b, U.tile, U.Lq);
        kt0 = hk.x / BN;
        kt_end = (hk.y + BN - 1) / BN;
      } else {
        query_tile_keys(U.tile, U.Lq, Lk, a.win, BN, kt0, nkt);
      }
      int kt_next = kt0;  // live-tile cursor (arbitrary mask)
      TileWalk tw;
      if constexpr (func) tw.init(a.fm, U.q0, U.b, U.tile, U.Lq);
      // arbitrary mask: this row's first endpoints, read once per unit
      int fe0 = 0, fe1 = 0, fe2 = 0;
      if constexpr (func) {
        const int64_t tr = static_cast<int64_t>(U.q0) + (i < U.Lq ? i : 0);
        fe0 = __ldg(a.fm.func + tr);
        if (a.fm.n >= 3) {
          fe1 = __ldg(a.fm.func + a.fm.len + tr);
          fe2 = __ldg(a.fm.func + 2 * a.fm.len + tr);
        }
      }
      const int64_t t_row = static_cast<int64_t>(U.q0) + (i < U.Lq ? i : 0);  // func row (any, if past Lq)
      // valid keys of this row: lo <= j < hi; every row of the warp sees
      // [lo_all, hi_all)
      const int lo = a.win.left < 0 ? 0 : i - a.win.left;
      const int hi = a.win.right < 0 ? Lk : min(Lk, i + a.win.right + 1);
      const int lo_all = a.win.left < 0 ? 0 : i_warp + 31 - a.win.left;
      const int hi_all = a.win.right < 0 ? Lk : min(Lk, i_warp + a.win.right + 1);
      for (int n = 0; n < U.n; ++n, ++g) {
        int kt = kt0 + n;
        if constexpr (func) {  // every warp walks every step to keep the cursor
          kt = tw.next(kt_next, kt_end, LBN);
          kt_next = kt + 1;
        }
        if (!SPLIT && static_cast<int>(g & 1) != par) continue;
        const int sb = g % NSB;
        // this warp's 64-column chunks of the step: its half (split steps) or all
        constexpr int C_N = SPLIT ? 1 : NCH;
        // arbitrary mask: the row's valid keys of each chunk, formed while S lands
        uint64_t fbs[C_N];
        if constexpr (func) {
#pragma unroll
          for (int ci = 0; ci < C_N; ++ci)
            fbs[ci] = func_row_bits3(a.fm, t_row, fe0, fe1, fe2, BN * kt + 64 * (SPLIT ? par : ci),
                                     Lk);
        }
        if (!wait_bar_warp(bar(SFULL + sb), (g / NSB) & 1, wc, 0x201)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int ci = 0; ci < C_N; ++ci) {
          const int c = SPLIT ? par : ci;
          const int jc = BN * kt + 64 * c;  // first key of this chunk
          const bool need_mask = jc < lo_all || jc + 64 > hi_all;
          uint32_t x[64];
          tmem_ld64(tS + sb * BN + 64 * c, x);
          uint32_t p[32];
          if (func && !__all_sync(0xffffffffu, fbs[ci] == ~0ull)) {
            // arbitrary mask, some key of the chunk invalid for some row
            const uint64_t fb = fbs[ci];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const uint32_t s0 = ((fb >> (2 * e)) & 1ull) ? x[2 * e] : 0u;
              const uint32_t s1 = ((fb >> (2 * e + 1)) & 1ull) ? x[2 * e + 1] : 0u;
              p[e] = silu_pair<BF16>(s0, s1, half_alpha);
            }
          } else if (func || !need_mask) {
#pragma unroll
            for (int e = 0; e < 32; ++e) p[e] = silu_pair<BF16>(x[2 * e], x[2 * e + 1], half_alpha);
          } else if (jc >= lo_all) {
            // only the upper bound (the diagonal or the sequence end) cuts
            // this chunk: every causal and full mask chunk
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int j = jc + 2 * e;
              const uint32_t s0 = j < hi ? x[2 * e] : 0u;  // SiLU(0) = 0
              const uint32_t s1 = j + 1 < hi ? x[2 * e + 1] : 0u;
              p[e] = silu_pair<BF16>(s0, s1, half_alpha);
            }
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int j = jc + 2 * e;
              const uint32_t s0 = (j >= lo && j < hi) ? x[2 * e] : 0u;
              const uint32_t s1 = (j + 1 >= lo && j + 1 < hi) ? x[2 * e + 1] : 0u;
              p[e] = silu_pair<BF16>(s0, s1, half_alpha);
            }
          }
          // split steps: P over this chunk's own first 32 columns; otherwise
          // columns [32 c, 32 c + 32), read by this chunk or the one before
          tmem_st32(tS + sb * BN + (SPLIT ? 64 : 32) * c, p);
        }
        tmem_st_wait();
        warp_arrive(bar(PFULL + sb));
      }
    }
  } else if (warp < kFwdPvWarp) {
    // ------------------------------------------------------------ O epilogue
    // Warp w owns TMEM lane quarter w % 4: it reads its 32 rows of O in
    // 64-column chunks, releases O once every chunk is in registers or
    // stored, and scales, rounds and stores the rows.
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const uint32_t tO = tmem + COL_O + (static_cast<uint32_t>(wq * 32) << 16);
    uint32_t oi = 0;
    bool ok = true;
    for (uint32_t uk = 0; ok; ++uk) {
      UnitInfo U;
      if (!unit_pop_warp(uq, uk, U, wc)) { ok = false; break; }
      if (U.n < 0) break;
      const int h = U.hz;
      const int i = kBM * U.tile + r;
      const int64_t grow = static_cast<int64_t>(U.q0) + i;
      const bool row_ok = i < U.Lq && grow < a.total_q;
      char* orow = static_cast<char*>(a.o0) +
                   (grow * a.o0_st + static_cast<int64_t>(h) * a.o0_sh) * 2;
      if (U.n <= 0) {
        if (row_ok) {
          if (D == 64 && a.d_out == 32) store_zero_n<32>(orow);  // zero-padded head dim 32
          else store_zero_n<D>(orow);
        }
        continue;
      }
      if (!wait_bar_warp(bar(OFULL), oi & 1, wc, 0x202)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t x[64];
        tmem_ld64(tO + 64 * c, x);
        if (c == D / 64 - 1) warp_arrive(bar(OEMPTY));  // every O column is read
        if (row_ok) {
          if (D == 64 && a.d_out == 32) store_row_head<32, 64, BF16>(orow, x, a.inv_L);
          else store_row_n<64, BF16>(orow + c * 128, x, a.inv_L);
        }
      }
      ++oi;
    }
  }

  // The role branches leave lanes of warps 0, 1 and 14 on different paths;
  // reconverge each warp so the aligned CTA barrier counts it exactly once
  // (otherwise it can release before the row warps finish reading TMEM).
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  release_work(a);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool BF16, bool FUNC>
cudaError_t launch_fwd_f(int grid, cudaStream_t st, bool pdl, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const AttnArgs& a) {
  auto kern = hstu_fwd_kernel<D, BF16, FUNC>;
  static bool attr_set = false;  // benign race: setting the attribute twice is harmless
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FwdCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_attn(kern, grid, kAttnThreads, FwdCfg<D>::SMEM, st, pdl, tq, tk, tv, a);
}

// The arbitrary-mask SiLU path is a separate instantiation, so that the
// window kernels keep their code size and registers.
template <int D, bool BF16>
cudaError_t launch_fwd_t(int grid, cudaStream_t st, bool pdl, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const AttnArgs& a) {
  if (a.fm.func != nullptr) return launch_fwd_f<D, BF16, true>(grid, st, pdl, tq, tk, tv, a);
  return launch_fwd_f<D, BF16, false>(grid, st, pdl, tq, tk, tv, a);
}

}  // namespace

cudaError_t launch_fwd(int D, bool bf16, int grid, cudaStream_t st, bool pdl, const CUtensorMap& tq,
                       const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a) {
  switch (D) {
    case 64: return bf16 ? launch_fwd_t<64, true>(grid, st, pdl, tq, tk, tv, a)
                         : launch_fwd_t<64, false>(grid, st, pdl, tq, tk, tv, a);
    case 128: return bf16 ? launch_fwd_t<128, true>(grid, st, pdl, tq, tk, tv, a)
                          : launch_fwd_t<128, false>(grid, st, pdl, tq, tk, tv, a);
    case 256: return bf16 ? launch_fwd_t<256, true>(grid, st, pdl, tq, tk, tv, a)
                          : launch_fwd_t<256, false>(grid, st, pdl, tq, tk, tv, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hstu
