// HSTU attention backward, dQ part: dQ_i = (alpha/L_scale) sum_j
// M_ij <dO_i, v_j> SiLU'(alpha q_i.k_j) k_j (chain rule of "HSTU Attention
// (Blackwell SM100/SM103)", Overview equations).
//
// Query-stationary and atomic-free: each 128-row query tile is owned by one
// CTA, which recomputes S = Q K^T and dP = dO V^T per key step, forms
// dS = M (.) dP (.) SiLU'(alpha S) in registers, stores it to TMEM as 16-bit,
// and accumulates dQ += dS K in TMEM.  The alpha/L_scale factor is applied
// once in the fp32 epilogue.
//   warp 0       TMA: Q and dO per unit, K and V per step (one barrier per
//                step for both).
//   warp 1       tcgen05 issuer of S_g and dP_g (once the row warps have loaded
//                S_{g-1} and dP_{g-1}).
//   warp 18      tcgen05 issuer of dQ += dS_g K_g (once dS_g is written).
//   warps 2-17   row work, four warps per TMEM lane quarter (one per quarter
//                of the key columns): load S and dP, release them (and the V
//                stage), SiLU' and mask, store dS; then the dQ epilogue.
// TMEM: S | dP | dQ | dS0 | dS1.
//
// A tcgen05.mma costs about 47 cycles of tensor-pipe intake whatever its size
// (M = 128) and the pipe queues only about one instruction ahead, so 128-key
// steps keep every instruction at N >= 128 (D = 256 uses 64-key steps to fit
// TMEM) and each issuing thread does little besides issuing: two issuers keep
// their barrier waits off each other's stream; releases that need no tensor
// ordering are signalled by a row warp.
#include "kernels.h"

namespace hstu {

namespace {

template <int D, bool BF16>
__global__ void __launch_bounds__(kDqThreads, 1)
    hstu_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
  using C = DqCfg<D>;
  constexpr int BN = C::BN, NQ = C::NQ, NK = C::NK, NV = C::NV, KCH = D / 64;
  constexpr int NF = NK < NV ? NK : NV;  // step barriers (K and V land on one)
  constexpr int RW = kRowWarps16;
  constexpr int CW = BN / 4;   // key columns per row warp
  constexpr int DW = D / 4;    // dQ columns per row warp
  constexpr int MMA_B = 2 + RW;  // warp of the dQ issuer
  constexpr uint32_t IDESC_S = idesc_f16(BF16, kBM, BN, false, false);
  constexpr uint32_t IDESC_DQ = idesc_f16(BF16, kBM, D, false, true);
  constexpr uint32_t COL_S = 0, COL_DP = BN, COL_DQ = 2 * BN, COL_DS = 2 * BN + D;
  constexpr uint32_t DS_BUF = BN / 2;  // packed dS columns per buffer
  static_assert(COL_DS + 2 * DS_BUF <= kTmemCols, "TMEM budget");
  static_assert(C::SMEM <= 232448, "shared memory budget");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sQ = base;                        // NQ x (Q, dO)
  const uint32_t sK = sQ + 2 * NQ * C::Q_BYTES;    // NK x K
  const uint32_t sV = sK + NK * C::KV_BYTES;       // NV x V

  enum {
    QFULL = 0, QEMPTY = QFULL + NQ, FULL = QEMPTY + NQ, KEMPTY = FULL + NF,
    VEMPTY = KEMPTY + NK, SPFULL = VEMPTY + NV, SPEMPTY = SPFULL + 1, DSFULL = SPEMPTY + 1,
    DSEMPTY = DSFULL + 2, DQFULL = DSEMPTY + 2, DQEMPTY = DQFULL + 1, UFULL = DQEMPTY + 1,
    UEMPTY = UFULL + kUnitRing, DRAIN = UEMPTY + kUnitRing, NBARS = DRAIN + 2
  };
  // control block: barriers | TMEM slot (8 B) | flags (16 B) | unit ring
  static_assert(NBARS * 8 + 24 + kUnitRing * sizeof(UnitInfo) <= kCtlBytes, "control block");
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + C::TILE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 2);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NQ; ++i) { mbar_init(bar(QFULL + i), 1); mbar_init(bar(QEMPTY + i), 1); }
    for (int i = 0; i < NF; ++i) mbar_init(bar(FULL + i), 1);
    for (int i = 0; i < NK; ++i) mbar_init(bar(KEMPTY + i), 1);
    for (int i = 0; i < NV; ++i) mbar_init(bar(VEMPTY + i), 1);
    mbar_init(bar(SPFULL), 1);
    mbar_init(bar(SPEMPTY), RW);
    for (int i = 0; i < 2; ++i) { mbar_init(bar(DSFULL + i), RW); mbar_init(bar(DSEMPTY + i), 1); }
    mbar_init(bar(DQFULL), 1);
    mbar_init(bar(DQEMPTY), RW);
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(bar(UFULL + i), 1);
      mbar_init(bar(UEMPTY + i), 2 + RW);
    }
    mbar_init(bar(DRAIN), 1);
    mbar_init(bar(DRAIN + 1), 1);
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q); tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v);
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
  const int n_units = *reinterpret_cast<volatile int*>(a.header + a.units_slot);
  const UnitQueue uq{reinterpret_cast<UnitInfo*>(const_cast<int*>(flags + 4)), bar(UFULL), bar(UEMPTY)};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t qi = 0, g = 0;
      bool ok = true;
      auto prefetch_kv = [&](int h, int row) {
#pragma unroll
        for (int c = 0; c < KCH; ++c) {
          tma_prefetch_3d(&tm_k, 64 * c, h, row);
          tma_prefetch_3d(&tm_v, 64 * c, h, row);
        }
      };
      int prev_n = kPrefetch;  // steps of the previous unit (the first unit is not warmed)
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
        const int kv_row0 = U.k0;
        const int qb = qi % NQ;
        if (!wait_bar(bar(QEMPTY + qb), ((qi / NQ) & 1) ^ 1, wc, 0x001)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(QFULL + qb), 2 * C::Q_BYTES);
        const uint32_t qt = sQ + qb * 2 * C::Q_BYTES, dot = qt + C::Q_BYTES;
#pragma unroll
        for (int c = 0; c < KCH; ++c) {
          tma_load_3d(qt + c * (kBM * 128), &tm_q, bar(QFULL + qb), 64 * c, h, q_row0);
          tma_load_3d(dot + c * (kBM * 128), &tm_do, bar(QFULL + qb), 64 * c, h, q_row0);
        }
        ++qi;
        // L2 warm-up runs kPrefetch steps ahead of the loads along the flat
        // stream (this unit's later K/V tiles, then the next unit's Q, dO and
        // first K/V tiles); what a short previous unit could not cover is
        // issued here.
        if (prev_n < kPrefetch)
          for (int m = 0; m < min(U.n, kPrefetch - prev_n); ++m) prefetch_kv(h, kv_row0 + BN * m);
        prev_n = U.n;
        for (int n = 0; n < U.n; ++n, ++g) {
          const int t = n + kPrefetch;
          if (t < U.n) {
            prefetch_kv(h, kv_row0 + BN * t);
          } else if (t - U.n < nx.n) {
            if (t == U.n) {
#pragma unroll
              for (int c = 0; c < KCH; ++c) {
                tma_prefetch_3d(&tm_q, 64 * c, nx.hz, nx.q0 + kBM * nx.tile);
                tma_prefetch_3d(&tm_do, 64 * c, nx.hz, nx.q0 + kBM * nx.tile);
              }
            }
            prefetch_kv(nx.hz, nx.k0 + BN * (t - U.n));
          }
          const int ks = g % NK, vs = g % NV, f = g % NF;
          if (!wait_bar(bar(KEMPTY + ks), ((g / NK) & 1) ^ 1, wc, 0x002) ||
              !wait_bar(bar(VEMPTY + vs), ((g / NV) & 1) ^ 1, wc, 0x003)) {
            ok = false;
            break;
          }
          const int row = kv_row0 + BN * n;
          mbar_arrive_expect_tx(bar(FULL + f), 2 * C::KV_BYTES);
#pragma unroll
          for (int c = 0; c < KCH; ++c) {
            tma_load_3d(sK + ks * C::KV_BYTES + c * (BN * 128), &tm_k, bar(FULL + f), 64 * c, h, row);
            tma_load_3d(sV + vs * C::KV_BYTES + c * (BN * 128), &tm_v, bar(FULL + f), 64 * c, h, row);
          }
        }
      }
      for (uint32_t i = qi > NQ ? qi - NQ : 0; i < qi; ++i)
        wait_bar(bar(QFULL + i % NQ), (i / NQ) & 1, drain, 0x0f1);
      for (uint32_t i = g > NF ? g - NF : 0; i < g; ++i)
        wait_bar(bar(FULL + i % NF), (i / NF) & 1, drain, 0x0f2);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S / dP issuer
    // Waits on TMA-filled stages need no tcgen05 fence (the async proxy both
    // writes and reads them); waits on the row warps' TMEM accesses do.
    if (lane == 0) {
      uint32_t qi = 0, g = 0;
      bool ok = true;
      for (uint32_t uk = 0; ok; ++uk) {
        UnitInfo U;
        if (!unit_pop(uq, uk, U, wc)) { ok = false; break; }
        if (U.n < 0) break;
        if (U.n <= 0) continue;
        const int qb = qi % NQ;
        if (!wait_bar(bar(QFULL + qb), (qi / NQ) & 1, wc, 0x104)) { ok = false; break; }
        const SDesc qd = kdesc(sQ + qb * 2 * C::Q_BYTES);
        const SDesc dod = kdesc(sQ + qb * 2 * C::Q_BYTES + C::Q_BYTES);
        for (int n = 0; n < U.n; ++n, ++g) {
          if (!wait_bar(bar(FULL + g % NF), (g / NF) & 1, wc, 0x106)) { ok = false; break; }
          // S and dP are single-buffered: the row warps must have loaded step g-1
          if (g > 0) {
            if (!wait_bar(bar(SPEMPTY), (g - 1) & 1, wc, 0x108)) { ok = false; break; }
            tc_fence_after();
          }
          const SDesc kd = kdesc(sK + (g % NK) * C::KV_BYTES);
          const SDesc vd = kdesc(sV + (g % NV) * C::KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + COL_S, desc_kmajor<kBM>(qd, kk), desc_kmajor<BN>(kd, kk), IDESC_S,
                   kk > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + COL_DP, desc_kmajor<kBM>(dod, kk), desc_kmajor<BN>(vd, kk), IDESC_S,
                   kk > 0 ? 1u : 0u);
          mma_commit(bar(SPFULL));
        }
        ++qi;
      }
      mma_commit(bar(DRAIN));
      wait_bar(bar(DRAIN), 0, drain, 0x1ff);
    }
  } else if (warp == MMA_B) {
    // ------------------------------------------------------------ dQ issuer
    if (lane == 0) {
      const uint32_t tDQ = tmem + COL_DQ;
      uint32_t g = 0, oi = 0;
      bool ok = true;
      for (uint32_t uk = 0; ok; ++uk) {
        UnitInfo U;
        if (!unit_pop(uq, uk, U, wc)) { ok = false; break; }
        if (U.n < 0) break;
        if (U.n <= 0) continue;
        for (int n = 0; n < U.n; ++n, ++g) {
          const int b = g & 1;
          if (!wait_bar(bar(DSFULL + b), (g >> 1) & 1, wc, 0x105)) { ok = false; break; }
          if (n == 0 && !wait_bar(bar(DQEMPTY), (oi & 1) ^ 1, wc, 0x103)) { ok = false; break; }
          tc_fence_after();
          const int ks = g % NK;
          const SDesc kd = mndesc<BN>(sK + ks * C::KV_BYTES);
          const uint32_t tDS = tmem + COL_DS + b * DS_BUF;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tDQ, tDS + 8 * kk, desc_mnmajor<BN>(kd, kk, 0), IDESC_DQ,
                   (n > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(KEMPTY + ks));
          mma_commit(bar(DSEMPTY + b));
          if (n == U.n - 1) mma_commit(bar(DQFULL));
        }
        ++oi;
      }
      mma_commit(bar(DRAIN + 1));
      wait_bar(bar(DRAIN + 1), 0, drain, 0x1fe);
    }
  } else {
    // ------------------------------------------------------------ SiLU' + epilogue
    // Sixteen warps: warp w owns TMEM lane quarter w % 4 (its 32 rows) and one
    // quarter of the key columns of each S / dP tile (and of the dQ columns).
    const int wq = warp & 3, cg = (warp - 2) >> 2;
    const int r = wq * 32 + lane;
    const bool releaser = warp == 2 && lane == 0;  // frees the V and Q stages
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + COL_S + lane_off + cg * CW, tDP = tmem + COL_DP + lane_off + cg * CW,
                   tDQ = tmem + COL_DQ + lane_off + cg * DW,
                   tDS = tmem + COL_DS + lane_off + cg * (CW / 2);
    const float half_alpha = 0.5f * a.alpha;
    const float out_scale = 0.5f * a.alpha * a.inv_L;  // dS is stored doubled
    uint32_t g = 0, oi = 0, qi = 0;
    bool ok = true;
    for (uint32_t uk = 0; ok; ++uk) {
      UnitInfo U;
      if (!unit_pop_warp(uq, uk, U, wc)) { ok = false; break; }
      if (U.n < 0) break;
      const int h = U.hz;
      const int q0 = U.q0, Lq = U.Lq, Lk = U.Lk;
      const int i = kBM * U.tile + r;
      const int i_warp = kBM * U.tile + wq * 32;
      const int64_t grow = static_cast<int64_t>(q0) + i;
      const bool row_ok = i < Lq && grow < a.total_q;
      char* orow = static_cast<char*>(a.o0) +
                   (grow * a.o0_st + static_cast<int64_t>(h) * a.o0_sh + cg * DW) * 2;
      if (U.n <= 0) {
        if (row_ok) store_zero_n<DW>(orow);
        continue;
      }
      const int qb = qi % NQ;
      const int lim = a.causal ? min(Lk, i + 1) : Lk;  // valid keys: j < lim
      for (int n = 0; n < U.n; ++n, ++g) {
        const int b = g & 1;
        if (!wait_bar_warp(bar(SPFULL), g & 1, wc, 0x201)) { ok = false; break; }
        tc_fence_after();
        uint32_t xs[CW], xp[CW];
        tmem_ld_x2<CW>(tS, tDP, xs, xp);
        warp_arrive(bar(SPEMPTY));  // S and dP of this step are in registers
        if (releaser) {
          // S_g and dP_g are complete: V_g and (after the last step) Q, dO are unused
          mbar_arrive(bar(VEMPTY + g % NV));
          if (n == U.n - 1) mbar_arrive(bar(QEMPTY + qb));
        }
        const int jc = BN * n + cg * CW;
        const bool need_mask = (a.causal && jc + CW - 1 > i_warp) || (jc + CW > Lk);
        uint32_t d[CW / 2];
        if (!need_mask) {
#pragma unroll
          for (int e = 0; e < CW / 2; ++e)
            d[e] = ds_pair<BF16>(xs[2 * e], xs[2 * e + 1], xp[2 * e], xp[2 * e + 1], half_alpha);
        } else {
#pragma unroll
          for (int e = 0; e < CW / 2; ++e) {
            const int j = jc + 2 * e;
            const bool v0 = j < lim, v1 = j + 1 < lim;
            d[e] = ds_pair<BF16>(v0 ? xs[2 * e] : 0u, v1 ? xs[2 * e + 1] : 0u, v0 ? xp[2 * e] : 0u,
                                 v1 ? xp[2 * e + 1] : 0u, half_alpha);
          }
        }
        // dS buffer b last held step g-2: free once dQ += dS_{g-2} K_{g-2} ran
        if (g >= 2 && !wait_bar_warp(bar(DSEMPTY + b), ((g >> 1) - 1) & 1, wc, 0x203)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st_w<CW / 2>(tDS + b * DS_BUF, d);
        tmem_st_wait();
        warp_arrive(bar(DSFULL + b));
      }
      if (!ok) break;
      if (!wait_bar_warp(bar(DQFULL), oi & 1, wc, 0x202)) { ok = false; break; }
      tc_fence_after();
      if constexpr (DW <= 32) {
        uint32_t x[DW];
        tmem_ld_w<DW>(tDQ, x);
        if (row_ok) store_row_n<DW, BF16>(orow, x, out_scale);
      } else {
#pragma unroll 1
        for (int c = 0; c < DW / 32; ++c) {
          uint32_t x[32];
          tmem_ld32(tDQ + 32 * c, x);
          if (row_ok) store_row_n<32, BF16>(orow + c * 64, x, out_scale);
        }
      }
      warp_arrive(bar(DQEMPTY));
      ++oi;
      ++qi;
    }
  }

  // The role branches leave lanes of warps 0, 1 (and 18) on different paths;
  // reconverge each warp so the aligned CTA barrier counts it exactly once
  // (otherwise it can release before the row warps finish reading TMEM).
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool BF16>
cudaError_t launch_dq_t(int grid, cudaStream_t st, bool pdl, const CUtensorMap& tq, const CUtensorMap& tdo,
                        const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a) {
  auto kern = hstu_bwd_dq_kernel<D, BF16>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DqCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_attn(kern, grid, kDqThreads, DqCfg<D>::SMEM, st, pdl, tq, tdo, tk, tv, a);
}

}  // namespace

cudaError_t launch_dq(int D, bool bf16, int grid, cudaStream_t st, bool pdl, const CUtensorMap& tq,
                      const CUtensorMap& tdo, const CUtensorMap& tk, const CUtensorMap& tv,
                      const AttnArgs& a) {
  switch (D) {
    case 64: return bf16 ? launch_dq_t<64, true>(grid, st, pdl, tq, tdo, tk, tv, a)
                         : launch_dq_t<64, false>(grid, st, pdl, tq, tdo, tk, tv, a);
    case 128: return bf16 ? launch_dq_t<128, true>(grid, st, pdl, tq, tdo, tk, tv, a)
                          : launch_dq_t<128, false>(grid, st, pdl, tq, tdo, tk, tv, a);
    case 256: return bf16 ? launch_dq_t<256, true>(grid, st, pdl, tq, tdo, tk, tv, a)
                          : launch_dq_t<256, false>(grid, st, pdl, tq, tdo, tk, tv, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hstu
