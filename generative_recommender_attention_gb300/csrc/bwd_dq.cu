// HSTU attention backward, dQ part: dQ_i = (alpha/L_scale) sum_j
// M_ij <dO_i, v_j> SiLU'(alpha q_i.k_j) k_j (chain rule of "HSTU Attention
// (Blackwell SM100/SM103)", Overview equations).
//
// Query-stationary and atomic-free: each 128-row query tile is owned by one
// CTA, which recomputes S = Q K^T and dP = dO V^T per 64-key step, forms
// dS = M (.) dP (.) SiLU'(alpha S) in registers, stores it to TMEM as 16-bit,
// and accumulates dQ += dS K in TMEM.  The alpha/L_scale factor is applied
// once in the fp32 epilogue.
//   warp 0      TMA: Q and dO per unit, K and V per step.
//   warp 1      tcgen05 issuer.  S and dP are double-buffered in TMEM and run
//               one step ahead: S_{g+1}, dP_{g+1} are queued before
//               dQ += dS_g K_g, so the tensor pipe has work while the row
//               warps form dS_g.
//   warps 2-9   row work (two warps per TMEM lane quarter, one per column
//               half): SiLU' and mask, then the dQ epilogue.
// TMEM: S0 | S1 | dP0 | dP1 | dQ | dS0 | dS1.  At D = 256 there is no room
// for separate dS buffers; dS_g is then written in place over the S_g
// columns its warp just read, and S_{g+2} (issued after dQ += dS_g K_g by
// the same thread, in order) overwrites it only after it is consumed.
#include "kernels.h"

namespace hstu {

namespace {

template <int D, bool BF16>
__global__ void __launch_bounds__(kAttnThreads, 1)
    hstu_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
  using C = DqCfg<D>;
  constexpr int BN = C::BN, NQ = C::NQ, NK = C::NK, NV = C::NV, KCH = D / 64;
  constexpr int CPW = BN / 2;  // key columns per row warp
  static_assert(CPW == 32, "one 32-column batch per row warp");
  static_assert(NK >= 2, "the next S is issued before the pending dQ += dS K");
  constexpr bool DS_ALIAS = 4 * BN + D + BN > kTmemCols;
  constexpr uint32_t IDESC_S = idesc_f16(BF16, kBM, BN, false, false);
  constexpr uint32_t IDESC_DQ = idesc_f16(BF16, kBM, D, false, true);
  constexpr uint32_t COL_S = 0, COL_DP = 2 * BN, COL_DQ = 4 * BN, COL_DS = 4 * BN + D;
  static_assert(COL_DQ + D + (DS_ALIAS ? 0 : BN) <= kTmemCols, "TMEM budget");
  // dS_g columns: a separate buffer of BN/2 packed columns, or the first
  // half of each row warp's own S columns.
  constexpr uint32_t DS_BUF = DS_ALIAS ? BN : BN / 2;         // stride between the two buffers
  constexpr uint32_t DS_HALF = DS_ALIAS ? CPW : CPW / 2;      // offset of column half 1
  constexpr uint32_t DS_BASE = DS_ALIAS ? COL_S : COL_DS;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sQ = base;                        // NQ x (Q, dO)
  const uint32_t sK = sQ + 2 * NQ * C::Q_BYTES;    // NK x K
  const uint32_t sV = sK + NK * C::KV_BYTES;       // NV x V

  enum {
    QFULL = 0, QEMPTY = QFULL + NQ, KFULL = QEMPTY + NQ, KEMPTY = KFULL + NK,
    VFULL = KEMPTY + NK, VEMPTY = VFULL + NV, SPFULL = VEMPTY + NV, DSFULL = SPFULL + 2,
    DQFULL = DSFULL + 2, DQEMPTY = DQFULL + 1, UFULL = DQEMPTY + 1, UEMPTY = UFULL + kUnitRing,
    DRAIN = UEMPTY + kUnitRing, NBARS = DRAIN + 1
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
    for (int i = 0; i < NK; ++i) { mbar_init(bar(KFULL + i), 1); mbar_init(bar(KEMPTY + i), 1); }
    for (int i = 0; i < NV; ++i) { mbar_init(bar(VFULL + i), 1); mbar_init(bar(VEMPTY + i), 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(SPFULL + i), 1);
      mbar_init(bar(DSFULL + i), kRowThreads);
    }
    mbar_init(bar(DQFULL), 1);
    mbar_init(bar(DQEMPTY), kRowThreads);
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(bar(UFULL + i), 1);
      mbar_init(bar(UEMPTY + i), kUnitConsumers);
    }
    mbar_init(bar(DRAIN), 1);
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q); tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) { tmem_alloc(smem_u32(tmem_slot), kTmemCols); tmem_relinquish(); }
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
      bool ok = true;
      // claim units one ahead: the next claim overlaps this unit's loads
      UnitInfo nx = load_unit_info(a.units, a.cu_q, a.cu_k, atomicAdd(a.header + a.next_slot, 1),
                                   n_units);
      for (uint32_t uk = 0; ok; ++uk) {
        const UnitInfo U = nx;
        if (!unit_push(uq, uk, U, wc)) { ok = false; break; }
        if (U.n < 0) break;
        nx = load_unit_info(a.units, a.cu_q, a.cu_k, atomicAdd(a.header + a.next_slot, 1), n_units);
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
        for (int n = 0; n < U.n; ++n) {
          const int row = kv_row0 + BN * n;
          if (!load_kv(&tm_k, sK, NK, ki, KFULL, KEMPTY, row, h, 0x002) ||
              !load_kv(&tm_v, sV, NV, vi, VFULL, VEMPTY, row, h, 0x003)) {
            ok = false;
            break;
          }
        }
      }
      for (uint32_t i = qi > NQ ? qi - NQ : 0; i < qi; ++i)
        wait_bar(bar(QFULL + i % NQ), (i / NQ) & 1, drain, 0x0f1);
      for (uint32_t i = ki > NK ? ki - NK : 0; i < ki; ++i)
        wait_bar(bar(KFULL + i % NK), (i / NK) & 1, drain, 0x0f2);
      for (uint32_t i = vi > NV ? vi - NV : 0; i < vi; ++i)
        wait_bar(bar(VFULL + i % NV), (i / NV) & 1, drain, 0x0f3);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Flat stream of steps g: S_g, dP_g, then dQ += dS_{g-1} K_{g-1}.
    if (lane == 0) {
      const uint32_t tDQ = tmem + COL_DQ;
      struct Pend {
        int valid, ks, first, last;
        uint32_t g, oi;
      } pd{0, 0, 0, 0, 0, 0};
      // dQ += dS_g K_g once the row warps have written dS_g
      auto issue_dq = [&](const Pend& p) -> bool {
        const int b = p.g & 1;
        if (!wait_bar(bar(DSFULL + b), (p.g >> 1) & 1, wc, 0x105)) return false;
        if (p.first && !wait_bar(bar(DQEMPTY), (p.oi & 1) ^ 1, wc, 0x103)) return false;
        tc_fence_after();
        const SDesc kd = mndesc<BN>(sK + p.ks * C::KV_BYTES);
        const uint32_t tDS = tmem + DS_BASE + b * DS_BUF;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const int key = 16 * kk;
          const uint32_t col = (key / CPW) * DS_HALF + (key % CPW) / 2;
          mma_ts(tDQ, tDS + col, desc_mnmajor<BN>(kd, kk, 0), IDESC_DQ,
                 (!p.first || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(KEMPTY + p.ks));
        if (p.last) mma_commit(bar(DQFULL));
        return true;
      };
      uint32_t qi = 0, ki = 0, vi = 0, g = 0, oi = 0;
      bool ok = true;
      for (uint32_t uk = 0; ok; ++uk) {
        UnitInfo U;
        if (!unit_pop(uq, uk, U, wc)) { ok = false; break; }
        if (U.n < 0) break;
        if (U.n <= 0) continue;
        const int qb = qi % NQ;
        if (!wait_bar(bar(QFULL + qb), (qi / NQ) & 1, wc, 0x104)) { ok = false; break; }
        tc_fence_after();
        const SDesc qd = kdesc(sQ + qb * 2 * C::Q_BYTES);
        const SDesc dod = kdesc(sQ + qb * 2 * C::Q_BYTES + C::Q_BYTES);
        for (int n = 0; n < U.n; ++n) {
          const int ks = ki % NK, vs = vi % NV, b = g & 1;
          // buffer b last held step g-2, whose dS was waited for (and, when
          // aliased, consumed by dQ) before step g-1's dQ was issued
          if (!wait_bar(bar(KFULL + ks), (ki / NK) & 1, wc, 0x106)) { ok = false; break; }
          tc_fence_after();
          const SDesc kd = kdesc(sK + ks * C::KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + COL_S + b * BN, desc_kmajor<kBM>(qd, kk), desc_kmajor<BN>(kd, kk),
                   IDESC_S, kk > 0 ? 1u : 0u);
          if (!wait_bar(bar(VFULL + vs), (vi / NV) & 1, wc, 0x107)) { ok = false; break; }
          tc_fence_after();
          const SDesc vd = kdesc(sV + vs * C::KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + COL_DP + b * BN, desc_kmajor<kBM>(dod, kk), desc_kmajor<BN>(vd, kk),
                   IDESC_S, kk > 0 ? 1u : 0u);
          mma_commit(bar(SPFULL + b));
          mma_commit(bar(VEMPTY + vs));
          if (n == U.n - 1) mma_commit(bar(QEMPTY + qb));
          if (pd.valid && !issue_dq(pd)) { ok = false; break; }
          pd = Pend{1, ks, n == 0, n == U.n - 1, g, oi};
          ++ki;
          ++vi;
          ++g;
        }
        ++qi;
        ++oi;
      }
      if (ok && pd.valid) issue_dq(pd);
      mma_commit(bar(DRAIN));
      wait_bar(bar(DRAIN), 0, drain, 0x1ff);
    }
  } else {
    // ------------------------------------------------------------ SiLU' + epilogue
    // Eight warps: warp w owns TMEM lane quarter w % 4 and one half of the key
    // columns of each S / dP tile (and of the dQ columns).
    const int wq = warp & 3, hc = (warp - 2) >> 2;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + COL_S + lane_off + hc * CPW, tDP = tmem + COL_DP + lane_off + hc * CPW,
                   tDQ = tmem + COL_DQ + lane_off, tDS = tmem + DS_BASE + lane_off + hc * DS_HALF;
    const float half_alpha = 0.5f * a.alpha;
    const float out_scale = 0.5f * a.alpha * a.inv_L;  // dS is stored doubled
    uint32_t g = 0, oi = 0;
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
                   (grow * a.o0_st + static_cast<int64_t>(h) * a.o0_sh + hc * (D / 2)) * 2;
      if (U.n <= 0) {
        if (row_ok)
          for (int c = 0; c < D / 64; ++c) store_zero32(orow + c * 64);
        continue;
      }
      const int lim = a.causal ? min(Lk, i + 1) : Lk;  // valid keys: j < lim
      for (int n = 0; n < U.n; ++n) {
        const int b = g & 1;
        if (!wait_bar_warp(bar(SPFULL + b), (g >> 1) & 1, wc, 0x201)) { ok = false; break; }
        tc_fence_after();
        const int jc = BN * n + hc * CPW;
        const bool need_mask = (a.causal && jc + CPW - 1 > i_warp) || (jc + CPW > Lk);
        uint32_t xs[CPW], xp[CPW];
        tmem_ld32x2(tS + b * BN, tDP + b * BN, xs, xp);
        uint32_t d[CPW / 2];
        if (!need_mask) {
#pragma unroll
          for (int e = 0; e < CPW / 2; ++e)
            d[e] = ds_pair<BF16>(xs[2 * e], xs[2 * e + 1], xp[2 * e], xp[2 * e + 1], half_alpha);
        } else {
#pragma unroll
          for (int e = 0; e < CPW / 2; ++e) {
            const int j = jc + 2 * e;
            const bool v0 = j < lim, v1 = j + 1 < lim;
            d[e] = ds_pair<BF16>(v0 ? xs[2 * e] : 0u, v1 ? xs[2 * e + 1] : 0u, v0 ? xp[2 * e] : 0u,
                                 v1 ? xp[2 * e + 1] : 0u, half_alpha);
          }
        }
        tmem_st16(tDS + b * DS_BUF, d);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(DSFULL + b));
        ++g;
      }
      if (!ok) break;
      if (!wait_bar_warp(bar(DQFULL), oi & 1, wc, 0x202)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t x[32];
        tmem_ld32(tDQ + hc * (D / 2) + 32 * c, x);
        if (row_ok) store_row32<BF16>(orow + c * 64, x, out_scale);
      }
      tc_fence_before();
      mbar_arrive(bar(DQEMPTY));
      ++oi;
    }
  }

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
  return launch_attn(kern, grid, DqCfg<D>::SMEM, st, pdl, tq, tdo, tk, tv, a);
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
