// HSTU attention backward, dK/dV part (chain rule of "HSTU Attention
// (Blackwell SM100/SM103)", Overview equations):
//   dV_j = (1/L_scale)     sum_i M_ij SiLU(alpha q_i.k_j) dO_i
//   dK_j = (alpha/L_scale) sum_i M_ij <dO_i, v_j> SiLU'(alpha q_i.k_j) q_i
//
// Key-stationary: each CTA owns a 128-row key tile (and, for D = 256, one
// 128-column half of dK/dV, so the accumulators fit in TMEM) and walks the
// 64-row query tiles that can see it.  Per step it recomputes S^T = K Q^T and
// dP^T = V dO^T into TMEM, forms A^T = M (.) SiLU(alpha S^T) and
// dS^T = M (.) dP^T (.) SiLU'(alpha S^T) in registers (one tanh per
// element), stores both to TMEM as 16-bit, and accumulates dV += A^T dO and
// dK += dS^T Q with the A operand read from TMEM.  No atomics.
//   warp 0      TMA: K and V per unit, Q and dO per step.
//   warp 1      tcgen05 issuer.  S^T and dP^T are double-buffered and run one
//               step ahead of the dV / dK accumulation, so the tensor pipe has
//               work while the row warps form A^T and dS^T.
//   warps 2-9   row work, two warps per TMEM lane quarter (one per column
//               half of each query tile).
// TMEM: S^T0 | S^T1 | dP^T0 | dP^T1 | dV | dK [| A^T0 | A^T1 | dS^T0 | dS^T1].
// When the separate A^T / dS^T buffers do not fit (D >= 128) they are written
// in place over the S^T / dP^T columns their warp just read; S^T_{g+2}
// (issued after the step-g accumulation by the same thread, in order)
// overwrites them only after they are consumed.
#include "kernels.h"

namespace hstu {

namespace {

template <int D, bool BF16>
__global__ void __launch_bounds__(kAttnThreads, 1)
    hstu_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_do, const AttnArgs a) {
  using C = DkdvCfg<D>;
  constexpr int BQ = C::BQ, DH = C::DH, SPLIT = C::SPLIT, NKV = C::NKV, NS = C::NS;
  constexpr int KCH = D / 64;
  constexpr int CPW = BQ / 2;
  static_assert(CPW == 32, "one 32-column batch per row warp");
  constexpr bool SERIAL = NS == 1;  // one Q/dO stage: accumulate before the next S^T
  constexpr bool ALIAS = 4 * BQ + 2 * DH + 2 * BQ > kTmemCols;
  constexpr uint32_t IDESC_S = idesc_f16(BF16, kBM, BQ, false, false);
  constexpr uint32_t IDESC_ACC = idesc_f16(BF16, kBM, DH, false, true);
  constexpr uint32_t COL_ST = 0, COL_DPT = 2 * BQ, COL_DV = 4 * BQ, COL_DK = 4 * BQ + DH,
                     COL_AT = 4 * BQ + 2 * DH, COL_DST = COL_AT + BQ;
  static_assert(COL_DK + DH + (ALIAS ? 0 : 2 * BQ) <= kTmemCols, "TMEM budget");
  // A^T / dS^T of step g: separate buffers of BQ/2 packed columns, or the
  // first half of each row warp's own S^T / dP^T columns.
  constexpr uint32_t P_BUF = ALIAS ? BQ : BQ / 2;
  constexpr uint32_t P_HALF = ALIAS ? CPW : CPW / 2;
  constexpr uint32_t A_BASE = ALIAS ? COL_ST : COL_AT;
  constexpr uint32_t D_BASE = ALIAS ? COL_DPT : COL_DST;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sKV = base;                          // NKV x (K, V)
  const uint32_t sQ = sKV + 2 * NKV * C::KV_BYTES;    // NS x Q
  const uint32_t sDO = sQ + NS * C::Q_BYTES;          // NS x dO

  enum {
    KVFULL = 0, KVEMPTY = KVFULL + NKV, QFULL = KVEMPTY + NKV, DOFULL = QFULL + NS,
    QEMPTY = DOFULL + NS, STFULL = QEMPTY + NS, ASFULL = STFULL + 2, ACCFULL = ASFULL + 2,
    ACCEMPTY = ACCFULL + 1, UFULL = ACCEMPTY + 1, UEMPTY = UFULL + kUnitRing,
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
    for (int i = 0; i < NKV; ++i) { mbar_init(bar(KVFULL + i), 1); mbar_init(bar(KVEMPTY + i), 1); }
    for (int i = 0; i < NS; ++i) {
      mbar_init(bar(QFULL + i), 1); mbar_init(bar(DOFULL + i), 1); mbar_init(bar(QEMPTY + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(STFULL + i), 1);
      mbar_init(bar(ASFULL + i), kRowThreads);
    }
    mbar_init(bar(ACCFULL), 1);
    mbar_init(bar(ACCEMPTY), kRowThreads);
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
    tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_q); tma_prefetch_desc(&tm_do);
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
      uint32_t kvi = 0, qi = 0;
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
        const int h = U.hz / SPLIT;
        const int k_row0 = U.k0 + kBM * U.tile;
        const int q_seq0 = U.q0;
        const int m0 = a.causal ? (kBM * U.tile) / BQ : 0;
        const int kb = kvi % NKV;
        if (!wait_bar(bar(KVEMPTY + kb), ((kvi / NKV) & 1) ^ 1, wc, 0x001)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(KVFULL + kb), 2 * C::KV_BYTES);
        const uint32_t kt = sKV + kb * 2 * C::KV_BYTES, vt = kt + C::KV_BYTES;
#pragma unroll
        for (int c = 0; c < KCH; ++c) {
          tma_load_3d(kt + c * (kBM * 128), &tm_k, bar(KVFULL + kb), 64 * c, h, k_row0);
          tma_load_3d(vt + c * (kBM * 128), &tm_v, bar(KVFULL + kb), 64 * c, h, k_row0);
        }
        ++kvi;
        for (int m = 0; m < U.n; ++m) {
          const int s = qi % NS;
          if (!wait_bar(bar(QEMPTY + s), ((qi / NS) & 1) ^ 1, wc, 0x002)) { ok = false; break; }
          const int row = q_seq0 + BQ * (m0 + m);
          mbar_arrive_expect_tx(bar(QFULL + s), C::Q_BYTES);
#pragma unroll
          for (int c = 0; c < KCH; ++c)
            tma_load_3d(sQ + s * C::Q_BYTES + c * (BQ * 128), &tm_q, bar(QFULL + s), 64 * c, h, row);
          mbar_arrive_expect_tx(bar(DOFULL + s), C::Q_BYTES);
#pragma unroll
          for (int c = 0; c < KCH; ++c)
            tma_load_3d(sDO + s * C::Q_BYTES + c * (BQ * 128), &tm_do, bar(DOFULL + s), 64 * c, h, row);
          ++qi;
        }
      }
      for (uint32_t i = kvi > NKV ? kvi - NKV : 0; i < kvi; ++i)
        wait_bar(bar(KVFULL + i % NKV), (i / NKV) & 1, drain, 0x0f1);
      for (uint32_t i = qi > NS ? qi - NS : 0; i < qi; ++i) {
        wait_bar(bar(QFULL + i % NS), (i / NS) & 1, drain, 0x0f2);
        wait_bar(bar(DOFULL + i % NS), (i / NS) & 1, drain, 0x0f3);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Flat stream of steps g: S^T_g, dP^T_g, then the step g-1 accumulation.
    if (lane == 0) {
      const uint32_t tDV = tmem + COL_DV, tDK = tmem + COL_DK;
      struct Pend {
        int valid, s, first, last, half;
        uint32_t g, oi;
      } pd{0, 0, 0, 0, 0, 0, 0};
      // dV += A^T dO, dK += dS^T Q over the step's queries, once A^T / dS^T exist
      auto issue_acc = [&](const Pend& p) -> bool {
        const int b = p.g & 1;
        if (!wait_bar(bar(ASFULL + b), (p.g >> 1) & 1, wc, 0x105)) return false;
        if (p.first && !wait_bar(bar(ACCEMPTY), (p.oi & 1) ^ 1, wc, 0x103)) return false;
        tc_fence_after();
        const SDesc qd = mndesc<BQ>(sQ + p.s * C::Q_BYTES), dod = mndesc<BQ>(sDO + p.s * C::Q_BYTES);
        const int n0 = p.half * DH;
        const uint32_t tAT = tmem + A_BASE + b * P_BUF, tDST = tmem + D_BASE + b * P_BUF;
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const int q = 16 * kk;
          const uint32_t col = (q / CPW) * P_HALF + (q % CPW) / 2;
          mma_ts(tDV, tAT + col, desc_mnmajor<BQ>(dod, kk, n0), IDESC_ACC,
                 (!p.first || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk) {
          const int q = 16 * kk;
          const uint32_t col = (q / CPW) * P_HALF + (q % CPW) / 2;
          mma_ts(tDK, tDST + col, desc_mnmajor<BQ>(qd, kk, n0), IDESC_ACC,
                 (!p.first || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar(QEMPTY + p.s));
        if (p.last) mma_commit(bar(ACCFULL));
        return true;
      };
      uint32_t kvi = 0, qi = 0, g = 0, oi = 0;
      bool ok = true;
      for (uint32_t uk = 0; ok; ++uk) {
        UnitInfo U;
        if (!unit_pop(uq, uk, U, wc)) { ok = false; break; }
        if (U.n < 0) break;
        if (U.n <= 0) continue;
        const int half = U.hz % SPLIT;
        const int kb = kvi % NKV;
        if (!wait_bar(bar(KVFULL + kb), (kvi / NKV) & 1, wc, 0x104)) { ok = false; break; }
        tc_fence_after();
        const SDesc kd = kdesc(sKV + kb * 2 * C::KV_BYTES);
        const SDesc vd = kdesc(sKV + kb * 2 * C::KV_BYTES + C::KV_BYTES);
        for (int m = 0; m < U.n; ++m) {
          const int s = qi % NS, b = g & 1;
          if (!wait_bar(bar(QFULL + s), (qi / NS) & 1, wc, 0x106)) { ok = false; break; }
          tc_fence_after();
          const SDesc qd = kdesc(sQ + s * C::Q_BYTES), dod = kdesc(sDO + s * C::Q_BYTES);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + COL_ST + b * BQ, desc_kmajor<kBM>(kd, kk), desc_kmajor<BQ>(qd, kk),
                   IDESC_S, kk > 0 ? 1u : 0u);
          if (!wait_bar(bar(DOFULL + s), (qi / NS) & 1, wc, 0x107)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + COL_DPT + b * BQ, desc_kmajor<kBM>(vd, kk), desc_kmajor<BQ>(dod, kk),
                   IDESC_S, kk > 0 ? 1u : 0u);
          mma_commit(bar(STFULL + b));
          if (m == U.n - 1) mma_commit(bar(KVEMPTY + kb));
          Pend cur{1, s, m == 0, m == U.n - 1, half, g, oi};
          if (SERIAL) {
            if (!issue_acc(cur)) { ok = false; break; }
          } else {
            if (pd.valid && !issue_acc(pd)) { ok = false; break; }
            pd = cur;
          }
          ++qi;
          ++g;
        }
        ++kvi;
        ++oi;
      }
      if (!SERIAL && ok && pd.valid) issue_acc(pd);
      mma_commit(bar(DRAIN));
      wait_bar(bar(DRAIN), 0, drain, 0x1ff);
    }
  } else {
    // ------------------------------------------------------------ A^T, dS^T + epilogue
    // Eight warps: warp w owns TMEM lane quarter w % 4 (32 key rows) and one
    // half of the query columns of each S^T / dP^T tile (and of dK / dV).
    const int wq = warp & 3, hc = (warp - 2) >> 2;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tST = tmem + COL_ST + lane_off + hc * CPW, tDPT = tmem + COL_DPT + lane_off + hc * CPW,
                   tDV = tmem + COL_DV + lane_off, tDK = tmem + COL_DK + lane_off,
                   tAT = tmem + A_BASE + lane_off + hc * P_HALF,
                   tDST = tmem + D_BASE + lane_off + hc * P_HALF;
    const float half_alpha = 0.5f * a.alpha;
    const float dk_scale = 0.5f * a.alpha * a.inv_L;  // dS^T is stored doubled
    uint32_t g = 0, oi = 0;
    bool ok = true;
    for (uint32_t uk = 0; ok; ++uk) {
      UnitInfo U;
      if (!unit_pop_warp(uq, uk, U, wc)) { ok = false; break; }
      if (U.n < 0) break;
      const int h = U.hz / SPLIT, half = U.hz % SPLIT;
      const int Lq = U.Lq, k0 = U.k0, Lk = U.Lk;
      const int j = kBM * U.tile + r;
      const int j_warp_last = kBM * U.tile + wq * 32 + 31;
      const int64_t grow = static_cast<int64_t>(k0) + j;
      const bool row_ok = j < Lk && grow < a.total_k;
      const int64_t col0 = static_cast<int64_t>(half) * DH + hc * (DH / 2);
      char* dvrow = static_cast<char*>(a.o0) + (grow * a.o0_st + static_cast<int64_t>(h) * a.o0_sh + col0) * 2;
      char* dkrow = static_cast<char*>(a.o1) + (grow * a.o1_st + static_cast<int64_t>(h) * a.o1_sh + col0) * 2;
      if (U.n <= 0) {
        if (row_ok)
          for (int c = 0; c < DH / 64; ++c) { store_zero32(dvrow + c * 64); store_zero32(dkrow + c * 64); }
        continue;
      }
      const int m0 = a.causal ? (kBM * U.tile) / BQ : 0;
      const int lo = a.causal ? j : 0;  // valid queries: lo <= i < Lq
      for (int m = 0; m < U.n; ++m) {
        const int b = g & 1;
        if (!wait_bar_warp(bar(STFULL + b), (g >> 1) & 1, wc, 0x201)) { ok = false; break; }
        tc_fence_after();
        const int ic = BQ * (m0 + m) + hc * CPW;  // first query of this warp's columns
        const bool need_mask = (ic + CPW > Lq) || (a.causal && j_warp_last > ic);
        uint32_t xs[32], xp[32];
        tmem_ld32x2(tST + b * BQ, tDPT + b * BQ, xs, xp);
        uint32_t pa[16], pd[16];
        if (!need_mask) {
#pragma unroll
          for (int e = 0; e < 16; ++e)
            a_ds_pair<BF16>(xs[2 * e], xs[2 * e + 1], xp[2 * e], xp[2 * e + 1], half_alpha, pa[e],
                            pd[e]);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int i = ic + 2 * e;
            const bool v0 = i >= lo && i < Lq, v1 = i + 1 >= lo && i + 1 < Lq;
            a_ds_pair<BF16>(v0 ? xs[2 * e] : 0u, v1 ? xs[2 * e + 1] : 0u, v0 ? xp[2 * e] : 0u,
                            v1 ? xp[2 * e + 1] : 0u, half_alpha, pa[e], pd[e]);
          }
        }
        tmem_st16(tAT + b * P_BUF, pa);
        tmem_st16(tDST + b * P_BUF, pd);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(ASFULL + b));
        ++g;
      }
      if (!ok) break;
      if (!wait_bar_warp(bar(ACCFULL), oi & 1, wc, 0x202)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < DH / 64; ++c) {
        uint32_t x[32];
        tmem_ld32(tDV + hc * (DH / 2) + 32 * c, x);
        if (row_ok) store_row32<BF16>(dvrow + c * 64, x, a.inv_L);
      }
#pragma unroll 1
      for (int c = 0; c < DH / 64; ++c) {
        uint32_t x[32];
        tmem_ld32(tDK + hc * (DH / 2) + 32 * c, x);
        if (row_ok) store_row32<BF16>(dkrow + c * 64, x, dk_scale);
      }
      tc_fence_before();
      mbar_arrive(bar(ACCEMPTY));
      ++oi;
    }
  }

  // Started early beside the dQ grid: finish only after it, so that work
  // queued behind this grid also sees dQ complete.
  if (a.pdl_wait == 2) grid_dependency_wait();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool BF16>
cudaError_t launch_dkdv_t(int grid, cudaStream_t st, bool pdl, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tq, const CUtensorMap& tdo, const AttnArgs& a) {
  auto kern = hstu_bwd_dkdv_kernel<D, BF16>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DkdvCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_attn(kern, grid, DkdvCfg<D>::SMEM, st, pdl, tk, tv, tq, tdo, a);
}

}  // namespace

cudaError_t launch_dkdv(int D, bool bf16, int grid, cudaStream_t st, bool pdl, const CUtensorMap& tk,
                        const CUtensorMap& tv, const CUtensorMap& tq, const CUtensorMap& tdo,
                        const AttnArgs& a) {
  switch (D) {
    case 64: return bf16 ? launch_dkdv_t<64, true>(grid, st, pdl, tk, tv, tq, tdo, a)
                         : launch_dkdv_t<64, false>(grid, st, pdl, tk, tv, tq, tdo, a);
    case 128: return bf16 ? launch_dkdv_t<128, true>(grid, st, pdl, tk, tv, tq, tdo, a)
                          : launch_dkdv_t<128, false>(grid, st, pdl, tk, tv, tq, tdo, a);
    case 256: return bf16 ? launch_dkdv_t<256, true>(grid, st, pdl, tk, tv, tq, tdo, a)
                          : launch_dkdv_t<256, false>(grid, st, pdl, tk, tv, tq, tdo, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hstu
