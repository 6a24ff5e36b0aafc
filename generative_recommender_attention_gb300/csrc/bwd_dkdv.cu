// HSTU attention backward, dK/dV part (chain rule of "HSTU Attention
// (Blackwell SM100/SM103)", Overview equations):
//   dV_j = (1/L_scale)     sum_i M_ij SiLU(alpha q_i.k_j) dO_i
//   dK_j = (alpha/L_scale) sum_i M_ij <dO_i, v_j> SiLU'(alpha q_i.k_j) q_i
//
// Key-stationary: each CTA owns a 128-row key tile (and, for D = 256, one
// 128-column half of dK/dV, so the accumulators fit in TMEM) and walks the
// query tiles that can see it.  Per step it recomputes S^T = K Q^T and
// dP^T = V dO^T into TMEM, forms A^T = M (.) SiLU(alpha S^T) and
// dS^T = M (.) dP^T (.) SiLU'(alpha S^T) in registers (one sigmoid per
// element), stores both to TMEM as 16-bit, and accumulates dV += A^T dO and
// dK += dS^T Q with the A operand read from TMEM.  No atomics.
//   warp 0      TMA: K and V per unit, Q and dO per step.
//   warp 1      tcgen05 issuer.
//   warps 2-9   row work, two warps per TMEM lane quarter (one per column
//               half of each query tile).
// TMEM: S^T | dP^T | dV | dK | A^T x2 | dS^T x2.
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
  constexpr bool SERIAL = NS == 1;
  constexpr uint32_t IDESC_S = idesc_f16(BF16, kBM, BQ, false, false);
  constexpr uint32_t IDESC_ACC = idesc_f16(BF16, kBM, DH, false, true);
  constexpr uint32_t COL_ST = 0, COL_DPT = BQ, COL_DV = 2 * BQ, COL_DK = 2 * BQ + DH,
                     COL_AT = 2 * BQ + 2 * DH, COL_DST = COL_AT + BQ;
  static_assert(COL_DST + BQ <= kTmemCols, "TMEM budget");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sKV = base;                          // NKV x (K, V)
  const uint32_t sQ = sKV + 2 * NKV * C::KV_BYTES;    // NS x Q
  const uint32_t sDO = sQ + NS * C::Q_BYTES;          // NS x dO

  enum {
    KVFULL = 0, KVEMPTY = KVFULL + NKV, QFULL = KVEMPTY + NKV, DOFULL = QFULL + NS,
    QEMPTY = DOFULL + NS, STFULL = QEMPTY + NS, ASFULL = STFULL + 1, ACCFULL = ASFULL + 2,
    ACCEMPTY = ACCFULL + 1, DRAIN = ACCEMPTY + 1, NBARS = DRAIN + 1
  };
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
    mbar_init(bar(STFULL), 1);
    mbar_init(bar(ASFULL), kRowThreads);
    mbar_init(bar(ASFULL + 1), kRowThreads);
    mbar_init(bar(ACCFULL), 1);
    mbar_init(bar(ACCEMPTY), kRowThreads);
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
  const int n_units = *reinterpret_cast<volatile int*>(a.header + a.units_slot);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t kvi = 0, qi = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const Unit U = load_unit(a.units, u);
        if (U.n <= 0) continue;
        const int h = U.hz / SPLIT;
        const int k_row0 = __ldg(a.cu_k + U.b) + kBM * U.tile;
        const int q_seq0 = __ldg(a.cu_q + U.b);
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
    if (lane == 0) {
      const uint32_t tST = tmem + COL_ST, tDPT = tmem + COL_DPT, tDV = tmem + COL_DV,
                     tDK = tmem + COL_DK, tAT = tmem + COL_AT, tDST = tmem + COL_DST;
      struct Pend {
        int valid, s, b, first, last, half;
        uint32_t g, oi;
      } pd{0, 0, 0, 0, 0, 0, 0, 0};
      // dV += A^T dO, dK += dS^T Q over this step's queries (its A^T/dS^T are ready)
      auto issue_acc = [&](const Pend& p) -> bool {
        if (p.first && !wait_bar(bar(ACCEMPTY), (p.oi & 1) ^ 1, wc, 0x103)) return false;
        tc_fence_after();
        const uint32_t qt = sQ + p.s * C::Q_BYTES, dot = sDO + p.s * C::Q_BYTES;
        const int n0 = p.half * DH;
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          mma_ts(tDV, tAT + p.b * (BQ / 2) + kk * 8, desc_mnmajor<BQ>(dot, kk, n0), IDESC_ACC,
                 (!p.first || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < BQ / 16; ++kk)
          mma_ts(tDK, tDST + p.b * (BQ / 2) + kk * 8, desc_mnmajor<BQ>(qt, kk, n0), IDESC_ACC,
                 (!p.first || kk > 0) ? 1u : 0u);
        mma_commit(bar(QEMPTY + p.s));
        if (p.last) mma_commit(bar(ACCFULL));
        return true;
      };
      uint32_t kvi = 0, qi = 0, g = 0, oi = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const Unit U = load_unit(a.units, u);
        if (U.n <= 0) continue;
        const int half = U.hz % SPLIT;
        const int kb = kvi % NKV;
        if (!wait_bar(bar(KVFULL + kb), (kvi / NKV) & 1, wc, 0x104)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kt = sKV + kb * 2 * C::KV_BYTES, vt = kt + C::KV_BYTES;
        for (int m = 0; m < U.n; ++m) {
          const int s = qi % NS, b = g & 1;
          if (pd.valid) {
            if (!wait_bar(bar(ASFULL + pd.b), (pd.g >> 1) & 1, wc, 0x105)) { ok = false; break; }
          }
          if (!wait_bar(bar(QFULL + s), (qi / NS) & 1, wc, 0x106)) { ok = false; break; }
          tc_fence_after();
          const uint32_t qt = sQ + s * C::Q_BYTES, dot = sDO + s * C::Q_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tST, desc_kmajor<kBM>(kt, kk), desc_kmajor<BQ>(qt, kk), IDESC_S, kk > 0 ? 1u : 0u);
          if (!wait_bar(bar(DOFULL + s), (qi / NS) & 1, wc, 0x107)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tDPT, desc_kmajor<kBM>(vt, kk), desc_kmajor<BQ>(dot, kk), IDESC_S, kk > 0 ? 1u : 0u);
          mma_commit(bar(STFULL));
          if (m == U.n - 1) mma_commit(bar(KVEMPTY + kb));
          Pend cur{1, s, b, m == 0, m == U.n - 1, half, g, oi};
          if (SERIAL) {
            if (!wait_bar(bar(ASFULL + b), (g >> 1) & 1, wc, 0x108)) { ok = false; break; }
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
      if (!SERIAL && ok && pd.valid) {
        if (wait_bar(bar(ASFULL + pd.b), (pd.g >> 1) & 1, wc, 0x109)) issue_acc(pd);
      }
      mma_commit(bar(DRAIN));
      wait_bar(bar(DRAIN), 0, drain, 0x1ff);
    }
  } else {
    // ------------------------------------------------------------ A^T, dS^T + epilogue
    // Eight warps: warp w owns TMEM lane quarter w % 4 (32 key rows) and one
    // half of the query columns of each S^T / dP^T tile (and of dK / dV).
    constexpr int CPW = BQ / 2;
    static_assert(CPW == 32, "one 32-column batch per warp");
    const int wq = warp & 3, hc = (warp - 2) >> 2;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tST = tmem + COL_ST + lane_off + hc * CPW, tDPT = tmem + COL_DPT + lane_off + hc * CPW,
                   tDV = tmem + COL_DV + lane_off, tDK = tmem + COL_DK + lane_off,
                   tAT = tmem + COL_AT + lane_off + hc * (CPW / 2),
                   tDST = tmem + COL_DST + lane_off + hc * (CPW / 2);
    const float half_alpha = 0.5f * a.alpha;
    const float dk_scale = 0.5f * a.alpha * a.inv_L;  // dS^T is stored doubled
    uint32_t g = 0, oi = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
      const Unit U = load_unit(a.units, u);
      const int h = U.hz / SPLIT, half = U.hz % SPLIT;
      const int q0 = __ldg(a.cu_q + U.b);
      const int Lq = __ldg(a.cu_q + U.b + 1) - q0;
      const int k0 = __ldg(a.cu_k + U.b);
      const int Lk = __ldg(a.cu_k + U.b + 1) - k0;
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
        if (!wait_bar_warp(bar(STFULL), g & 1, wc, 0x201)) { ok = false; break; }
        tc_fence_after();
        const int ic = BQ * (m0 + m) + hc * CPW;  // first query of this warp's columns
        const bool need_mask = (ic + CPW > Lq) || (a.causal && j_warp_last > ic);
        uint32_t xs[32], xp[32];
        tmem_ld32x2(tST, tDPT, xs, xp);
        uint32_t pa[16], pd[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float av[2], dv[2];
#pragma unroll
          for (int t2 = 0; t2 < 2; ++t2) {
            float sv = __uint_as_float(xs[2 * e + t2]), pv = __uint_as_float(xp[2 * e + t2]);
            if (need_mask) {
              const int i = ic + 2 * e + t2;
              if (i < lo || i >= Lq) { sv = 0.f; pv = 0.f; }
            }
            const float hh = sv * half_alpha;
            const float tt = tanh_approx(hh);
            av[t2] = fmaf(hh, tt, hh);     // SiLU(x)
            dv[t2] = dsilu2(hh, tt, pv);   // 2 dP^T SiLU'(x)
          }
          pa[e] = pack2<BF16>(av[0], av[1]);
          pd[e] = pack2<BF16>(dv[0], dv[1]);
        }
        tmem_st16(tAT + b * (BQ / 2), pa);
        tmem_st16(tDST + b * (BQ / 2), pd);
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

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool BF16>
cudaError_t launch_dkdv_t(int grid, cudaStream_t st, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tq, const CUtensorMap& tdo, const AttnArgs& a) {
  auto kern = hstu_bwd_dkdv_kernel<D, BF16>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DkdvCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<grid, kAttnThreads, DkdvCfg<D>::SMEM, st>>>(tk, tv, tq, tdo, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dkdv(int D, bool bf16, int grid, cudaStream_t st, const CUtensorMap& tk,
                        const CUtensorMap& tv, const CUtensorMap& tq, const CUtensorMap& tdo,
                        const AttnArgs& a) {
  switch (D) {
    case 64: return bf16 ? launch_dkdv_t<64, true>(grid, st, tk, tv, tq, tdo, a)
                         : launch_dkdv_t<64, false>(grid, st, tk, tv, tq, tdo, a);
    case 128: return bf16 ? launch_dkdv_t<128, true>(grid, st, tk, tv, tq, tdo, a)
                          : launch_dkdv_t<128, false>(grid, st, tk, tv, tq, tdo, a);
    case 256: return bf16 ? launch_dkdv_t<256, true>(grid, st, tk, tv, tq, tdo, a)
                          : launch_dkdv_t<256, false>(grid, st, tk, tv, tq, tdo, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hstu
