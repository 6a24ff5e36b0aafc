// HSTU attention backward, dQ part: dQ_i = (alpha/L_scale) sum_j
// M_ij <dO_i, v_j> SiLU'(alpha q_i.k_j) k_j (chain rule of "HSTU Attention
// (Blackwell SM100/SM103)", Overview equations).
//
// Query-stationary and atomic-free: each 128-row query tile is owned by one
// CTA, which recomputes S = Q K^T and dP = dO V^T per key tile, forms
// dS = M (.) dP (.) SiLU'(alpha S) in registers, stores it to TMEM as 16-bit,
// and accumulates dQ += dS K in TMEM.  The alpha/L_scale factor is applied
// once in the fp32 epilogue.
//   warp 0      TMA: Q and dO per unit, K and V per step.
//   warp 1      tcgen05 issuer.
//   warps 2-9   row work (two warps per TMEM lane quarter, one per column
//               half): SiLU' and mask, then the dQ epilogue.
// TMEM: S | dP | dQ | dS0, dS1.
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
  static_assert(NK >= 2, "the next S is issued before the pending dQ += dS K");
  constexpr uint32_t IDESC_S = idesc_f16(BF16, kBM, BN, false, false);
  constexpr uint32_t IDESC_DQ = idesc_f16(BF16, kBM, D, false, true);
  constexpr uint32_t COL_S = 0, COL_DP = BN, COL_DQ = 2 * BN, COL_DS = 2 * BN + D;
  static_assert(COL_DS + BN <= kTmemCols, "TMEM budget");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  const uint32_t sQ = base;                        // NQ x (Q, dO)
  const uint32_t sK = sQ + 2 * NQ * C::Q_BYTES;    // NK x K
  const uint32_t sV = sK + NK * C::KV_BYTES;       // NV x V

  enum {
    QFULL = 0, QEMPTY = QFULL + NQ, KFULL = QEMPTY + NQ, KEMPTY = KFULL + NK,
    VFULL = KEMPTY + NK, VEMPTY = VFULL + NV, SPFULL = VEMPTY + NV, DSFULL = SPFULL + 1,
    DQFULL = DSFULL + 2, DQEMPTY = DQFULL + 1, DRAIN = DQEMPTY + 1, NBARS = DRAIN + 1
  };
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + C::TILE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 2);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < NQ; ++i) { mbar_init(bar(QFULL + i), 1); mbar_init(bar(QEMPTY + i), 1); }
    for (int i = 0; i < NK; ++i) { mbar_init(bar(KFULL + i), 1); mbar_init(bar(KEMPTY + i), 1); }
    for (int i = 0; i < NV; ++i) { mbar_init(bar(VFULL + i), 1); mbar_init(bar(VEMPTY + i), 1); }
    mbar_init(bar(SPFULL), 1);
    mbar_init(bar(DSFULL), kRowThreads);
    mbar_init(bar(DSFULL + 1), kRowThreads);
    mbar_init(bar(DQFULL), 1);
    mbar_init(bar(DQEMPTY), kRowThreads);
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
  const int n_units = *reinterpret_cast<volatile int*>(a.header + a.units_slot);

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
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const Unit U = load_unit(a.units, u);
        if (U.n <= 0) continue;
        const int h = U.hz;
        const int q_row0 = __ldg(a.cu_q + U.b) + kBM * U.tile;
        const int kv_row0 = __ldg(a.cu_k + U.b);
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
    // Step n: [wait dS_{n-1}] S_n, dP_n, then the pending dQ += dS_{n-1} K_{n-1}.
    if (lane == 0) {
      const uint32_t tS = tmem + COL_S, tDP = tmem + COL_DP, tDQ = tmem + COL_DQ,
                     tDS = tmem + COL_DS;
      struct Pend {
        int valid, ks, b, first, last;
        uint32_t g, oi;
      } pd{0, 0, 0, 0, 0, 0, 0};
      // dQ += dS_g K_g (the step's dS has been waited for already)
      auto issue_dq = [&](const Pend& p) -> bool {
        if (p.first && !wait_bar(bar(DQEMPTY), (p.oi & 1) ^ 1, wc, 0x103)) return false;
        tc_fence_after();
        const uint32_t kt = sK + p.ks * C::KV_BYTES;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tDQ, tDS + p.b * (BN / 2) + kk * 8, desc_mnmajor<BN>(kt, kk, 0), IDESC_DQ,
                 (!p.first || kk > 0) ? 1u : 0u);
        mma_commit(bar(KEMPTY + p.ks));
        if (p.last) mma_commit(bar(DQFULL));
        return true;
      };
      uint32_t qi = 0, ki = 0, vi = 0, g = 0, oi = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
        const Unit U = load_unit(a.units, u);
        if (U.n <= 0) continue;
        const int qb = qi % NQ;
        if (!wait_bar(bar(QFULL + qb), (qi / NQ) & 1, wc, 0x104)) { ok = false; break; }
        tc_fence_after();
        const uint32_t qt = sQ + qb * 2 * C::Q_BYTES, dot = qt + C::Q_BYTES;
        for (int n = 0; n < U.n; ++n) {
          const int ks = ki % NK, vs = vi % NV, b = g & 1;
          // S and dP of the previous step must have been read before they are overwritten
          if (pd.valid) {
            if (!wait_bar(bar(DSFULL + pd.b), (pd.g >> 1) & 1, wc, 0x105)) { ok = false; break; }
          }
          if (!wait_bar(bar(KFULL + ks), (ki / NK) & 1, wc, 0x106)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kt = sK + ks * C::KV_BYTES, vt = sV + vs * C::KV_BYTES;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tS, desc_kmajor<kBM>(qt, kk), desc_kmajor<BN>(kt, kk), IDESC_S, kk > 0 ? 1u : 0u);
          if (!wait_bar(bar(VFULL + vs), (vi / NV) & 1, wc, 0x107)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tDP, desc_kmajor<kBM>(dot, kk), desc_kmajor<BN>(vt, kk), IDESC_S, kk > 0 ? 1u : 0u);
          mma_commit(bar(SPFULL));
          mma_commit(bar(VEMPTY + vs));
          if (n == U.n - 1) mma_commit(bar(QEMPTY + qb));
          if (pd.valid && !issue_dq(pd)) { ok = false; break; }
          pd = Pend{1, ks, b, n == 0, n == U.n - 1, g, oi};
          ++ki;
          ++vi;
          ++g;
        }
        ++qi;
        ++oi;
      }
      if (ok && pd.valid) {
        if (wait_bar(bar(DSFULL + pd.b), (pd.g >> 1) & 1, wc, 0x109)) issue_dq(pd);
      }
      mma_commit(bar(DRAIN));
      wait_bar(bar(DRAIN), 0, drain, 0x1ff);
    }
  } else {
    // ------------------------------------------------------------ SiLU' + epilogue
    // Eight warps: warp w owns TMEM lane quarter w % 4 and one half of the key
    // columns of each S / dP tile (and of the dQ columns).
    constexpr int CPW = BN / 2;
    const int wq = warp & 3, hc = (warp - 2) >> 2;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + COL_S + lane_off + hc * CPW, tDP = tmem + COL_DP + lane_off + hc * CPW,
                   tDQ = tmem + COL_DQ + lane_off, tDS = tmem + COL_DS + lane_off + hc * (CPW / 2);
    const float half_alpha = 0.5f * a.alpha;
    const float out_scale = 0.5f * a.alpha * a.inv_L;  // dS is stored doubled
    uint32_t g = 0, oi = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < n_units; u += gridDim.x) {
      const Unit U = load_unit(a.units, u);
      const int h = U.hz;
      const int q0 = __ldg(a.cu_q + U.b);
      const int Lq = __ldg(a.cu_q + U.b + 1) - q0;
      const int Lk = __ldg(a.cu_k + U.b + 1) - __ldg(a.cu_k + U.b);
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
        if (!wait_bar_warp(bar(SPFULL), g & 1, wc, 0x201)) { ok = false; break; }
        tc_fence_after();
        const int jc = BN * n + hc * CPW;
        const bool need_mask = (a.causal && jc + CPW - 1 > i_warp) || (jc + CPW > Lk);
#pragma unroll
        for (int sc = 0; sc < CPW / 32; ++sc) {
          uint32_t xs[32], xp[32];
          tmem_ld32x2(tS + 32 * sc, tDP + 32 * sc, xs, xp);
          uint32_t d[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float v[2];
#pragma unroll
            for (int t2 = 0; t2 < 2; ++t2) {
              float sv = __uint_as_float(xs[2 * e + t2]), pv = __uint_as_float(xp[2 * e + t2]);
              if (need_mask && jc + 32 * sc + 2 * e + t2 >= lim) { sv = 0.f; pv = 0.f; }
              const float hh = sv * half_alpha;
              v[t2] = dsilu2(hh, tanh_approx(hh), pv);
            }
            d[e] = pack2<BF16>(v[0], v[1]);
          }
          tmem_st16(tDS + b * (BN / 2) + 16 * sc, d);
        }
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
cudaError_t launch_dq_t(int grid, cudaStream_t st, const CUtensorMap& tq, const CUtensorMap& tdo,
                        const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a) {
  auto kern = hstu_bwd_dq_kernel<D, BF16>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DqCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<grid, kAttnThreads, DqCfg<D>::SMEM, st>>>(tq, tdo, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dq(int D, bool bf16, int grid, cudaStream_t st, const CUtensorMap& tq,
                      const CUtensorMap& tdo, const CUtensorMap& tk, const CUtensorMap& tv,
                      const AttnArgs& a) {
  switch (D) {
    case 64: return bf16 ? launch_dq_t<64, true>(grid, st, tq, tdo, tk, tv, a)
                         : launch_dq_t<64, false>(grid, st, tq, tdo, tk, tv, a);
    case 128: return bf16 ? launch_dq_t<128, true>(grid, st, tq, tdo, tk, tv, a)
                          : launch_dq_t<128, false>(grid, st, tq, tdo, tk, tv, a);
    case 256: return bf16 ? launch_dq_t<256, true>(grid, st, tq, tdo, tk, tv, a)
                          : launch_dq_t<256, false>(grid, st, tq, tdo, tk, tv, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hstu
