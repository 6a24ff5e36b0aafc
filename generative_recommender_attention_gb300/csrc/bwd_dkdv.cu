// HSTU attention backward, dK/dV part (chain rule of "HSTU Attention
// (Blackwell SM100/SM103)", Overview equations):
//   dV_j = (1/L_scale)     sum_i M_ij SiLU(alpha q_i.k_j) dO_i
//   dK_j = (alpha/L_scale) sum_i M_ij <dO_i, v_j> SiLU'(alpha q_i.k_j) q_i
//
// Key-stationary: each CTA owns a 128-row key tile and walks the 64-row
// query tiles that can see it.  Per half-step h it recomputes
// S^T = K Q^T and dP^T = V dO^T into TMEM, forms A^T = M (.) SiLU(alpha S^T)
// and dS^T = M (.) dP^T (.) SiLU'(alpha S^T) in registers (one tanh per
// element), writes both back in place as 16-bit, and accumulates
// dV += A^T dO and dK += dS^T Q with the A operand read from TMEM.  No
// atomics.  Each dS block (64 queries x 128 keys, query-major) is also
// stored to the workspace, where the dQ phase reads it for dQ = dS K; keys
// past the sequence end store zeros there, so they add nothing to dQ.  A
// thread holds one key row of dS^T; neighbouring lanes swap halves of their
// packed pairs so that every 4-byte store writes two keys of one query and
// a warp's store covers two contiguous 64-byte runs.
//   warp 0       TMA: K and V per unit, Q and dO per half-step (separate
//                rings: Q is released after dK, dO after dV); at D <= 128
//                also the TMA stores of finished dK / dV tiles.
//   warp 1       tcgen05 issuer of the dV chain: S^T_h into S^T buffer h % 2,
//                and dV += A^T_h dO_h as soon as A^T_h is written, followed
//                at once by S^T_{h+2} into the same buffer (MMAs from one
//                thread execute in order, so S^T_{h+2} cannot overwrite A^T_h
//                before dV_h has read it, and no release barrier is needed).
//   warp 10      the same for the dK chain: dP^T_h, dK += dS^T_h Q_h,
//                dP^T_{h+2}.
//   warps 2-9    row work, two warps per TMEM lane quarter (one per half of
//                the query columns): A^T_h from S^T_h as soon as S^T_h
//                lands (so dV_h overlaps dP^T_h), then dS^T_h from dP^T_h.
// Epilogue: once a unit's last MMAs complete, the row warps read dV and dK
// from TMEM and release them at once.  At D <= 128 they write the two tiles
// (scaled, 16-bit, in the TMA box layout) into the unit's own K / V buffer,
// which no MMA reads any more, and the producer issues TMA stores of them
// before it loads the unit after next into that buffer; per-row stores of
// 64-byte pieces (one cache line per lane) kept the row warps from the next
// unit for several thousand cycles.  Ragged last tiles and D = 256 (one
// K/V buffer) keep the per-row stores.
// D = 256: the dV and dK accumulators (256 fp32 columns each) do not fit in
// TMEM together, so the key tiles are walked twice, in two phases of the
// launch: a dV pass (S^T, A^T, dV += A^T dO: no V tile and no dP^T, so its
// shared memory holds three Q and two dO stages) and a dK pass (S^T, dP^T,
// dS^T, dK += dS^T Q, with dO released right after dP^T, so one dO stage
// overlaps the next load).  The passes are list B's two halves; together
// they do five of the six products that splitting the head into two
// 128-column halves (each recomputing S^T and dP^T) took, and neither
// waits for a Q / dO load with a single stage of both.
// After its last dK/dV unit the CTA drains, re-initialises its barriers and
// runs dQ units (bwd_dq.cuh) in the same shared memory and TMEM; each waits
// for the readiness count of its sequence and head (ready_target), which
// the row warps raise once per unit after fencing their dS stores.
// TMEM: S^T0 | S^T1 | dP^T0 | dP^T1 | dV | dK.  The two dependency chains
// (S^T -> A^T -> dV -> S^T and dP^T -> dS^T -> dK -> dP^T) run side by side,
// two half-steps deep, one per issuing thread, so while one thread waits
// for the row warps the other keeps the tensor pipe fed.
// The N = 64 S^T / dP^T MMAs run at about two thirds of the tensor rate; that
// costs less than serialising the row work with 128-query steps, for which
// TMEM has no room to double-buffer.
#include "bwd_dq.cuh"

namespace hstu {

namespace {

// First 64-query block a key tile visits (count: U.n): the window's rule, or
// under an arbitrary mask the start of the hull the scheduler recorded (the
// unit then visits the U.n live blocks of the hull).
__device__ __forceinline__ int unit_first_qblock(const AttnArgs& a, const UnitInfo& U, int bq) {
  if (a.fm.func != nullptr) return a.fm.kt_range[kt_slot(U.k0, U.b, U.tile)].x;
  int m0, cnt;
  key_tile_queries(U.tile, U.Lq, U.Lk, a.win, bq, m0, cnt);
  return m0;
}

// Arbitrary mask: the end of that hull.
__device__ __forceinline__ int unit_qblock_end(const AttnArgs& a, const UnitInfo& U) {
  const int2 r = a.fm.kt_range[kt_slot(U.k0, U.b, U.tile)];
  return r.x + r.y;
}

// A key tile whose 128 rows all belong to its sequence (and to the tensor)
// can leave through a TMA store of the whole tile; a ragged last tile is
// stored row by row, since the box would also cover the next sequence.
__device__ __forceinline__ bool tile_full(const UnitInfo& U, int64_t total_k) {
  const int end = kBM * (U.tile + 1);
  return end <= U.Lk && static_cast<int64_t>(U.k0) + end <= total_k;
}

// One dK/dV phase of the backward kernel over list `a` (or the half of it
// that a.part names): the role code of every warp.  PASS: both
// accumulators (D <= 128), or the dV or dK pass (D = 256).  The caller has
// allocated TMEM and waited for the previous grid; the phase initialises
// its barriers at `bars`, and on return the block has synchronised and the
// barriers are invalidated (every MMA, TMEM read and copy has completed).
template <int D, bool BF16, bool FUNC, int PASS>
__device__ __forceinline__ void dkdv_phase(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                           const CUtensorMap* tm_q, const CUtensorMap* tm_do,
                                           const CUtensorMap* tm_dk, const CUtensorMap* tm_dv,
                                           const AttnArgs& a, uint32_t base, uint64_t* bars,
                                           volatile int* flags, UnitInfo* ring, uint32_t tmem) {
  using C = DkdvCfg<D, PASS>;
  constexpr int BQ = C::BQ, DH = C::DH, SPLIT = C::SPLIT, NKV = C::NKV;
  constexpr int NSQ = C::NSQ, NSD = C::NSD;
  constexpr int KCH = D / 64;
  constexpr bool DO_V = PASS != kPassDK;  // accumulates dV
  constexpr bool DO_K = PASS != kPassDV;  // forms dP^T and dS^T, accumulates dK
  constexpr int RW = kDkdvRowWarps;
  constexpr int WPQ = RW / 4;    // row warps per TMEM lane quarter
  constexpr int CW = BQ / WPQ;   // query columns per row warp
  constexpr int DW = DH / WPQ;  // dK / dV columns per row warp
  constexpr int MMA_B = 2 + RW;  // warp of the dK chain's issuer
  // With two (K, V) buffers, a unit's dV / dK leave through its own K / V
  // buffer: the row warps stage them there once the unit's MMAs are done,
  // and the producer writes them out with TMA stores before it loads the
  // unit after next into that buffer.
  constexpr bool STAGE = NKV == 2;
  static_assert(!STAGE || PASS == kPassBoth, "staging holds both tiles");
  // Score tiles issued ahead of the accumulation that frees their buffer.
  // Both accumulators: step h + LOOK needs a Q / dO stage that only step
  // h + LOOK - NS releases, so LOOK < NS, or the two issuers could wait on
  // each other.  The dV pass releases Q with S^T, the dK pass dO with dP^T,
  // so those rings never hold up the look-ahead; the dK pass's Q ring (two
  // stages) still limits it to one.
  constexpr int LOOK = PASS == kPassDV ? 2 : PASS == kPassDK ? 1 : (NSQ >= 3 ? 2 : 1);
  static_assert(PASS != kPassBoth || NSQ != NSD || LOOK < NSQ || NSQ == 1,
                "look-ahead must leave a free stage");
  static_assert(PASS != kPassDK || LOOK < NSQ, "look-ahead must leave a free Q stage");
  constexpr uint32_t IDESC_S = idesc_f16(BF16, kBM, BQ, false, false);
  constexpr uint32_t IDESC_ACC = idesc_f16(BF16, kBM, DH, false, true);
  constexpr uint32_t COL_ST = 0, COL_DPT = 2 * BQ, COL_DV = 4 * BQ,
                     COL_DK = 4 * BQ + (DO_V ? DH : 0);
  static_assert((DO_K ? COL_DK : COL_DV) + DH <= kTmemCols, "TMEM budget");
  static_assert(C::TILE_BYTES <= BwdCfg<D>::TILE_BYTES, "tile area");
  static_assert(CW == 32, "one query per lane in the arbitrary-mask transpose");
  static_assert(BQ == kDsQueries && kBM == kDsKeys && CW % 8 == 0 && CW <= 32,
                "one stored dS block per half-step");

  const uint32_t sKV = base;                          // NKV x (K[, V])
  const uint32_t sQ = sKV + NKV * C::KV_STRIDE;       // NSQ x Q
  const uint32_t sDO = sQ + NSQ * C::Q_BYTES;         // NSD x dO

  enum {
    KVFULL = 0, KVEMPTY = KVFULL + NKV, QFULL = KVEMPTY + NKV, QEMPTY = QFULL + NSQ,
    DOFULL = QEMPTY + NSQ, DOEMPTY = DOFULL + NSD, SFULL = DOEMPTY + NSD, PFULL = SFULL + 2,
    AFULL = PFULL + 2, DSFULL = AFULL + 2,
    ACCFULL = DSFULL + 2, ACCEMPTY = ACCFULL + 1, STAGED = ACCEMPTY + 1, UFULL = STAGED + 2,
    UEMPTY = UFULL + kUnitRing, DRAIN = UEMPTY + kUnitRing, NBARS = DRAIN + 2
  };
  static_assert(NBARS <= BwdCfg<D>::kBars, "barrier area");
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    // K / V: released by each issuer that reads them (the dV pass: the dV
    // chain only); Q by its last reader (dK, or S^T in the dV pass); dO by
    // dV and dP^T (both accumulators), else by its one reader
    constexpr int kv_readers = PASS == kPassDV ? 1 : 2;
    for (int i = 0; i < NKV; ++i) {
      mbar_init(bar(KVFULL + i), 1);
      mbar_init(bar(KVEMPTY + i), kv_readers);
    }
    for (int i = 0; i < NSQ; ++i) { mbar_init(bar(QFULL + i), 1); mbar_init(bar(QEMPTY + i), 1); }
    for (int i = 0; i < NSD; ++i) {
      mbar_init(bar(DOFULL + i), 1);
      mbar_init(bar(DOEMPTY + i), PASS == kPassBoth ? 2 : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(SFULL + i), 1);
      mbar_init(bar(PFULL + i), 1);
      mbar_init(bar(AFULL + i), RW);
      mbar_init(bar(DSFULL + i), RW);
    }
    mbar_init(bar(ACCFULL), PASS == kPassBoth ? 2 : 1);  // the accumulating chains
    mbar_init(bar(ACCEMPTY), RW);
    mbar_init(bar(STAGED), RW);
    mbar_init(bar(STAGED + 1), RW);
    for (int i = 0; i < kUnitRing; ++i) {
      mbar_init(bar(UFULL + i), 1);
      mbar_init(bar(UEMPTY + i), 2 + RW);
    }
    mbar_init(bar(DRAIN), 1);
    mbar_init(bar(DRAIN + 1), 1);
    fence_mbar_init();
  }
  __syncwarp();  // thread 0's set-up above diverged warp 0
  __syncthreads();
  const WaitCtl wc{a.header, flags, a.timeout_ns};
  const WaitCtl drain{a.header, flags + 1, a.timeout_ns};
  // list B whole, or one of its halves (D = 256: the dV pass takes the first)
  const int n_all = work_units(a);
  const int n_units = a.part != 0 ? n_all / 2 : n_all;
  const int4* ulist = a.units + (a.part == 2 ? 2 * static_cast<int64_t>(n_units) : 0);
  const UnitQueue uq{ring, bar(UFULL), bar(UEMPTY)};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t kvi = 0, qi = 0;
      bool ok = true;
      int prev_n = kPrefetchQ;  // steps of the previous unit (the first unit is not warmed)
      auto prefetch_qdo = [&](int h, int row) {
#pragma unroll
        for (int c = 0; c < KCH; ++c) {
          tma_prefetch_3d(tm_q, 64 * c, h, row);
          tma_prefetch_3d(tm_do, 64 * c, h, row);
        }
      };
      // Staged output tiles of K/V buffers 0 and 1: first key row (-1: the
      // row warps stored that unit row by row) and head.
      int st_row0 = -1, st_hd0 = 0, st_row1 = -1, st_hd1 = 0;
      // A unit reads its K / V tiles and writes its dK / dV tiles once: those
      // lines leave L2 first, so that more of the dS blocks stay there until
      // the dQ units read them (Q / dO tiles, which the other key tiles of the
      // group read again, keep the normal priority).  Measured: recsys 127.5
      // against 129.9 us per step, no workload slower.
      const uint64_t stream_policy = l2_policy_evict_first();
      // Writes out the dV / dK tiles that the u-th unit (with key steps)
      // staged in its K/V buffer, and waits until TMA has read them.
      auto store_staged = [&](uint32_t u, const WaitCtl& w) -> bool {
        const int kb = static_cast<int>(u & 1u);
        if (!wait_bar(bar(STAGED + kb), (u >> 1) & 1u, w, 0x005)) return false;
        const int row = kb ? st_row1 : st_row0, hd = kb ? st_hd1 : st_hd0;
        if (row >= 0) {
          const uint32_t kt = sKV + kb * C::KV_STRIDE, vt = kt + C::KV_BYTES;
#pragma unroll
          for (int c = 0; c < KCH; ++c) {
            tma_store_3d_hint(tm_dk, kt + c * (kBM * 128), 64 * c, hd, row, stream_policy);
            tma_store_3d_hint(tm_dv, vt + c * (kBM * 128), 64 * c, hd, row, stream_policy);
          }
          bulk_commit_group();
          bulk_wait_read_all();
        }
        return true;
      };
      // Units are claimed one ahead: the next claim overlaps this unit's
      // loads.  Every dK/dV unit, the first included, comes from the counter,
      // so only CTAs already running hold one: the dQ units that wait for
      // them never wait on a CTA that has not started.
      UnitInfo nx = load_unit_info(ulist, atomicAdd(a.header + a.next_slot, 1), n_units);
      for (uint32_t uk = 0; ok; ++uk) {
        UnitInfo U = nx;
        if (U.n > 0 && DO_K) {
          // first stored dS block of this key tile (the units that form dS^T
          // store it); -1 when the metadata outgrew the workspace
          const int b0 = __ldg(a.ds_base + U.b), b1 = __ldg(a.ds_base + U.b + 1);
          const int blk = b0 + (U.hz / SPLIT) * ((b1 - b0) / a.H) +
                          ds_block_off(U.tile, U.Lq, U.Lk, a.win);
          // an arbitrary mask stores its live blocks at their places in the hull
          const int span = FUNC ? unit_qblock_end(a, U) - unit_first_qblock(a, U, BQ) : U.n;
          U.ds = (blk >= 0 && static_cast<int64_t>(blk) + span <= a.ds_cap) ? blk : -1;
        }
        if (!unit_push(uq, uk, U, wc)) { ok = false; break; }
        if (U.n < 0) break;
        nx = load_unit_info(ulist, atomicAdd(a.header + a.next_slot, 1), n_units);
        if (U.n <= 0) continue;
        const int h = U.hz / SPLIT;
        const int k_row0 = U.k0 + kBM * U.tile;
        const int q_seq0 = U.q0;
        const int m0 = unit_first_qblock(a, U, BQ);  // query tiles m0 .. m0 + U.n - 1
        const int m_end = FUNC ? unit_qblock_end(a, U) : 0;
        int m_next = m0;  // live-block cursor (arbitrary mask)
        BlockWalk bw;  // the live blocks, 32 at a time
        bw.init();
        const int kb = kvi % NKV;
        if constexpr (STAGE) {
          // buffer kb last held the unit before the previous one
          if (kvi >= 2 && !store_staged(kvi - 2, wc)) { ok = false; break; }
          const int row = tile_full(U, a.total_k) ? k_row0 : -1;
          if (kb) { st_row1 = row; st_hd1 = h; } else { st_row0 = row; st_hd0 = h; }
        } else {
          if (!wait_bar(bar(KVEMPTY + kb), ((kvi / NKV) & 1) ^ 1, wc, 0x001)) { ok = false; break; }
        }
        mbar_arrive_expect_tx(bar(KVFULL + kb), C::KV_STRIDE);
        const uint32_t kt = sKV + kb * C::KV_STRIDE, vt = kt + C::KV_BYTES;
#pragma unroll
        for (int c = 0; c < KCH; ++c) {
          tma_load_3d_hint(kt + c * (kBM * 128), tm_k, bar(KVFULL + kb), 64 * c, h, k_row0,
                           stream_policy);
          if constexpr (C::LOAD_V)
            tma_load_3d_hint(vt + c * (kBM * 128), tm_v, bar(KVFULL + kb), 64 * c, h, k_row0,
                             stream_policy);
        }
        ++kvi;
        // L2 warm-up runs kPrefetchQ steps ahead of the loads along the flat
        // stream (this unit's later Q/dO tiles, then the next unit's K, V and
        // first Q/dO tiles); what a short previous unit could not cover is
        // issued here.
        if (prev_n < kPrefetchQ)
          for (int m = 0; m < min(U.n, kPrefetchQ - prev_n); ++m) prefetch_qdo(h, q_seq0 + BQ * (m0 + m));
        prev_n = U.n;
        int nx_m0 = -1;  // the next unit's first query block, read when first needed
        for (int m = 0; m < U.n; ++m) {
          const int sq = qi % NSQ, sd = qi % NSD;
          int qm = m0 + m;
          if constexpr (FUNC) {
            qm = bw.next<false>(a.fm, U.q0, U.b, U.tile, m_next, m_end);
            m_next = qm + 1;
          }
          const int row = q_seq0 + BQ * qm;
          if (!wait_bar(bar(QEMPTY + sq), ((qi / NSQ) & 1) ^ 1, wc, 0x002)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(QFULL + sq), C::Q_BYTES);
#pragma unroll
          for (int c = 0; c < KCH; ++c)
            tma_load_3d(sQ + sq * C::Q_BYTES + c * (BQ * 128), tm_q, bar(QFULL + sq), 64 * c, h, row);
          if (!wait_bar(bar(DOEMPTY + sd), ((qi / NSD) & 1) ^ 1, wc, 0x004)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(DOFULL + sd), C::Q_BYTES);
#pragma unroll
          for (int c = 0; c < KCH; ++c)
            tma_load_3d(sDO + sd * C::Q_BYTES + c * (BQ * 128), tm_do, bar(DOFULL + sd), 64 * c, h,
                        row);
          ++qi;
          // the L2 warm-up of step m + kPrefetchQ, after this step's loads (under an
          // arbitrary mask the next unit's first block is a global read)
          const int t = m + kPrefetchQ;
          if (t < U.n) {
            prefetch_qdo(h, q_seq0 + BQ * (m0 + t));
          } else if (t - U.n < nx.n) {
            const int nh = nx.hz / SPLIT;
            if (t == U.n) {
#pragma unroll
              for (int c = 0; c < KCH; ++c) {
                tma_prefetch_3d(tm_k, 64 * c, nh, nx.k0 + kBM * nx.tile);
                if constexpr (C::LOAD_V) tma_prefetch_3d(tm_v, 64 * c, nh, nx.k0 + kBM * nx.tile);
              }
            }
            if (nx_m0 < 0) nx_m0 = unit_first_qblock(a, nx, BQ);
            prefetch_qdo(nh, nx.q0 + BQ * (nx_m0 + t - U.n));
          }
        }
      }
      if constexpr (STAGE) {
        if (ok)
          for (uint32_t u = kvi > 2 ? kvi - 2 : 0; u < kvi; ++u)
            if (!store_staged(u, wc)) break;
        bulk_wait_all();  // the output writes are complete before the block exits
      }
      for (uint32_t i = kvi > NKV ? kvi - NKV : 0; i < kvi; ++i)
        wait_bar(bar(KVFULL + i % NKV), (i / NKV) & 1, drain, 0x0f1);
      for (uint32_t i = qi > NSQ ? qi - NSQ : 0; i < qi; ++i)
        wait_bar(bar(QFULL + i % NSQ), (i / NSQ) & 1, drain, 0x0f2);
      for (uint32_t i = qi > NSD ? qi - NSD : 0; i < qi; ++i)
        wait_bar(bar(DOFULL + i % NSD), (i / NSD) & 1, drain, 0x0f3);
    }
  } else if (warp == 1 || warp == MMA_B) {
    // ------------------------------------------------------------ chain issuers
    // Warp 1: S^T = K Q^T and dV += A^T dO.  Warp MMA_B: dP^T = V dO^T and
    // dK += dS^T Q.  In the dV pass the dK chain only keeps pace with the
    // unit ring; in the dK pass the dV chain issues S^T only.  Waits on
    // TMA-filled stages need no tcgen05 fence; waits on the row warps' TMEM
    // accesses do.
    if (lane == 0) {
      const bool vchain = warp == 1;
      const bool accumulates = vchain ? DO_V : DO_K;
      const bool idle = !vchain && !DO_K;  // the dK chain in the dV pass
      // score MMA: A = K or V tile (K-major), B = Q or dO stage (K-major)
      const int kv_off = vchain ? 0 : C::KV_BYTES;
      const uint32_t sB = vchain ? sQ : sDO;
      const int bfull = vchain ? QFULL : DOFULL;
      const int nsb = vchain ? NSQ : NSD;  // the score's B-operand ring
      const uint32_t tScore = tmem + (vchain ? COL_ST : COL_DPT);
      const int score_full = vchain ? SFULL : PFULL;
      // accumulation: A = the 16-bit operand written over the score buffer,
      // B = dO or Q stage (MN-major), into dV or dK
      const uint32_t sAccB = vchain ? sDO : sQ;
      const int accbfull = vchain ? DOFULL : QFULL;
      const int nsa = vchain ? NSD : NSQ;  // the accumulation's B-operand ring
      const int ready = vchain ? AFULL : DSFULL;
      const uint32_t tAcc = tmem + (vchain ? COL_DV : COL_DK);
      uint32_t kvi = 0, h = 0, oi = 0;
      bool ok = true;
      auto score = [&](uint32_t hh, const SDesc& ad) -> bool {
        const int s = hh % nsb, b = hh & 1;
        if (!wait_bar(bar(bfull + s), (hh / nsb) & 1, wc, vchain ? 0x106 : 0x107)) return false;
        const SDesc bd = kdesc(sB + s * C::Q_BYTES);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tScore + b * BQ, desc_kmajor<kBM>(ad, kk), desc_kmajor<BQ>(bd, kk), IDESC_S,
                 kk > 0 ? 1u : 0u);
        mma_commit(bar(score_full + b));
        if (!vchain) mma_commit(bar(DOEMPTY + s));  // dP^T is the dK chain's only dO reader
        if (vchain && PASS == kPassDV) mma_commit(bar(QEMPTY + s));  // the dV pass's only Q reader
        return true;
      };
      for (uint32_t uk = 0; ok; ++uk) {
        UnitInfo U;
        if (!unit_pop(uq, uk, U, wc)) { ok = false; break; }
        if (U.n < 0) break;
        if (U.n <= 0 || idle) continue;
        const int kb = kvi % NKV;
        if (!wait_bar(bar(KVFULL + kb), (kvi / NKV) & 1, wc, 0x104)) { ok = false; break; }
        const SDesc ad = kdesc(sKV + kb * C::KV_STRIDE + kv_off);
        // the first LOOK score tiles of the unit; later ones follow the
        // accumulation (or, without one, the row warps' read) that frees
        // their buffer
        for (int m = 0; m < U.n && m < LOOK && ok; ++m) ok = score(h + m, ad);
        for (int m = 0; m < U.n && ok; ++m, ++h) {
          const int b = h & 1;
          if (!wait_bar(bar(ready + b), (h >> 1) & 1, wc, vchain ? 0x105 : 0x10a)) { ok = false; break; }
          tc_fence_after();
          if (accumulates) {
            const int s = h % nsa;
            if (!wait_bar(bar(accbfull + s), (h / nsa) & 1, wc, 0x10b)) { ok = false; break; }
            if (m == 0 && !wait_bar(bar(ACCEMPTY), (oi & 1) ^ 1, wc, 0x103)) { ok = false; break; }
            tc_fence_after();
            const SDesc bd = mndesc<BQ>(sAccB + s * C::Q_BYTES);
            // A^T / dS^T of queries [16 kk, 16 kk + 16) sit packed in the first
            // half of their row warp's own CW columns
#pragma unroll
            for (int kk = 0; kk < BQ / 16; ++kk)
              mma_ts(tAcc, tScore + b * BQ + (16 * kk / CW) * CW + (16 * kk % CW) / 2,
                     desc_mnmajor<BQ>(bd, kk, 0), IDESC_ACC, (m > 0 || kk > 0) ? 1u : 0u);
            mma_commit(bar((vchain ? DOEMPTY : QEMPTY) + s));
            if (m == U.n - 1) mma_commit(bar(ACCFULL));
          }
          if (m + LOOK < U.n && !score(h + LOOK, ad)) { ok = false; break; }
        }
        if (!STAGE) mma_commit(bar(KVEMPTY + kb));  // staged: the epilogue frees it
        ++kvi;
        if (accumulates) ++oi;
      }
      mma_commit(bar(DRAIN + (vchain ? 0 : 1)));
      wait_bar(bar(DRAIN + (vchain ? 0 : 1)), 0, drain, vchain ? 0x1ff : 0x1fe);
    }
  } else {
    // ------------------------------------------------------------ A^T, dS^T + epilogue
    // Warp w owns TMEM lane quarter w % 4 (32 key rows) and one share of the
    // query columns of each S^T / dP^T tile (and of dK / dV).
    const int wq = warp & 3, cg = (warp - 2) >> 2;
    const int r = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tST = tmem + COL_ST + lane_off + cg * CW,
                   tDPT = tmem + COL_DPT + lane_off + cg * CW,
                   tDV = tmem + COL_DV + lane_off + cg * DW, tDK = tmem + COL_DK + lane_off + cg * DW;
    const int q_first = cg * CW;
    const float half_alpha = 0.5f * a.alpha;
    const float dk_scale = 0.5f * a.alpha * a.inv_L;  // dS^T is stored doubled
    uint32_t h = 0, oi = 0;
    bool ok = true;
    // This warp's dS stores of unit V are issued: fence them and count the
    // unit toward the readiness of its sequence and head.
    auto count_unit = [&](const UnitInfo& V) {
      if (a.ready == nullptr) return;
      __threadfence();
      __syncwarp();
      if (lane == 0) atomicAdd(a.ready + V.b * a.H + V.hz / SPLIT, 1);
    };
    // this lane's dV / dK row pieces of unit V, for the per-row stores
    // (formed only where they are used, so no pointer stays live across the
    // steps); returns whether the row exists
    auto out_rows = [&](const UnitInfo& V, char*& dvrow, char*& dkrow) -> bool {
      const int jj = kBM * V.tile + r;
      const int64_t grow = static_cast<int64_t>(V.k0) + jj;
      const int64_t hd = V.hz / SPLIT;
      const int64_t col0 = cg * DW;
      dvrow = static_cast<char*>(a.o0) + (grow * a.o0_st + hd * a.o0_sh + col0) * 2;
      dkrow = static_cast<char*>(a.o1) + (grow * a.o1_st + hd * a.o1_sh + col0) * 2;
      // columns past d_out (a zero-padded head dim 32) are not stored
      return jj < V.Lk && grow < a.total_k && col0 < a.d_out;
    };
    // Epilogue of unit V (the oi-th unit with key steps): wait for its last
    // MMAs, read dV and dK out of TMEM, release them, write them out.
    auto epilogue = [&](const UnitInfo& V) -> bool {
      if (!wait_bar_warp(bar(ACCFULL), oi & 1, wc, 0x202)) return false;
      tc_fence_after();
      const bool staged = STAGE && tile_full(V, a.total_k);
      if (staged) {
        // dV into the V half and dK into the K half of the unit's (K, V)
        // buffer, which no MMA reads any more (ACCFULL covers them all)
        const uint32_t kt = sKV + (oi & 1u) * C::KV_STRIDE, vt = kt + C::KV_BYTES;
#pragma unroll
        for (int c = 0; c < DW / 32; ++c) {
          uint32_t xv[32], xk[32];
          tmem_ld32x2(tDV + 32 * c, tDK + 32 * c, xv, xk);
          stage_row32<BF16>(vt, r, cg * DW + 32 * c, xv, a.inv_L);
          stage_row32<BF16>(kt, r, cg * DW + 32 * c, xk, dk_scale);
        }
      } else if constexpr (DW <= 32) {
        char *dvrow, *dkrow;
        const bool row_ok = out_rows(V, dvrow, dkrow);
        uint32_t x[DW];
        if constexpr (DO_V) {
          tmem_ld_w<DW>(tDV, x);
          if (row_ok) store_row_n<DW, BF16>(dvrow, x, a.inv_L);
        }
        if constexpr (DO_K) {
          tmem_ld_w<DW>(tDK, x);
          if (row_ok) store_row_n<DW, BF16>(dkrow, x, dk_scale);
        }
      } else {
        char *dvrow, *dkrow;
        const bool row_ok = out_rows(V, dvrow, dkrow);
#pragma unroll 1
        for (int c = 0; c < DW / 32; ++c) {
          uint32_t x[32];
          if constexpr (DO_V) {
            tmem_ld32(tDV + 32 * c, x);
            if (row_ok) store_row_n<32, BF16>(dvrow + c * 64, x, a.inv_L);
          }
          if constexpr (DO_K) {
            tmem_ld32(tDK + 32 * c, x);
            if (row_ok) store_row_n<32, BF16>(dkrow + c * 64, x, dk_scale);
          }
        }
      }
      warp_arrive(bar(ACCEMPTY));
      if constexpr (STAGE) {
        fence_proxy_async_smem();  // staged tiles become visible to the TMA store
        warp_arrive(bar(STAGED + (oi & 1u)));
      }
      ++oi;
      return true;
    };
    for (uint32_t uk = 0; ok; ++uk) {
      UnitInfo U;
      if (!unit_pop_warp(uq, uk, U, wc)) { ok = false; break; }
      if (U.n < 0) break;
      const int Lq = U.Lq, Lk = U.Lk;
      const int j = kBM * U.tile + r;
      const int j_warp_last = kBM * U.tile + wq * 32 + 31;
      if (U.n <= 0) {  // no key steps: zeros, no TMEM
        char *dvrow, *dkrow;
        if (out_rows(U, dvrow, dkrow)) {
          if (DO_V) store_zero_n<DW>(dvrow);
          if (DO_K) store_zero_n<DW>(dkrow);
        }
        count_unit(U);
        continue;
      }
      const int m0 = unit_first_qblock(a, U, BQ);  // query tiles m0 .. m0 + U.n - 1
      constexpr bool func = FUNC;  // arbitrary mask: a separate instantiation
      const int m_end = func ? unit_qblock_end(a, U) : 0;
      int m_next = m0;  // live-block cursor (arbitrary mask)
      BlockWalk bw;  // the live blocks and their full class, 32 at a time
      bw.init();
      // arbitrary mask: the first three endpoints of this lane's query row,
      // loaded one step ahead so their latency hides behind a half-step
      int qm_ahead = 0, e0 = 0, e1 = 0, e2 = 0;
      bool full_ahead = false;  // its block sees every key of the tile (no per-element mask)
      auto ends = [&](int qm, int& f0, int& f1, int& f2) {
        const int iq = BQ * qm + q_first + lane;
        const int64_t t = static_cast<int64_t>(U.q0) + (iq < Lq ? iq : 0);
        f0 = __ldg(a.fm.func + t);
        f1 = f2 = 0;
        if (a.fm.n >= 3) {
          f1 = __ldg(a.fm.func + a.fm.len + t);
          f2 = __ldg(a.fm.func + 2 * a.fm.len + t);
        }
      };
      if constexpr (func) {
        qm_ahead = bw.next<true>(a.fm, U.q0, U.b, U.tile, m_next, m_end);
        m_next = qm_ahead + 1;
        full_ahead = bw.is_full(qm_ahead);
        ends(qm_ahead, e0, e1, e2);
      }
      // valid queries of this key row: lo <= i < hi; every key row of the
      // warp is seen by queries [lo_all, hi_all)
      const int lo = a.win.right < 0 ? 0 : j - a.win.right;
      const int hi = a.win.left < 0 ? Lq : min(Lq, j + a.win.left + 1);
      const int lo_all = a.win.right < 0 ? 0 : j_warp_last - a.win.right;
      const int hi_all = a.win.left < 0 ? Lq : min(Lq, j_warp_last - 31 + a.win.left + 1);
      // dS blocks of this key tile: one per half-step, stored by the units
      // that form dS^T; this lane writes keys (r & ~1, r | 1) of query rows
      // q, q + 2, ..., q = cg * CW + (r & 1), at q * 256 + (r & ~1) * 2
      char* ds_row = nullptr;
      if (DO_K && U.ds >= 0)  // set by the producer when the blocks fit
        ds_row = static_cast<char*>(a.ds) + static_cast<int64_t>(U.ds) * kDsBlockBytes +
                 (cg * CW + (r & 1)) * (kDsKeys * 2) + (r & ~1) * 2;
      const bool key_ok = j < Lk;
      for (int m = 0; m < U.n; ++m, ++h) {
        const int b = h & 1;
        int qm = m0 + m;  // this step's query block
        int f0 = 0, f1 = 0, f2 = 0;
        bool full = false;
        if constexpr (func) {
          qm = qm_ahead;
          full = full_ahead;
          f0 = e0; f1 = e1; f2 = e2;
          if (m + 1 < U.n) {  // the next step's block, class and endpoints
            qm_ahead = bw.next<true>(a.fm, U.q0, U.b, U.tile, m_next, m_end);
            m_next = qm_ahead + 1;
            full_ahead = bw.is_full(qm_ahead);
            ends(qm_ahead, e0, e1, e2);
          }
        }
        const int ic = BQ * qm + q_first;  // first query of this warp's columns
        const bool need_mask = ic < lo_all || ic + CW > hi_all;
        // valid queries of this warp's columns (bit e: query ic + e), the run
        // of bits [lo - ic, hi - ic) clamped to [0, CW)
        uint32_t valid = CW == 32 ? 0xffffffffu : (1u << CW) - 1u;
        if (func && full) {
          // arbitrary mask, a full block: every query of it sees every key
          // row of the tile (keys past Lk are never stored); only the
          // sequence end cuts the columns
          const int nq = Lq - ic;
          valid = nq >= CW ? valid : nq <= 0 ? 0u : (1u << nq) - 1u;
        } else if constexpr (func) {
          // arbitrary mask: lane l forms query ic + l's valid keys among the
          // warp's 32 key rows from its endpoints; 32 ballots transpose them
          // into each key row's valid queries
          const int jw = j_warp_last - 31, iq = ic + lane;
          const uint32_t mq = iq < Lq ? static_cast<uint32_t>(func_row_bits3(
                                            a.fm, static_cast<int64_t>(U.q0) + iq, f0, f1, f2,
                                            jw, Lk))
                                      : 0u;
          uint32_t mine = 0;
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const uint32_t col = __ballot_sync(0xffffffffu, (mq >> k) & 1u);
            if (lane == k) mine = col;
          }
          valid = mine;
        } else if (need_mask) {
          const int e0 = min(max(lo - ic, 0), CW), e1 = min(max(hi - ic, 0), CW);
          const uint32_t below_e1 = e1 >= 32 ? 0xffffffffu : (1u << e1) - 1u;
          const uint32_t below_e0 = e0 >= 32 ? 0xffffffffu : (1u << e0) - 1u;
          valid = below_e1 & ~below_e0;
        }
        // A^T = SiLU(alpha S^T) as soon as S^T lands; h and tanh(h) are kept
        // for dS^T
        if (!wait_bar_warp(bar(SFULL + b), (h >> 1) & 1, wc, 0x201)) { ok = false; break; }
        tc_fence_after();
        float hv[CW], tv[CW];
        {
          uint32_t xs[CW];
          tmem_ld_w<CW>(tST + b * BQ, xs);
#pragma unroll
          for (int e = 0; e < CW; ++e) {
            hv[e] = ((valid >> e) & 1u) ? __uint_as_float(xs[e]) * half_alpha : 0.f;  // SiLU(0) = 0
            tv[e] = tanh_approx(hv[e]);
          }
        }
        if constexpr (DO_V) {
          uint32_t pk[CW / 2];
#pragma unroll
          for (int e = 0; e < CW / 2; ++e)
            pk[e] = pack2<BF16>(fmaf(hv[2 * e], tv[2 * e], hv[2 * e]),
                                fmaf(hv[2 * e + 1], tv[2 * e + 1], hv[2 * e + 1]));
          tmem_st_w<CW / 2>(tST + b * BQ, pk);   // in place over this warp's S^T columns
          tmem_st_wait();
        }
        // A^T written (or, in the dK pass, S^T read): the buffer is free
        warp_arrive(bar(AFULL + b));
        if constexpr (!DO_K) continue;
        // dS^T = dP^T SiLU'(alpha S^T) (doubled), masked entries exactly 0
        if (!wait_bar_warp(bar(PFULL + b), (h >> 1) & 1, wc, 0x203)) { ok = false; break; }
        tc_fence_after();
        uint32_t pd[CW / 2];
        {
          uint32_t xp[CW];
          tmem_ld_w<CW>(tDPT + b * BQ, xp);
#pragma unroll
          for (int e = 0; e < CW / 2; ++e) {
            const float d0 = ((valid >> (2 * e)) & 1u) ? __uint_as_float(xp[2 * e]) : 0.f;
            const float d1 = ((valid >> (2 * e + 1)) & 1u) ? __uint_as_float(xp[2 * e + 1]) : 0.f;
            pd[e] = pack2<BF16>(dsilu2(hv[2 * e], tv[2 * e], d0),
                                dsilu2(hv[2 * e + 1], tv[2 * e + 1], d1));
          }
        }
        tmem_st_w<CW / 2>(tDPT + b * BQ, pd);  // in place over this warp's dP^T columns
        tmem_st_wait();
        warp_arrive(bar(DSFULL + b));  // dK += dS^T Q may start; the global copy follows
        if (ds_row != nullptr) {
          // pd[e] = (dS[q0 + 2e][r], dS[q0 + 2e + 1][r]); the even lane keeps
          // query q0 + 2e for keys (r, r + 1), the odd lane query q0 + 2e + 1
          uint32_t* dst =
              reinterpret_cast<uint32_t*>(ds_row + static_cast<int64_t>(qm - m0) * kDsBlockBytes);
          const bool odd = (lane & 1) != 0;
#pragma unroll
          for (int e = 0; e < CW / 2; ++e) {
            const uint32_t mine = key_ok ? pd[e] : 0u;
            const uint32_t other = __shfl_xor_sync(0xffffffffu, mine, 1);
            dst[e * kDsKeys] = __byte_perm(mine, other, odd ? 0x3276u : 0x5410u);
          }
        }
      }
      if (!ok) break;
      count_unit(U);
      if (!epilogue(U)) { ok = false; break; }
    }
  }

  // The role branches leave lanes of warps 0, 1 and 10 on different paths;
  // reconverge each warp so the aligned CTA barrier counts it exactly once
  // (otherwise it can release before the row warps finish reading TMEM).
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // every phase of these barriers has completed: retire them for the next phase
  if (threadIdx.x == 0)
    for (int i = 0; i < NBARS; ++i) mbar_inval(bar(i));
  __syncwarp();
}

// The backward kernel: this CTA's dK/dV units (list B: args `a`, and at
// D = 256 its dV pass `a` then its dK pass `a2`), then its dQ units (list A,
// args `aq`; bwd_dq.cuh), in one launch.  Each phase takes over the tile
// area, the barrier words and TMEM once the one before has drained.
template <int D, bool BF16, bool FUNC>
__global__ void __launch_bounds__(kDkdvThreads, 1)
    hstu_bwd_kernel(const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dk,
                    const __grid_constant__ CUtensorMap tm_dv,
                    const __grid_constant__ CUtensorMap tm_ds, const AttnArgs a,
                    const AttnArgs a2, const AttnArgs aq) {
  using B = BwdCfg<D>;
  static_assert(dq::Bars<D>::NBARS <= B::kBars, "dQ phase barriers");
  // control block: barriers | TMEM slot (8 B) | flags (16 B) | unit ring
  static_assert(B::kBars * 8 + 24 + kUnitRing * sizeof(UnitInfo) <= kCtlBytes, "control block");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base_ptr + B::TILE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + B::kBars);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 2);
  UnitInfo* ring = reinterpret_cast<UnitInfo*>(const_cast<int*>(flags + 4));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    flags[0] = 0;
    flags[1] = 0;
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_q); tma_prefetch_desc(&tm_do);
    if (D <= 128) { tma_prefetch_desc(&tm_dk); tma_prefetch_desc(&tm_dv); }
    tma_prefetch_desc(&tm_ds);
  }
  if (warp == 1) { tmem_alloc(smem_u32(tmem_slot), kTmemCols); tmem_relinquish(); }
  __syncwarp();  // thread 0's set-up above diverged warp 0
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // everything below reads what earlier grids wrote (work lists, inputs)
  if (a.pdl_wait == 1) grid_dependency_wait();
  if (threadIdx.x == 0) grid_launch_dependents();

  // ---------------------------------------------------------------- dK/dV phases
  if constexpr (D == 256) {
    dkdv_phase<D, BF16, FUNC, kPassDV>(&tm_k, &tm_v, &tm_q, &tm_do, &tm_dk, &tm_dv, a, base, bars,
                                       flags, ring, tmem);
    if (flags[0] == 0)
      dkdv_phase<D, BF16, FUNC, kPassDK>(&tm_k, &tm_v, &tm_q, &tm_do, &tm_dk, &tm_dv, a2, base,
                                         bars, flags, ring, tmem);
  } else {
    dkdv_phase<D, BF16, FUNC, kPassBoth>(&tm_k, &tm_v, &tm_q, &tm_do, &tm_dk, &tm_dv, a, base,
                                         bars, flags, ring, tmem);
  }

  // ---------------------------------------------------------------- dQ phase
  // A CTA whose dK/dV phases gave up skips it (the dQ units that wait for its
  // counts then give up too, after the wait limit).
  const bool dkdv_ok = flags[0] == 0;
  if (threadIdx.x == 0) dq::init_bars<D>(bars);
  __syncwarp();
  __syncthreads();
  if (dkdv_ok) dq::run<D, BF16>(&tm_ds, &tm_k, aq, base, bars, flags, ring, tmem);
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // planned calls: the last CTA leaves the unit counters at zero and
  // advances the readiness epoch (every CTA has made its last claim and
  // passed its last readiness wait by then)
  if (a.planned && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.header + kHdrDone, 1) == static_cast<int>(gridDim.x) - 1) {
      atomicExch(a.header + a.next_slot, 0);
      if (D == 256) atomicExch(a.header + a2.next_slot, 0);
      atomicExch(a.header + aq.next_slot, 0);
      atomicAdd(a.header + kHdrEpoch, 1);
      atomicExch(a.header + kHdrDone, 0);
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool BF16, bool FUNC>
cudaError_t launch_bwd_f(int grid, cudaStream_t st, bool pdl, const BwdMaps& m, const AttnArgs& a,
                         const AttnArgs& a2, const AttnArgs& aq) {
  auto kern = hstu_bwd_kernel<D, BF16, FUNC>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         BwdCfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_attn(kern, grid, kDkdvThreads, BwdCfg<D>::SMEM, st, pdl, m.k, m.v, m.q, m.dout,
                     m.dk, m.dv, m.ds, a, a2, aq);
}

// The arbitrary-mask path (its endpoint loads and ballot transpose) is a
// separate instantiation, so that the window kernels keep their registers.
template <int D, bool BF16>
cudaError_t launch_bwd_t(int grid, cudaStream_t st, bool pdl, const BwdMaps& m, const AttnArgs& a,
                         const AttnArgs& a2, const AttnArgs& aq) {
  if (a.fm.func != nullptr) return launch_bwd_f<D, BF16, true>(grid, st, pdl, m, a, a2, aq);
  return launch_bwd_f<D, BF16, false>(grid, st, pdl, m, a, a2, aq);
}

}  // namespace

cudaError_t launch_bwd(int D, bool bf16, int grid, cudaStream_t st, bool pdl, const BwdMaps& m,
                       const AttnArgs& a, const AttnArgs& a2, const AttnArgs& aq) {
  switch (D) {
    case 64: return bf16 ? launch_bwd_t<64, true>(grid, st, pdl, m, a, a2, aq)
                         : launch_bwd_t<64, false>(grid, st, pdl, m, a, a2, aq);
    case 128: return bf16 ? launch_bwd_t<128, true>(grid, st, pdl, m, a, a2, aq)
                          : launch_bwd_t<128, false>(grid, st, pdl, m, a, a2, aq);
    case 256: return bf16 ? launch_bwd_t<256, true>(grid, st, pdl, m, a, a2, aq)
                          : launch_bwd_t<256, false>(grid, st, pdl, m, a, a2, aq);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace hstu
