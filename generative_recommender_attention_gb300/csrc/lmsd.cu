// HSTU LayerNorm-Multiply-SiLU-Dropout (page "HSTU LayerNorm-Multiply-SiLU-
// Dropout (LMSD)", Overview): per row of x (N, D), bf16,
//   xhat = (x - mean) rstd,  l = xhat * weight + bias,  a = SiLU(u) or u,
//   y = [dropout(a) if concat_u, dropout(x) if concat_x, dropout(l * a)],
// inverted dropout with one int8 mask per element (bit 0 main, bit 1 x
// segment, bit 2 u segment; set = kept), row mean and rstd saved for the
// backward.  The op is HBM-bound: one warp per row, 16-byte loads and stores
// (8 bf16 per lane per chunk) kept packed in registers, fp32 arithmetic.  The
// forward loads the next row of its warp while it computes the current one.
// The backward makes two passes over each row (the row means of dxhat and
// dxhat xhat, then dx and du); dweight and dbias are column sums
// over rows, reduced deterministically: each warp adds its rows' terms to
// its own shared-memory accumulators, each block sums its warps in a fixed
// order into a partial row of the workspace, and a second kernel sums the
// partials in block order.
//
// Dropout decisions: Philox4x32-10 (Salmon et al., SC 2011), implemented
// here from its definition.  One call decides 8 elements: element
// e = row * D + col of segment k uses the 16-bit half e % 2 (low first) of
// word (e % 8) / 2 of Philox(counter (e / 8 low, high, k, 0), key (seed low,
// high)) and is kept iff that half >= floor(p 2^16).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "hstu_lmsd.h"

namespace {

constexpr int kLmsdWarps = 8;          // rows in flight per block

struct Philox4 {
  uint32_t v[4];
};

// Round keys of one seed: round r uses (seed low + r W0, seed high + r W1).
// Computed on the host and passed in the kernel parameters, so the rounds
// read them as constants.
struct PhiloxKeys {
  uint32_t k[20];
};

PhiloxKeys philox_keys(uint64_t seed) {
  PhiloxKeys p;
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  for (int r = 0; r < 10; ++r) {
    p.k[2 * r] = k0;
    p.k[2 * r + 1] = k1;
    k0 += 0x9E3779B9u;  // key increments
    k1 += 0xBB67AE85u;
  }
  return p;
}

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2,
                                                 uint32_t c3, const PhiloxKeys& key) {
  constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;   // round multipliers
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(kM0, c0), lo0 = kM0 * c0;
    const uint32_t hi1 = __umulhi(kM1, c2), lo1 = kM1 * c2;
    const uint32_t n0 = hi1 ^ c1 ^ key.k[2 * r], n2 = hi0 ^ c3 ^ key.k[2 * r + 1];
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
  }
  return Philox4{{c0, c1, c2, c3}};
}

// The Philox words deciding the 8 elements e0 .. e0 + 7 (e0 a multiple of 8)
// of segment k.
__device__ __forceinline__ Philox4 draw8(uint64_t e0, uint32_t k, const PhiloxKeys& key) {
  const uint64_t g = e0 >> 3;
  return philox4x32_10(static_cast<uint32_t>(g), static_cast<uint32_t>(g >> 32), k, 0u, key);
}

// Element 2 j + h of a draw is kept iff its 16-bit half of word j (h = 0:
// low) is at least thr = floor(p 2^16); the kernels pass thr_hi = thr << 16.

__device__ __forceinline__ float2 bf2(uint32_t w) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
}

// 32-bit word j (two bf16, element 2 j in the low half) of a 16-byte chunk.
__device__ __forceinline__ uint32_t word(const uint4& v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = bf2(v[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over the 32 / RPW lanes that share a row (RPW rows per warp).
template <int RPW>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
  for (int o = 16 / RPW; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// sigmoid(u) = 1 / (1 + e^-u) with the fast exponential and reciprocal
// (e^-u = inf for u < -88 gives 0, the limit).
__device__ __forceinline__ float sigmoid(float u) { return __fdividef(1.f, 1.f + __expf(-u)); }

__device__ __forceinline__ uint4 ld16(const __nv_bfloat16* p, int ch) {
  return __ldg(reinterpret_cast<const uint4*>(p) + ch);
}

struct FwdArgs {
  const __nv_bfloat16* x;
  int64_t xs;
  const __nv_bfloat16* u;
  int64_t us;
  const __nv_bfloat16* w;
  const __nv_bfloat16* b;
  int64_t n;
  int d;
  float eps;
  float p;          // dropout ratio (fp32)
  uint32_t thr_hi;  // keep iff the 16-bit half << 16 >= thr_hi (0 without dropout)
  float scale;      // 1 / (1 - p)
  int silu, concat_u, concat_x;
  PhiloxKeys keys;
  __nv_bfloat16* y;
  float* mean;
  float* rstd;
  int8_t* mask;
};

// Blocks of 8 warps resident per SM (the register budget of the kernels
// below), by 8-element chunks per lane.
__host__ __device__ constexpr int fwd_blocks_per_sm(int nc) { return nc <= 1 ? 4 : nc == 2 ? 3 : 2; }
__host__ __device__ constexpr int bwd_blocks_per_sm(int nc) { return nc <= 2 ? 4 : 2; }

// NC: 8-element chunks per lane (D <= 256 NC).  Lanes past the row's last
// chunk hold zeros.  RPW = 2 (rows of at most 16 chunks, D <= 128): each
// half-warp takes a row, so no lane idles.
template <int NC, int RPW>
__global__ void __launch_bounds__(32 * kLmsdWarps, fwd_blocks_per_sm(NC))
    hstu_lmsd_fwd_kernel(FwdArgs a) {
  static_assert(RPW == 1 || (RPW == 2 && NC == 1), "two rows per warp only for one chunk");
  const int lane = RPW == 2 ? (threadIdx.x & 15) : (threadIdx.x & 31);  // lane within the row
  const int nch = a.d / 8;
  const int S = 1 + a.concat_u + a.concat_x;
  const bool drop = a.p > 0.f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kLmsdWarps * RPW;
  int64_t base = (static_cast<int64_t>(blockIdx.x) * kLmsdWarps + (threadIdx.x >> 5)) * RPW;
  int64_t row = base + (RPW == 2 ? (threadIdx.x & 31) >> 4 : 0);
  auto load = [&](int64_t r, uint4 (&xo)[NC], uint4 (&uo)[NC]) {
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int ch = lane + 32 * c;
      xo[c] = uo[c] = make_uint4(0u, 0u, 0u, 0u);
      if (r < a.n && ch < nch) {
        xo[c] = ld16(a.x + r * a.xs, ch);
        uo[c] = ld16(a.u + r * a.us, ch);
      }
    }
  };
  uint4 xv[NC], uv[NC];
  load(row, xv, uv);
  for (; base < a.n; base += stride, row += stride) {
    const bool live = row < a.n;  // (a half-warp's second row can be past the end)
    uint4 xn[NC], un[NC];
    load(row + stride, xn, un);  // the warp's next row, in flight during this one
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      float f[8];
      unpack8(xv[c], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) s += f[i];
    }
    const float mean = row_sum<RPW>(s) / a.d;
    float v = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      if (lane + 32 * c >= nch) continue;
      float f[8];
      unpack8(xv[c], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) v += (f[i] - mean) * (f[i] - mean);
    }
    const float rstd = rsqrtf(row_sum<RPW>(v) / a.d + a.eps);
    if (!live) continue;
    if (lane == 0) { a.mean[row] = mean; a.rstd[row] = rstd; }
    uint4* yrow = reinterpret_cast<uint4*>(a.y + row * static_cast<int64_t>(S) * a.d);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int ch = lane + 32 * c;
      if (ch >= nch) continue;
      // without dropout every draw is 0 and thr_hi 0: everything is kept
      Philox4 r0{}, r1{}, r2{};
      if (drop) {
        const uint64_t e0 = static_cast<uint64_t>(row) * a.d + 8 * ch;
        r0 = draw8(e0, 0u, a.keys);
        if (a.concat_x) r1 = draw8(e0, 1u, a.keys);
        if (a.concat_u) r2 = draw8(e0, 2u, a.keys);
      }
      const float sc = drop ? a.scale : 1.f;
      const uint4 wv = ld16(a.w, ch), bv = ld16(a.b, ch);
      // keep masks, two elements per word: 0xffff in each 16-bit half whose
      // draw is at least the threshold (a segment that is not written keeps
      // nothing); one SIMD compare decides two elements
      const uint32_t thr2 = (a.thr_hi >> 16) * 0x00010001u;
      uint32_t ya[4], yx[4], ym[4], k0[4], k1[4], k2[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        k0[j] = __vcmpgeu2(r0.v[j], thr2);
        k1[j] = a.concat_x ? __vcmpgeu2(r1.v[j], thr2) : 0u;
        k2[j] = a.concat_u ? __vcmpgeu2(r2.v[j], thr2) : 0u;
        const float2 x2 = bf2(word(xv[c], j)), u2 = bf2(word(uv[c], j));
        const float2 w2 = bf2(word(wv, j)), b2 = bf2(word(bv, j));
        const float xs[2] = {x2.x, x2.y}, us[2] = {u2.x, u2.y};
        const float ws[2] = {w2.x, w2.y}, bs[2] = {b2.x, b2.y};
        float oa[2], ox[2], om[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float act = a.silu ? us[h] * sigmoid(us[h]) : us[h];
          const float l = (xs[h] - mean) * rstd * ws[h] + bs[h];
          oa[h] = act * sc;
          ox[h] = xs[h] * sc;
          om[h] = l * act * sc;
        }
        // a dropped element is +0 (its 16 bits cleared)
        ya[j] = pack2(oa[0], oa[1]) & k2[j];
        yx[j] = pack2(ox[0], ox[1]) & k1[j];
        ym[j] = pack2(om[0], om[1]) & k0[j];
      }
      // mask bytes of elements 4 i .. 4 i + 3: bit k set where segment k keeps
      // it; each byte of a permuted keep word is 0xff or 0
      uint32_t mw[2];
#pragma unroll
      for (int i = 0; i < 2; ++i)
        mw[i] = (__byte_perm(k0[2 * i], k0[2 * i + 1], 0x6420u) & 0x01010101u) |
                (__byte_perm(k1[2 * i], k1[2 * i + 1], 0x6420u) & 0x02020202u) |
                (__byte_perm(k2[2 * i], k2[2 * i + 1], 0x6420u) & 0x04040404u);
      if (drop) reinterpret_cast<uint2*>(a.mask + row * a.d)[ch] = make_uint2(mw[0], mw[1]);
      int seg = 0;
      if (a.concat_u) yrow[seg++ * nch + ch] = make_uint4(ya[0], ya[1], ya[2], ya[3]);
      if (a.concat_x) yrow[seg++ * nch + ch] = make_uint4(yx[0], yx[1], yx[2], yx[3]);
      yrow[seg * nch + ch] = make_uint4(ym[0], ym[1], ym[2], ym[3]);
    }
#pragma unroll
    for (int c = 0; c < NC; ++c) { xv[c] = xn[c]; uv[c] = un[c]; }
  }
}

struct BwdArgs {
  const __nv_bfloat16* dy;
  int64_t dys;
  const __nv_bfloat16* x;
  int64_t xs;
  const __nv_bfloat16* u;
  int64_t us;
  const __nv_bfloat16* w;
  const __nv_bfloat16* b;
  const float* mean;
  const float* rstd;
  const int8_t* mask;
  int64_t n;
  int d;
  float scale;  // 1 / (1 - p), or 1
  int drop, silu, concat_u, concat_x, dweight;
  __nv_bfloat16* dx;
  int64_t dxs;
  __nv_bfloat16* du;
  int64_t dus;
  float* part;  // gridDim.x rows of [dweight partial (d) | dbias partial (d)]
};

// Shared-memory column accumulators of one warp: [dweight | dbias][NC][8][32
// lanes], so that lane l's columns 8 (l + 32 c) + i sit in its own bank.
template <int NC>
__host__ __device__ constexpr int acc_floats() { return 2 * NC * 8 * 32; }
template <int NC>
__device__ __forceinline__ int acc_slot(int which, int c, int i, int lane) {
  return ((which * NC + c) * 8 + i) * 32 + lane;
}

// Two passes over a row: the first forms the row means of dxh = dl * weight
// and dxh * xhat and adds the row's dweight / dbias terms to the warp's
// accumulators; the second reads the row again (from L1 / L2) and writes dx
// and du, which keeps registers for more warps.
template <int NC, int RPW>
__global__ void __launch_bounds__(32 * kLmsdWarps, bwd_blocks_per_sm(NC))
    hstu_lmsd_bwd_kernel(BwdArgs a) {
  static_assert(RPW == 1 || (RPW == 2 && NC == 1), "two rows per warp only for one chunk");
  extern __shared__ float acc_all[];  // [warp][acc_floats<NC>()]
  const int wl = threadIdx.x & 31, warp = threadIdx.x >> 5;   // lane in the warp
  const int lane = RPW == 2 ? (wl & 15) : wl;                  // lane within the row
  float* acc = acc_all + warp * acc_floats<NC>();
  for (int k = wl; k < acc_floats<NC>(); k += 32) acc[k] = 0.f;  // warp-private
  const int nch = a.d / 8;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kLmsdWarps * RPW;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  int64_t row = (static_cast<int64_t>(blockIdx.x) * kLmsdWarps + warp) * RPW +
                (RPW == 2 ? wl >> 4 : 0);
  for (int64_t base = row - (RPW == 2 ? wl >> 4 : 0); base < a.n; base += stride, row += stride) {
    const bool live = row < a.n;  // (a half-warp's second row can be past the end)
    const float mean = live ? __ldg(a.mean + row) : 0.f, rstd = live ? __ldg(a.rstd + row) : 0.f;
    const __nv_bfloat16* dyrow = a.dy + row * a.dys;
    uint4 xv[NC], uv[NC], dmv[NC], duv[NC], dxv[NC];
    uint64_t mv[NC];
    auto load = [&](int c) {
      const int ch = lane + 32 * c;
      xv[c] = uv[c] = dmv[c] = duv[c] = dxv[c] = zero;
      mv[c] = 0;
      if (ch >= nch || !live) return;
      xv[c] = ld16(a.x + row * a.xs, ch);
      uv[c] = ld16(a.u + row * a.us, ch);
      int seg = 0;
      if (a.concat_u) duv[c] = ld16(dyrow, seg++ * nch + ch);
      if (a.concat_x) dxv[c] = ld16(dyrow, seg++ * nch + ch);
      dmv[c] = ld16(dyrow, seg * nch + ch);
      mv[c] = a.drop ? __ldg(reinterpret_cast<const unsigned long long*>(a.mask + row * a.d) + ch)
                     : ~0ull;
    };
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int ch = lane + 32 * c;
      if (ch >= nch || !live) continue;
      load(c);
      const uint4 wv = ld16(a.w, ch);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 x2 = bf2(word(xv[c], j)), u2 = bf2(word(uv[c], j));
        const float2 d2 = bf2(word(dmv[c], j)), w2 = bf2(word(wv, j));
        const float xs[2] = {x2.x, x2.y}, us[2] = {u2.x, u2.y};
        const float ds[2] = {d2.x, d2.y}, ws[2] = {w2.x, w2.y};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int i = 2 * j + h;
          const float xh = (xs[h] - mean) * rstd;
          const float act = a.silu ? us[h] * sigmoid(us[h]) : us[h];
          const float g = ((mv[c] >> (8 * i)) & 1u) ? ds[h] * a.scale : 0.f;
          const float dl = g * act, dxh = dl * ws[h];
          s1 += dxh;
          s2 += dxh * xh;
          acc[acc_slot<NC>(0, c, i, wl)] += dl * xh;
          acc[acc_slot<NC>(1, c, i, wl)] += dl;
        }
      }
    }
    const float m1 = row_sum<RPW>(s1) / a.d, m2 = row_sum<RPW>(s2) / a.d;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int ch = lane + 32 * c;
      if (ch >= nch || !live) continue;
      load(c);  // again: from L1 / L2
      const uint4 wv = ld16(a.w, ch), bv = ld16(a.b, ch);
      uint32_t ox[4], ou[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 x2 = bf2(word(xv[c], j)), u2 = bf2(word(uv[c], j));
        const float2 d2 = bf2(word(dmv[c], j)), w2 = bf2(word(wv, j)), b2 = bf2(word(bv, j));
        const float2 yu2 = bf2(word(duv[c], j)), yx2 = bf2(word(dxv[c], j));
        const float xs[2] = {x2.x, x2.y}, us[2] = {u2.x, u2.y}, ds[2] = {d2.x, d2.y};
        const float ws[2] = {w2.x, w2.y}, bs[2] = {b2.x, b2.y};
        const float yus[2] = {yu2.x, yu2.y}, yxs[2] = {yx2.x, yx2.y};
        float rx[2], ru[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t mb = static_cast<uint32_t>(mv[c] >> (8 * (2 * j + h)));
          const float xh = (xs[h] - mean) * rstd;
          const float l = xh * ws[h] + bs[h];
          const float sg = a.silu ? sigmoid(us[h]) : 0.f;
          const float act = a.silu ? us[h] * sg : us[h];
          const float g = (mb & 1u) ? ds[h] * a.scale : 0.f;
          const float dxh = g * act * ws[h];
          const float da = g * l + ((mb & 4u) ? yus[h] * a.scale : 0.f);
          rx[h] = rstd * (dxh - m1 - xh * m2) + ((mb & 2u) ? yxs[h] * a.scale : 0.f);
          ru[h] = a.silu ? da * sg * (1.f + us[h] * (1.f - sg)) : da;
        }
        ox[j] = pack2(rx[0], rx[1]);
        ou[j] = pack2(ru[0], ru[1]);
      }
      reinterpret_cast<uint4*>(a.dx + row * a.dxs)[ch] = make_uint4(ox[0], ox[1], ox[2], ox[3]);
      reinterpret_cast<uint4*>(a.du + row * a.dus)[ch] = make_uint4(ou[0], ou[1], ou[2], ou[3]);
    }
  }
  // column partials: the block's warps in a fixed order, one partial row per block
  __syncthreads();
  for (int col = threadIdx.x; col < 2 * a.d; col += blockDim.x) {
    const int which = col >= a.d ? 1 : 0, cc = col - which * a.d, ch = cc >> 3;
    const int slot = acc_slot<NC>(which, ch >> 5, cc & 7, ch & 31);
    float t = 0.f;
    for (int k = 0; k < kLmsdWarps; ++k) {
      t += acc_all[k * acc_floats<NC>() + slot];
      if (RPW == 2) t += acc_all[k * acc_floats<NC>() + slot + 16];  // the other half-warp
    }
    a.part[static_cast<int64_t>(blockIdx.x) * 2 * a.d + col] = t;
  }
}

// Column sums of the per-block partials, one warp per column: lane l adds
// partials l, l + 32, ... in order, then a fixed shuffle tree adds the lanes
// (the same order on every run): dweight, dbias.
__global__ void hstu_lmsd_colsum_kernel(const float* part, int blocks, int d, int dweight,
                                        __nv_bfloat16* dw, __nv_bfloat16* db) {
  const int col = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (col >= 2 * d) return;
  float t = 0.f;
  for (int k = lane; k < blocks; k += 32) t += part[static_cast<int64_t>(k) * 2 * d + col];
  t = warp_sum(t);
  if (lane != 0) return;
  if (col < d) {
    if (dweight) dw[col] = __float2bfloat16_rn(t);
  } else {
    db[col - d] = __float2bfloat16_rn(t);
  }
}

// Persistent grids: `per_sm` blocks of 8 rows per SM, the blocks that fit.
int lmsd_grid(int64_t n, int per_sm, int rpw) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t rows = static_cast<int64_t>(kLmsdWarps) * rpw;  // rows in flight per block
  const int64_t want = (n + rows - 1) / rows;
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  return static_cast<int>(want < cap ? want : cap);
}
int chunks_per_lane(int32_t d) { return (d / 8 + 31) / 32; }

// Rows of at most 16 chunks (D <= 128) go two to a warp, a half-warp each.
int rows_per_warp(int32_t d) { return d / 8 <= 16 ? 2 : 1; }

// Bytes of the backward's shared-memory column accumulators.
size_t bwd_smem(int nc) { return static_cast<size_t>(kLmsdWarps) * 2 * nc * 8 * 32 * sizeof(float); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

hstu_lmsd_status_t check_rows(const void* p, int64_t stride, int64_t n, int64_t width) {
  if (n > 0 && p == nullptr) return HSTU_LMSD_ERR_INVALID_ARG;
  if (!aligned16(p)) return HSTU_LMSD_ERR_MISALIGNED;
  if (stride < width) return HSTU_LMSD_ERR_INVALID_ARG;
  if ((stride * 2) % 16 != 0) return HSTU_LMSD_ERR_MISALIGNED;
  return HSTU_LMSD_OK;
}

hstu_lmsd_status_t check_common(int64_t n, int32_t d, float p) {
  if (n < 0 || d < 8 || d >= 1024 || d % 8 != 0) return HSTU_LMSD_ERR_UNSUPPORTED;
  if (n * static_cast<int64_t>(d) > (int64_t(1) << 31)) return HSTU_LMSD_ERR_UNSUPPORTED;
  if (!std::isfinite(p) || p < 0.f || p >= 1.f) return HSTU_LMSD_ERR_INVALID_ARG;
  return HSTU_LMSD_OK;
}

}  // namespace

extern "C" {

hstu_lmsd_status_t hstu_lmsd_fwd(const void* x, int64_t x_stride, const void* u, int64_t u_stride,
                                 const void* weight, const void* bias, int64_t n, int32_t d,
                                 float eps, float dropout_ratio, int32_t apply_u_silu,
                                 int32_t concat_u, int32_t concat_x, int64_t seed, void* y,
                                 float* mean, float* rstd, int8_t* mask, cudaStream_t stream) {
  hstu_lmsd_status_t s = check_common(n, d, dropout_ratio);
  if (s != HSTU_LMSD_OK) return s;
  if (!std::isfinite(eps) || eps <= 0.f) return HSTU_LMSD_ERR_INVALID_ARG;
  const int S = 1 + (concat_u != 0) + (concat_x != 0);
  if ((s = check_rows(x, x_stride, n, d)) != HSTU_LMSD_OK) return s;
  if ((s = check_rows(u, u_stride, n, d)) != HSTU_LMSD_OK) return s;
  if ((s = check_rows(y, int64_t(S) * d, n, int64_t(S) * d)) != HSTU_LMSD_OK) return s;
  if ((s = check_rows(weight, d, 1, d)) != HSTU_LMSD_OK) return s;
  if ((s = check_rows(bias, d, 1, d)) != HSTU_LMSD_OK) return s;
  if (n > 0 && (mean == nullptr || rstd == nullptr)) return HSTU_LMSD_ERR_INVALID_ARG;
  const bool drop = dropout_ratio > 0.f;
  if (drop && n > 0 && mask == nullptr) return HSTU_LMSD_ERR_INVALID_ARG;
  if (drop && !aligned16(mask)) return HSTU_LMSD_ERR_MISALIGNED;
  if (n == 0) return HSTU_LMSD_OK;
  FwdArgs a{};
  a.x = static_cast<const __nv_bfloat16*>(x); a.xs = x_stride;
  a.u = static_cast<const __nv_bfloat16*>(u); a.us = u_stride;
  a.w = static_cast<const __nv_bfloat16*>(weight); a.b = static_cast<const __nv_bfloat16*>(bias);
  a.n = n; a.d = d; a.eps = eps; a.p = dropout_ratio;
  a.thr_hi = drop ? static_cast<uint32_t>(std::floor(static_cast<double>(dropout_ratio) * 65536.0))
                       << 16
                 : 0u;
  a.scale = drop ? 1.f / (1.f - dropout_ratio) : 1.f;
  a.silu = apply_u_silu != 0; a.concat_u = concat_u != 0; a.concat_x = concat_x != 0;
  a.keys = philox_keys(static_cast<uint64_t>(seed));
  a.y = static_cast<__nv_bfloat16*>(y); a.mean = mean; a.rstd = rstd; a.mask = mask;
  const int nc = chunks_per_lane(d);
  const int rpw = rows_per_warp(d);
  auto kern = rpw == 2 ? hstu_lmsd_fwd_kernel<1, 2>
            : nc == 1 ? hstu_lmsd_fwd_kernel<1, 1> : nc == 2 ? hstu_lmsd_fwd_kernel<2, 1>
            : nc == 3 ? hstu_lmsd_fwd_kernel<3, 1> : hstu_lmsd_fwd_kernel<4, 1>;
  kern<<<lmsd_grid(n, fwd_blocks_per_sm(nc), rpw), 32 * kLmsdWarps, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? HSTU_LMSD_OK : HSTU_LMSD_ERR_CUDA;
}

size_t hstu_lmsd_bwd_workspace_size(int64_t n, int32_t d) {
  if (n < 0 || d < 8 || d >= 1024 || d % 8 != 0) return 0;
  return static_cast<size_t>(lmsd_grid(n < 1 ? 1 : n, bwd_blocks_per_sm(chunks_per_lane(d)),
                                      rows_per_warp(d))) * 2 *
         d * sizeof(float);
}

hstu_lmsd_status_t hstu_lmsd_bwd(const void* dy, int64_t dy_stride, const void* x,
                                 int64_t x_stride, const void* u, int64_t u_stride,
                                 const void* weight, const void* bias, const float* mean,
                                 const float* rstd, const int8_t* mask, int64_t n, int32_t d,
                                 float dropout_ratio, int32_t apply_u_silu, int32_t concat_u,
                                 int32_t concat_x, int32_t compute_dweight, void* dx,
                                 int64_t dx_stride, void* du, int64_t du_stride, void* dweight,
                                 void* dbias, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
  hstu_lmsd_status_t s = check_common(n, d, dropout_ratio);
  if (s != HSTU_LMSD_OK) return s;
  const int S = 1 + (concat_u != 0) + (concat_x != 0);
  if ((s = check_rows(dy, dy_stride, n, int64_t(S) * d)) != HSTU_LMSD_OK) return s;
  if ((s = check_rows(x, x_stride, n, d)) != HSTU_LMSD_OK) return s;
  if ((s = check_rows(u, u_stride, n, d)) != HSTU_LMSD_OK) return s;
  if ((s = check_rows(dx, dx_stride, n, d)) != HSTU_LMSD_OK) return s;
  if ((s = check_rows(du, du_stride, n, d)) != HSTU_LMSD_OK) return s;
  if ((s = check_rows(weight, d, 1, d)) != HSTU_LMSD_OK) return s;
  if ((s = check_rows(bias, d, 1, d)) != HSTU_LMSD_OK) return s;
  if (compute_dweight && (s = check_rows(dweight, d, 1, d)) != HSTU_LMSD_OK) return s;
  if ((s = check_rows(dbias, d, 1, d)) != HSTU_LMSD_OK) return s;
  if (n > 0 && (mean == nullptr || rstd == nullptr)) return HSTU_LMSD_ERR_INVALID_ARG;
  const bool drop = dropout_ratio > 0.f;
  if (drop && n > 0 && mask == nullptr) return HSTU_LMSD_ERR_INVALID_ARG;
  if (drop && !aligned16(mask)) return HSTU_LMSD_ERR_MISALIGNED;
  const size_t need = hstu_lmsd_bwd_workspace_size(n, d);
  if (workspace == nullptr || workspace_bytes < need) return HSTU_LMSD_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return HSTU_LMSD_ERR_MISALIGNED;
  const int nc = chunks_per_lane(d);
  const int rpw = rows_per_warp(d);
  const int grid = n > 0 ? lmsd_grid(n, bwd_blocks_per_sm(nc), rpw) : 1;
  const size_t smem = bwd_smem(nc);
  auto kern = rpw == 2 ? hstu_lmsd_bwd_kernel<1, 2>
            : nc == 1 ? hstu_lmsd_bwd_kernel<1, 1> : nc == 2 ? hstu_lmsd_bwd_kernel<2, 1>
            : nc == 3 ? hstu_lmsd_bwd_kernel<3, 1> : hstu_lmsd_bwd_kernel<4, 1>;
  static bool attr[6] = {false, false, false, false, false, false};
  const int ki = rpw == 2 ? 5 : nc;
  if (!attr[ki]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return HSTU_LMSD_ERR_CUDA;
    attr[ki] = true;
  }
  BwdArgs a{};
  a.dy = static_cast<const __nv_bfloat16*>(dy); a.dys = dy_stride;
  a.x = static_cast<const __nv_bfloat16*>(x); a.xs = x_stride;
  a.u = static_cast<const __nv_bfloat16*>(u); a.us = u_stride;
  a.w = static_cast<const __nv_bfloat16*>(weight); a.b = static_cast<const __nv_bfloat16*>(bias);
  a.mean = mean; a.rstd = rstd; a.mask = mask; a.n = n; a.d = d;
  a.scale = drop ? 1.f / (1.f - dropout_ratio) : 1.f;
  a.drop = drop; a.silu = apply_u_silu != 0; a.concat_u = concat_u != 0;
  a.concat_x = concat_x != 0; a.dweight = compute_dweight != 0;
  a.dx = static_cast<__nv_bfloat16*>(dx); a.dxs = dx_stride;
  a.du = static_cast<__nv_bfloat16*>(du); a.dus = du_stride;
  a.part = static_cast<float*>(workspace);
  if (n > 0) kern<<<grid, 32 * kLmsdWarps, smem, stream>>>(a);
  else cudaMemsetAsync(workspace, 0, need, stream);
  hstu_lmsd_colsum_kernel<<<(2 * d * 32 + 255) / 256, 256, 0, stream>>>(
      a.part, grid, d, a.dweight, static_cast<__nv_bfloat16*>(dweight),
      static_cast<__nv_bfloat16*>(dbias));
  return cudaGetLastError() == cudaSuccess ? HSTU_LMSD_OK : HSTU_LMSD_ERR_CUDA;
}

}  // extern "C"
