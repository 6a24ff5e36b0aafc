// HSTU LayerNorm-Multiply-SiLU-Dropout (page "HSTU LayerNorm-Multiply-SiLU-
// Dropout (LMSD)", Overview): per row of x (N, D), bf16,
//   xhat = (x - mean) rstd,  l = xhat * weight + bias,  a = SiLU(u) or u,
//   y = [dropout(a) if concat_u, dropout(x) if concat_x, dropout(l * a)],
// inverted dropout with one int8 mask per element (bit 0 main, bit 1 x
// segment, bit 2 u segment; set = kept), row mean and rstd saved for the
// backward.  The op is HBM-bound: one warp per row, 16-byte loads and stores
// (8 bf16 per lane per chunk), fp32 arithmetic, no shared memory in the
// forward.  The backward forms dx and du per row the same way; dweight and
// dbias are column sums over rows, reduced deterministically: each warp sums
// its rows in registers, each block sums its warps in a fixed order into a
// partial row of the workspace, and a second kernel sums the partials in
// block order.
//
// Dropout decisions: Philox4x32-10 (Salmon et al., SC 2011), implemented
// here from its definition; element e = row * D + col of segment k uses word
// e % 4 of Philox(counter (e / 4 low, high, k, 0), key (seed low, high)) and
// is kept iff the word >= floor(p 2^32).
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

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2,
                                                 uint32_t c3, uint32_t k0, uint32_t k1) {
  constexpr uint32_t kM0 = 0xD2511F53u, kM1 = 0xCD9E8D57u;   // round multipliers
  constexpr uint32_t kW0 = 0x9E3779B9u, kW1 = 0xBB67AE85u;   // key increments
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t hi0 = __umulhi(kM0, c0), lo0 = kM0 * c0;
    const uint32_t hi1 = __umulhi(kM1, c2), lo1 = kM1 * c2;
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    k0 += kW0;
    k1 += kW1;
  }
  return Philox4{{c0, c1, c2, c3}};
}

// Keep bits of 8 consecutive elements starting at flat index e0 (a multiple
// of 8) of segment k.
__device__ __forceinline__ uint32_t keep8(uint64_t e0, uint32_t k, uint64_t seed, uint32_t thr) {
  const uint64_t g = e0 >> 2;
  const Philox4 a = philox4x32_10(static_cast<uint32_t>(g), static_cast<uint32_t>(g >> 32), k, 0u,
                                  static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  const Philox4 b = philox4x32_10(static_cast<uint32_t>(g + 1),
                                  static_cast<uint32_t>((g + 1) >> 32), k, 0u,
                                  static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32));
  uint32_t bits = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    bits |= (a.v[i] >= thr ? 1u : 0u) << i;
    bits |= (b.v[i] >= thr ? 1u : 0u) << (4 + i);
  }
  return bits;
}

__device__ __forceinline__ void unpack8(const uint4& w, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 w;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return w;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float silu(float u) { return u / (1.f + __expf(-u)); }
__device__ __forceinline__ float silu_grad(float u) {
  const float s = 1.f / (1.f + __expf(-u));
  return s * (1.f + u * (1.f - s));
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
  uint32_t thr;     // keep iff word >= thr
  float scale;      // 1 / (1 - p)
  int silu, concat_u, concat_x;
  uint64_t seed;
  __nv_bfloat16* y;
  float* mean;
  float* rstd;
  int8_t* mask;
};

// NC: 8-element chunks per lane (D <= 256 NC, so a row's x stays in registers).
template <int NC>
__global__ void __launch_bounds__(32 * kLmsdWarps) hstu_lmsd_fwd_kernel(FwdArgs a) {
  const int lane = threadIdx.x & 31;
  const int nch = a.d / 8;
  const int S = 1 + a.concat_u + a.concat_x;
  const bool drop = a.p > 0.f;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kLmsdWarps;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kLmsdWarps + (threadIdx.x >> 5);
       row < a.n; row += stride) {
    float x[NC][8];
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int ch = lane + 32 * c;
      if (ch < nch) {
        unpack8(reinterpret_cast<const uint4*>(a.x + row * a.xs)[ch], x[c]);
#pragma unroll
        for (int i = 0; i < 8; ++i) s += x[c][i];
      }
    }
    const float mean = warp_sum(s) / a.d;
    float v = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c)
      if (lane + 32 * c < nch) {
#pragma unroll
        for (int i = 0; i < 8; ++i) v += (x[c][i] - mean) * (x[c][i] - mean);
      }
    const float rstd = rsqrtf(warp_sum(v) / a.d + a.eps);
    if (lane == 0) { a.mean[row] = mean; a.rstd[row] = rstd; }
    uint4* yrow = reinterpret_cast<uint4*>(a.y + row * static_cast<int64_t>(S) * a.d);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int ch = lane + 32 * c;
      if (ch >= nch) continue;
      const uint64_t e0 = static_cast<uint64_t>(row) * a.d + 8 * ch;
      uint32_t k0 = 0xffu, k1 = 0xffu, k2 = 0xffu;
      if (drop) {
        k0 = keep8(e0, 0u, a.seed, a.thr);
        if (a.concat_x) k1 = keep8(e0, 1u, a.seed, a.thr);
        if (a.concat_u) k2 = keep8(e0, 2u, a.seed, a.thr);
        uint64_t m = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint64_t byte = ((k0 >> i) & 1u) | (a.concat_x ? ((k1 >> i) & 1u) << 1 : 0u) |
                                (a.concat_u ? ((k2 >> i) & 1u) << 2 : 0u);
          m |= byte << (8 * i);
        }
        reinterpret_cast<uint64_t*>(a.mask + row * a.d)[ch] = m;
      }
      const float sc = drop ? a.scale : 1.f;
      float u[8], w[8], bb[8], act[8], out[8];
      unpack8(reinterpret_cast<const uint4*>(a.u + row * a.us)[ch], u);
      unpack8(reinterpret_cast<const uint4*>(a.w)[ch], w);
      unpack8(reinterpret_cast<const uint4*>(a.b)[ch], bb);
#pragma unroll
      for (int i = 0; i < 8; ++i) act[i] = a.silu ? silu(u[i]) : u[i];
      int seg = 0;
      if (a.concat_u) {
#pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = ((k2 >> i) & 1u) ? act[i] * sc : 0.f;
        yrow[seg * nch + ch] = pack8(out);
        ++seg;
      }
      if (a.concat_x) {
#pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = ((k1 >> i) & 1u) ? x[c][i] * sc : 0.f;
        yrow[seg * nch + ch] = pack8(out);
        ++seg;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float l = (x[c][i] - mean) * rstd * w[i] + bb[i];
        out[i] = ((k0 >> i) & 1u) ? l * act[i] * sc : 0.f;
      }
      yrow[seg * nch + ch] = pack8(out);
    }
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

// One row term of the backward at element i of a chunk: returns dl (the
// gradient of l), and the pieces of dx and du.
struct BwdTerms {
  float xh, dl, da, dxh, dx_extra;
};

__device__ __forceinline__ BwdTerms bwd_terms(const BwdArgs& a, float x, float u, float w, float b,
                                              float mean, float rstd, float dm, float dyu,
                                              float dyx, uint32_t mb) {
  BwdTerms t;
  const float s0 = (mb & 1u) ? a.scale : 0.f;
  const float sx = (mb & 2u) ? a.scale : 0.f;
  const float su = (mb & 4u) ? a.scale : 0.f;
  t.xh = (x - mean) * rstd;
  const float l = t.xh * w + b;
  const float act = a.silu ? silu(u) : u;
  const float g = dm * s0;  // gradient of l * a
  t.dl = g * act;
  t.da = g * l + (a.concat_u ? dyu * su : 0.f);
  t.dxh = t.dl * w;
  t.dx_extra = a.concat_x ? dyx * sx : 0.f;
  return t;
}

// Loads chunk ch of a row's inputs: x, u, the dy segments, the mask bytes.
__device__ __forceinline__ void bwd_load(const BwdArgs& a, int64_t row, int ch, int nch,
                                         float (&x)[8], float (&u)[8], float (&dm)[8],
                                         float (&dyu)[8], float (&dyx)[8], uint64_t& m) {
  const uint4* dyrow = reinterpret_cast<const uint4*>(a.dy + row * a.dys);
  unpack8(reinterpret_cast<const uint4*>(a.x + row * a.xs)[ch], x);
  unpack8(reinterpret_cast<const uint4*>(a.u + row * a.us)[ch], u);
  int seg = 0;
  if (a.concat_u) unpack8(dyrow[seg++ * nch + ch], dyu);
  if (a.concat_x) unpack8(dyrow[seg++ * nch + ch], dyx);
  unpack8(dyrow[seg * nch + ch], dm);
  m = a.drop ? reinterpret_cast<const uint64_t*>(a.mask + row * a.d)[ch] : ~0ull;
}

// Two passes per row: the first forms the row means of dxh and dxh xhat and
// the dweight / dbias contributions, the second reloads the row (from L1 /
// L2) and writes dx and du, so that only the column accumulators stay in
// registers across rows.
template <int NC>
__global__ void __launch_bounds__(32 * kLmsdWarps) hstu_lmsd_bwd_kernel(BwdArgs a) {
  extern __shared__ float red[];  // [warp][2 d]
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nch = a.d / 8;
  float gw[NC][8], gb[NC][8];
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int i = 0; i < 8; ++i) { gw[c][i] = 0.f; gb[c][i] = 0.f; }
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kLmsdWarps;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kLmsdWarps + warp; row < a.n;
       row += stride) {
    const float mean = a.mean[row], rstd = a.rstd[row];
    float s1 = 0.f, s2 = 0.f;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int ch = lane + 32 * c;
      if (ch >= nch) continue;
      float x[8], u[8], dm[8], dyu[8], dyx[8], w[8], b[8];
      uint64_t m;
      bwd_load(a, row, ch, nch, x, u, dm, dyu, dyx, m);
      unpack8(reinterpret_cast<const uint4*>(a.w)[ch], w);
      unpack8(reinterpret_cast<const uint4*>(a.b)[ch], b);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const BwdTerms t = bwd_terms(a, x[i], u[i], w[i], b[i], mean, rstd, dm[i], dyu[i], dyx[i],
                                     static_cast<uint32_t>(m >> (8 * i)) & 0xffu);
        gw[c][i] += t.dl * t.xh;
        gb[c][i] += t.dl;
        s1 += t.dxh;
        s2 += t.dxh * t.xh;
      }
    }
    const float m1 = warp_sum(s1) / a.d, m2 = warp_sum(s2) / a.d;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int ch = lane + 32 * c;
      if (ch >= nch) continue;
      float x[8], u[8], dm[8], dyu[8], dyx[8], w[8], b[8], ox[8], ou[8];
      uint64_t m;
      bwd_load(a, row, ch, nch, x, u, dm, dyu, dyx, m);
      unpack8(reinterpret_cast<const uint4*>(a.w)[ch], w);
      unpack8(reinterpret_cast<const uint4*>(a.b)[ch], b);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const BwdTerms t = bwd_terms(a, x[i], u[i], w[i], b[i], mean, rstd, dm[i], dyu[i], dyx[i],
                                     static_cast<uint32_t>(m >> (8 * i)) & 0xffu);
        ox[i] = rstd * (t.dxh - m1 - t.xh * m2) + t.dx_extra;
        ou[i] = a.silu ? t.da * silu_grad(u[i]) : t.da;
      }
      reinterpret_cast<uint4*>(a.dx + row * a.dxs)[ch] = pack8(ox);
      reinterpret_cast<uint4*>(a.du + row * a.dus)[ch] = pack8(ou);
    }
  }
  // column partials: warps in a fixed order, then one partial row per block
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int ch = lane + 32 * c;
    if (ch >= nch) continue;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      red[warp * 2 * a.d + 8 * ch + i] = gw[c][i];
      red[warp * 2 * a.d + a.d + 8 * ch + i] = gb[c][i];
    }
  }
  __syncthreads();
  for (int col = threadIdx.x; col < 2 * a.d; col += blockDim.x) {
    float t = 0.f;
    for (int k = 0; k < kLmsdWarps; ++k) t += red[k * 2 * a.d + col];
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

// Persistent grids: `per_sm` blocks of 8 rows per SM (the backward keeps it
// small, each block adds a row of column partials).
int lmsd_grid(int64_t n, int per_sm) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (n + kLmsdWarps - 1) / kLmsdWarps;
  const int64_t cap = static_cast<int64_t>(sms) * per_sm;
  return static_cast<int>(want < cap ? want : cap);
}
constexpr int kFwdBlocksPerSm = 8, kBwdBlocksPerSm = 2;

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
  const double t = std::floor(static_cast<double>(dropout_ratio) * 4294967296.0);
  a.thr = static_cast<uint32_t>(t > 4294967295.0 ? 4294967295.0 : t);
  a.scale = drop ? 1.f / (1.f - dropout_ratio) : 1.f;
  a.silu = apply_u_silu != 0; a.concat_u = concat_u != 0; a.concat_x = concat_x != 0;
  a.seed = static_cast<uint64_t>(seed);
  a.y = static_cast<__nv_bfloat16*>(y); a.mean = mean; a.rstd = rstd; a.mask = mask;
  const int nc = (d / 8 + 31) / 32;
  auto kern = nc == 1 ? hstu_lmsd_fwd_kernel<1> : nc == 2 ? hstu_lmsd_fwd_kernel<2>
            : nc == 3 ? hstu_lmsd_fwd_kernel<3> : hstu_lmsd_fwd_kernel<4>;
  kern<<<lmsd_grid(n, kFwdBlocksPerSm), 32 * kLmsdWarps, 0, stream>>>(a);
  return cudaGetLastError() == cudaSuccess ? HSTU_LMSD_OK : HSTU_LMSD_ERR_CUDA;
}

size_t hstu_lmsd_bwd_workspace_size(int64_t n, int32_t d) {
  if (n < 0 || d < 8 || d >= 1024 || d % 8 != 0) return 0;
  return static_cast<size_t>(lmsd_grid(n < 1 ? 1 : n, kBwdBlocksPerSm)) * 2 * d * sizeof(float);
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
  const int grid = n > 0 ? lmsd_grid(n, kBwdBlocksPerSm) : 1;
  const size_t smem = static_cast<size_t>(kLmsdWarps) * 2 * d * sizeof(float);
  const int nc = (d / 8 + 31) / 32;
  auto kern = nc == 1 ? hstu_lmsd_bwd_kernel<1> : nc == 2 ? hstu_lmsd_bwd_kernel<2>
            : nc == 3 ? hstu_lmsd_bwd_kernel<3> : hstu_lmsd_bwd_kernel<4>;
  static bool attr[5] = {false, false, false, false, false};
  if (!attr[nc]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kLmsdWarps * 2 * 1024 * sizeof(float))) !=
        cudaSuccess)
      return HSTU_LMSD_ERR_CUDA;
    attr[nc] = true;
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
