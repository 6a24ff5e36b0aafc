// Shared definitions of the HSTU attention kernels: workspace layout, kernel
// parameter blocks, bounded barrier waits, element conversion.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "ptx.cuh"

namespace hstu {

// ---------------------------------------------------------------- workspace
// Bytes [0, 256): header of int32 words.  Then list A (query-tile work units)
// and, for the backward, list B (key-tile work units), int4 each.  A plan
// (one schedule shared by forward and backward calls) adds list F, the
// forward's query tiles, and records the sizes it was made for.
enum HeaderWord : int {
  kHdrStatus = 0,     // 0 = ok, else an hstu_status_t recorded on the device
  kHdrUnitsA = 1,     // number of units in list A
  kHdrUnitsB = 2,     // number of units in list B
  kHdrWhere = 3,      // which wait gave up (role * 256 + barrier id), for debugging
  kHdrOverflow = 4,   // units dropped because the metadata exceeded the totals (list A)
  kHdrOverflowB = 5,  // same, list B
  kHdrNextA = 6,      // next unclaimed unit of list A (atomic counter)
  kHdrNextB = 7,      // next unclaimed unit of list B
  kHdrUnitsF = 8,     // plan: number of units in list F
  kHdrNextF = 9,      // plan: next unclaimed unit of list F
  kHdrOverflowF = 10, // plan: units dropped from list F
  kHdrDone = 11,      // plan: CTAs of the running kernel that have finished
  kHdrEpoch = 12,     // backward: calls completed since the readiness counts were zeroed
  kHdrNextB2 = 13,    // next unclaimed unit of list B's second half (D = 256: the dK pass)
  kHdrKey = 16,       // plan: kPlanKeyInts words (16-byte aligned), the sizes the plan was made for
};
constexpr int kPlanKeyInts = 10;
static_assert(kPlanKeyInts <= 12, "the plan key is read as three int4");
constexpr int kHeaderBytes = 256;
constexpr int kStatusTimeout = 5;     // == HSTU_ERR_DEVICE_TIMEOUT
constexpr int kStatusBadMeta = 1;     // == HSTU_ERR_INVALID_ARG

// Query tiles are always 128 rows (the tcgen05 M of every kernel).
constexpr int kBM = 128;

// Work unit: x = sequence, y = tile index inside the sequence,
// z = head (times the D split for list B, plus the split index),
// w = number of inner tiles the unit iterates over (0 = write zeros).
struct Unit {
  int b, tile, hz, n;
};

__device__ __forceinline__ Unit load_unit(const int4* units, int u) {
  int4 v = __ldg(units + u);
  return Unit{v.x, v.y, v.z, v.w};
}

// ---------------------------------------------------------------- waits
// Every barrier wait is bounded: after `timeout_ns` the waiting thread records
// HSTU_ERR_DEVICE_TIMEOUT in the workspace, raises the block's abort flag and
// returns false; every other wait in the block then returns false at once,
// so the block drains its own copies and exits.  Nothing traps or spins
// forever.
struct WaitCtl {
  int* status;                 // workspace header (global)
  volatile int* abort_flag;    // shared
  uint64_t timeout_ns;
};

// The slow path takes its controls by value so that nothing is spilled to
// the stack (local memory misses a nearly cache-less L1 when shared memory
// takes the whole carve-out).
static __device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, int* status,
                                              volatile int* abort_flag, uint64_t timeout_ns,
                                              int where) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        atomicCAS(status + kHdrStatus, 0, kStatusTimeout);
        atomicExch(status + kHdrWhere, where);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                         int where) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, c.status, c.abort_flag, c.timeout_ns, where);
}

// Bounded wait until a global counter that other CTAs raise has grown by
// `target` past `start` (acquire at GPU scope; modulo 2^32, so a count may
// wrap), with the same give-up rules as a barrier wait.  On success the
// counted data may be read by TMA.
static __device__ __noinline__ bool wait_count(const int* cnt, uint32_t start, uint32_t target,
                                               int* status, volatile int* abort_flag,
                                               uint64_t timeout_ns, int where) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (static_cast<uint32_t>(ld_acquire_gpu(cnt)) - start >= target) {
      fence_proxy_async_global();
      return true;
    }
    if ((it & 15u) == 0u) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        atomicCAS(status + kHdrStatus, 0, kStatusTimeout);
        atomicExch(status + kHdrWhere, where);
        return false;
      }
    }
    __nanosleep(64);
  }
}

// Work-unit record plus the packed-sequence offsets and lengths it needs,
// loaded together so a role can prefetch the next unit while it works on
// the current one (the loads are independent global reads).
// `ds` is filled in by kernels that need it (dK/dV: the unit's first stored
// dS block, -1 for none).
struct UnitInfo {
  int b, tile, hz, n;
  int q0, Lq, k0, Lk;
  int ds;
};

__device__ __forceinline__ UnitInfo load_unit_info(const int4* units, int u, int n_units) {
  UnitInfo r{0, 0, 0, -1, 0, 0, 0, 0, -1};  // n = -1: no more units
  if (u < n_units) {
    const int4 v = units[2 * u], w = units[2 * u + 1];
    r.b = v.x; r.tile = v.y; r.hz = v.z; r.n = v.w;
    r.q0 = w.x; r.Lq = w.y; r.k0 = w.z; r.Lk = w.w;
  }
  return r;
}

// Warp-uniform wait for the four row warps: lane 0 polls with the bounded
// wait and broadcasts the outcome, so a give-up never splits a warp in front
// of a .sync.aligned tcgen05 instruction.  On success the other lanes then
// observe the (already completed) phase themselves, which gives each of them
// the barrier's acquire ordering.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                              int where) {
  bool ok = true;
  if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, c, where);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (ok) {
    for (uint32_t it = 0; it < (1u << 20) && !mbar_try_wait(bar, parity); ++it) {
    }
  }
  return ok;
}

// ---------------------------------------------------------------- dynamic units
// The producer thread claims units from the work list with an atomic counter
// (so a CTA that finishes early takes the next unit, longest first) and hands
// each one to the MMA thread and the row warps through a small ring in
// shared memory.  An entry with n = -1 ends the stream.
constexpr int kUnitRing = 4;

struct UnitQueue {
  UnitInfo* ring;       // kUnitRing entries in shared memory
  uint32_t full, empty; // first barrier of each kUnitRing-long barrier array
};

// Producer: publish unit k (waits until consumers released the slot's last use).
__device__ __forceinline__ bool unit_push(const UnitQueue& q, uint32_t k, const UnitInfo& u,
                                          const WaitCtl& wc) {
  const uint32_t s = k % kUnitRing;
  if (!wait_bar(q.empty + 8 * s, ((k / kUnitRing) & 1) ^ 1, wc, 0x00a)) return false;
  q.ring[s] = u;
  mbar_arrive(q.full + 8 * s);
  return true;
}

// Single consumer thread (the MMA issuer).
__device__ __forceinline__ bool unit_pop(const UnitQueue& q, uint32_t k, UnitInfo& u,
                                         const WaitCtl& wc) {
  const uint32_t s = k % kUnitRing;
  if (!wait_bar(q.full + 8 * s, (k / kUnitRing) & 1, wc, 0x10a)) return false;
  u = q.ring[s];
  mbar_arrive(q.empty + 8 * s);
  return true;
}

// Whole row warp (warp-uniform); lane 0 releases the slot for the warp.
__device__ __forceinline__ bool unit_pop_warp(const UnitQueue& q, uint32_t k, UnitInfo& u,
                                              const WaitCtl& wc) {
  const uint32_t s = k % kUnitRing;
  if (!wait_bar_warp(q.full + 8 * s, (k / kUnitRing) & 1, wc, 0x20a)) return false;
  u = q.ring[s];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(q.empty + 8 * s);
  return true;
}

// Programmatic dependent launch: wait for the grid this one depends on (its
// writes become visible), and let the next dependent grid start launching.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- conversion
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// SiLU(x) = x * sigmoid(x) = h + h * tanh(h), h = x / 2: one MUFU op.
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// sigmoid(x) = 1/2 + tanh(x/2)/2.
__device__ __forceinline__ float sigmoid_fast(float x) {
  return fmaf(0.5f, tanh_approx(0.5f * x), 0.5f);
}

// TMEM column batches of compile-time width: N in {32, 64} loads, {16, 32} stores.
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 64) tmem_ld64(taddr, r);
  else tmem_ld32(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 32) tmem_st32(taddr, r);
  else tmem_st16(taddr, r);
}

// SiLU of two scaled scores, rounded and packed: h = x/2, SiLU(x) = h + h tanh(h).
template <bool BF16>
__device__ __forceinline__ uint32_t silu_pair(uint32_t s0, uint32_t s1, float half_alpha) {
  const float h0 = __uint_as_float(s0) * half_alpha;
  const float h1 = __uint_as_float(s1) * half_alpha;
  return pack2<BF16>(fmaf(h0, tanh_approx(h0), h0), fmaf(h1, tanh_approx(h1), h1));
}

// Twice the score gradient of one element: with h = x/2 and t = tanh(h),
// SiLU'(x) = sigmoid(x) (1 + x (1 - sigmoid(x))) = (1 + t)(1 + h (1 - t)) / 2,
// so 2 dP SiLU'(x) = dP (1 + t)(1 + h (1 - t)); the 1/2 goes to the epilogue.
// Equivalently 2 SiLU'(x) = 1 + t + h (1 - t^2): three FMAs.
__device__ __forceinline__ float dsilu2(float h, float t, float dp) {
  const float a = fmaf(-t, t, 1.f);  // 1 - t^2
  const float v = fmaf(h, a, t);     // t + h (1 - t^2)
  return fmaf(dp, v, dp);            // dp (1 + v)
}

// dS pair (doubled) from raw scores s and dP of two elements; a masked
// element enters as s = dP = 0 and leaves as exactly 0.
template <bool BF16>
__device__ __forceinline__ uint32_t ds_pair(uint32_t s0, uint32_t s1, uint32_t p0, uint32_t p1,
                                            float half_alpha) {
  const float h0 = __uint_as_float(s0) * half_alpha, h1 = __uint_as_float(s1) * half_alpha;
  return pack2<BF16>(dsilu2(h0, tanh_approx(h0), __uint_as_float(p0)),
                     dsilu2(h1, tanh_approx(h1), __uint_as_float(p1)));
}

// A^T pair (SiLU) and dS^T pair (doubled) of two elements sharing one tanh each.
template <bool BF16>
__device__ __forceinline__ void a_ds_pair(uint32_t s0, uint32_t s1, uint32_t p0, uint32_t p1,
                                          float half_alpha, uint32_t& a, uint32_t& d) {
  const float h0 = __uint_as_float(s0) * half_alpha, h1 = __uint_as_float(s1) * half_alpha;
  const float t0 = tanh_approx(h0), t1 = tanh_approx(h1);
  a = pack2<BF16>(fmaf(h0, t0, h0), fmaf(h1, t1, h1));
  d = pack2<BF16>(dsilu2(h0, t0, __uint_as_float(p0)), dsilu2(h1, t1, __uint_as_float(p1)));
}

// Store 32 fp32 values (one TMEM chunk of one row) as 32 16-bit elements,
// scaled by `scale`, with four 16-byte stores.
template <bool BF16>
__device__ __forceinline__ void store_row32(void* dst, const uint32_t (&x)[32], float scale) {
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    uint4 w;
    w.x = pack2<BF16>(__uint_as_float(x[8 * v + 0]) * scale, __uint_as_float(x[8 * v + 1]) * scale);
    w.y = pack2<BF16>(__uint_as_float(x[8 * v + 2]) * scale, __uint_as_float(x[8 * v + 3]) * scale);
    w.z = pack2<BF16>(__uint_as_float(x[8 * v + 4]) * scale, __uint_as_float(x[8 * v + 5]) * scale);
    w.w = pack2<BF16>(__uint_as_float(x[8 * v + 6]) * scale, __uint_as_float(x[8 * v + 7]) * scale);
    p[v] = w;
  }
}

__device__ __forceinline__ void store_zero32(void* dst) {
  uint4* p = reinterpret_cast<uint4*>(dst);
  const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int v = 0; v < 4; ++v) p[v] = z;
}

// Compile-time-width variants used by the 16-row-warp kernels.
template <int N>
__device__ __forceinline__ void tmem_ld_x2(uint32_t ta, uint32_t tb, uint32_t (&a)[N],
                                           uint32_t (&b)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  if constexpr (N == 32) tmem_ld32x2(ta, tb, a, b);
  else tmem_ld16x2(ta, tb, a, b);
}
template <int N>
__device__ __forceinline__ void tmem_ld_w(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  if constexpr (N == 32) tmem_ld32(taddr, r);
  else tmem_ld16(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st_w(uint32_t taddr, const uint32_t (&r)[N]) {
  static_assert(N == 8 || N == 16 || N == 32, "8, 16 or 32 columns");
  if constexpr (N == 32) tmem_st32(taddr, r);
  else if constexpr (N == 16) tmem_st16(taddr, r);
  else tmem_st8(taddr, r);
}

// N fp32 values (N a multiple of 8) scaled, rounded to 16 bits and stored
// with 16-byte writes; dst is 16-byte aligned.
template <int N, bool BF16>
__device__ __forceinline__ void store_row_n(void* dst, const uint32_t (&x)[N], float scale) {
  static_assert(N % 8 == 0, "whole 16-byte groups");
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int v = 0; v < N / 8; ++v) {
    uint4 w;
    w.x = pack2<BF16>(__uint_as_float(x[8 * v + 0]) * scale, __uint_as_float(x[8 * v + 1]) * scale);
    w.y = pack2<BF16>(__uint_as_float(x[8 * v + 2]) * scale, __uint_as_float(x[8 * v + 3]) * scale);
    w.z = pack2<BF16>(__uint_as_float(x[8 * v + 4]) * scale, __uint_as_float(x[8 * v + 5]) * scale);
    w.w = pack2<BF16>(__uint_as_float(x[8 * v + 6]) * scale, __uint_as_float(x[8 * v + 7]) * scale);
    p[v] = w;
  }
}
// 32 fp32 values of row r (columns col .. col + 31, col a multiple of 32)
// scaled, rounded to 16 bits and written into a shared-memory tile laid out
// like the TMA box: 64-column chunks of [128 rows][128 bytes], 128-byte
// swizzle (16-byte unit u of row r sits at unit u ^ (r & 7)), so a TMA store
// of the tile writes the rows out and the eight lanes of each store phase hit
// distinct banks.
template <bool BF16>
__device__ __forceinline__ void stage_row32(uint32_t tile, int r, int col, const uint32_t (&x)[32],
                                            float scale) {
  const uint32_t row_base = tile + static_cast<uint32_t>(col >> 6) * (kBM * 128) +
                            static_cast<uint32_t>(r) * 128;
  const int u0 = (col & 63) >> 3;
#pragma unroll
  for (int v = 0; v < 4; ++v) {
    const uint32_t w0 = pack2<BF16>(__uint_as_float(x[8 * v + 0]) * scale, __uint_as_float(x[8 * v + 1]) * scale);
    const uint32_t w1 = pack2<BF16>(__uint_as_float(x[8 * v + 2]) * scale, __uint_as_float(x[8 * v + 3]) * scale);
    const uint32_t w2 = pack2<BF16>(__uint_as_float(x[8 * v + 4]) * scale, __uint_as_float(x[8 * v + 5]) * scale);
    const uint32_t w3 = pack2<BF16>(__uint_as_float(x[8 * v + 6]) * scale, __uint_as_float(x[8 * v + 7]) * scale);
    st_shared_v4(row_base + (static_cast<uint32_t>((u0 + v) ^ (r & 7)) << 4), w0, w1, w2, w3);
  }
}

// The first N of M fp32 values, scaled, rounded and stored (N a multiple of 8).
template <int N, int M, bool BF16>
__device__ __forceinline__ void store_row_head(void* dst, const uint32_t (&x)[M], float scale) {
  static_assert(N % 8 == 0 && N <= M, "whole 16-byte groups of the row");
  uint4* p = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int v = 0; v < N / 8; ++v) {
    uint4 w;
    w.x = pack2<BF16>(__uint_as_float(x[8 * v + 0]) * scale, __uint_as_float(x[8 * v + 1]) * scale);
    w.y = pack2<BF16>(__uint_as_float(x[8 * v + 2]) * scale, __uint_as_float(x[8 * v + 3]) * scale);
    w.z = pack2<BF16>(__uint_as_float(x[8 * v + 4]) * scale, __uint_as_float(x[8 * v + 5]) * scale);
    w.w = pack2<BF16>(__uint_as_float(x[8 * v + 6]) * scale, __uint_as_float(x[8 * v + 7]) * scale);
    p[v] = w;
  }
}

template <int N>
__device__ __forceinline__ void store_zero_n(void* dst) {
  static_assert(N % 8 == 0, "whole 16-byte groups");
  uint4* p = reinterpret_cast<uint4*>(dst);
  const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int v = 0; v < N / 8; ++v) p[v] = z;
}

// Row-warp barrier arrival: every lane's TMEM accesses are complete (waited
// for by the caller), then one arrival per warp.
__device__ __forceinline__ void warp_arrive(uint32_t bar) {
  tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// K-major operand descriptor: tile of ROWS rows by D columns, stored as D/64
// chunks of [ROWS][64] 16-bit elements with the 128-byte swizzle (the TMA box
// layout).  kk selects the 16-element K step.
// `base` is kdesc(tile).
__device__ __forceinline__ SDesc kdesc(uint32_t tile) { return sdesc_split(tile, 16, 1024); }
template <int ROWS>
__device__ __forceinline__ SDesc desc_kmajor(SDesc base, int kk) {
  return sdesc_add(base, static_cast<uint32_t>(kk >> 2) * (ROWS * 128) +
                             static_cast<uint32_t>(kk & 3) * 32);
}

// MN-major B operand read from the same tile layout: K runs down the ROWS
// (16 rows per step kk), N runs along the columns starting at column n0
// (a multiple of 64); 64-column chunks are ROWS*128 bytes apart (LBO) and
// 8-row groups 1024 bytes apart (SBO).  `base` is mndesc<ROWS>(tile).
template <int ROWS>
__device__ __forceinline__ SDesc mndesc(uint32_t tile) {
  return sdesc_split(tile, ROWS * 128, 1024);
}
template <int ROWS>
__device__ __forceinline__ SDesc desc_mnmajor(SDesc base, int kk, int n0) {
  return sdesc_add(base, static_cast<uint32_t>(n0 >> 6) * (ROWS * 128) +
                             static_cast<uint32_t>(kk) * 2048);
}

}  // namespace hstu
