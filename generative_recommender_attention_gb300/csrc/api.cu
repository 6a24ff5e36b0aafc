// Host side of the C ABI in hstu_attn.h: argument validation, TMA tensor-map
// encoding, work-list scheduling and kernel launches.  No allocation, no
// host copy of device metadata, no synchronization (except in the explicit
// status query).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "hstu_attn.h"
#include "kernels.h"

using namespace hstu;

namespace {

constexpr uint64_t kWaitTimeoutNs = 4000000000ull;  // 4 s per barrier wait
constexpr int kMaxDevices = 64;

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------- device info
struct DevInfo {
  int sm_count = 0;
  int major = 0, minor = 0;
  int max_smem_optin = 0;
};

bool device_info(DevInfo* out) {
  static DevInfo cache[kMaxDevices];
  static bool valid[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(mu);
  if (!valid[dev]) {
    DevInfo d;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
      return false;
    cache[dev] = d;
    valid[dev] = true;
  }
  *out = cache[dev];
  return true;
}

// ---------------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D map over a (T, H, D) tensor with a box of 64 elements x 1 head x
// box_rows tokens, 128-byte swizzle; rows past T read as zeros.
bool encode_thd(CUtensorMap* m, const void* ptr, int64_t T, int H, int D, int64_t st, int64_t sh,
                int box_rows, bool bf16) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(std::max<int64_t>(T, 1))};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(sh * 2), static_cast<cuuint64_t>(st * 2)};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                  const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over the dS blocks: (128 keys, 64 queries, block), box of 64 keys
// x 64 queries of one block, 128-byte swizzle.
bool encode_ds(CUtensorMap* m, void* ptr, int64_t blocks, bool bf16) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDsKeys), static_cast<cuuint64_t>(kDsQueries),
                        static_cast<cuuint64_t>(std::max<int64_t>(blocks, 1))};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kDsKeys * 2),
                           static_cast<cuuint64_t>(kDsBlockBytes)};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kDsQueries), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                  ptr, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- validation
bool supported_dim(int D) { return D == 32 || D == 64 || D == 128 || D == 256; }
// Head dim 32 runs through the D = 64 kernels: the tensor maps keep the true
// head dim, the 64-wide boxes read its columns 32-63 as zeros (out-of-range
// fill), which add nothing to any product, and the outputs are clipped to 32
// columns.
int kernel_dim(int D) { return D == 32 ? 64 : D; }

// Checks one (T, H, D) tensor with element strides (st, sh, 1).
hstu_status_t check_tensor(const void* ptr, int64_t st, int64_t sh, int64_t T, int H, int D) {
  if (T == 0) return HSTU_OK;
  if (ptr == nullptr) return HSTU_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return HSTU_ERR_MISALIGNED;
  if (st <= 0 || sh <= 0) return HSTU_ERR_INVALID_ARG;
  if ((st * 2) % 16 != 0 || (sh * 2) % 16 != 0) return HSTU_ERR_MISALIGNED;
  if (st * 2 >= (int64_t(1) << 40) || sh * 2 >= (int64_t(1) << 40)) return HSTU_ERR_INVALID_ARG;
  // no two logical elements at one address: sort dims by stride, each stride
  // must exceed the span of the smaller ones.
  struct Dim { int64_t stride, size; } d[3] = {{1, D}, {sh, H}, {st, T}};
  std::sort(d, d + 3, [](const Dim& x, const Dim& y) { return x.stride < y.stride; });
  int64_t span = 0;
  for (auto& x : d) {
    if (x.size <= 1) continue;
    if (x.stride <= span) return HSTU_ERR_INVALID_ARG;
    span += x.stride * (x.size - 1);
  }
  return HSTU_OK;
}

struct Common {
  DevInfo dev;
  float inv_L;
  bool bf16;
  Window win;
};

hstu_status_t check_common(int32_t batch, int64_t total_q, int64_t total_k, int32_t H, int32_t D,
                           hstu_dtype_t dtype, int32_t max_q, int32_t max_k, float alpha,
                           int32_t scaling, int32_t wl, int32_t wr, const int32_t* cu_q,
                           const int32_t* cu_k, Common* c) {
  if (batch < 0 || total_q < 0 || total_k < 0 || H <= 0 || max_q < 0 || max_k < 0)
    return HSTU_ERR_INVALID_ARG;
  if (total_q > INT32_MAX || total_k > INT32_MAX) return HSTU_ERR_INVALID_ARG;
  if (!(dtype == HSTU_FP16 || dtype == HSTU_BF16)) return HSTU_ERR_UNSUPPORTED;
  if (!supported_dim(D)) return HSTU_ERR_UNSUPPORTED;
  if (max_q > max_k) return HSTU_ERR_INVALID_ARG;
  if (!std::isfinite(alpha)) return HSTU_ERR_INVALID_ARG;
  if (scaling < 0) return HSTU_ERR_INVALID_ARG;
  if (wl < -1 || wr < -1) return HSTU_ERR_INVALID_ARG;  // -1: no bound on that side
  const int32_t L = scaling > 0 ? scaling : max_q;
  if (batch > 0 && total_q > 0 && L <= 0) return HSTU_ERR_INVALID_ARG;
  if (batch > 0 && (cu_q == nullptr || cu_k == nullptr)) return HSTU_ERR_INVALID_ARG;
  c->inv_L = L > 0 ? 1.0f / static_cast<float>(L) : 0.f;
  c->bf16 = dtype == HSTU_BF16;
  c->win = Window{wl, wr};
  return HSTU_OK;
}

int64_t cap_a(int32_t batch, int64_t total_q, int32_t H) {
  return static_cast<int64_t>(H) * (cdiv(total_q, kBM) + batch);
}
int64_t cap_b(int32_t batch, int64_t total_k, int32_t H, int32_t D) {
  const int split = D == 256 ? 2 : 1;
  return static_cast<int64_t>(H) * split * (cdiv(total_k, kBM) + batch);
}

int bn_for(int D) { return D == 256 ? 64 : 128; }

// Backward workspace: header | list A | list B | ds_base (B + 1 ints) |
// readiness counts (B x H ints) | dS blocks.  The dS capacity bounds sum_b H ceil(Lk_b/128) ceil(Lq_b/64) from
// the sizes alone (every Lq_b <= max_seqlen_q), so the host never needs the
// sequence lengths.
struct BwdLayout {
  size_t units_b, ds_base, ready, ds, total;
  int64_t ds_blocks;
};

bool bwd_layout(int32_t batch, int64_t total_q, int64_t total_k, int32_t H, int32_t D,
                int32_t max_q, BwdLayout* L) {
  const int64_t capA = cap_a(batch, total_q, H), capB = cap_b(batch, total_k, H, D);
  L->units_b = kHeaderBytes + 32 * static_cast<size_t>(capA);
  L->ds_base = L->units_b + 32 * static_cast<size_t>(capB);
  L->ready = L->ds_base + 4 * (static_cast<size_t>(batch) + 1);
  L->ds = (L->ready + 4 * static_cast<size_t>(batch) * H + 1023) & ~size_t(1023);
  L->ds_blocks = static_cast<int64_t>(H) * cdiv(std::max<int32_t>(max_q, 0), kDsQueries) *
                 (cdiv(total_k, kDsKeys) + batch);
  if (L->ds_blocks > INT32_MAX) return false;  // block indices are int32 on the device
  L->total = L->ds + static_cast<size_t>(L->ds_blocks) * kDsBlockBytes;
  return true;
}

// A plan is the backward workspace followed by list F, the forward's query
// tiles.  Its header records the sizes it was made for (plan_key), which
// every planned kernel compares with its own before it starts.
size_t plan_list_f(const BwdLayout& L) { return (L.total + 255) & ~size_t(255); }

constexpr int kPlanMagic = 0x504c414e;

void plan_key(int32_t batch, int64_t total_q, int64_t total_k, int32_t H, int32_t D, int32_t max_q,
              int32_t max_k, Window w, int* key) {
  const int k[kPlanKeyInts] = {kPlanMagic, batch, static_cast<int>(total_q),
                               static_cast<int>(total_k), H, D, max_q, max_k, w.left, w.right};
  std::memcpy(key, k, sizeof(k));
}

// Arbitrary mask: the key hull of every query-block slot, and (backward)
// the query-block hull of every key-tile slot, appended to the workspace.
// Layout: qb_range | kt_range (backward) | qb_bits | qb_full, each 256-byte
// aligned (qb_bits and qb_full have the same size).
int func_kt_words(int32_t max_k) {
  return static_cast<int>(std::max<int64_t>(1, cdiv(cdiv(std::max<int32_t>(max_k, 1), kBM), 32)));
}
size_t func_bits_off(int32_t batch, int64_t total_q, int64_t total_k, bool bwd) {
  const size_t qb = 8 * static_cast<size_t>(total_q / 64 + batch + 1);
  const size_t kt = bwd ? 8 * static_cast<size_t>(total_k / kBM + batch + 1) : 0;
  return ((qb + 255) & ~size_t(255)) + ((kt + 255) & ~size_t(255));
}
size_t func_bits_bytes(int32_t batch, int64_t total_q, int32_t max_k) {
  const size_t n = 4 * static_cast<size_t>(func_kt_words(max_k)) *
                   static_cast<size_t>(total_q / 64 + batch + 1);
  return (n + 255) & ~size_t(255);
}
size_t func_extra(int32_t batch, int64_t total_q, int64_t total_k, int32_t max_k, bool bwd) {
  return func_bits_off(batch, total_q, total_k, bwd) + 2 * func_bits_bytes(batch, total_q, max_k);
}

// Arbitrary-mask arguments of a call (func null: none).
struct FuncArgs {
  const int32_t* func;
  int32_t n;
  int64_t len;
};

// Shared memory of the scheduler block: one int per cost bucket, then (for
// up to kSchedCacheSeqs sequences) one 16-byte record per sequence.
bool sched_smem(int cmax, int batch, int64_t cap, const DevInfo& dev, int* bytes, int* cache,
                int* stage_units) {
  *cache = batch <= kSchedCacheSeqs ? 1 : 0;
  int b = sched_hist_ints(cmax) * 4 + (*cache ? 16 * batch : 0);
  if (b > dev.max_smem_optin - 1024) return false;
  // a list of up to kSchedStageUnits records is staged in shared memory
  // and leaves in one coalesced copy
  *stage_units = static_cast<int>(std::min<int64_t>(
      cap, std::min<int64_t>(kSchedStageUnits, (dev.max_smem_optin - 1024 - b) / 32)));
  b += 32 * std::max(*stage_units, 0);
  // the opt-in limit less the kernel's static shared memory, set once
  static bool set = false;
  if (b > 48 * 1024 && !set) {
    if (cudaFuncSetAttribute(hstu_sched_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dev.max_smem_optin - 1024) != cudaSuccess)
      return false;
    set = true;
  }
  *bytes = b;
  return true;
}

}  // namespace

extern "C" {

int32_t hstu_attn_version(void) { return 100; }

const char* hstu_attn_status_string(hstu_status_t s) {
  switch (s) {
    case HSTU_OK: return "ok";
    case HSTU_ERR_INVALID_ARG: return "invalid argument";
    case HSTU_ERR_UNSUPPORTED: return "unsupported configuration";
    case HSTU_ERR_MISALIGNED: return "pointer or stride not 16-byte aligned";
    case HSTU_ERR_CUDA: return "CUDA error";
    case HSTU_ERR_DEVICE_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

size_t hstu_attn_workspace_size(int32_t batch, int64_t total_q, int64_t total_k,
                                int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q,
                                int32_t max_seqlen_k, int32_t is_bwd) {
  if (batch < 0 || total_q < 0 || total_k < 0 || num_heads <= 0 || !supported_dim(head_dim) ||
      max_seqlen_q < 0 || max_seqlen_k < 0)
    return 0;
  if (!is_bwd) {
    // a unit record is two int4 (32 bytes)
    const size_t bytes = kHeaderBytes + 32 * static_cast<size_t>(cap_a(batch, total_q, num_heads));
    return (bytes + 255) & ~size_t(255);
  }
  BwdLayout L;
  if (!bwd_layout(batch, total_q, total_k, num_heads, head_dim, max_seqlen_q, &L)) return 0;
  return (L.total + 255) & ~size_t(255);
}

size_t hstu_attn_workspace_size_func(int32_t batch, int64_t total_q, int64_t total_k,
                                     int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q,
                                     int32_t max_seqlen_k, int32_t is_bwd) {
  const size_t base = hstu_attn_workspace_size(batch, total_q, total_k, num_heads, head_dim,
                                               max_seqlen_q, max_seqlen_k, is_bwd);
  if (base == 0) return 0;
  return base + func_extra(batch, total_q, total_k, max_seqlen_k, is_bwd != 0);
}

size_t hstu_attn_plan_workspace_size(int32_t batch, int64_t total_q, int64_t total_k,
                                     int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q,
                                     int32_t max_seqlen_k) {
  if (hstu_attn_workspace_size(batch, total_q, total_k, num_heads, head_dim, max_seqlen_q,
                               max_seqlen_k, 1) == 0)
    return 0;
  BwdLayout L;
  if (!bwd_layout(batch, total_q, total_k, num_heads, head_dim, max_seqlen_q, &L)) return 0;
  const size_t bytes = plan_list_f(L) + 32 * static_cast<size_t>(cap_a(batch, total_q, num_heads));
  return (bytes + 255) & ~size_t(255);
}

}  // extern "C"

namespace {

// Records events[i] on `stream` when a profiling caller supplied them.
struct EventMarks {
  cudaEvent_t* ev;
  int n;
  // Events between the kernels would serialise them: chain the grids with
  // programmatic dependent launch only when no events are recorded.
  bool pdl() const { return ev == nullptr; }
  bool mark(int i, cudaStream_t st) const {
    return ev == nullptr || i >= n || cudaEventRecord(ev[i], st) == cudaSuccess;
  }
};

// Validates the arbitrary-mask arguments and builds the device view over
// the workspace tail that starts at `tail` (bytes into the workspace).
hstu_status_t func_setup(const FuncArgs* fn, int32_t batch, int64_t total_q, int64_t total_k,
                         int32_t max_k, char* ws, size_t tail, bool bwd, Common* c,
                         FuncMask* fm) {
  *fm = FuncMask{};
  if (fn == nullptr) return HSTU_OK;
  if (fn->n < 1 || fn->n % 2 != 1 || fn->len < total_q) return HSTU_ERR_INVALID_ARG;
  if (batch > 0 && total_q > 0 && fn->func == nullptr) return HSTU_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(fn->func) % 4 != 0) return HSTU_ERR_MISALIGNED;
  c->win = Window{-1, -1};  // the endpoints decide; the dS blocks use the full layout
  fm->func = fn->func;
  fm->n = fn->n;
  fm->len = fn->len;
  fm->qb_range = reinterpret_cast<int2*>(ws + tail);
  if (bwd)
    fm->kt_range = reinterpret_cast<int2*>(
        ws + tail + ((8 * static_cast<size_t>(total_q / 64 + batch + 1) + 255) & ~size_t(255)));
  fm->qb_bits = reinterpret_cast<uint32_t*>(ws + tail + func_bits_off(batch, total_q, total_k, bwd));
  fm->qb_full = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(fm->qb_bits) +
                                            func_bits_bytes(batch, total_q, max_k));
  fm->kt_words = func_kt_words(max_k);
  return HSTU_OK;
}

// A paged K/V cache: contiguous (num_pages, 2, 128, H, D) storage and the
// device page tables.
struct PagedKV {
  const void* kv;
  int64_t num_pages;
  const int32_t* page_ids;
  const int32_t* page_indptrs;
};

hstu_status_t fwd_impl(hstu_cten_t q, hstu_cten_t k, hstu_cten_t v, hstu_ten_t out,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
                       int64_t total_q, int64_t total_k, int32_t num_heads, int32_t head_dim,
                       hstu_dtype_t dtype, int32_t max_seqlen_q, int32_t max_seqlen_k,
                       float alpha, int32_t scaling_seqlen, int32_t window_left,
                       int32_t window_right, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream, const EventMarks& em,
                       const PagedKV* paged = nullptr, const FuncArgs* fn = nullptr,
                       bool planned = false) {
  Common c;
  hstu_status_t s = check_common(batch, total_q, total_k, num_heads, head_dim, dtype, max_seqlen_q,
                                 max_seqlen_k, alpha, scaling_seqlen, window_left, window_right,
                                 cu_seqlens_q, cu_seqlens_k, &c);
  if (s != HSTU_OK) return s;
  const int H = num_heads, D = head_dim;
  if ((s = check_tensor(q.ptr, q.stride_t, q.stride_h, total_q, H, D)) != HSTU_OK) return s;
  if (paged == nullptr) {
    if ((s = check_tensor(k.ptr, k.stride_t, k.stride_h, total_k, H, D)) != HSTU_OK) return s;
    if ((s = check_tensor(v.ptr, v.stride_t, v.stride_h, total_k, H, D)) != HSTU_OK) return s;
  } else {
    if (paged->num_pages <= 0 || paged->num_pages > (INT32_MAX / 256)) return HSTU_ERR_INVALID_ARG;
    if (batch > 0 && (paged->page_ids == nullptr || paged->page_indptrs == nullptr))
      return HSTU_ERR_INVALID_ARG;
    if ((s = check_tensor(paged->kv, int64_t(H) * D, D, paged->num_pages * 256, H, D)) != HSTU_OK)
      return s;
  }
  if ((s = check_tensor(out.ptr, out.stride_t, out.stride_h, total_q, H, D)) != HSTU_OK) return s;
  if (batch == 0 || total_q == 0) return HSTU_OK;
  const size_t base_need =
      planned ? hstu_attn_plan_workspace_size(batch, total_q, total_k, H, D, max_seqlen_q,
                                              max_seqlen_k)
              : hstu_attn_workspace_size(batch, total_q, total_k, H, D, max_seqlen_q, max_seqlen_k,
                                         0);
  if (base_need == 0) return HSTU_ERR_INVALID_ARG;
  const size_t need =
      base_need + (fn ? func_extra(batch, total_q, total_k, max_seqlen_k, false) : 0);
  if (workspace == nullptr || workspace_bytes < need) return HSTU_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return HSTU_ERR_MISALIGNED;
  FuncMask fm;
  if ((s = func_setup(fn, batch, total_q, total_k, max_seqlen_k, static_cast<char*>(workspace),
                      base_need, false,
                      &c, &fm)) != HSTU_OK)
    return s;
  if (!device_info(&c.dev)) return HSTU_ERR_CUDA;
  if (c.dev.major != 10 || c.dev.minor != 3) return HSTU_ERR_UNSUPPORTED;

  const int BN = bn_for(D);
  const int64_t capA = cap_a(batch, total_q, H);
  const int cmax = static_cast<int>(std::max<int64_t>(1, cdiv(max_seqlen_k, BN)));
  int sched_bytes, sched_cache, sched_stage;
  if (!sched_smem(cmax, batch, capA, c.dev, &sched_bytes, &sched_cache, &sched_stage))
    return HSTU_ERR_UNSUPPORTED;

  CUtensorMap tq, tk, tv;
  const void* kptr = total_k > 0 ? k.ptr : q.ptr;  // stand-in, never read when total_k == 0
  const void* vptr = total_k > 0 ? v.ptr : q.ptr;
  const int64_t kst = total_k > 0 ? k.stride_t : q.stride_t, ksh = total_k > 0 ? k.stride_h : q.stride_h;
  const int64_t vst = total_k > 0 ? v.stride_t : q.stride_t, vsh = total_k > 0 ? v.stride_h : q.stride_h;
  if (!encode_thd(&tq, q.ptr, total_q, H, D, q.stride_t, q.stride_h, kBM, c.bf16))
    return HSTU_ERR_CUDA;
  if (paged != nullptr) {
    // one map over the whole cache, 256 rows per page (128 K rows, then 128 V rows)
    if (!encode_thd(&tk, paged->kv, paged->num_pages * 256, H, D, int64_t(H) * D, D, BN, c.bf16))
      return HSTU_ERR_CUDA;
    tv = tk;
  } else if (!encode_thd(&tk, kptr, total_k, H, D, kst, ksh, BN, c.bf16) ||
             !encode_thd(&tv, vptr, total_k, H, D, vst, vsh, BN, c.bf16)) {
    return HSTU_ERR_CUDA;
  }

  int* header = static_cast<int*>(workspace);
  int4* units = reinterpret_cast<int4*>(static_cast<char*>(workspace) + kHeaderBytes);
  if (planned) {
    BwdLayout L;
    if (!bwd_layout(batch, total_q, total_k, H, D, max_seqlen_q, &L)) return HSTU_ERR_UNSUPPORTED;
    units = reinterpret_cast<int4*>(static_cast<char*>(workspace) + plan_list_f(L));
  }
  SchedArgs sa{};
  sa.cu_q = cu_seqlens_q; sa.cu_k = cu_seqlens_k; sa.B = batch; sa.H = H; sa.win = c.win;
  sa.bn_a = BN; sa.cmax_a = cmax; sa.cap_a = static_cast<int>(capA); sa.units_a = units;
  sa.header = header; sa.cache_seqs = sched_cache; sa.stage_units = sched_stage; sa.fm = fm;
  if (!em.mark(0, stream)) return HSTU_ERR_CUDA;
  if (fm.func != nullptr &&
      launch_func_ranges(cu_seqlens_q, cu_seqlens_k, batch,
                         static_cast<int>(cdiv(std::max<int32_t>(max_seqlen_q, 1), 64)), fm, stream,
                         em.pdl()) != cudaSuccess)
    return HSTU_ERR_CUDA;
  if (!planned && launch_sched(1, sched_bytes, stream, em.pdl(), sa) != cudaSuccess)
    return HSTU_ERR_CUDA;
  if (!em.mark(1, stream)) return HSTU_ERR_CUDA;

  AttnArgs a{};
  a.total_q = total_q; a.total_k = total_k;
  a.H = H; a.win = c.win; a.d_out = D; a.alpha = alpha; a.inv_L = c.inv_L; a.header = header;
  a.units = units;
  a.units_slot = planned ? kHdrUnitsF : kHdrUnitsA;
  a.next_slot = planned ? kHdrNextF : kHdrNextA;
  a.planned = planned ? 1 : 0;
  if (planned) plan_key(batch, total_q, total_k, H, D, max_seqlen_q, max_seqlen_k, c.win, a.key);
  a.timeout_ns = kWaitTimeoutNs; a.pdl_wait = 1;
  a.o0 = out.ptr; a.o0_st = out.stride_t; a.o0_sh = out.stride_h;
  a.fm = fm;
  if (paged != nullptr) {
    a.page_ids = paged->page_ids;
    a.page_indptrs = paged->page_indptrs;
  }
  const int grid = static_cast<int>(std::min<int64_t>(c.dev.sm_count, capA));
  if (launch_fwd(kernel_dim(D), c.bf16, grid, stream, em.pdl(), tq, tk, tv, a) != cudaSuccess)
    return HSTU_ERR_CUDA;
  if (!em.mark(2, stream)) return HSTU_ERR_CUDA;
  return HSTU_OK;
}

hstu_status_t bwd_impl(hstu_cten_t dout, hstu_cten_t q, hstu_cten_t k, hstu_cten_t v,
                       hstu_ten_t dq, hstu_ten_t dk, hstu_ten_t dv, const int32_t* cu_seqlens_q,
                       const int32_t* cu_seqlens_k, int32_t batch, int64_t total_q,
                       int64_t total_k, int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
                       int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
                       int32_t scaling_seqlen, int32_t window_left, int32_t window_right,
                       void* workspace,
                       size_t workspace_bytes, cudaStream_t stream, const EventMarks& em,
                       const FuncArgs* fn = nullptr, bool planned = false) {
  Common c;
  hstu_status_t s = check_common(batch, total_q, total_k, num_heads, head_dim, dtype, max_seqlen_q,
                                 max_seqlen_k, alpha, scaling_seqlen, window_left, window_right,
                                 cu_seqlens_q, cu_seqlens_k, &c);
  if (s != HSTU_OK) return s;
  const int H = num_heads, D = head_dim;
  if ((s = check_tensor(dout.ptr, dout.stride_t, dout.stride_h, total_q, H, D)) != HSTU_OK) return s;
  if ((s = check_tensor(q.ptr, q.stride_t, q.stride_h, total_q, H, D)) != HSTU_OK) return s;
  if ((s = check_tensor(k.ptr, k.stride_t, k.stride_h, total_k, H, D)) != HSTU_OK) return s;
  if ((s = check_tensor(v.ptr, v.stride_t, v.stride_h, total_k, H, D)) != HSTU_OK) return s;
  if ((s = check_tensor(dq.ptr, dq.stride_t, dq.stride_h, total_q, H, D)) != HSTU_OK) return s;
  if ((s = check_tensor(dk.ptr, dk.stride_t, dk.stride_h, total_k, H, D)) != HSTU_OK) return s;
  if ((s = check_tensor(dv.ptr, dv.stride_t, dv.stride_h, total_k, H, D)) != HSTU_OK) return s;
  if (batch == 0 || (total_q == 0 && total_k == 0)) return HSTU_OK;
  BwdLayout lay;
  if (!bwd_layout(batch, total_q, total_k, H, D, max_seqlen_q, &lay)) return HSTU_ERR_UNSUPPORTED;
  const size_t base_need =
      planned ? hstu_attn_plan_workspace_size(batch, total_q, total_k, H, D, max_seqlen_q,
                                              max_seqlen_k)
              : hstu_attn_workspace_size(batch, total_q, total_k, H, D, max_seqlen_q, max_seqlen_k,
                                         1);
  if (base_need == 0) return HSTU_ERR_INVALID_ARG;
  const size_t need =
      base_need + (fn ? func_extra(batch, total_q, total_k, max_seqlen_k, true) : 0);
  if (workspace == nullptr || workspace_bytes < need) return HSTU_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return HSTU_ERR_MISALIGNED;
  FuncMask fm;
  if ((s = func_setup(fn, batch, total_q, total_k, max_seqlen_k, static_cast<char*>(workspace),
                      base_need, true,
                      &c, &fm)) != HSTU_OK)
    return s;
  if (!device_info(&c.dev)) return HSTU_ERR_CUDA;
  if (c.dev.major != 10 || c.dev.minor != 3) return HSTU_ERR_UNSUPPORTED;

  const int BN = kDsKeys;                                         // dQ unit key tile
  const int BQ = DkdvCfg<128, kPassBoth>::BQ;  // dK/dV query tile (every D)
  const int split = D == 256 ? 2 : 1;
  const int64_t capA = cap_a(batch, total_q, H);
  const int64_t capB = cap_b(batch, total_k, H, D);
  const int cmaxA = static_cast<int>(std::max<int64_t>(1, cdiv(max_seqlen_k, BN)));
  const int cmaxB = static_cast<int>(std::max<int64_t>(1, cdiv(max_seqlen_q, BQ)));
  int sched_bytes, sched_cache, sched_stage;
  if (!sched_smem(std::max(cmaxA, cmaxB), batch, std::max(capA, capB), c.dev, &sched_bytes,
                  &sched_cache, &sched_stage))
    return HSTU_ERR_UNSUPPORTED;

  // Stand-ins for empty sides: valid maps that no unit ever reads through.
  const bool hq = total_q > 0, hk = total_k > 0;
  const hstu_cten_t qx = hq ? q : k, dox = hq ? dout : k, kx = hk ? k : q, vx = hk ? v : q;
  CUtensorMap m_k128, m_v128, m_q64, m_do64, m_ds;
  char* ws = static_cast<char*>(workspace);
  if (!encode_thd(&m_k128, kx.ptr, total_k, H, D, kx.stride_t, kx.stride_h, kBM, c.bf16) ||
      !encode_thd(&m_v128, vx.ptr, total_k, H, D, vx.stride_t, vx.stride_h, kBM, c.bf16) ||
      !encode_thd(&m_q64, qx.ptr, total_q, H, D, qx.stride_t, qx.stride_h, BQ, c.bf16) ||
      !encode_thd(&m_do64, dox.ptr, total_q, H, D, dox.stride_t, dox.stride_h, BQ, c.bf16) ||
      !encode_ds(&m_ds, ws + lay.ds, lay.ds_blocks, c.bf16))
    return HSTU_ERR_CUDA;

  int* header = reinterpret_cast<int*>(ws);
  int4* unitsA = reinterpret_cast<int4*>(ws + kHeaderBytes);
  int4* unitsB = reinterpret_cast<int4*>(ws + lay.units_b);
  int* ds_base = reinterpret_cast<int*>(ws + lay.ds_base);
  int* ready = reinterpret_cast<int*>(ws + lay.ready);
  SchedArgs sa{};
  sa.cu_q = cu_seqlens_q; sa.cu_k = cu_seqlens_k; sa.B = batch; sa.H = H; sa.win = c.win;
  sa.bn_a = BN; sa.cmax_a = cmaxA; sa.cap_a = static_cast<int>(capA); sa.units_a = unitsA;
  sa.bq_b = BQ; sa.split_b = split; sa.cmax_b = cmaxB; sa.cap_b = static_cast<int>(capB);
  sa.units_b = unitsB; sa.header = header;
  sa.ds_base = ds_base; sa.ds_cap = static_cast<int>(lay.ds_blocks); sa.cache_seqs = sched_cache;
  sa.stage_units = sched_stage;
  sa.ready = ready;
  sa.fm = fm;
  if (!em.mark(0, stream)) return HSTU_ERR_CUDA;
  if (fm.func != nullptr &&
      launch_func_ranges(cu_seqlens_q, cu_seqlens_k, batch,
                         static_cast<int>(cdiv(std::max<int32_t>(max_seqlen_q, 1), 64)), fm, stream,
                         em.pdl()) != cudaSuccess)
    return HSTU_ERR_CUDA;
  if (!planned && launch_sched(2, sched_bytes, stream, em.pdl(), sa) != cudaSuccess)
    return HSTU_ERR_CUDA;
  if (!em.mark(1, stream)) return HSTU_ERR_CUDA;

  AttnArgs a{};
  a.total_q = total_q; a.total_k = total_k;
  a.H = H; a.win = c.win; a.d_out = D; a.alpha = alpha; a.inv_L = c.inv_L; a.header = header;
  a.planned = planned ? 1 : 0;
  if (planned) plan_key(batch, total_q, total_k, H, D, max_seqlen_q, max_seqlen_k, c.win, a.key);
  a.timeout_ns = kWaitTimeoutNs; a.pdl_wait = 1;
  a.ds = ws + lay.ds; a.ds_base = ds_base; a.ds_cap = static_cast<int>(lay.ds_blocks);
  a.ready = ready;
  a.fm = fm;
  // One launch: each CTA takes dK/dV units (list B), which also store the
  // dS blocks, then dQ units (list A), each of which waits until the dS
  // blocks of its sequence and head are complete.
  AttnArgs ak = a;
  ak.units = unitsB; ak.units_slot = kHdrUnitsB; ak.next_slot = kHdrNextB;
  ak.o0 = dv.ptr; ak.o0_st = dv.stride_t; ak.o0_sh = dv.stride_h;
  ak.o1 = dk.ptr; ak.o1_st = dk.stride_t; ak.o1_sh = dk.stride_h;
  // D = 256: list B's first half is the dV pass, its second half the dK pass
  AttnArgs ak2 = ak;
  if (D == 256) {
    ak.part = 1;
    ak2.part = 2;
    ak2.next_slot = kHdrNextB2;
  }
  AttnArgs aq = a;
  aq.units = unitsA; aq.units_slot = kHdrUnitsA; aq.next_slot = kHdrNextA;
  aq.o0 = dq.ptr; aq.o0_st = dq.stride_t; aq.o0_sh = dq.stride_h;
  const int grid = static_cast<int>(std::min<int64_t>(c.dev.sm_count, std::max(capA, capB)));
  BwdMaps m;
  m.k = m_k128; m.v = m_v128; m.q = m_q64; m.dout = m_do64; m.ds = m_ds;
  // whole key tiles of dK / dV leave through TMA stores
  const hstu_ten_t dkx = hk ? dk : dq, dvx = hk ? dv : dq;
  if (!encode_thd(&m.dk, dkx.ptr, hk ? total_k : total_q, H, D, dkx.stride_t, dkx.stride_h, kBM,
                  c.bf16) ||
      !encode_thd(&m.dv, dvx.ptr, hk ? total_k : total_q, H, D, dvx.stride_t, dvx.stride_h, kBM,
                  c.bf16))
    return HSTU_ERR_CUDA;
  if (launch_bwd(kernel_dim(D), c.bf16, grid, stream, em.pdl(), m, ak, ak2, aq) != cudaSuccess)
    return HSTU_ERR_CUDA;
  if (!em.mark(2, stream) || !em.mark(3, stream)) return HSTU_ERR_CUDA;
  return HSTU_OK;
}

}  // namespace

extern "C" {

hstu_status_t hstu_attn_fwd(hstu_cten_t q, hstu_cten_t k, hstu_cten_t v, hstu_ten_t out,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            int32_t batch, int64_t total_q, int64_t total_k, int32_t num_heads,
                            int32_t head_dim, hstu_dtype_t dtype, int32_t max_seqlen_q,
                            int32_t max_seqlen_k, float alpha, int32_t scaling_seqlen,
                            int32_t window_left, int32_t window_right, void* workspace,
                            size_t workspace_bytes,
                            cudaStream_t stream) {
  return fwd_impl(q, k, v, out, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, num_heads,
                  head_dim, dtype, max_seqlen_q, max_seqlen_k, alpha, scaling_seqlen, window_left,
                  window_right,
                  workspace, workspace_bytes, stream, EventMarks{nullptr, 0});
}

hstu_status_t hstu_attn_fwd_profiled(hstu_cten_t q, hstu_cten_t k, hstu_cten_t v, hstu_ten_t out,
                                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                     int32_t batch, int64_t total_q, int64_t total_k,
                                     int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
                                     int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
                                     int32_t scaling_seqlen, int32_t window_left,
                                     int32_t window_right,
                       void* workspace,
                                     size_t workspace_bytes, cudaStream_t stream,
                                     cudaEvent_t* events, int32_t n_events) {
  if (events == nullptr || n_events < 0) return HSTU_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, out, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, num_heads,
                  head_dim, dtype, max_seqlen_q, max_seqlen_k, alpha, scaling_seqlen, window_left,
                  window_right,
                  workspace, workspace_bytes, stream, EventMarks{events, n_events});
}

hstu_status_t hstu_attn_bwd(hstu_cten_t dout, hstu_cten_t q, hstu_cten_t k, hstu_cten_t v,
                            hstu_ten_t dq, hstu_ten_t dk, hstu_ten_t dv,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            int32_t batch, int64_t total_q, int64_t total_k, int32_t num_heads,
                            int32_t head_dim, hstu_dtype_t dtype, int32_t max_seqlen_q,
                            int32_t max_seqlen_k, float alpha, int32_t scaling_seqlen,
                            int32_t window_left, int32_t window_right, void* workspace,
                            size_t workspace_bytes,
                            cudaStream_t stream) {
  return bwd_impl(dout, q, k, v, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                  num_heads, head_dim, dtype, max_seqlen_q, max_seqlen_k, alpha, scaling_seqlen,
                  window_left, window_right, workspace, workspace_bytes, stream,
                  EventMarks{nullptr, 0});
}

hstu_status_t hstu_attn_bwd_profiled(hstu_cten_t dout, hstu_cten_t q, hstu_cten_t k,
                                     hstu_cten_t v, hstu_ten_t dq, hstu_ten_t dk, hstu_ten_t dv,
                                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                     int32_t batch, int64_t total_q, int64_t total_k,
                                     int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
                                     int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
                                     int32_t scaling_seqlen, int32_t window_left,
                                     int32_t window_right,
                       void* workspace,
                                     size_t workspace_bytes, cudaStream_t stream,
                                     cudaEvent_t* events, int32_t n_events) {
  if (events == nullptr || n_events < 0) return HSTU_ERR_INVALID_ARG;
  return bwd_impl(dout, q, k, v, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                  num_heads, head_dim, dtype, max_seqlen_q, max_seqlen_k, alpha, scaling_seqlen,
                  window_left, window_right, workspace, workspace_bytes, stream,
                  EventMarks{events, n_events});
}

hstu_status_t hstu_attn_plan(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                             int32_t batch, int64_t total_q, int64_t total_k, int32_t num_heads,
                             int32_t head_dim, int32_t max_seqlen_q, int32_t max_seqlen_k,
                             int32_t window_left, int32_t window_right, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
  Common c;
  // the dtype, alpha and L_scale do not enter a schedule: any valid ones
  hstu_status_t s = check_common(batch, total_q, total_k, num_heads, head_dim, HSTU_BF16,
                                 max_seqlen_q, max_seqlen_k, 1.f, 0, window_left, window_right,
                                 cu_seqlens_q, cu_seqlens_k, &c);
  if (s != HSTU_OK) return s;
  if (batch == 0 || (total_q == 0 && total_k == 0)) return HSTU_OK;  // planned calls do nothing
  const int H = num_heads, D = head_dim;
  BwdLayout lay;
  if (!bwd_layout(batch, total_q, total_k, H, D, max_seqlen_q, &lay)) return HSTU_ERR_UNSUPPORTED;
  const size_t need =
      hstu_attn_plan_workspace_size(batch, total_q, total_k, H, D, max_seqlen_q, max_seqlen_k);
  if (need == 0) return HSTU_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < need) return HSTU_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return HSTU_ERR_MISALIGNED;
  if (!device_info(&c.dev)) return HSTU_ERR_CUDA;
  if (c.dev.major != 10 || c.dev.minor != 3) return HSTU_ERR_UNSUPPORTED;

  const int BN = kDsKeys, BNF = bn_for(D);
  const int BQ = DkdvCfg<128, kPassBoth>::BQ;
  const int64_t capA = cap_a(batch, total_q, H), capB = cap_b(batch, total_k, H, D);
  const int cmaxA = static_cast<int>(std::max<int64_t>(1, cdiv(max_seqlen_k, BN)));
  const int cmaxB = static_cast<int>(std::max<int64_t>(1, cdiv(max_seqlen_q, BQ)));
  const int cmaxF = static_cast<int>(std::max<int64_t>(1, cdiv(max_seqlen_k, BNF)));
  int sched_bytes, sched_cache, sched_stage;
  if (!sched_smem(std::max(cmaxF, std::max(cmaxA, cmaxB)), batch, std::max(capA, capB), c.dev,
                  &sched_bytes, &sched_cache, &sched_stage))
    return HSTU_ERR_UNSUPPORTED;
  char* ws = static_cast<char*>(workspace);
  SchedArgs sa{};
  sa.cu_q = cu_seqlens_q; sa.cu_k = cu_seqlens_k; sa.B = batch; sa.H = H; sa.win = c.win;
  sa.bn_a = BN; sa.cmax_a = cmaxA; sa.cap_a = static_cast<int>(capA);
  sa.units_a = reinterpret_cast<int4*>(ws + kHeaderBytes);
  sa.bq_b = BQ; sa.split_b = D == 256 ? 2 : 1; sa.cmax_b = cmaxB; sa.cap_b = static_cast<int>(capB);
  sa.units_b = reinterpret_cast<int4*>(ws + lay.units_b);
  sa.bn_f = BNF; sa.cmax_f = cmaxF; sa.cap_f = static_cast<int>(capA);
  sa.units_f = reinterpret_cast<int4*>(ws + plan_list_f(lay));
  sa.header = reinterpret_cast<int*>(ws);
  sa.ds_base = reinterpret_cast<int*>(ws + lay.ds_base);
  sa.ready = reinterpret_cast<int*>(ws + lay.ready);
  sa.ds_cap = static_cast<int>(lay.ds_blocks);
  sa.cache_seqs = sched_cache;
  sa.stage_units = sched_stage;
  plan_key(batch, total_q, total_k, H, D, max_seqlen_q, max_seqlen_k, c.win, sa.key);
  return launch_sched(3, sched_bytes, stream, true, sa) == cudaSuccess ? HSTU_OK : HSTU_ERR_CUDA;
}

hstu_status_t hstu_attn_fwd_planned(hstu_cten_t q, hstu_cten_t k, hstu_cten_t v, hstu_ten_t out,
                                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                    int32_t batch, int64_t total_q, int64_t total_k,
                                    int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
                                    int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
                                    int32_t scaling_seqlen, int32_t window_left,
                                    int32_t window_right, void* plan, size_t plan_bytes,
                                    cudaStream_t stream) {
  return fwd_impl(q, k, v, out, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, num_heads,
                  head_dim, dtype, max_seqlen_q, max_seqlen_k, alpha, scaling_seqlen, window_left,
                  window_right, plan, plan_bytes, stream, EventMarks{nullptr, 0}, nullptr, nullptr,
                  true);
}

hstu_status_t hstu_attn_bwd_planned(hstu_cten_t dout, hstu_cten_t q, hstu_cten_t k, hstu_cten_t v,
                                    hstu_ten_t dq, hstu_ten_t dk, hstu_ten_t dv,
                                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                    int32_t batch, int64_t total_q, int64_t total_k,
                                    int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
                                    int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
                                    int32_t scaling_seqlen, int32_t window_left,
                                    int32_t window_right, void* plan, size_t plan_bytes,
                                    cudaStream_t stream) {
  return bwd_impl(dout, q, k, v, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                  num_heads, head_dim, dtype, max_seqlen_q, max_seqlen_k, alpha, scaling_seqlen,
                  window_left, window_right, plan, plan_bytes, stream, EventMarks{nullptr, 0},
                  nullptr, true);
}

hstu_status_t hstu_attn_last_device_status(const void* workspace, cudaStream_t stream) {
  if (workspace == nullptr) return HSTU_ERR_INVALID_ARG;
  int h[16];
  if (cudaMemcpyAsync(h, workspace, sizeof(h), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return HSTU_ERR_CUDA;
  if (h[kHdrStatus] != 0) return static_cast<hstu_status_t>(h[kHdrStatus]);
  if (h[kHdrOverflow] != 0 || h[kHdrOverflowB] != 0 || h[kHdrOverflowF] != 0)
    return HSTU_ERR_INVALID_ARG;
  return HSTU_OK;
}

hstu_status_t hstu_attn_selftest_timeout(void* workspace, uint32_t timeout_us, cudaStream_t stream) {
  if (workspace == nullptr || timeout_us == 0 || timeout_us > 10000000u) return HSTU_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return HSTU_ERR_MISALIGNED;
  if (launch_selftest_timeout(static_cast<int*>(workspace), uint64_t(timeout_us) * 1000u, stream) !=
      cudaSuccess)
    return HSTU_ERR_CUDA;
  return HSTU_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- no-allocation forward
// Some callers cannot allocate device memory when they call us: for example a
// plugin inside an inference engine whose execute hook only receives buffers
// the engine planned in advance, or a service that fixes its device-memory
// budget at start-up and forbids allocation afterwards.  Such a caller cannot
// provide the workspace hstu_attn_fwd asks for.  This variant keeps that
// workspace (the tile schedule and the status words) in a fixed-size array
// in the library's own device memory instead; every GPU that loads the
// library holds one such array until the process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(2) << 20;  // 2 MiB: up to 65,528 work units
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (host code may not use the symbol's name as a device pointer).
bool noalloc_scratch(void** out) {
  static void* ptr[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(mu);
  if (ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return false;
    ptr[dev] = p;
  }
  *out = ptr[dev];
  return true;
}

}  // namespace

extern "C" hstu_status_t hstu_attn_fwd_func(
    hstu_cten_t q, hstu_cten_t k, hstu_cten_t v, hstu_ten_t out, const int32_t* cu_seqlens_q,
    const int32_t* cu_seqlens_k, int32_t batch, int64_t total_q, int64_t total_k,
    int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype, int32_t max_seqlen_q,
    int32_t max_seqlen_k, float alpha, int32_t scaling_seqlen, const int32_t* func, int32_t func_n,
    int64_t func_len, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  const FuncArgs fn{func, func_n, func_len};
  return fwd_impl(q, k, v, out, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, num_heads,
                  head_dim, dtype, max_seqlen_q, max_seqlen_k, alpha, scaling_seqlen, -1, -1,
                  workspace, workspace_bytes, stream, EventMarks{nullptr, 0}, nullptr, &fn);
}

extern "C" hstu_status_t hstu_attn_bwd_func(
    hstu_cten_t dout, hstu_cten_t q, hstu_cten_t k, hstu_cten_t v, hstu_ten_t dq, hstu_ten_t dk,
    hstu_ten_t dv, const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
    int64_t total_q, int64_t total_k, int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
    int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha, int32_t scaling_seqlen,
    const int32_t* func, int32_t func_n, int64_t func_len, void* workspace,
    size_t workspace_bytes, cudaStream_t stream) {
  const FuncArgs fn{func, func_n, func_len};
  return bwd_impl(dout, q, k, v, dq, dk, dv, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k,
                  num_heads, head_dim, dtype, max_seqlen_q, max_seqlen_k, alpha, scaling_seqlen,
                  -1, -1, workspace, workspace_bytes, stream, EventMarks{nullptr, 0}, &fn);
}

extern "C" hstu_status_t hstu_attn_fwd_paged(
    hstu_cten_t q, const void* paged_kv, int64_t num_pages, const int32_t* page_ids,
    const int32_t* page_indptrs, hstu_ten_t out, const int32_t* cu_seqlens_q,
    const int32_t* cu_seqlens_k, int32_t batch, int64_t total_q, int32_t num_heads,
    int32_t head_dim, hstu_dtype_t dtype, int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
    int32_t scaling_seqlen, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (paged_kv == nullptr) return HSTU_ERR_INVALID_ARG;
  const PagedKV pg{paged_kv, num_pages, page_ids, page_indptrs};
  const hstu_cten_t none{nullptr, 0, 0};
  // causal only; total_k bounds the keys the pages can hold
  return fwd_impl(q, none, none, out, cu_seqlens_q, cu_seqlens_k, batch, total_q,
                  num_pages * 128, num_heads, head_dim, dtype, max_seqlen_q, max_seqlen_k, alpha,
                  scaling_seqlen, -1, 0, workspace, workspace_bytes, stream,
                  EventMarks{nullptr, 0}, &pg);
}

extern "C" hstu_status_t hstu_attn_fwd_noalloc(
    hstu_cten_t q, hstu_cten_t k, hstu_cten_t v, hstu_ten_t out, const int32_t* cu_seqlens_q,
    const int32_t* cu_seqlens_k, int32_t batch, int64_t total_q, int64_t total_k,
    int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype, int32_t max_seqlen_q,
    int32_t max_seqlen_k, float alpha, int32_t scaling_seqlen, int32_t window_left,
    int32_t window_right,
    cudaStream_t stream) {
  const size_t need = hstu_attn_workspace_size(batch, total_q, total_k, num_heads, head_dim,
                                               max_seqlen_q, max_seqlen_k, 0);
  if (need == 0) return supported_dim(head_dim) ? HSTU_ERR_INVALID_ARG : HSTU_ERR_UNSUPPORTED;
  if (need > kNoAllocScratchBytes) return HSTU_ERR_INVALID_ARG;  // schedule would not fit
  void* scratch = nullptr;
  if (!noalloc_scratch(&scratch)) return HSTU_ERR_CUDA;
  // The scheduler kernel rewrites the header and the whole work list at the
  // start of every call, so nothing in the array has to be cleared first.
  return fwd_impl(q, k, v, out, cu_seqlens_q, cu_seqlens_k, batch, total_q, total_k, num_heads,
                  head_dim, dtype, max_seqlen_q, max_seqlen_k, alpha, scaling_seqlen, window_left,
                  window_right,
                  scratch, kNoAllocScratchBytes, stream, EventMarks{nullptr, 0});
}

// The status words of the no-allocation forward live in the same fixed
// array, so the caller cannot name them; this reads them the way
// hstu_attn_last_device_status reads a workspace's.
extern "C" hstu_status_t hstu_attn_noalloc_last_device_status(cudaStream_t stream) {
  void* scratch = nullptr;
  if (!noalloc_scratch(&scratch)) return HSTU_ERR_CUDA;
  return hstu_attn_last_device_status(scratch, stream);
}
