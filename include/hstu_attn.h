/*
 * hstu_attn.h: C ABI of the GB300 (sm_103a) HSTU attention library.
 *
 * Operation ("HSTU Attention (Blackwell SM100/SM103)", section Overview):
 * for every packed sequence and head h,
 *     S_h = alpha * Q_h K_h^T
 *     A_h = (1 / L_scale) * (M (.) SiLU(S_h))
 *     O_h = A_h V_h
 * with no row softmax; the heads' outputs are concatenated.  The backward
 * returns dQ, dK, dV from dO (same page, section "High-level functions"):
 *     dV = A^T dO,   dS = M (.) (dO V^T) (.) SiLU'(S) / L_scale,
 *     dQ = alpha dS K,   dK = alpha dS^T Q.
 *
 * Layout (same page, section "Tensor layout"): packed variable-length THD
 * tensors.  q, dO, out, dq are (T_q, H, D); k, v, dk, dv are (T_k, H, D);
 * all share one dtype, FP16 or BF16.  cu_seqlens_q / cu_seqlens_k are int32
 * (B + 1,) cumulative lengths starting at 0 that delimit each sequence.
 * Q, K and V have the same number of heads (MHA only: no GQA/MQA).
 *
 * Mask (same page, section "Mask support"): the token window
 * window_size = (window_left, window_right), -1 meaning no bound on that
 * side.  Key j is valid for query i (indices local to the sequence) iff
 * j >= i - window_left (when window_left >= 0) and j <= i + window_right
 * (when window_right >= 0), aligned top-left on the diagonal j = i, which is
 * kept.  Causal = window (-1, 0); full = window (-1, -1); finite bounds give
 * the local / sliding window.  Keys outside the sequence never count.  A query row with no valid key gets a zero output and
 * a zero dQ; a key that no query sees gets zero dK and dV (same page, section
 * "Mask support": keyless rows are written as zeros, no output memset needed).
 *
 * Ownership and calling rules, common to every entry point:
 *  - The caller owns every buffer.  The library never allocates device or
 *    host memory and keeps no per-call state outside the caller's workspace.
 *  - All tensor pointers and cu_seqlens are DEVICE pointers.  Their values
 *    (cu_seqlens) are trusted and never copied to the host (same page,
 *    section "Tensor layout").  Work is enqueued asynchronously on `stream`.
 *  - Outputs are overwritten; every logical output element is written.
 *  - Each tensor is described by a base pointer and two element strides
 *    (token, head); the last (D) dimension is contiguous.  Base pointers and
 *    both strides (in bytes) must be multiples of 16 (the page requires
 *    16-byte aligned bases; the strides feed the tensor-memory-access unit).
 *    A tensor's strides must not map two logical elements to one address.
 *    Storage spans of distinct tensors are not compared: outputs must not
 *    overlap live inputs.  dk and dv may be disjoint views of one packed KV
 *    allocation (same page, section "High-level functions").
 *  - Return codes: HSTU_OK, or an error with nothing enqueued (argument
 *    errors) or with a launch error (HSTU_ERR_CUDA).
 */
#ifndef HSTU_ATTN_H_
#define HSTU_ATTN_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HSTU_OK = 0,
  HSTU_ERR_INVALID_ARG = 1,    /* bad sizes, null pointers, max_seqlen_q > max_seqlen_k,
                                  scaling_seqlen < 0, non-finite alpha, a window bound
                                  below -1, overlapping strides, workspace too small */
  HSTU_ERR_UNSUPPORTED = 2,    /* head_dim or dtype outside the built set, device not sm_103 */
  HSTU_ERR_MISALIGNED = 3,     /* base pointer or stride not a multiple of 16 bytes */
  HSTU_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed */
  HSTU_ERR_DEVICE_TIMEOUT = 5  /* a kernel wait ran past its limit (read back by
                                  hstu_attn_last_device_status) */
} hstu_status_t;

typedef enum { HSTU_FP16 = 0, HSTU_BF16 = 1 } hstu_dtype_t;

/* Read-only THD tensor: element (t, h, d) is at ptr[t*stride_t + h*stride_h + d]. */
typedef struct {
  const void* ptr;
  int64_t stride_t;
  int64_t stride_h;
} hstu_cten_t;

/* Writable THD tensor, same addressing. */
typedef struct {
  void* ptr;
  int64_t stride_t;
  int64_t stride_h;
} hstu_ten_t;

/*
 * Device workspace size, in bytes, that hstu_attn_fwd (is_bwd = 0) or
 * hstu_attn_bwd (is_bwd = 1) needs for these sizes; pass the same
 * max_seqlen_q / max_seqlen_k as to the call.  The workspace holds the
 * device-built tile schedule and status words, and for the backward the
 * intermediate dS = M (.) (dO V^T) (.) SiLU'(S) in blocks of 128 keys x 64
 * queries (16-bit), bounded from the sizes alone by
 *     num_heads * ceil(max_seqlen_q / 64) * (ceil(total_k / 128) + batch)
 * blocks of 16 KiB (the host never reads the sequence lengths).  It must be
 * 256-byte aligned and may be reused by later calls on the same stream.
 * Returns 0 for invalid sizes, or when the dS block count exceeds 2^31 - 1.
 */
size_t hstu_attn_workspace_size(int32_t batch, int64_t total_q, int64_t total_k,
                                int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q,
                                int32_t max_seqlen_k, int32_t is_bwd);

/*
 * Forward: out = HSTU-MHA(q, k, v) (page "HSTU Attention (Blackwell
 * SM100/SM103)", sections Overview and "High-level functions").
 *   q, out: (total_q, num_heads, head_dim); k, v: (total_k, num_heads, head_dim).
 *   batch B >= 0; cu_seqlens_q/k: device int32 (B+1,), cu[0] = 0,
 *     cu_seqlens_q[B] <= total_q, cu_seqlens_k[B] <= total_k.
 *   max_seqlen_q <= max_seqlen_k, each >= the longest sequence on its side.
 *   alpha: score scale, finite.  scaling_seqlen: L_scale; 0 selects
 *     max_seqlen_q, negative is an error (the page requires it positive).
 *   window_left, window_right: the mask window, each -1 (no bound) or >= 0;
 *     (-1, 0) causal, (-1, -1) full; a bound below -1 is an error.
 *   head_dim in {32, 64, 128, 256} (32 runs on the 64-wide kernels with the
 *     head dimension zero-padded on chip); dtype FP16 or BF16.
 * B == 0 or total_q == 0 is a no-op returning HSTU_OK.
 */
hstu_status_t hstu_attn_fwd(hstu_cten_t q, hstu_cten_t k, hstu_cten_t v, hstu_ten_t out,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            int32_t batch, int64_t total_q, int64_t total_k,
                            int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
                            int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
                            int32_t scaling_seqlen, int32_t window_left,
                            int32_t window_right, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/*
 * Backward: (dq, dk, dv) from dout (page "HSTU Attention (Blackwell
 * SM100/SM103)", section "High-level functions").  Arguments as for the
 * forward, which must have used the same alpha, scaling_seqlen, mask and
 * sequence metadata.  dout, dq: (total_q, H, D); dk, dv: (total_k, H, D).
 * No forward output or statistic is needed: S is recomputed.  A key-stationary
 * kernel forms dK, dV and the dS blocks (stored in the workspace); a second
 * kernel reduces dQ = alpha dS K per query tile without atomics, so results
 * do not depend on scheduling.  A sequence longer than max_seqlen_q makes the
 * dS blocks overflow the workspace: the stores past its end are skipped and
 * hstu_attn_last_device_status reports HSTU_ERR_INVALID_ARG.
 */
hstu_status_t hstu_attn_bwd(hstu_cten_t dout, hstu_cten_t q, hstu_cten_t k, hstu_cten_t v,
                            hstu_ten_t dq, hstu_ten_t dk, hstu_ten_t dv,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            int32_t batch, int64_t total_q, int64_t total_k,
                            int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
                            int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
                            int32_t scaling_seqlen, int32_t window_left,
                            int32_t window_right, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/*
 * Arbitrary mask (page "HSTU Attention (Blackwell SM100/SM103)", section
 * "Mask support", func_tensor): forward and backward with the same arguments
 * as hstu_attn_fwd / hstu_attn_bwd, the window replaced by
 *   func: device int32 endpoints, row n of query token t at
 *     func[n * func_len + t] (the page's (1, N, L) tensor); func_n = N, odd,
 *     >= 1; func_len = L >= total_q (the page's 256 padding columns are
 *     accepted and unused).  Query token t's valid keys are
 *     [0, F0) U [F1, F2) U [F3, F4) ... of its endpoints F_n (key indices
 *     local to the sequence; intervals may overlap or come in any order),
 *     cut to the sequence's keys.  Values are trusted and never copied to
 *     the host.
 *   workspace: hstu_attn_workspace_size_func(...) bytes (the regular size
 *     plus the per-tile key and query ranges and live-tile bitmaps the
 *     library derives from the endpoints on every call, so in-place changes
 *     of func are seen, also under CUDA graph replay).
 * Each unit visits the live tiles of the hull its rows can see (a tile is
 * live when some row of a 64-row query block sees one of its 128 keys) and
 * applies the exact predicate inside them.  Errors as for hstu_attn_fwd/_bwd, plus
 * HSTU_ERR_INVALID_ARG for an even or non-positive func_n or
 * func_len < total_q, HSTU_ERR_MISALIGNED for a func pointer that is not
 * 4-byte aligned.
 */
size_t hstu_attn_workspace_size_func(int32_t batch, int64_t total_q, int64_t total_k,
                                     int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q,
                                     int32_t max_seqlen_k, int32_t is_bwd);
hstu_status_t hstu_attn_fwd_func(hstu_cten_t q, hstu_cten_t k, hstu_cten_t v, hstu_ten_t out,
                                 const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                 int32_t batch, int64_t total_q, int64_t total_k,
                                 int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
                                 int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
                                 int32_t scaling_seqlen, const int32_t* func, int32_t func_n,
                                 int64_t func_len, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);
hstu_status_t hstu_attn_bwd_func(hstu_cten_t dout, hstu_cten_t q, hstu_cten_t k, hstu_cten_t v,
                                 hstu_ten_t dq, hstu_ten_t dk, hstu_ten_t dv,
                                 const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                 int32_t batch, int64_t total_q, int64_t total_k,
                                 int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
                                 int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
                                 int32_t scaling_seqlen, const int32_t* func, int32_t func_n,
                                 int64_t func_len, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/*
 * Forward over a paged K/V cache (page "HSTU Attention (Blackwell
 * SM100/SM103)", section "Mask support", paged-KV paragraph; the page's
 * paged path is causal only and has no backward, and so has this one).
 *   paged_kv: device, contiguous (num_pages, 2, 128, num_heads, head_dim) in
 *     dtype, 16-byte aligned; [p][0] holds K and [p][1] V of 128 consecutive
 *     keys.  num_pages > 0.
 *   page_ids: device int32; page_indptrs: device int32 (batch + 1,).  Key j
 *     of sequence b lives in row j % 128 of page
 *     page_ids[page_indptrs[b] + j / 128].  Values are trusted (never copied to
 *     the host, never range-checked), as the page requires.
 *   cu_seqlens_k: its differences give each sequence's key count Lk_b (its
 *     offsets are not used: the storage is the pages).  max_seqlen_k >= every
 *     Lk_b, max_seqlen_q <= max_seqlen_k.
 *   Rows of a page past its sequence's last key are multiplied by exact
 *     zeros, so they must hold finite values (NaN or Inf there would leak).
 *   Other arguments as for hstu_attn_fwd with window (-1, 0); workspace:
 *     hstu_attn_workspace_size(batch, total_q, 0, num_heads, head_dim,
 *     max_seqlen_q, max_seqlen_k, 0) bytes.
 */
hstu_status_t hstu_attn_fwd_paged(hstu_cten_t q, const void* paged_kv, int64_t num_pages,
                                  const int32_t* page_ids, const int32_t* page_indptrs,
                                  hstu_ten_t out, const int32_t* cu_seqlens_q,
                                  const int32_t* cu_seqlens_k, int32_t batch, int64_t total_q,
                                  int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
                                  int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
                                  int32_t scaling_seqlen, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream);

/*
 * Profiling variants: identical to hstu_attn_fwd / hstu_attn_bwd (same
 * arguments, results and errors), and they additionally record the first
 * `n_events` of these caller-created CUDA events on `stream`:
 *   forward:  events[0] before the scheduler launch, events[1] after it,
 *             events[2] after the forward kernel;
 *   backward: events[0] before the scheduler launch, events[1] after it,
 *             events[2] and events[3] after the backward kernel (dK/dV then dQ units
 *             in one launch; the two are recorded back to back).
 * Elapsed times between consecutive events are per-kernel device times.
 * events must be non-null (HSTU_ERR_INVALID_ARG otherwise).
 */
hstu_status_t hstu_attn_fwd_profiled(hstu_cten_t q, hstu_cten_t k, hstu_cten_t v, hstu_ten_t out,
                                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                     int32_t batch, int64_t total_q, int64_t total_k,
                                     int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
                                     int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
                                     int32_t scaling_seqlen, int32_t window_left,
                                     int32_t window_right, void* workspace,
                                     size_t workspace_bytes, cudaStream_t stream,
                                     cudaEvent_t* events, int32_t n_events);
hstu_status_t hstu_attn_bwd_profiled(hstu_cten_t dout, hstu_cten_t q, hstu_cten_t k,
                                     hstu_cten_t v, hstu_ten_t dq, hstu_ten_t dk, hstu_ten_t dv,
                                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                     int32_t batch, int64_t total_q, int64_t total_k,
                                     int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
                                     int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
                                     int32_t scaling_seqlen, int32_t window_left,
                                     int32_t window_right, void* workspace,
                                     size_t workspace_bytes, cudaStream_t stream,
                                     cudaEvent_t* events, int32_t n_events);

/*
 * Forward without a workspace argument; it allocates nothing.  The pages
 * have no counterpart: it exists for callers that cannot allocate device
 * memory when they call in (e.g. a plugin of an inference engine whose
 * execute hook only gets buffers planned ahead, or a service that fixes its
 * memory budget at start-up) and so cannot pass the workspace hstu_attn_fwd
 * needs.  Arguments and results are those of hstu_attn_fwd; the caller still
 * passes every input and output.
 *
 * The schedule lives in a 2 MiB array in the library's own device memory
 * (one per GPU that loads the library, held until exit).  Problems whose
 * schedule exceeds it, hstu_attn_workspace_size(..., is_bwd = 0) > 2 MiB,
 * i.e. more than 65,528 work units (num_heads * (ceil(total_q / 128) + batch)),
 * return HSTU_ERR_INVALID_ARG.  The first call on a device looks the array's
 * address up (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  All calls share the one array and each
 * call rewrites it from the start, so calls that can overlap on the GPU (for
 * example on two streams) race: serialize them.  Uses no cudaMalloc, no
 * cudaFree and no allocating library routine.
 */
hstu_status_t hstu_attn_fwd_noalloc(hstu_cten_t q, hstu_cten_t k, hstu_cten_t v, hstu_ten_t out,
                                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                    int32_t batch, int64_t total_q, int64_t total_k,
                                    int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
                                    int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
                                    int32_t scaling_seqlen, int32_t window_left,
                                    int32_t window_right, cudaStream_t stream);

/*
 * Device-side status of the most recent hstu_attn_fwd_noalloc call on the
 * current device, in the order of `stream`: the same report as
 * hstu_attn_last_device_status gives for a workspace (HSTU_OK, or
 * HSTU_ERR_INVALID_ARG for metadata past the sizes, HSTU_ERR_DEVICE_TIMEOUT
 * for a wait that gave up), read from the library's fixed array, which the
 * caller cannot name.  Copies 64 bytes to the host and synchronizes
 * `stream`: for debugging and tests, not for the hot path.  The pages have
 * no counterpart.
 */
hstu_status_t hstu_attn_noalloc_last_device_status(cudaStream_t stream);

/*
 * Plans: one schedule for every call on one batch layout.
 *
 * A training step runs the forward and the backward of every layer on the
 * same packed batch, and the work lists (the tiles of every sequence, sorted
 * longest first) depend only on the layout: cu_seqlens, the sizes and the
 * window.  hstu_attn_plan builds the forward's and the backward's lists in
 * one launch; hstu_attn_fwd_planned / hstu_attn_bwd_planned then start their
 * kernels directly, with no scheduling launch of their own.  Results are
 * those of hstu_attn_fwd / hstu_attn_bwd, bit for bit.
 *
 *   workspace (the plan): hstu_attn_plan_workspace_size(...) bytes,
 *     256-byte aligned, caller-owned; it also serves as the backward's
 *     workspace (dS blocks).  Returns 0 for invalid or unsupported sizes.
 *   hstu_attn_plan: reads cu_seqlens on the device; arguments and errors as
 *     for hstu_attn_bwd (without the tensors, dtype, alpha or
 *     scaling_seqlen, which do not enter a schedule).
 *   hstu_attn_fwd_planned / hstu_attn_bwd_planned: the arguments of
 *     hstu_attn_fwd / hstu_attn_bwd, with the plan as the workspace.  Their
 *     cu_seqlens must hold the values the plan was built from; their sizes
 *     (batch, totals, heads, head_dim, max_seqlen_q/k, window) must be the
 *     plan's: each kernel compares them with those the plan recorded and, if
 *     they differ, writes nothing and records HSTU_ERR_INVALID_ARG for
 *     hstu_attn_last_device_status.  Arbitrary masks and paged K/V are not
 *     planned.
 * Any number of planned calls may share a plan, in stream order (each
 * kernel leaves the plan ready for the next).  Calls sharing a plan on
 * different streams race: serialize them.  After a device-side error
 * (HSTU_ERR_DEVICE_TIMEOUT) build the plan again.
 */
size_t hstu_attn_plan_workspace_size(int32_t batch, int64_t total_q, int64_t total_k,
                                     int32_t num_heads, int32_t head_dim, int32_t max_seqlen_q,
                                     int32_t max_seqlen_k);
hstu_status_t hstu_attn_plan(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                             int32_t batch, int64_t total_q, int64_t total_k, int32_t num_heads,
                             int32_t head_dim, int32_t max_seqlen_q, int32_t max_seqlen_k,
                             int32_t window_left, int32_t window_right, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream);
hstu_status_t hstu_attn_fwd_planned(hstu_cten_t q, hstu_cten_t k, hstu_cten_t v, hstu_ten_t out,
                                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                    int32_t batch, int64_t total_q, int64_t total_k,
                                    int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
                                    int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
                                    int32_t scaling_seqlen, int32_t window_left,
                                    int32_t window_right, void* plan, size_t plan_bytes,
                                    cudaStream_t stream);
hstu_status_t hstu_attn_bwd_planned(hstu_cten_t dout, hstu_cten_t q, hstu_cten_t k, hstu_cten_t v,
                                    hstu_ten_t dq, hstu_ten_t dk, hstu_ten_t dv,
                                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                    int32_t batch, int64_t total_q, int64_t total_k,
                                    int32_t num_heads, int32_t head_dim, hstu_dtype_t dtype,
                                    int32_t max_seqlen_q, int32_t max_seqlen_k, float alpha,
                                    int32_t scaling_seqlen, int32_t window_left,
                                    int32_t window_right, void* plan, size_t plan_bytes,
                                    cudaStream_t stream);

/* Static text for a status code. */
const char* hstu_attn_status_string(hstu_status_t status);

/*
 * Synchronizes `stream` and returns the device-side status that the last
 * call using `workspace` recorded: HSTU_OK, or HSTU_ERR_DEVICE_TIMEOUT when a
 * kernel gave up a wait (it then wrote no further output and exited).
 * For tests and debugging; costs a stream synchronization.
 */
hstu_status_t hstu_attn_last_device_status(const void* workspace, cudaStream_t stream);

/*
 * Self-test of the bounded-wait machinery: launches one block that waits on
 * a barrier nothing will ever complete, with a limit of `timeout_us`
 * microseconds (1..10,000,000).  The kernel records HSTU_ERR_DEVICE_TIMEOUT in
 * `workspace` and returns; no fault, no hang.  Read the result with
 * hstu_attn_last_device_status.  workspace: >= 256 bytes, device.
 */
hstu_status_t hstu_attn_selftest_timeout(void* workspace, uint32_t timeout_us,
                                         cudaStream_t stream);

/* Library version, e.g. 100 for 0.1.0. */
int32_t hstu_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HSTU_ATTN_H_ */
