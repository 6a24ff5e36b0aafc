/*
 * hstu_lmsd.h: C ABI of the GB300 (sm_103a) HSTU LayerNorm-Multiply-SiLU-
 * Dropout (LMSD) kernels, in the same library as hstu_attn.h.
 *
 * Operation (page "HSTU LayerNorm-Multiply-SiLU-Dropout (LMSD)", Overview):
 * for every row of x (N, D),
 *     xhat = (x - mean(x)) rstd,   rstd = 1 / sqrt(var(x) + eps)  (biased var)
 *     l    = xhat * weight + bias
 *     a    = SiLU(u) when apply_u_silu, else u
 *     y    = [dropout(a) if concat_u, dropout(x) if concat_x, dropout(l * a)]
 * Inverted dropout: an element is kept with probability 1 - p and scaled by
 * 1 / (1 - p).  The int8 mask has one byte per input element: bit 0 the
 * mandatory l * a result, bit 1 the x segment, bit 2 the activated-u segment;
 * a set bit means kept; disabled segments leave their bits clear.  With
 * p = 0 no random numbers are drawn and no mask is written.
 *
 * Random numbers: Philox4x32-10 (Salmon et al., SC 2011), one call per 8
 * elements.  The element at flat index e = row * D + col of segment k
 * (0 main, 1 x, 2 u) is decided by the 16-bit half e % 2 (0 = low) of word
 * (e % 8) / 2 of Philox(counter = (e / 8 mod 2^32, e / 8 >> 32, k, 0),
 * key = (seed mod 2^32, seed >> 32)) and kept iff that half is at least
 * floor(p * 2^16), so the drop rate is p to within 2^-16.  (The page fixes
 * Philox but not the counter layout; this one is a reading.)
 *
 * Backward (chain rule; the page gives the API): with s_k = mask bit k /
 * (1 - p), or 1 when p = 0,
 *     dm = dy_main s_0,  dl = dm a,  da = dm l + dy_u s_2 (if concat_u)
 *     du = da SiLU'(u) (if apply_u_silu) else da
 *     dx = rstd (dl w - mean(dl w) - xhat mean(dl w xhat)) + dy_x s_1 (if concat_x)
 *     dweight = sum over rows of dl xhat,  dbias = sum over rows of dl,
 * the sums reduced in a fixed order (deterministic).
 *
 * Layout (same page, "Tensor shapes and layouts"): all tensors BF16 except
 * mean, rstd (fp32) and mask (int8); D divisible by 8 with 8 <= D < 1024;
 * N * D <= 2^31.  x, u, dx, du: (N, D) with a row stride (in elements) >= D;
 * y: contiguous (N, S * D), S = 1 + concat_u + concat_x; dy: (N, S * D) with
 * a row stride >= S * D; weight, bias, dweight, dbias: (D,); mean, rstd:
 * (N,); mask: contiguous (N, D).  Every pointer and every row (stride * 2
 * bytes) 16-byte aligned.  All pointers are device pointers; outputs must not
 * overlap inputs or one another.  Calls are asynchronous on `stream`; the
 * library allocates nothing (the backward takes a caller-owned workspace).
 */
#ifndef HSTU_LMSD_H_
#define HSTU_LMSD_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HSTU_LMSD_OK = 0,
  HSTU_LMSD_ERR_INVALID_ARG = 1,   /* null pointers, p outside [0, 1), eps <= 0, short strides,
                                      workspace too small */
  HSTU_LMSD_ERR_UNSUPPORTED = 2,   /* D outside 8..1016 or not a multiple of 8, N D > 2^31 */
  HSTU_LMSD_ERR_MISALIGNED = 3,    /* a pointer or row not 16-byte aligned */
  HSTU_LMSD_ERR_CUDA = 4           /* a launch failed */
} hstu_lmsd_status_t;

/*
 * Forward.  dropout_ratio is taken as fp32 and must lie in [0, 1); mask may
 * be NULL when it is 0.  n == 0 is a no-op returning HSTU_LMSD_OK.
 */
hstu_lmsd_status_t hstu_lmsd_fwd(const void* x, int64_t x_stride, const void* u,
                                 int64_t u_stride, const void* weight, const void* bias,
                                 int64_t n, int32_t d, float eps, float dropout_ratio,
                                 int32_t apply_u_silu, int32_t concat_u, int32_t concat_x,
                                 int64_t seed, void* y, float* mean, float* rstd, int8_t* mask,
                                 cudaStream_t stream);

/* Workspace bytes of hstu_lmsd_bwd (fp32 column partials), 0 for bad sizes. */
size_t hstu_lmsd_bwd_workspace_size(int64_t n, int32_t d);

/*
 * Backward.  Forward and backward must use the same dropout_ratio,
 * apply_u_silu, concat_u, concat_x, saved mean/rstd and mask (the page's
 * rule).  compute_dweight = 0 skips writing dweight (which may then be NULL).
 */
hstu_lmsd_status_t hstu_lmsd_bwd(const void* dy, int64_t dy_stride, const void* x,
                                 int64_t x_stride, const void* u, int64_t u_stride,
                                 const void* weight, const void* bias, const float* mean,
                                 const float* rstd, const int8_t* mask, int64_t n, int32_t d,
                                 float dropout_ratio, int32_t apply_u_silu, int32_t concat_u,
                                 int32_t concat_x, int32_t compute_dweight, void* dx,
                                 int64_t dx_stride, void* du, int64_t du_stride, void* dweight,
                                 void* dbias, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* HSTU_LMSD_H_ */
