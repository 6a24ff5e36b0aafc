/*
 * HSTU attention: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker that the CUDA path is
 * compared against.  Only the tests, the smoke check and the benchmark's CPU
 * baseline / reference arm may build, load or call it.  It shares no code,
 * header, table or helper with the CUDA library.
 *
 * What it computes ("HSTU Attention (Blackwell SM100/SM103)", section
 * Overview, the three displayed equations): for every packed sequence b and
 * head h,
 *     S = alpha * Q K^T,
 *     A = (1 / L_scale) * (M (.) SiLU(S)),
 *     O = A V,
 * with no softmax.  Tensors are packed THD, (T, H, D) row-major, sequences
 * delimited by cumulative lengths cu_seqlens (same page, section "Tensor
 * layout").  Indices i (query) and j (key) below are local to the sequence.
 *
 * Mask M (same page, section "Mask support"): window_size = (left, right)
 * is the token-window mask, -1 meaning no bound on that side: key j is valid
 * for query i iff j >= i - left (when left >= 0) and j <= i + right (when
 * right >= 0).  Window (-1, 0) is causal, (-1, -1) full, finite bounds the
 * local / sliding window.  The window is read as aligned top-left, on the
 * diagonal j = i (the cuDNN "Attention" page: diagonal_alignment TOP_LEFT
 * with right bound 0 is the standard causal mask), with the diagonal kept.
 * In every mode a key must also lie inside the sequence: j < Lk.  A masked
 * score contributes exactly zero (M multiplies SiLU(S)).
 *
 * Arbitrary mask (same section, func_tensor): with func given (N int32
 * endpoint rows of length func_len, N odd; row n of query token t at
 * func[n * func_len + t]), query token t's valid keys are the union
 * [0, F0) U [F1, F2) U [F3, F4) ... of its endpoints F_n, key indices local
 * to the sequence, each interval taken on its own (they may overlap or come
 * in any order), still cut to j < Lk.  The window is then ignored.
 *
 * Backward: the pages give the API (section "High-level functions") but not
 * the formulas.  They follow from the forward equations by the chain rule:
 *     dV_j  = sum_i A_ij dO_i
 *     dA_ij = <dO_i, v_j>
 *     dS_ij = M_ij * dA_ij * SiLU'(S_ij) / L_scale,
 *             SiLU'(x) = sigma(x) * (1 + x * (1 - sigma(x)))
 *     dQ_i  = alpha * sum_j dS_ij k_j
 *     dK_j  = alpha * sum_i dS_ij q_i
 *
 * Every output row is computed on its own, straight from these sums, in the
 * order they are written; nothing is blocked, fused or reordered.  The row
 * entry points exist so that tests can check sampled rows of large problems.
 * Rows that lie in no sequence (token index >= cu_seqlens[B]) are set to 0.
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC hstu_oracle.c -lm
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* SiLU(x) = x * sigma(x). */
static double silu(double x) { return x * sigmoid(x); }

/* d/dx [x sigma(x)] = sigma(x) + x sigma(x) (1 - sigma(x)). */
static double silu_grad(double x) {
    double s = sigmoid(x);
    return s * (1.0 + x * (1.0 - s));
}

static int mask_valid(int64_t i, int64_t j, int64_t Lk, int left, int right) {
    if (j >= Lk) return 0;
    if (left >= 0 && j < i - left) return 0;
    if (right >= 0 && j > i + right) return 0;
    return 1;
}

/* Arbitrary mask: key j against the endpoints of query token t. */
typedef struct {
    const int32_t *func; /* NULL: the window decides */
    int n;
    int64_t len;
} Func;

static int func_valid(const Func *f, int64_t t, int64_t j, int64_t Lk) {
    if (j >= Lk) return 0;
    if (j < f->func[t]) return 1; /* [0, F0) */
    for (int m = 1; m + 1 < f->n; m += 2) {
        int64_t lo = f->func[(int64_t)m * f->len + t];
        int64_t hi = f->func[(int64_t)(m + 1) * f->len + t];
        if (lo <= j && j < hi) return 1;
    }
    return 0;
}

static int valid(const Func *f, int64_t t, int64_t i, int64_t j, int64_t Lk, int left,
                 int right) {
    return f->func ? func_valid(f, t, j, Lk) : mask_valid(i, j, Lk, left, right);
}

static double dot(const double *a, const double *b, int D) {
    double s = 0.0;
    for (int d = 0; d < D; ++d) s += a[d] * b[d];
    return s;
}

/* Sequence b that holds token t: the last b with cu[b] <= t, and t < cu[b+1].
 * Returns -1 when t lies in no sequence. */
static int64_t find_seq(const int32_t *cu, int64_t B, int64_t t) {
    if (B <= 0 || t < cu[0] || t >= cu[B]) return -1;
    int64_t lo = 0, hi = B; /* invariant: cu[lo] <= t < cu[hi] */
    while (hi - lo > 1) {
        int64_t mid = lo + (hi - lo) / 2;
        if (cu[mid] <= t) lo = mid; else hi = mid;
    }
    return lo;
}

static const double *row(const double *x, int64_t t, int64_t h, int64_t H, int D) {
    return x + (t * H + h) * (int64_t)D;
}

static int set_threads(int threads) {
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
    return omp_get_max_threads();
#else
    (void)threads;
    return 1;
#endif
}

/* Number of threads the next parallel region will use (1 without OpenMP). */
int hstu_oracle_threads(int threads) { return set_threads(threads); }

/* O rows for n (token, head) pairs; out is (n, D). */
int hstu_oracle_fwd_rows(const double *q, const double *k, const double *v,
                         const int32_t *cu_q, const int32_t *cu_k, int64_t B,
                         int64_t H, int D, double alpha, double L_scale,
                         int left, int right,
                         const int32_t *func, int func_n, int64_t func_len,
                         const int64_t *tok, const int64_t *head,
                         int64_t n, double *out, int threads) {
    set_threads(threads);
    const Func f = {func, func_n, func_len};
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < n; ++r) {
        double *o = out + r * (int64_t)D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        int64_t b = find_seq(cu_q, B, tok[r]);
        if (b < 0) continue;
        int64_t h = head[r];
        int64_t i = tok[r] - cu_q[b];
        int64_t ok = cu_k[b], Lk = (int64_t)cu_k[b + 1] - cu_k[b];
        const double *qi = row(q, tok[r], h, H, D);
        for (int64_t j = 0; j < Lk; ++j) {
            if (!valid(&f, tok[r], i, j, Lk, left, right)) continue;
            const double *kj = row(k, ok + j, h, H, D);
            const double *vj = row(v, ok + j, h, H, D);
            double s = alpha * dot(qi, kj, D);
            double a = silu(s) / L_scale;
            for (int d = 0; d < D; ++d) o[d] += a * vj[d];
        }
    }
    return 0;
}

/* dQ rows for n (token, head) pairs of the query side; dq is (n, D). */
int hstu_oracle_dq_rows(const double *dout, const double *q, const double *k,
                        const double *v, const int32_t *cu_q,
                        const int32_t *cu_k, int64_t B, int64_t H, int D,
                        double alpha, double L_scale, int left, int right,
                        const int32_t *func, int func_n, int64_t func_len,
                        const int64_t *tok, const int64_t *head, int64_t n,
                        double *dq, int threads) {
    set_threads(threads);
    const Func f = {func, func_n, func_len};
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < n; ++r) {
        double *g = dq + r * (int64_t)D;
        for (int d = 0; d < D; ++d) g[d] = 0.0;
        int64_t b = find_seq(cu_q, B, tok[r]);
        if (b < 0) continue;
        int64_t h = head[r];
        int64_t i = tok[r] - cu_q[b];
        int64_t ok = cu_k[b], Lk = (int64_t)cu_k[b + 1] - cu_k[b];
        const double *qi = row(q, tok[r], h, H, D);
        const double *doi = row(dout, tok[r], h, H, D);
        for (int64_t j = 0; j < Lk; ++j) {
            if (!valid(&f, tok[r], i, j, Lk, left, right)) continue;
            const double *kj = row(k, ok + j, h, H, D);
            const double *vj = row(v, ok + j, h, H, D);
            double s = alpha * dot(qi, kj, D);
            double dA = dot(doi, vj, D);
            double dS = dA * silu_grad(s) / L_scale;
            for (int d = 0; d < D; ++d) g[d] += alpha * dS * kj[d];
        }
    }
    return 0;
}

/* dK and dV rows for n (token, head) pairs of the key side; (n, D) each. */
int hstu_oracle_dkdv_rows(const double *dout, const double *q, const double *k,
                          const double *v, const int32_t *cu_q,
                          const int32_t *cu_k, int64_t B, int64_t H, int D,
                          double alpha, double L_scale, int left, int right,
                          const int32_t *func, int func_n, int64_t func_len,
                          const int64_t *tok, const int64_t *head, int64_t n,
                          double *dk, double *dv, int threads) {
    set_threads(threads);
    const Func f = {func, func_n, func_len};
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < n; ++r) {
        double *gk = dk + r * (int64_t)D;
        double *gv = dv + r * (int64_t)D;
        for (int d = 0; d < D; ++d) { gk[d] = 0.0; gv[d] = 0.0; }
        int64_t b = find_seq(cu_k, B, tok[r]);
        if (b < 0) continue;
        int64_t h = head[r];
        int64_t j = tok[r] - cu_k[b];
        int64_t oq = cu_q[b], Lq = (int64_t)cu_q[b + 1] - cu_q[b];
        int64_t Lk = (int64_t)cu_k[b + 1] - cu_k[b];
        const double *kj = row(k, tok[r], h, H, D);
        const double *vj = row(v, tok[r], h, H, D);
        for (int64_t i = 0; i < Lq; ++i) {
            if (!valid(&f, oq + i, i, j, Lk, left, right)) continue;
            const double *qi = row(q, oq + i, h, H, D);
            const double *doi = row(dout, oq + i, h, H, D);
            double s = alpha * dot(qi, kj, D);
            double a = silu(s) / L_scale;
            for (int d = 0; d < D; ++d) gv[d] += a * doi[d];
            double dA = dot(doi, vj, D);
            double dS = dA * silu_grad(s) / L_scale;
            for (int d = 0; d < D; ++d) gk[d] += alpha * dS * qi[d];
        }
    }
    return 0;
}
