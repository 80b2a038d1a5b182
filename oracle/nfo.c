/*
 * nfo.c -- fp64 CPU oracle for the normalization-fused bf16 GEMM.
 *
 * TEST INFRASTRUCTURE: only tests, the smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code with the CUDA library.
 *
 * Each function writes out the plain definition of its operation in double
 * precision: widen the bf16 inputs exactly, form the product with plain
 * loops, then apply the normalization as defined, with no blocking, no fusion
 * and no reordering beyond what the definition states.
 *
 * Definitions followed ("Towards Free Normalization: Fusing Normalization
 * into GEMM and Attention Kernels"):
 *   - §2, Lazy Pre-Norm: C = rmsnorm(A) @ B, with rmsnorm(A) = A * rstd(A)
 *     row-wise and rstd(A) = rsqrt(sum(A^2 over the row) / row length + eps).
 *   - §3, Multi-CTA Norm: C = norm(A @ B), the norm taken over each full
 *     output row of length N.
 *   - LayerNorm as torch.nn.LayerNorm (linked from the blog's Introduction):
 *     biased variance (divide by N), eps inside the square root, then
 *     elementwise gain gamma and bias beta.
 *   - RMSNorm with a gain: y = x / sqrt(mean(x^2) + eps) * gamma (the
 *     FusedRMSNorm+MatMul article, §3.1 "数学原理重述").
 */
#include "nfo.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> double, exact (bf16 is the top half of an fp32). */
static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int check_rows(const int64_t* rows, int64_t nrows, int64_t M) {
    if (!rows) return 0;
    if (nrows < 0) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -1;
    return 0;
}

static int64_t row_count(const int64_t* rows, int64_t nrows, int64_t M) {
    return rows ? nrows : M;
}

static int64_t row_index(const int64_t* rows, int64_t r) {
    return rows ? rows[r] : r;
}

/* z[j] = sum_k x[k] * W[k][j] for one row x of length K (fp64). */
static void row_times_w(const double* x, const uint16_t* W, int64_t N, int64_t K,
                        double* z) {
    for (int64_t j = 0; j < N; ++j) z[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double xk = x[k];
        const uint16_t* wk = W + k * N;
        for (int64_t j = 0; j < N; ++j) z[j] += xk * bf16_to_double(wk[j]);
    }
}

static void load_row(const uint16_t* A, int64_t i, int64_t len, double* out) {
    const uint16_t* a = A + i * len;
    for (int64_t k = 0; k < len; ++k) out[k] = bf16_to_double(a[k]);
}

/* LayerNorm of one row v (length n) as torch.nn.LayerNorm defines it:
 * two passes, biased variance, eps inside the root. */
static void layernorm_row(const double* v, int64_t n, const uint16_t* gamma,
                          const uint16_t* beta, double eps, double* y,
                          double* mean_out, double* rstd_out) {
    double s = 0.0;
    for (int64_t j = 0; j < n; ++j) s += v[j];
    const double mu = s / (double)n;
    double ss = 0.0;
    for (int64_t j = 0; j < n; ++j) ss += (v[j] - mu) * (v[j] - mu);
    const double var = ss / (double)n;
    const double rstd = 1.0 / sqrt(var + eps);
    for (int64_t j = 0; j < n; ++j) {
        double t = (v[j] - mu) * rstd;
        if (gamma) t *= bf16_to_double(gamma[j]);
        if (beta) t += bf16_to_double(beta[j]);
        y[j] = t;
    }
    if (mean_out) *mean_out = mu;
    if (rstd_out) *rstd_out = rstd;
}

/* RMSNorm of one row v (length n): v / sqrt(mean(v^2) + eps) * gamma. */
static void rmsnorm_row(const double* v, int64_t n, const uint16_t* gamma,
                        double eps, double* y, double* rstd_out) {
    double ss = 0.0;
    for (int64_t j = 0; j < n; ++j) ss += v[j] * v[j];
    const double rstd = 1.0 / sqrt(ss / (double)n + eps);
    for (int64_t j = 0; j < n; ++j) {
        double t = v[j] * rstd;
        if (gamma) t *= bf16_to_double(gamma[j]);
        y[j] = t;
    }
    if (rstd_out) *rstd_out = rstd;
}

int nfo_gemm_plain(const uint16_t* X, const uint16_t* W, int64_t M, int64_t N,
                   int64_t K, const int64_t* rows, int64_t nrows, double* Y) {
    if (!X || !W || !Y || M < 0 || N <= 0 || K <= 0) return -1;
    if (check_rows(rows, nrows, M)) return -1;
    const int64_t R = row_count(rows, nrows, M);
    int bad = 0;
#pragma omp parallel
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)K);
        if (!x) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < R; ++r) {
            if (!x) continue;
            load_row(X, row_index(rows, r), K, x);
            row_times_w(x, W, N, K, Y + r * N);
        }
        free(x);
    }
    return bad ? -1 : 0;
}

int nfo_gemm_prenorm_rms(const uint16_t* X, const uint16_t* W, int64_t M,
                         int64_t N, int64_t K, double eps, const int64_t* rows,
                         int64_t nrows, double* Y, double* rstd_out) {
    if (!X || !W || !Y || M < 0 || N <= 0 || K <= 0 || !(eps >= 0.0)) return -1;
    if (check_rows(rows, nrows, M)) return -1;
    const int64_t R = row_count(rows, nrows, M);
    int bad = 0;
#pragma omp parallel
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)K);
        if (!x) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < R; ++r) {
            if (!x) continue;
            load_row(X, row_index(rows, r), K, x);
            /* rstd over the full row of X (length K) ... */
            double ss = 0.0;
            for (int64_t k = 0; k < K; ++k) ss += x[k] * x[k];
            const double rstd = 1.0 / sqrt(ss / (double)K + eps);
            /* ... rmsnorm(X) materialised in fp64 ... */
            for (int64_t k = 0; k < K; ++k) x[k] *= rstd;
            /* ... then the product with W. */
            row_times_w(x, W, N, K, Y + r * N);
            if (rstd_out) rstd_out[r] = rstd;
        }
        free(x);
    }
    return bad ? -1 : 0;
}

int nfo_gemm_postnorm_ln(const uint16_t* X, const uint16_t* W,
                         const uint16_t* gamma, const uint16_t* beta,
                         int64_t M, int64_t N, int64_t K, double eps,
                         const int64_t* rows, int64_t nrows, double* Y,
                         double* mean_out, double* rstd_out) {
    if (!X || !W || !Y || M < 0 || N <= 0 || K <= 0 || !(eps >= 0.0)) return -1;
    if (check_rows(rows, nrows, M)) return -1;
    const int64_t R = row_count(rows, nrows, M);
    int bad = 0;
#pragma omp parallel
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)K);
        double* z = (double*)malloc(sizeof(double) * (size_t)N);
        if (!x || !z) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < R; ++r) {
            if (!x || !z) continue;
            load_row(X, row_index(rows, r), K, x);
            row_times_w(x, W, N, K, z);                       /* Z = X W */
            layernorm_row(z, N, gamma, beta, eps, Y + r * N,  /* norm(Z) */
                          mean_out ? mean_out + r : NULL,
                          rstd_out ? rstd_out + r : NULL);
        }
        free(x);
        free(z);
    }
    return bad ? -1 : 0;
}

int nfo_gemm_postnorm_rms(const uint16_t* X, const uint16_t* W,
                          const uint16_t* gamma, int64_t M, int64_t N,
                          int64_t K, double eps, const int64_t* rows,
                          int64_t nrows, double* Y, double* rstd_out) {
    if (!X || !W || !Y || M < 0 || N <= 0 || K <= 0 || !(eps >= 0.0)) return -1;
    if (check_rows(rows, nrows, M)) return -1;
    const int64_t R = row_count(rows, nrows, M);
    int bad = 0;
#pragma omp parallel
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)K);
        double* z = (double*)malloc(sizeof(double) * (size_t)N);
        if (!x || !z) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < R; ++r) {
            if (!x || !z) continue;
            load_row(X, row_index(rows, r), K, x);
            row_times_w(x, W, N, K, z);
            rmsnorm_row(z, N, gamma, eps, Y + r * N,
                        rstd_out ? rstd_out + r : NULL);
        }
        free(x);
        free(z);
    }
    return bad ? -1 : 0;
}

int nfo_gemm_postnorm_res(const uint16_t* X, const uint16_t* W,
                          const uint16_t* Rs, const uint16_t* gamma,
                          const uint16_t* beta, int64_t M, int64_t N,
                          int64_t K, int kind, double eps,
                          const int64_t* rows, int64_t nrows, double* Y,
                          double* H_out, double* mean_out, double* rstd_out) {
    if (!X || !W || !Rs || !Y || M < 0 || N <= 0 || K <= 0 || !(eps >= 0.0)) return -1;
    if (kind != NFO_NORM_LN && kind != NFO_NORM_RMS) return -1;
    if (check_rows(rows, nrows, M)) return -1;
    const int64_t R = row_count(rows, nrows, M);
    int bad = 0;
#pragma omp parallel
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)K);
        double* h = (double*)malloc(sizeof(double) * (size_t)N);
        if (!x || !h) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < R; ++r) {
            if (!x || !h) continue;
            const int64_t i = row_index(rows, r);
            load_row(X, i, K, x);
            row_times_w(x, W, N, K, h);                        /* X W */
            const uint16_t* ri = Rs + i * N;
            for (int64_t j = 0; j < N; ++j) h[j] += bf16_to_double(ri[j]);  /* + residual */
            if (H_out) memcpy(H_out + r * N, h, sizeof(double) * (size_t)N);
            if (kind == NFO_NORM_LN)
                layernorm_row(h, N, gamma, beta, eps, Y + r * N, mean_out ? mean_out + r : NULL,
                              rstd_out ? rstd_out + r : NULL);
            else
                rmsnorm_row(h, N, gamma, eps, Y + r * N, rstd_out ? rstd_out + r : NULL);
        }
        free(x);
        free(h);
    }
    return bad ? -1 : 0;
}

int nfo_norm_rows(const uint16_t* in, const uint16_t* gamma,
                  const uint16_t* beta, int64_t R, int64_t C, int kind,
                  double eps, const int64_t* rows, int64_t nrows, double* out,
                  double* mean_out, double* rstd_out) {
    if (!in || !out || R < 0 || C <= 0 || !(eps >= 0.0)) return -1;
    if (kind != NFO_NORM_LN && kind != NFO_NORM_RMS) return -1;
    if (check_rows(rows, nrows, R)) return -1;
    const int64_t n = row_count(rows, nrows, R);
    int bad = 0;
#pragma omp parallel
    {
        double* v = (double*)malloc(sizeof(double) * (size_t)C);
        if (!v) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < n; ++r) {
            if (!v) continue;
            load_row(in, row_index(rows, r), C, v);
            if (kind == NFO_NORM_LN)
                layernorm_row(v, C, gamma, beta, eps, out + r * C,
                              mean_out ? mean_out + r : NULL,
                              rstd_out ? rstd_out + r : NULL);
            else
                rmsnorm_row(v, C, gamma, eps, out + r * C,
                            rstd_out ? rstd_out + r : NULL);
        }
        free(v);
    }
    return bad ? -1 : 0;
}

/* Backward of one normalized row of length n, given that row's forward
 * statistics: g = dy * gamma, xhat = (z - mean) * rstd (LN) or z * rstd
 * (RMS); dz = rstd * (g - mean(g) - xhat * mean(g * xhat)), the mean(g)
 * term for LN only.  g and xh are scratch rows of length n. */
static void norm_bwd_row(const double* dy, const double* z, int64_t n,
                         const uint16_t* gamma, int kind, double mean, double rstd,
                         double* g, double* xh, double* dz) {
    double sg = 0.0, sgx = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        g[j] = gamma ? dy[j] * bf16_to_double(gamma[j]) : dy[j];
        xh[j] = (kind == NFO_NORM_LN ? z[j] - mean : z[j]) * rstd;
        sg += g[j];
        sgx += g[j] * xh[j];
    }
    const double mg = kind == NFO_NORM_LN ? sg / (double)n : 0.0;
    const double mgx = sgx / (double)n;
    for (int64_t j = 0; j < n; ++j) dz[j] = rstd * (g[j] - mg - xh[j] * mgx);
}

int nfo_gemm_postnorm_bwd(const uint16_t* A, const uint16_t* B, const uint16_t* Z,
                          const uint16_t* gamma, const double* mean,
                          const double* rstd, int64_t M, int64_t N, int64_t K,
                          int kind, const int64_t* rows, int64_t nrows, double* dZ) {
    if (!A || !B || !Z || !rstd || !dZ || M < 0 || N <= 0 || K <= 0) return -1;
    if (kind != NFO_NORM_LN && kind != NFO_NORM_RMS) return -1;
    if (kind == NFO_NORM_LN && !mean) return -1;
    if (check_rows(rows, nrows, M)) return -1;
    const int64_t R = row_count(rows, nrows, M);
    int bad = 0;
#pragma omp parallel
    {
        double* a = (double*)malloc(sizeof(double) * (size_t)K);
        double* buf = (double*)malloc(sizeof(double) * (size_t)N * 4);
        if (!a || !buf) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < R; ++r) {
            if (!a || !buf) continue;
            const int64_t i = row_index(rows, r);
            double* dy = buf;
            double* z = buf + N;
            load_row(A, i, K, a);
            row_times_w(a, B, N, K, dy);
            load_row(Z, i, N, z);
            norm_bwd_row(dy, z, N, gamma, kind, kind == NFO_NORM_LN ? mean[i] : 0.0, rstd[i],
                         buf + 2 * N, buf + 3 * N, dZ + r * N);
        }
        free(a);
        free(buf);
    }
    return bad ? -1 : 0;
}

int nfo_norm_rows_bwd(const uint16_t* dY, const uint16_t* Z, const uint16_t* gamma,
                      const double* mean, const double* rstd, int64_t R, int64_t C,
                      int kind, const int64_t* rows, int64_t nrows, double* dZ) {
    if (!dY || !Z || !rstd || !dZ || R < 0 || C <= 0) return -1;
    if (kind != NFO_NORM_LN && kind != NFO_NORM_RMS) return -1;
    if (kind == NFO_NORM_LN && !mean) return -1;
    if (check_rows(rows, nrows, R)) return -1;
    const int64_t n = row_count(rows, nrows, R);
    int bad = 0;
#pragma omp parallel
    {
        double* buf = (double*)malloc(sizeof(double) * (size_t)C * 4);
        if (!buf) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < n; ++r) {
            if (!buf) continue;
            const int64_t i = row_index(rows, r);
            load_row(dY, i, C, buf);
            load_row(Z, i, C, buf + C);
            norm_bwd_row(buf, buf + C, C, gamma, kind, kind == NFO_NORM_LN ? mean[i] : 0.0, rstd[i],
                         buf + 2 * C, buf + 3 * C, dZ + r * C);
        }
        free(buf);
    }
    return bad ? -1 : 0;
}

int nfo_prenorm_rms_bwd_da(const uint16_t* A, const uint16_t* B, const double* rstd,
                           const uint16_t* dC, int64_t M, int64_t N, int64_t K,
                           const int64_t* rows, int64_t nrows, double* dA) {
    if (!A || !B || !rstd || !dC || !dA || M < 0 || N <= 0 || K <= 0) return -1;
    if (check_rows(rows, nrows, M)) return -1;
    const int64_t R = row_count(rows, nrows, M);
    int bad = 0;
#pragma omp parallel
    {
        double* buf = (double*)malloc(sizeof(double) * (size_t)(N + 4 * K));
        if (!buf) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < R; ++r) {
            if (!buf) continue;
            const int64_t i = row_index(rows, r);
            double* dc = buf;
            double* dxh = buf + N;
            double* a = buf + N + K;
            load_row(dC, i, N, dc);
            /* dXhat[i,k] = sum_n dC[i,n] * B[k,n] */
            for (int64_t k = 0; k < K; ++k) {
                const uint16_t* bk = B + k * N;
                double t = 0.0;
                for (int64_t n = 0; n < N; ++n) t += dc[n] * bf16_to_double(bk[n]);
                dxh[k] = t;
            }
            load_row(A, i, K, a);
            norm_bwd_row(dxh, a, K, NULL, NFO_NORM_RMS, 0.0, rstd[i], buf + N + 2 * K, buf + N + 3 * K,
                         dA + r * K);
        }
        free(buf);
    }
    return bad ? -1 : 0;
}

int nfo_prenorm_rms_bwd_db(const uint16_t* A, const double* rstd, const uint16_t* dC,
                           int64_t M, int64_t N, int64_t K, const int64_t* krows,
                           int64_t nkrows, double* dB) {
    if (!A || !rstd || !dC || !dB || M < 0 || N <= 0 || K <= 0) return -1;
    if (check_rows(krows, nkrows, K)) return -1;
    const int64_t R = row_count(krows, nkrows, K);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; ++r) {
        const int64_t k = row_index(krows, r);
        double* out = dB + r * N;
        for (int64_t n = 0; n < N; ++n) out[n] = 0.0;
        /* dB[k,n] = sum_i (A[i,k] * rstd_i) * dC[i,n] */
        for (int64_t i = 0; i < M; ++i) {
            const double xh = bf16_to_double(A[i * K + k]) * rstd[i];
            const uint16_t* dci = dC + i * N;
            for (int64_t n = 0; n < N; ++n) out[n] += xh * bf16_to_double(dci[n]);
        }
    }
    return 0;
}

static double activation(double x, int act) {
    if (act == NFO_ACT_GELU_TANH)
        return 0.5 * x * (1.0 + tanh(sqrt(2.0 / 3.14159265358979323846) * (x + 0.044715 * x * x * x)));
    if (act == NFO_ACT_SILU) return x / (1.0 + exp(-x));
    return x;
}

int nfo_flashnorm_attn_fwd(const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                           const int32_t* q_len, int64_t B, int64_t Lq, int64_t Lkv,
                           int64_t H, int64_t D, int act, double eps1, double eps2,
                           double* Out) {
    if (!Q || !K || !V || !Out || B < 0 || Lq < 0 || Lkv <= 0 || H <= 0 || D <= 0) return -1;
    if (act != NFO_ACT_IDENTITY && act != NFO_ACT_GELU_TANH && act != NFO_ACT_SILU) return -1;
    if (!(eps1 >= 0.0) || !(eps2 >= 0.0)) return -1;
    if (q_len)
        for (int64_t b = 0; b < B; ++b)
            if (q_len[b] < 0 || q_len[b] > Lq) return -1;
    const int64_t HD = H * D;
    const int64_t tokens = B * Lq;
    int bad = 0;
#pragma omp parallel
    {
        double* q = (double*)malloc(sizeof(double) * (size_t)HD);
        double* ln = (double*)malloc(sizeof(double) * (size_t)HD);
        double* o = (double*)malloc(sizeof(double) * (size_t)HD);
        double* s = (double*)malloc(sizeof(double) * (size_t)Lkv);
        if (!q || !ln || !o || !s) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t i = 0; i < tokens; ++i) {
            if (!q || !ln || !o || !s) continue;
            const int64_t b = i / Lq, t = i - b * Lq;
            if (t >= (q_len ? q_len[b] : Lq)) continue;
            load_row(Q, i, HD, q);
            layernorm_row(q, HD, NULL, NULL, eps1, ln, NULL, NULL);      /* ln_q over all heads */
            for (int64_t h = 0; h < H; ++h) {
                const double* lh = ln + h * D;
                for (int64_t j = 0; j < Lkv; ++j) {                      /* p_j = act(ln_q_h . k_j) */
                    const uint16_t* kj = K + ((b * Lkv + j) * H + h) * D;
                    double acc = 0.0;
                    for (int64_t d = 0; d < D; ++d) acc += lh[d] * bf16_to_double(kj[d]);
                    s[j] = activation(acc, act);
                }
                for (int64_t d = 0; d < D; ++d) o[h * D + d] = lh[d];    /* residual 1 */
                for (int64_t j = 0; j < Lkv; ++j) {                      /* + p . V */
                    const uint16_t* vj = V + ((b * Lkv + j) * H + h) * D;
                    for (int64_t d = 0; d < D; ++d) o[h * D + d] += s[j] * bf16_to_double(vj[d]);
                }
            }
            double* out = Out + i * HD;
            rmsnorm_row(o, HD, NULL, eps2, out, NULL);                   /* RMSNorm over all heads */
            for (int64_t k = 0; k < HD; ++k) out[k] += q[k];             /* residual 2 */
        }
        free(q);
        free(ln);
        free(o);
        free(s);
    }
    return bad ? -1 : 0;
}

int nfo_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void nfo_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
