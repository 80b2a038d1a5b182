/*
 * nfo.h -- fp64 CPU oracle for the normalization-fused bf16 GEMM.
 *
 * TEST INFRASTRUCTURE. Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library. The CUDA library never
 * calls it and the two share no source, header, table or helper.
 *
 * Conventions shared by every function:
 *   - X is M x K, W is K x N, gamma and beta have N entries; all are row-major
 *     bfloat16 given as raw uint16 bit patterns and widened to double exactly.
 *   - `rows` lists the output rows to compute (nrows of them, each in [0, M));
 *     rows == NULL means all rows 0..M-1 (nrows is then ignored).  Results are
 *     written densely: output row r of Y (N doubles) belongs to X row rows[r].
 *   - gamma / beta may be NULL (no gain / no bias).  mean / rstd outputs may
 *     be NULL.
 *   - eps is added inside the square root, to the mean (of squares or of
 *     squared deviations).
 *   - Return value: 0 on success, -1 on an invalid argument.
 *
 * Source: "Towards Free Normalization: Fusing Normalization into GEMM and
 * Attention Kernels" (PyTorch blog), §2 Lazy Pre-Norm and §3 Multi-CTA Norm;
 * LayerNorm as torch.nn.LayerNorm, which that blog's Introduction links.
 */
#ifndef NFO_H
#define NFO_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NFO_NORM_LN 0
#define NFO_NORM_RMS 1

/* Y = X W (fp64 sums of exact products). */
int nfo_gemm_plain(const uint16_t* X, const uint16_t* W, int64_t M, int64_t N,
                   int64_t K, const int64_t* rows, int64_t nrows, double* Y);

/* Y = rmsnorm(X) W with rmsnorm(X)[i,k] = X[i,k] * r_i and
 * r_i = 1 / sqrt(sum_k X[i,k]^2 / K + eps): normalize first, then multiply
 * (blog §2, definition of C = rmsnorm(A) @ B). rstd_out[r] = r_i. */
int nfo_gemm_prenorm_rms(const uint16_t* X, const uint16_t* W, int64_t M,
                         int64_t N, int64_t K, double eps, const int64_t* rows,
                         int64_t nrows, double* Y, double* rstd_out);

/* Z = X W; Y = (Z - mu_i) / sqrt(var_i + eps) * gamma_j + beta_j with
 * mu_i = mean_j Z[i,j] and var_i = mean_j (Z[i,j] - mu_i)^2 (blog §3,
 * C = norm(A @ B), LayerNorm over N). */
int nfo_gemm_postnorm_ln(const uint16_t* X, const uint16_t* W,
                         const uint16_t* gamma, const uint16_t* beta,
                         int64_t M, int64_t N, int64_t K, double eps,
                         const int64_t* rows, int64_t nrows, double* Y,
                         double* mean_out, double* rstd_out);

/* Z = X W; Y = Z / sqrt(mean_j Z[i,j]^2 + eps) * gamma_j (blog §3 with RMSNorm). */
int nfo_gemm_postnorm_rms(const uint16_t* X, const uint16_t* W,
                          const uint16_t* gamma, int64_t M, int64_t N,
                          int64_t K, double eps, const int64_t* rows,
                          int64_t nrows, double* Y, double* rstd_out);

/* Residual add before the norm: H = X W + Rs (Rs: M x N, bf16), then
 * Y = LayerNorm(H) * gamma + beta (kind 0) or RMSNorm(H) * gamma (kind 1),
 * over N.  H_out (may be NULL) receives H itself, the updated residual stream
 * that the next layer reads.  Sources: chapter 8 "Element-wise 与算子融合"
 * of the CUDA book, §8.4 (residual add followed by RMSNorm, the updated
 * residual written back) and §8.5.1 (the residual add taken into a GEMM's
 * epilogue); the norm over the GEMM output as blog §3. */
int nfo_gemm_postnorm_res(const uint16_t* X, const uint16_t* W,
                          const uint16_t* Rs, const uint16_t* gamma,
                          const uint16_t* beta, int64_t M, int64_t N,
                          int64_t K, int kind, double eps,
                          const int64_t* rows, int64_t nrows, double* Y,
                          double* H_out, double* mean_out, double* rstd_out);

/* LayerNorm (kind 0) or RMSNorm (kind 1) of each row of `in` (R x C), the
 * unfused normalization kernel of the blog's §1 baseline. beta is ignored for
 * RMSNorm; mean_out is left untouched for RMSNorm. */
int nfo_norm_rows(const uint16_t* in, const uint16_t* gamma,
                  const uint16_t* beta, int64_t R, int64_t C, int kind,
                  double eps, const int64_t* rows, int64_t nrows, double* out,
                  double* mean_out, double* rstd_out);

/* Backward of the row normalization, from the row statistics the forward
 * pass saved (blog §3 "What about backward? Fusion regrouping"):
 *   g = dY * gamma;  xhat = (Z - mean_i) * rstd_i (LN) or Z * rstd_i (RMS);
 *   LN:  dZ = rstd_i * (g - mean_j g - xhat * mean_j(g * xhat))
 *   RMS: dZ = rstd_i * (g - xhat * mean_j(g * xhat))
 * With Z's own statistics this is the gradient of sum(dY * norm(Z)) with
 * respect to Z.  mean and rstd hold one value per row of Z, indexed by the
 * row itself (mean is unused, and may be NULL, for RMS); gamma may be NULL.
 *
 * nfo_gemm_postnorm_bwd: dY = A B (A is M x K, B is K x N; fp64, never
 * rounded), then dZ as above, Z being M x N: the norm's backward fused into
 * the epilogue of the GEMM that produces its incoming gradient. */
int nfo_gemm_postnorm_bwd(const uint16_t* A, const uint16_t* B, const uint16_t* Z,
                          const uint16_t* gamma, const double* mean,
                          const double* rstd, int64_t M, int64_t N, int64_t K,
                          int kind, const int64_t* rows, int64_t nrows, double* dZ);

/* nfo_norm_rows_bwd: dZ as above for each row of dY (R x C, bf16), the
 * unfused normalization-backward kernel. */
int nfo_norm_rows_bwd(const uint16_t* dY, const uint16_t* Z, const uint16_t* gamma,
                      const double* mean, const double* rstd, int64_t R, int64_t C,
                      int kind, const int64_t* rows, int64_t nrows, double* dZ);

/* Lazy Pre-Norm backward (blog §2, limitation 3: the backward rebuilds
 * rmsnorm(A) from A and the saved rstd).  Forward: C = xhat B with
 * xhat[i,k] = A[i,k] * rstd_i.  Given dC (M x N):
 *   dXhat = dC B^T;  dA[i,k] = rstd_i * (dXhat[i,k] - xhat[i,k] * mean_k(dXhat * xhat))
 *   dB[k,n] = sum_i xhat[i,k] * dC[i,n].
 * A is M x K, B is K x N, dC is M x N (bf16), rstd has M entries.
 * nfo_prenorm_rms_bwd_da writes the listed rows of dA (`rows` over M);
 * nfo_prenorm_rms_bwd_db writes the listed rows of dB (`krows` over K). */
int nfo_prenorm_rms_bwd_da(const uint16_t* A, const uint16_t* B, const double* rstd,
                           const uint16_t* dC, int64_t M, int64_t N, int64_t K,
                           const int64_t* rows, int64_t nrows, double* dA);
int nfo_prenorm_rms_bwd_db(const uint16_t* A, const double* rstd, const uint16_t* dC,
                           int64_t M, int64_t N, int64_t K, const int64_t* krows,
                           int64_t nkrows, double* dB);

/* FlashNormAttention forward (blog §4, the fused short-K/V GDPA pseudocode):
 * for each batch b and query token t < q_len[b] (q = Q[b, t, :, :], H*D values)
 *   ln_q = LayerNorm(q) over all H*D values (biased variance, eps1, no affine)
 *   for each head h:  p   = act(ln_q[h] . K[b, :, h, :]^T)             (Lkv values)
 *                     o_h = p . V[b, :, h, :] + ln_q[h]                  (residual 1)
 *   out = RMSNorm(o) over all H*D values (eps2, no affine) + q          (residual 2)
 * Every intermediate stays in fp64, as the pseudocode keeps it: nothing is
 * rounded between the input's bf16 values and the fp64 result.  act:
 * NFO_ACT_IDENTITY, NFO_ACT_GELU_TANH (x/2 (1 + tanh(sqrt(2/pi) (x + 0.044715
 * x^3)))) or NFO_ACT_SILU (x / (1 + e^-x)).
 * Q: [B, Lq, H, D], K and V: [B, Lkv, H, D], bf16; q_len: B entries in
 * [0, Lq] (NULL: Lq each).  Out: [B, Lq, H, D] fp64; rows t >= q_len[b] are
 * not written. */
#define NFO_ACT_IDENTITY 0
#define NFO_ACT_GELU_TANH 1
#define NFO_ACT_SILU 2
int nfo_flashnorm_attn_fwd(const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                           const int32_t* q_len, int64_t B, int64_t Lq, int64_t Lkv,
                           int64_t H, int64_t D, int act, double eps1, double eps2,
                           double* Out);

/* Threads used by the loops over rows (OpenMP). */
int nfo_max_threads(void);
void nfo_set_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
