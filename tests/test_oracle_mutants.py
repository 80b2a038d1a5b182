"""Plant plausible mistakes in copies of the oracle and check that the pins
catch every one.  Each mutant is compiled from a patched copy of
``oracle/nfo.c`` in a temporary directory (the committed oracle is never
touched) and judged in a subprocess, so a mutant that crashes counts as caught.
CPU only."""
import concurrent.futures as cf
import json
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))

# (name, text in nfo.c, replacement).  Each text must occur exactly once.
MUTANTS = [
    ("prenorm_divides_by_K_minus_1", "ss / (double)K + eps", "ss / (double)(K - 1) + eps"),
    ("prenorm_eps_outside_root", "1.0 / sqrt(ss / (double)K + eps)", "1.0 / sqrt(ss / (double)K) + eps"),
    ("prenorm_drops_normalization", "for (int64_t k = 0; k < K; ++k) x[k] *= rstd;", ""),
    ("prenorm_rstd_squared", "for (int64_t k = 0; k < K; ++k) x[k] *= rstd;",
     "for (int64_t k = 0; k < K; ++k) x[k] *= rstd * rstd;"),
    ("matmul_transposed_W", "z[j] += xk * bf16_to_double(wk[j]);",
     "z[j] += xk * bf16_to_double(W[j * N + k]);"),
    ("matmul_skips_last_k", "for (int64_t k = 0; k < K; ++k) {\n        const double xk",
     "for (int64_t k = 0; k < K - 1; ++k) {\n        const double xk"),
    ("ln_unbiased_variance", "const double var = ss / (double)n;",
     "const double var = ss / (double)(n - 1);"),
    ("ln_mean_divisor", "const double mu = s / (double)n;", "const double mu = s / (double)(n + 1);"),
    ("ln_no_mean_subtraction", "double t = (v[j] - mu) * rstd;", "double t = v[j] * rstd;"),
    ("ln_beta_sign", "if (beta) t += bf16_to_double(beta[j]);", "if (beta) t -= bf16_to_double(beta[j]);"),
    ("ln_gamma_added", "if (gamma) t *= bf16_to_double(gamma[j]);\n        if (beta)",
     "if (gamma) t += bf16_to_double(gamma[j]);\n        if (beta)"),
    ("ln_eps_outside_root", "const double rstd = 1.0 / sqrt(var + eps);",
     "const double rstd = 1.0 / sqrt(var) + eps;"),
    ("rms_sum_not_squares", "for (int64_t j = 0; j < n; ++j) ss += v[j] * v[j];",
     "for (int64_t j = 0; j < n; ++j) ss += v[j] * (v[j] < 0 ? -v[j] : v[j]);"),
    ("rms_eps_scaled", "const double rstd = 1.0 / sqrt(ss / (double)n + eps);",
     "const double rstd = 1.0 / sqrt((ss + eps) / (double)n);"),
    ("rms_gamma_dropped", "if (gamma) t *= bf16_to_double(gamma[j]);\n        y[j] = t;\n    }\n    if (rstd_out) *rstd_out = rstd;\n}\n\nint",
     "y[j] = t;\n    }\n    if (rstd_out) *rstd_out = rstd;\n}\n\nint"),
    ("bf16_decode_shift", "((uint32_t)b) << 16", "((uint32_t)b) << 15"),
    ("plain_ignores_row_list", "load_row(X, row_index(rows, r), K, x);\n            row_times_w(x, W, N, K, Y + r * N);",
     "load_row(X, r, K, x);\n            row_times_w(x, W, N, K, Y + r * N);"),
    ("postln_wrong_rstd_slot", "rstd_out ? rstd_out + r : NULL);\n        }\n        free(x);\n        free(z);\n    }\n    return bad ? -1 : 0;\n}\n\nint nfo_gemm_postnorm_rms",
     "rstd_out ? rstd_out : NULL);\n        }\n        free(x);\n        free(z);\n    }\n    return bad ? -1 : 0;\n}\n\nint nfo_gemm_postnorm_rms"),
    ("bwd_drops_mean_g", "const double mg = kind == NFO_NORM_LN ? sg / (double)n : 0.0;", "const double mg = 0.0;"),
    ("bwd_mean_g_for_rms", "const double mg = kind == NFO_NORM_LN ? sg / (double)n : 0.0;",
     "const double mg = sg / (double)n;"),
    ("bwd_drops_xhat_term", "dz[j] = rstd * (g[j] - mg - xh[j] * mgx);", "dz[j] = rstd * (g[j] - mg);"),
    ("bwd_xhat_term_sign", "dz[j] = rstd * (g[j] - mg - xh[j] * mgx);", "dz[j] = rstd * (g[j] - mg + xh[j] * mgx);"),
    ("bwd_no_rstd", "dz[j] = rstd * (g[j] - mg - xh[j] * mgx);", "dz[j] = (g[j] - mg - xh[j] * mgx);"),
    ("bwd_ignores_gamma", "g[j] = gamma ? dy[j] * bf16_to_double(gamma[j]) : dy[j];", "g[j] = dy[j];"),
    ("bwd_xhat_not_centred", "xh[j] = (kind == NFO_NORM_LN ? z[j] - mean : z[j]) * rstd;", "xh[j] = z[j] * rstd;"),
    ("bwd_divisor", "const double mgx = sgx / (double)n;", "const double mgx = sgx / (double)(n - 1);"),
    ("bwd_z_ignores_row_list", "load_row(Z, i, N, z);", "load_row(Z, r, N, z);"),
    ("bwd_stats_dense_index", "mean[i] : 0.0, rstd[i],\n                         buf + 2 * N", "mean[r] : 0.0, rstd[r],\n                         buf + 2 * N"),
    ("prebwd_db_no_rstd", "const double xh = bf16_to_double(A[i * K + k]) * rstd[i];",
     "const double xh = bf16_to_double(A[i * K + k]);"),
    ("prebwd_db_transposed_dC", "for (int64_t n = 0; n < N; ++n) out[n] += xh * bf16_to_double(dci[n]);",
     "for (int64_t n = 0; n < N; ++n) out[n] += xh * bf16_to_double(dC[n * N + i % N]);"),
    ("prebwd_da_B_not_transposed", "for (int64_t n = 0; n < N; ++n) t += dc[n] * bf16_to_double(bk[n]);",
     "for (int64_t n = 0; n < N; ++n) t += dc[n] * bf16_to_double(B[(n % K) * N + k % N]);"),
    ("prebwd_da_wrong_rstd_row", "norm_bwd_row(dxh, a, K, NULL, NFO_NORM_RMS, 0.0, rstd[i],",
     "norm_bwd_row(dxh, a, K, NULL, NFO_NORM_RMS, 0.0, rstd[r],"),
    ("res_not_added", "for (int64_t j = 0; j < N; ++j) h[j] += bf16_to_double(ri[j]);", ""),
    ("res_subtracted", "h[j] += bf16_to_double(ri[j]);", "h[j] -= bf16_to_double(ri[j]);"),
    ("res_dense_row_index", "const uint16_t* ri = Rs + i * N;", "const uint16_t* ri = Rs + r * N;"),
    ("res_transposed", "h[j] += bf16_to_double(ri[j]);", "h[j] += bf16_to_double(Rs[(j % M) * N + i % N]);"),
    ("res_h_before_add",
     "for (int64_t j = 0; j < N; ++j) h[j] += bf16_to_double(ri[j]);  /* + residual */\n            if (H_out) memcpy(H_out + r * N, h, sizeof(double) * (size_t)N);",
     "if (H_out) memcpy(H_out + r * N, h, sizeof(double) * (size_t)N);\n            for (int64_t j = 0; j < N; ++j) h[j] += bf16_to_double(ri[j]);"),
    ("res_rms_uses_ln", "rmsnorm_row(h, N, gamma, eps, Y + r * N, rstd_out ? rstd_out + r : NULL);",
     "layernorm_row(h, N, gamma, NULL, eps, Y + r * N, NULL, rstd_out ? rstd_out + r : NULL);"),
    ("fna_no_residual1", "for (int64_t d = 0; d < D; ++d) o[h * D + d] = lh[d];    /* residual 1 */",
     "for (int64_t d = 0; d < D; ++d) o[h * D + d] = 0.0;"),
    ("fna_no_residual2", "for (int64_t k = 0; k < HD; ++k) out[k] += q[k];             /* residual 2 */", ""),
    ("fna_ln_per_head", "layernorm_row(q, HD, NULL, NULL, eps1, ln, NULL, NULL);",
     "for (int64_t h2 = 0; h2 < H; ++h2) layernorm_row(q + h2 * D, D, NULL, NULL, eps1, ln + h2 * D, NULL, NULL);"),
    ("fna_rms_per_head", "rmsnorm_row(o, HD, NULL, eps2, out, NULL);",
     "for (int64_t h2 = 0; h2 < H; ++h2) rmsnorm_row(o + h2 * D, D, NULL, eps2, out + h2 * D, NULL);"),
    ("fna_wrong_k_head", "const uint16_t* kj = K + ((b * Lkv + j) * H + h) * D;",
     "const uint16_t* kj = K + ((b * Lkv + j) * H + (h + 1) % H) * D;"),
    # a kernel's bf16 tensor-core operands carried into the oracle: p or ln_q
    # rounded to bf16 (nearest even; normal range) before its matmul
    ("fna_p_rounded_bf16", "s[j] = activation(acc, act);",
     "{ const double a_ = activation(acc, act); int e_; (void)frexp(a_, &e_);"
     " s[j] = a_ == 0.0 ? 0.0 : ldexp(rint(ldexp(a_, 8 - e_)), e_ - 8); }"),
    ("fna_lnq_rounded_bf16", "acc += lh[d] * bf16_to_double(kj[d]);",
     "{ int e_; (void)frexp(lh[d], &e_);"
     " acc += (lh[d] == 0.0 ? 0.0 : ldexp(rint(ldexp(lh[d], 8 - e_)), e_ - 8)) * bf16_to_double(kj[d]); }"),
    ("fna_gelu_coefficient", "(x + 0.044715 * x * x * x)", "(x + 0.04715 * x * x * x)"),
    ("fna_silu_sign", "return x / (1.0 + exp(-x));", "return x / (1.0 + exp(x));"),
    ("fna_v_transposed", "const uint16_t* vj = V + ((b * Lkv + j) * H + h) * D;",
     "const uint16_t* vj = V + ((b * Lkv + (j + 1) % Lkv) * H + h) * D;"),
]


def _judge(name, old, new, workdir):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutant {name}: anchor text must occur exactly once"
    d = os.path.join(workdir, name)
    os.makedirs(d, exist_ok=True)
    path = os.path.join(d, "nfo.c")
    with open(path, "w") as fh:
        fh.write(src.replace(old, new))
    lib = os.path.join(d, "libnfo_mutant.so")
    subprocess.run(["gcc", *oracle.CFLAGS, "-I", os.path.dirname(oracle._SRC), path, "-o", lib,
                    "-lm"], check=True, capture_output=True, text=True)
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run([sys.executable, os.path.join(HERE, "oracle_pins.py"), lib],
                       capture_output=True, text=True, timeout=600, env=env)
    if p.returncode != 0:
        return name, True, f"crashed (rc={p.returncode})"
    res = json.loads(p.stdout.strip().splitlines()[-1])
    failed = [r[0] for r in res if not r[1]]
    return name, bool(failed), ",".join(failed)


@pytest.mark.slow
def test_every_mutant_is_caught(tmp_path):
    workers = max(1, min(8, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(lambda m: _judge(*m, str(tmp_path)), MUTANTS))
    missed = [n for n, caught, _ in results if not caught]
    assert not missed, f"pins missed mutants: {missed}; results: {results}"


def test_unmutated_copy_passes(tmp_path):
    """Control: the same harness passes on an unmodified copy."""
    name, caught, detail = _judge("control", "((uint32_t)b) << 16", "((uint32_t)b) << 16",
                                  str(tmp_path))
    assert not caught, f"unmodified oracle failed pins: {detail}"
