"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each pin takes an ``oracle.Oracle`` and raises ``AssertionError`` on a
mismatch.  They are chosen so that a plausible slip anywhere in the oracle (a
dropped term, a wrong sign, divisor or index, a transposed operand, eps in the
wrong place) fails at least one of them; ``test_oracle_mutants.py`` plants such
slips in copies of the oracle and checks exactly that.

What each pin compares against:
  * brute force   -- exact rational arithmetic (``fractions``) for sums and
                     products and 60-digit ``decimal`` square roots, on tiny
                     shapes;
  * torch float64 -- ``torch.nn.functional.layer_norm`` / ``rms_norm`` and
                     ``@`` on the CPU, the library special cases;
  * identity      -- (A * rstd[:, None]) @ B == (A @ B) * rstd[:, None], the
                     blog's §2 "Proof";
  * invariants    -- normalized rows have mean 0 / variance (or mean square)
                     var/(var+eps) = 1 - eps*rstd^2;
  * closed forms  -- hand-derived results under ``tests/golden/``;
  * reductions    -- W = I and permutation W, unit gain and zero bias,
                     power-of-two row scales, row-subset consistency;
  * backward      -- exact rationals, torch float64 autograd through
                     layer_norm / rms_norm, and the closed-form invariants of a
                     normalization's gradient (LN rows sum to 0, the
                     xhat-weighted sum is N rstd^3 eps mean(g xhat)).

Run as a script (``python tests/oracle_pins.py LIB.so``) it loads the given
library, runs every pin and prints a JSON list of results.
"""
from __future__ import annotations

import json
import math
import os
import sys
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

import nf_inputs  # noqa: E402
from nf_inputs import bf16_round, bf16_to_f64  # noqa: E402

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
getcontext().prec = 60


# ---------------------------------------------------------------- helpers
def _frac_matrix(bits: np.ndarray):
    """bf16 bits -> nested lists of exact Fractions."""
    vals = bf16_to_f64(bits)
    return [[Fraction(float(v)) for v in row] for row in np.atleast_2d(vals)]


def _dec(f: Fraction) -> Decimal:
    return Decimal(f.numerator) / Decimal(f.denominator)


def _rsqrt(f: Fraction) -> Decimal:
    return Decimal(1) / _dec(f).sqrt()


def _tiny_cases():
    """Tiny problems with awkward rows: zero, constant, mixed sign, large."""
    cases = []
    for seed, (M, K, N) in enumerate([(3, 5, 4), (4, 8, 6), (2, 1, 3), (5, 7, 8)]):
        inp = nf_inputs.make_inputs(M, K, N, seed=100 + seed, gamma=True, beta=True,
                                    w_var=0.5)
        X = inp["X"].copy()
        if M >= 3:
            X[1, :] = 0                                   # zero row
            X[2, :] = bf16_round(np.full(K, 1.5))         # constant row
        cases.append((X, inp["W"], inp["gamma"], inp["beta"]))
    return cases


def _close(got, exact, bound, what):
    got = float(got)
    err = abs(Decimal(repr(got)) - exact)
    assert err <= Decimal(repr(float(bound))), f"{what}: got {got!r}, exact {exact}, err {err}"


# ---------------------------------------------------------------- brute force
def pin_bruteforce_plain(o):
    for X, W, _, _ in _tiny_cases():
        M, K = X.shape
        N = W.shape[1]
        Y = o.gemm_plain(X, W)
        xf, wf = _frac_matrix(X), _frac_matrix(W)
        for i in range(M):
            for j in range(N):
                exact = sum((xf[i][k] * wf[k][j] for k in range(K)), Fraction(0))
                mag = sum(abs(xf[i][k] * wf[k][j]) for k in range(K))
                _close(Y[i, j], _dec(exact), 1e-15 * float(mag) + 1e-300, f"plain[{i},{j}]")


def pin_bruteforce_prenorm(o):
    for eps in (1e-6, 0.5):
        for X, W, _, _ in _tiny_cases():
            M, K = X.shape
            N = W.shape[1]
            Y, rstd = o.gemm_prenorm_rms(X, W, eps)
            xf, wf = _frac_matrix(X), _frac_matrix(W)
            e = Fraction(eps)
            for i in range(M):
                ms = sum((x * x for x in xf[i]), Fraction(0)) / K
                r = _rsqrt(ms + e)
                _close(rstd[i], r, 1e-14 * float(r), f"pre rstd[{i}]")
                for j in range(N):
                    dot = sum((xf[i][k] * wf[k][j] for k in range(K)), Fraction(0))
                    mag = sum(abs(xf[i][k] * wf[k][j]) for k in range(K))
                    _close(Y[i, j], _dec(dot) * r, 1e-14 * float(mag) * float(r) + 1e-300,
                           f"pre[{i},{j}] eps={eps}")


def _ln_exact(z, eps, g=None, b=None):
    n = len(z)
    mu = sum(z, Fraction(0)) / n
    var = sum(((v - mu) ** 2 for v in z), Fraction(0)) / n
    r = _rsqrt(var + Fraction(eps))
    y = []
    for j, v in enumerate(z):
        t = _dec(v - mu) * r
        if g is not None:
            t *= _dec(g[j])
        if b is not None:
            t += _dec(b[j])
        y.append(t)
    return y, _dec(mu), r


def _rms_exact(z, eps, g=None):
    n = len(z)
    ms = sum((v * v for v in z), Fraction(0)) / n
    r = _rsqrt(ms + Fraction(eps))
    y = []
    for j, v in enumerate(z):
        t = _dec(v) * r
        if g is not None:
            t *= _dec(g[j])
        y.append(t)
    return y, r


def pin_bruteforce_postnorm(o):
    for eps in (1e-5, 0.5):
        for X, W, G, B in _tiny_cases():
            M, K = X.shape
            N = W.shape[1]
            xf, wf = _frac_matrix(X), _frac_matrix(W)
            gf, bf = _frac_matrix(G)[0], _frac_matrix(B)[0]
            for affine in (False, True):
                g = G if affine else None
                b = B if affine else None
                Yl, mean, rstd = o.gemm_postnorm_ln(X, W, eps, g, b)
                Yr, rstd_r = o.gemm_postnorm_rms(X, W, eps, g)
                for i in range(M):
                    z = [sum((xf[i][k] * wf[k][j] for k in range(K)), Fraction(0))
                         for j in range(N)]
                    mag = max(float(sum(abs(xf[i][k] * wf[k][j]) for k in range(K)))
                              for j in range(N))
                    y, mu, r = _ln_exact(z, eps, gf if affine else None, bf if affine else None)
                    _close(mean[i], mu, 1e-14 * mag + 1e-300, f"ln mean[{i}]")
                    _close(rstd[i], r, 1e-12 * float(r), f"ln rstd[{i}]")
                    for j in range(N):
                        _close(Yl[i, j], y[j], 1e-13 * (1 + mag * float(r)) * 2,
                               f"post-ln[{i},{j}] eps={eps} affine={affine}")
                    y2, r2 = _rms_exact(z, eps, gf if affine else None)
                    _close(rstd_r[i], r2, 1e-13 * float(r2), f"rms rstd[{i}]")
                    for j in range(N):
                        _close(Yr[i, j], y2[j], 1e-13 * (1 + mag * float(r2)) * 2,
                               f"post-rms[{i},{j}] eps={eps} affine={affine}")


def pin_bruteforce_norm_rows(o):
    for eps in (1e-5, 0.5):
        for X, _, _, _ in _tiny_cases():
            R, C = X.shape
            G = bf16_round(np.linspace(0.5, 1.5, C))
            B = bf16_round(np.linspace(-0.25, 0.25, C))
            xf = _frac_matrix(X)
            gf, bf = _frac_matrix(G)[0], _frac_matrix(B)[0]
            yl, mean, rstd = o.norm_rows(X, 0, eps, G, B)
            yr, _, rstd_r = o.norm_rows(X, 1, eps, G, None)
            for i in range(R):
                mag = float(max(abs(v) for v in xf[i])) + 1e-300
                y, mu, r = _ln_exact(xf[i], eps, gf, bf)
                _close(mean[i], mu, 1e-15 * mag, "norm_rows mean")
                _close(rstd[i], r, 1e-13 * float(r), "norm_rows ln rstd")
                for j in range(C):
                    _close(yl[i, j], y[j], 1e-13 * (1 + mag * float(r)), f"norm_rows ln[{i},{j}]")
                y2, r2 = _rms_exact(xf[i], eps, gf)
                _close(rstd_r[i], r2, 1e-13 * float(r2), "norm_rows rms rstd")
                for j in range(C):
                    _close(yr[i, j], y2[j], 1e-13 * (1 + mag * float(r2)), f"norm_rows rms[{i},{j}]")


# ---------------------------------------------------------------- torch fp64
def pin_torch_f64(o):
    import torch
    import torch.nn.functional as F
    for (M, K, N, eps) in [(37, 72, 40, 1e-5), (19, 136, 24, 1e-6), (8, 8, 264, 1e-5)]:
        inp = nf_inputs.make_inputs(M, K, N, seed=M + K + N, gamma=True, beta=True)
        X, W, G, B = inp["X"], inp["W"], inp["gamma"], inp["beta"]
        x = torch.from_numpy(bf16_to_f64(X))
        w = torch.from_numpy(bf16_to_f64(W))
        g = torch.from_numpy(bf16_to_f64(G))
        b = torch.from_numpy(bf16_to_f64(B))
        z = x @ w
        scale = (x.abs() @ w.abs()).max().item()

        def cmp(got, want, tol, what):
            err = np.max(np.abs(np.asarray(got) - want.numpy()))
            assert err <= tol, f"{what}: max err {err} > {tol}"

        cmp(o.gemm_plain(X, W), z, 1e-13 * scale, "plain vs torch")
        Yp, rp = o.gemm_prenorm_rms(X, W, eps)
        cmp(Yp, F.rms_norm(x, (K,), eps=eps) @ w, 1e-13 * scale, "prenorm vs torch")
        cmp(rp, torch.rsqrt((x * x).mean(-1) + eps), 1e-13, "prenorm rstd vs torch")
        for gg, bb in ((None, None), (g, b)):
            Yl, mean, rstd = o.gemm_postnorm_ln(X, W, eps, G if gg is not None else None,
                                                B if bb is not None else None)
            cmp(Yl, F.layer_norm(z, (N,), gg, bb, eps), 1e-11, "post-ln vs torch")
            cmp(mean, z.mean(-1), 1e-13 * scale, "post-ln mean vs torch")
            cmp(rstd, torch.rsqrt(z.var(-1, unbiased=False) + eps), 1e-10, "post-ln rstd")
            Yr, rr = o.gemm_postnorm_rms(X, W, eps, G if gg is not None else None)
            cmp(Yr, F.rms_norm(z, (N,), gg, eps), 1e-11, "post-rms vs torch")
        yl, mean, rstd = o.norm_rows(X, 0, eps, None, None)
        cmp(yl, F.layer_norm(x, (K,), None, None, eps), 1e-11, "norm_rows ln vs torch")
        Gk = bf16_round(np.linspace(0.5, 1.5, K))
        Bk = bf16_round(np.linspace(-1.0, 1.0, K))
        gk = torch.from_numpy(bf16_to_f64(Gk))
        bk = torch.from_numpy(bf16_to_f64(Bk))
        yl, mean, rstd = o.norm_rows(X, 0, eps, Gk, Bk)
        cmp(yl, F.layer_norm(x, (K,), gk, bk, eps), 1e-11, "norm_rows ln affine vs torch")
        cmp(mean, x.mean(-1), 1e-14, "norm_rows mean vs torch")
        yr, _, _ = o.norm_rows(X, 1, eps, Gk, None)
        cmp(yr, F.rms_norm(x, (K,), gk, eps), 1e-11, "norm_rows rms vs torch")


# ---------------------------------------------------------------- identity
def pin_lazy_identity(o):
    """Blog §2 "Proof": (A*rstd) @ B == (A @ B) * rstd for a row-wise scale."""
    inp = nf_inputs.make_inputs(64, 192, 96, seed=7, x_dist="row_scaled")
    X, W = inp["X"], inp["W"]
    Yp, rstd = o.gemm_prenorm_rms(X, W, 1e-6)
    Z = o.gemm_plain(X, W)
    x = bf16_to_f64(X)
    scale = (np.abs(x) @ np.abs(bf16_to_f64(W))) * rstd[:, None]
    err = np.abs(Yp - Z * rstd[:, None])
    assert np.all(err <= 1e-13 * scale + 1e-300), f"lazy identity: max err {err.max()}"
    # rstd follows the rstd formula of §2 over the full row of X (length K).
    want = 1.0 / np.sqrt((x * x).sum(-1) / x.shape[1] + 1e-6)
    assert np.allclose(rstd, want, rtol=1e-13, atol=0), "rstd formula"


# ---------------------------------------------------------------- invariants
def pin_invariants(o):
    M, K, N = 48, 128, 136
    for eps in (1e-5, 1e-2):
        inp = nf_inputs.make_inputs(M, K, N, seed=11)
        X, W = inp["X"], inp["W"]
        Yl, mean, rstd = o.gemm_postnorm_ln(X, W, eps)
        assert np.all(np.abs(Yl.mean(-1)) <= 1e-13), "LN rows must have mean 0"
        var_out = (Yl * Yl).mean(-1)
        assert np.allclose(var_out, 1.0 - eps * rstd ** 2, rtol=1e-12, atol=0), \
            "LN rows must have variance var/(var+eps)"
        Z = o.gemm_plain(X, W)
        assert np.allclose(mean, Z.mean(-1), rtol=0, atol=1e-13), "LN mean_out"
        Yr, rr = o.gemm_postnorm_rms(X, W, eps)
        assert np.allclose((Yr * Yr).mean(-1), 1.0 - eps * rr ** 2, rtol=1e-12, atol=0), \
            "RMS rows must have mean square ms/(ms+eps)"
        # Pre-norm with W = I reproduces RMSNorm(X): mean square ms/(ms+eps) over K.
        I = bf16_round(np.eye(K))
        Yp, rp = o.gemm_prenorm_rms(X, I, eps)
        assert np.allclose((Yp * Yp).mean(-1), 1.0 - eps * rp ** 2, rtol=1e-12, atol=0), \
            "pre-RMS with W=I must give unit mean square"


# ---------------------------------------------------------------- reductions
def pin_reductions(o):
    M, K = 24, 96
    eps = 1e-5
    inp = nf_inputs.make_inputs(M, K, K, seed=5, gamma=True, beta=True)
    X, G, B = inp["X"], inp["gamma"], inp["beta"]
    I = bf16_round(np.eye(K))
    a, ma, ra = o.gemm_postnorm_ln(X, I, eps, G, B)
    b, mb, rb = o.norm_rows(X, 0, eps, G, B)
    assert np.array_equal(a, b) and np.array_equal(ma, mb) and np.array_equal(ra, rb), \
        "post-LN with W=I must equal LayerNorm(X)"
    a, ra = o.gemm_postnorm_rms(X, I, eps, G)
    b, _, rb = o.norm_rows(X, 1, eps, G)
    assert np.array_equal(a, b) and np.array_equal(ra, rb), "post-RMS with W=I"
    a, ra = o.gemm_prenorm_rms(X, I, eps)
    b, _, rb = o.norm_rows(X, 1, eps)
    assert np.allclose(a, b, rtol=0, atol=1e-15) and np.allclose(ra, rb, rtol=1e-15), \
        "pre-RMS with W=I must equal RMSNorm(X)"
    # unit gain and zero bias are the no-affine result
    one = bf16_round(np.ones(K))
    zero = bf16_round(np.zeros(K))
    a, _, _ = o.gemm_postnorm_ln(X, I, eps, one, zero)
    b, _, _ = o.gemm_postnorm_ln(X, I, eps)
    assert np.array_equal(a, b), "gamma=1, beta=0 must equal no affine"
    # a (non-symmetric) permutation W permutes columns: pins the W index order
    perm = np.roll(np.arange(K), 1)
    P = np.zeros((K, K))
    P[np.arange(K), perm] = 1.0
    Yp = o.gemm_plain(X, bf16_round(P))
    x = bf16_to_f64(X)
    want = np.zeros_like(x)
    want[:, perm] = x
    assert np.array_equal(Yp, want), "X @ P must move column k to perm[k]"
    # a non-square W with a distinct value per (k, j) pins the W index order
    Kp, Np = 6, 4
    Wr = bf16_round(np.arange(Kp * Np, dtype=np.float64).reshape(Kp, Np))
    Xr = bf16_round(np.eye(Kp)[:3])                 # rows e_0, e_1, e_2
    assert np.array_equal(o.gemm_plain(Xr, Wr), bf16_to_f64(Wr)[:3]), "e_k @ W = W[k,:]"


def pin_power_of_two_scale(o):
    """Scaling a row by 2^p is exact in bf16; the normalized result changes only
    through eps, by the closed-form factor sqrt(q + eps) / sqrt(q + eps / s^2)."""
    M, K, N = 16, 64, 80
    eps = 1e-3
    inp = nf_inputs.make_inputs(M, K, N, seed=9)
    X, W = inp["X"], inp["W"]
    x = bf16_to_f64(X)
    s = 2.0 ** np.arange(-4, 4).repeat(2)[:M]
    Xs = bf16_round(x * s[:, None])
    assert np.array_equal(bf16_to_f64(Xs), x * s[:, None])
    Y0, r0 = o.gemm_prenorm_rms(X, W, eps)
    Y1, r1 = o.gemm_prenorm_rms(Xs, W, eps)
    ms = (x * x).mean(-1)
    f = np.sqrt(ms + eps) / np.sqrt(ms + eps / s ** 2)
    assert np.allclose(Y1, Y0 * f[:, None], rtol=1e-12, atol=1e-14), "pre-RMS scale law"
    L0, _, _ = o.gemm_postnorm_ln(X, W, eps)
    L1, _, _ = o.gemm_postnorm_ln(Xs, W, eps)
    z = o.gemm_plain(X, W)
    var = z.var(-1)
    f = np.sqrt(var + eps) / np.sqrt(var + eps / s ** 2)
    assert np.allclose(L1, L0 * f[:, None], rtol=1e-11, atol=1e-13), "post-LN scale law"


def pin_row_subset(o):
    M, K, N = 40, 64, 72
    inp = nf_inputs.make_inputs(M, K, N, seed=3, gamma=True, beta=True)
    X, W, G, B = inp["X"], inp["W"], inp["gamma"], inp["beta"]
    rows = np.array([39, 0, 17, 17, 5])
    full = o.gemm_postnorm_ln(X, W, 1e-5, G, B)
    part = o.gemm_postnorm_ln(X, W, 1e-5, G, B, rows=rows)
    for f, p in zip(full, part):
        assert np.array_equal(f[rows], p), "row subset must equal the full result's rows"
    full = o.gemm_prenorm_rms(X, W, 1e-6)
    part = o.gemm_prenorm_rms(X, W, 1e-6, rows=rows)
    for f, p in zip(full, part):
        assert np.array_equal(f[rows], p), "prenorm row subset"
    full = o.gemm_plain(X, W)
    assert np.array_equal(full[rows], o.gemm_plain(X, W, rows=rows)), "plain row subset"
    full = o.gemm_postnorm_rms(X, W, 1e-5, G)
    part = o.gemm_postnorm_rms(X, W, 1e-5, G, rows=rows)
    for f, p in zip(full, part):
        assert np.array_equal(f[rows], p), "post-rms row subset"
    full = o.norm_rows(X, 0, 1e-5, G[:K].copy(), B[:K].copy())
    part = o.norm_rows(X, 0, 1e-5, G[:K].copy(), B[:K].copy(), rows=rows)
    for f, p in zip(full, part):
        assert np.array_equal(f[rows], p), "norm_rows row subset"


# ---------------------------------------------------------------- closed forms
def _golden_cases():
    with open(os.path.join(GOLDEN, "closed_forms.json")) as fh:
        return json.load(fh)["cases"]


def _pin_closed_form_fna(o, case, env):
    """FlashNormAttention forward on a hand-derived case (inputs exact in bf16)."""
    arrs = {}
    for k in ("Q", "K", "V"):
        a = np.array(case[k], dtype=np.float64)
        arrs[k] = bf16_round(a)
        assert np.array_equal(bf16_to_f64(arrs[k]), a), f"{case['name']}: fixture {k} must be exact in bf16"
    env = dict(env)
    for name, expr in case.get("let", []):
        env[name] = eval(expr, env)  # noqa: S307
    want = np.array([eval(e, env) for e in case["Y"]]).reshape(np.array(case["Q"]).shape)  # noqa: S307
    got = o.flashnorm_attn_fwd(arrs["Q"], arrs["K"], arrs["V"], int(case["act"]), float(case["eps1"]),
                               float(case["eps2"]))
    assert np.allclose(got, want, rtol=1e-14, atol=1e-14), \
        f"closed form {case['name']}: got {got.ravel().tolist()} want {want.ravel().tolist()}"


def pin_closed_forms(o):
    env = {"sqrt": math.sqrt, "exp": math.exp, "tanh": math.tanh, "pi": math.pi}
    for case in _golden_cases():
        if case["op"] == "fna":
            _pin_closed_form_fna(o, case, env)
            continue
        X = bf16_round(np.array(case["X"], dtype=np.float64))
        assert np.array_equal(bf16_to_f64(X), np.array(case["X"], dtype=np.float64)), \
            f"{case['name']}: fixture X must be exact in bf16"
        eps = float(case["eps"])
        want = np.array([[eval(e, env) for e in row] for row in case["Y"]])  # noqa: S307
        op = case["op"]
        if op == "norm_rows_ln":
            got, _, _ = o.norm_rows(X, 0, eps)
        elif op == "norm_rows_rms":
            got, _, _ = o.norm_rows(X, 1, eps)
        else:
            W = bf16_round(np.array(case["W"], dtype=np.float64))
            if op == "pre_rms":
                got, _ = o.gemm_prenorm_rms(X, W, eps)
            elif op == "post_ln":
                got, _, _ = o.gemm_postnorm_ln(X, W, eps)
            elif op == "post_rms":
                got, _ = o.gemm_postnorm_rms(X, W, eps)
            elif op == "plain":
                got = o.gemm_plain(X, W)
            else:
                raise AssertionError(f"unknown op {op}")
        assert np.allclose(got, want, rtol=1e-14, atol=1e-14), \
            f"closed form {case['name']}: got {got.tolist()} want {want.tolist()}"


# ---------------------------------------------------------------- backward
# The norm's backward fused into the epilogue of the GEMM that produces its
# incoming gradient (blog §3 "What about backward? Fusion regrouping"), and
# the unfused row kernel, both from the forward's saved row statistics.
def _bwd_cases():
    """Tiny problems: A (M x K), B (K x N), Z (M x N), gamma, and dyadic row
    statistics (exact in binary; the formula takes any statistics)."""
    cases = []
    for seed, (M, K, N) in enumerate([(3, 5, 4), (4, 8, 6), (2, 1, 3)]):
        inp = nf_inputs.make_inputs(M, K, N, seed=200 + seed, gamma=True, w_var=0.5)
        rng = np.random.default_rng(300 + seed)
        Z = bf16_round(rng.normal(0.5, 1.5, size=(M, N)))
        mean = np.array([0.125 * (i - 1) for i in range(M)])
        rstd = np.array([0.75 + 0.25 * i for i in range(M)])
        cases.append((inp["X"], inp["W"], Z, inp["gamma"], mean, rstd))
    return cases


def _bwd_exact(dy, z, g, kind, mean, rstd):
    """dz of one row in exact rationals, written from the chain rule through
    y = xhat * g with xhat = (z - mean) * rstd (LN) or z * rstd (RMS)."""
    n = len(dy)
    gg = [dy[j] * (g[j] if g is not None else 1) for j in range(n)]
    xh = [((z[j] - mean) if kind == 0 else z[j]) * rstd for j in range(n)]
    mg = sum(gg, Fraction(0)) / n if kind == 0 else Fraction(0)
    mgx = sum((gg[j] * xh[j] for j in range(n)), Fraction(0)) / n
    return [rstd * (gg[j] - mg - xh[j] * mgx) for j in range(n)]


def pin_bruteforce_norm_bwd(o):
    for A, B, Z, gamma, mean, rstd in _bwd_cases():
        M, K = A.shape
        N = B.shape[1]
        af, bf, zf = _frac_matrix(A), _frac_matrix(B), _frac_matrix(Z)
        gf = _frac_matrix(gamma)[0]
        dyf = [[sum((af[i][k] * bf[k][j] for k in range(K)), Fraction(0)) for j in range(N)]
               for i in range(M)]
        dY16 = bf16_round(np.array([[float(v) for v in row] for row in dyf]))
        d16 = _frac_matrix(dY16)
        for kind in (0, 1):
            for use_g in (False, True):
                m = mean if kind == 0 else None
                g = gamma if use_g else None
                fused = o.gemm_postnorm_bwd(A, B, Z, kind, m, rstd, g)
                unfused = o.norm_rows_bwd(dY16, Z, kind, m, rstd, g)
                for i in range(M):
                    mu, r = Fraction(float(mean[i])), Fraction(float(rstd[i]))
                    want_f = _bwd_exact(dyf[i], zf[i], gf if use_g else None, kind, mu, r)
                    want_u = _bwd_exact(d16[i], zf[i], gf if use_g else None, kind, mu, r)
                    scale = 1e-13 * (1 + max(float(abs(v)) for v in want_f + want_u))
                    for j in range(N):
                        _close(fused[i, j], _dec(want_f[j]), scale, f"bwd fused kind={kind}[{i},{j}]")
                        _close(unfused[i, j], _dec(want_u[j]), scale, f"bwd rows kind={kind}[{i},{j}]")


def pin_torch_autograd_bwd(o):
    """torch float64 autograd through F.layer_norm / F.rms_norm, with the
    statistics of Z itself."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(41)
    M, K, N = 7, 33, 40
    A = bf16_round(rng.normal(size=(M, K)))
    B = bf16_round(rng.normal(0, 0.3, size=(K, N)))
    Z = bf16_round(rng.normal(0.3, 2.0, size=(M, N)))
    G = bf16_round(rng.normal(1.0, 0.3, size=N))
    eps = 1e-3
    dY = torch.from_numpy(bf16_to_f64(A)) @ torch.from_numpy(bf16_to_f64(B))
    for kind in (0, 1):
        for use_g in (False, True):
            z = torch.from_numpy(bf16_to_f64(Z)).requires_grad_(True)
            w = torch.from_numpy(bf16_to_f64(G)) if use_g else None
            if kind == 0:
                y = F.layer_norm(z, (N,), w, None, eps)
                mu = z.detach().mean(-1)
                rs = 1.0 / torch.sqrt(z.detach().var(-1, unbiased=False) + eps)
            else:
                y = F.rms_norm(z, (N,), w, eps)
                mu = None
                rs = 1.0 / torch.sqrt((z.detach() ** 2).mean(-1) + eps)
            (y * dY).sum().backward()
            want = z.grad.numpy()
            got = o.gemm_postnorm_bwd(A, B, Z, kind, None if mu is None else mu.numpy(), rs.numpy(),
                                      G if use_g else None)
            assert np.allclose(got, want, rtol=1e-10, atol=1e-11 * np.abs(want).max()), \
                f"autograd kind={kind} gamma={use_g}: max err {np.abs(got - want).max()}"


def pin_norm_bwd_invariants(o):
    """With Z's own statistics: LN gradient rows sum to 0; for both norms
    sum_j dz_j * xhat_j = N * rstd^3 * eps * mean_j(g_j * xhat_j)."""
    rng = np.random.default_rng(43)
    R, C = 6, 48
    Z = bf16_round(rng.normal(-0.7, 1.3, size=(R, C)))
    dY = bf16_round(rng.normal(size=(R, C)))
    G = bf16_round(rng.normal(1.0, 0.2, size=C))
    z, dy, g = bf16_to_f64(Z), bf16_to_f64(dY), bf16_to_f64(G)
    for eps in (1e-5, 0.25):
        for kind in (0, 1):
            _, mean, rstd = o.norm_rows(Z, kind, eps)
            dz = o.norm_rows_bwd(dY, Z, kind, mean, rstd, G)
            xh = ((z - mean[:, None]) if kind == 0 else z) * rstd[:, None]
            gx = (dy * g * xh).mean(-1)
            scale = np.abs(dz).max()
            if kind == 0:
                assert np.abs(dz.sum(-1)).max() <= 1e-12 * C * scale, f"LN bwd row sums eps={eps}"
            want = C * rstd ** 3 * eps * gx
            got = (dz * xh).sum(-1)
            assert np.allclose(got, want, rtol=1e-9, atol=1e-12 * C * scale), \
                f"bwd orthogonality kind={kind} eps={eps}: {got} vs {want}"


def pin_norm_bwd_reductions(o):
    """B = I and B = a column permutation reduce the fused backward to the row
    kernel on A; gamma = 1 equals no gamma; a row list gives the same rows."""
    rng = np.random.default_rng(47)
    M, N = 5, 12
    A = bf16_round(rng.normal(size=(M, N)))
    Z = bf16_round(rng.normal(0.2, 1.0, size=(M, N)))
    mean = rng.normal(size=M)
    rstd = rng.uniform(0.5, 2.0, size=M)
    I = bf16_round(np.eye(N))
    perm = np.roll(np.arange(N), 5)
    P = np.ascontiguousarray(bf16_round(np.eye(N)[:, perm]))  # (A @ P)[:, j] = A[:, perm[j]]
    ones = bf16_round(np.ones(N))
    G = bf16_round(rng.normal(1.0, 0.5, size=N))
    for kind in (0, 1):
        m = mean if kind == 0 else None
        rows = o.norm_rows_bwd(A, Z, kind, m, rstd, G)
        assert np.array_equal(o.gemm_postnorm_bwd(A, I, Z, kind, m, rstd, G), rows), f"B=I kind={kind}"
        Ap = np.ascontiguousarray(A[:, perm])
        assert np.array_equal(o.gemm_postnorm_bwd(A, P, Z, kind, m, rstd, G),
                              o.norm_rows_bwd(Ap, Z, kind, m, rstd, G)), f"B=P kind={kind}"
        assert np.array_equal(o.gemm_postnorm_bwd(A, I, Z, kind, m, rstd, ones),
                              o.gemm_postnorm_bwd(A, I, Z, kind, m, rstd, None)), f"gamma=1 kind={kind}"
        sub = np.array([4, 0, 2])
        full = o.gemm_postnorm_bwd(A, P, Z, kind, m, rstd, G)
        assert np.array_equal(o.gemm_postnorm_bwd(A, P, Z, kind, m, rstd, G, rows=sub), full[sub]), \
            f"row list kind={kind}"
        assert np.array_equal(o.norm_rows_bwd(A, Z, kind, m, rstd, G, rows=sub), rows[sub]), \
            f"row list (rows kernel) kind={kind}"


def pin_prenorm_bwd_bruteforce(o):
    """Lazy Pre-Norm backward in exact rationals on tiny problems."""
    for seed, (M, K, N) in enumerate([(3, 5, 4), (4, 6, 3), (2, 1, 2)]):
        inp = nf_inputs.make_inputs(M, K, N, seed=400 + seed, w_var=0.5)
        A, B = inp["X"], inp["W"]
        dC = bf16_round(np.random.default_rng(500 + seed).normal(size=(M, N)))
        rstd = np.array([0.5 + 0.25 * i for i in range(M)])
        af, bf, cf = _frac_matrix(A), _frac_matrix(B), _frac_matrix(dC)
        rf = [Fraction(float(v)) for v in rstd]
        dA = o.prenorm_rms_bwd_da(A, B, rstd, dC)
        dB = o.prenorm_rms_bwd_db(A, rstd, dC)
        for i in range(M):
            dxh = [sum((cf[i][n] * bf[k][n] for n in range(N)), Fraction(0)) for k in range(K)]
            want = _bwd_exact(dxh, af[i], None, 1, Fraction(0), rf[i])
            scale = 1e-13 * (1 + max(float(abs(v)) for v in want))
            for k in range(K):
                _close(dA[i, k], _dec(want[k]), scale, f"pre bwd dA[{i},{k}]")
        for k in range(K):
            for n in range(N):
                want = sum((af[i][k] * rf[i] * cf[i][n] for i in range(M)), Fraction(0))
                mag = sum(abs(af[i][k] * rf[i] * cf[i][n]) for i in range(M))
                _close(dB[k, n], _dec(want), 1e-14 * float(mag) + 1e-300, f"pre bwd dB[{k},{n}]")


def pin_prenorm_bwd_autograd(o):
    """torch float64 autograd through C = rms_norm(A) @ B, with A's own rstd."""
    import torch
    import torch.nn.functional as F
    rng = np.random.default_rng(53)
    M, K, N = 9, 40, 24
    A = bf16_round(rng.normal(0.2, 1.3, size=(M, K)))
    B = bf16_round(rng.normal(0, 0.2, size=(K, N)))
    dC = bf16_round(rng.normal(size=(M, N)))
    eps = 1e-2
    a = torch.from_numpy(bf16_to_f64(A)).requires_grad_(True)
    b = torch.from_numpy(bf16_to_f64(B)).requires_grad_(True)
    c = F.rms_norm(a, (K,), None, eps) @ b
    (c * torch.from_numpy(bf16_to_f64(dC))).sum().backward()
    rstd = (1.0 / torch.sqrt((a.detach() ** 2).mean(-1) + eps)).numpy()
    got_a = o.prenorm_rms_bwd_da(A, B, rstd, dC)
    got_b = o.prenorm_rms_bwd_db(A, rstd, dC)
    assert np.allclose(got_a, a.grad.numpy(), rtol=1e-10, atol=1e-12), "pre-norm bwd dA vs autograd"
    assert np.allclose(got_b, b.grad.numpy(), rtol=1e-10, atol=1e-12), "pre-norm bwd dB vs autograd"


def pin_prenorm_bwd_reductions(o):
    """dC = 1: dB rows are the column sums of xhat; the dA rows' xhat-weighted
    sums follow the normalization-gradient closed form; row lists agree."""
    rng = np.random.default_rng(59)
    M, K, N = 6, 16, 5
    A = bf16_round(rng.normal(size=(M, K)))
    B = bf16_round(rng.normal(0, 0.3, size=(K, N)))
    eps = 0.1
    a = bf16_to_f64(A)
    ms = (a * a).mean(-1)
    rstd = 1.0 / np.sqrt(ms + eps)
    ones = bf16_round(np.ones((M, N)))
    xh = a * rstd[:, None]
    dB = o.prenorm_rms_bwd_db(A, rstd, ones)
    assert np.allclose(dB, np.repeat(xh.sum(0)[:, None], N, axis=1), rtol=1e-13, atol=1e-13), "dB with dC = 1"
    dC = bf16_round(rng.normal(size=(M, N)))
    dA = o.prenorm_rms_bwd_da(A, B, rstd, dC)
    dxh = bf16_to_f64(dC) @ bf16_to_f64(B).T
    want = K * rstd ** 3 * eps * (dxh * xh).mean(-1)
    assert np.allclose((dA * xh).sum(-1), want, rtol=1e-9, atol=1e-12), "dA orthogonality"
    sub = np.array([5, 1])
    assert np.array_equal(o.prenorm_rms_bwd_da(A, B, rstd, dC, rows=sub), dA[sub]), "dA row list"
    ksub = np.array([3, 0, 15])
    full_b = o.prenorm_rms_bwd_db(A, rstd, dC)
    assert np.array_equal(o.prenorm_rms_bwd_db(A, rstd, dC, krows=ksub), full_b[ksub]), "dB row list"


# ---------------------------------------------------------------- residual add
def _res_cases():
    """(M, K, N, eps, X, W, Rs, gamma, beta): non-square shapes so that a
    transposed residual cannot pass."""
    out = []
    for (M, K, N, eps) in [(37, 72, 40, 1e-5), (19, 24, 136, 1e-6), (8, 8, 264, 1e-5)]:
        inp = nf_inputs.make_inputs(M, K, N, seed=3 * M + N, gamma=True, beta=True)
        Rs = nf_inputs.make_inputs(M, N, 8, seed=M + 5 * N)["X"]
        out.append((M, K, N, eps, inp["X"], inp["W"], Rs, inp["gamma"], inp["beta"]))
    return out


def pin_residual_torch(o):
    """H = X W + R and its LayerNorm / RMSNorm against torch CPU float64."""
    import torch
    import torch.nn.functional as F
    for (M, K, N, eps, X, W, Rs, G, B) in _res_cases():
        x, w, r = (torch.from_numpy(bf16_to_f64(a)) for a in (X, W, Rs))
        g, b = torch.from_numpy(bf16_to_f64(G)), torch.from_numpy(bf16_to_f64(B))
        h = x @ w + r
        scale = (x.abs() @ w.abs() + r.abs()).max().item()
        for gg, bb in ((None, None), (G, B)):
            tg = g if gg is not None else None
            tb = b if bb is not None else None
            Y, H, mean, rstd = o.gemm_postnorm_res(X, W, Rs, 0, eps, gg, bb)
            assert np.max(np.abs(H - h.numpy())) <= 1e-13 * scale, "residual H vs torch"
            assert np.max(np.abs(Y - F.layer_norm(h, (N,), tg, tb, eps).numpy())) <= 1e-11, "res LN vs torch"
            assert np.max(np.abs(mean - h.mean(-1).numpy())) <= 1e-13 * scale, "res LN mean"
            want_r = torch.rsqrt(h.var(-1, unbiased=False) + eps).numpy()
            assert np.max(np.abs(rstd - want_r) / want_r) <= 1e-10, "res LN rstd"
            Y, H, mean, rstd = o.gemm_postnorm_res(X, W, Rs, 1, eps, gg, None)
            assert mean is None
            assert np.max(np.abs(Y - F.rms_norm(h, (N,), tg, eps).numpy())) <= 1e-11, "res RMS vs torch"
            want_r = torch.rsqrt((h * h).mean(-1) + eps).numpy()
            assert np.max(np.abs(rstd - want_r) / want_r) <= 1e-12, "res RMS rstd"


def pin_residual_reductions(o):
    """W = 0: the result is the row norm of R alone (and H = R); R = 0: the
    post-norm GEMM; a row list selects rows of X and of R alike; LayerNorm is
    blind to a constant added to a row of R, which moves H by that constant."""
    for (M, K, N, eps, X, W, Rs, G, B) in _res_cases():
        Z0 = bf16_round(np.zeros((K, N)))
        Y, H, mean, rstd = o.gemm_postnorm_res(X, Z0, Rs, 0, eps, G, B)
        y2, m2, r2 = o.norm_rows(Rs, 0, eps, G, B)
        assert np.array_equal(Y, y2) and np.array_equal(mean, m2) and np.array_equal(rstd, r2), \
            "W = 0: LayerNorm(R)"
        assert np.array_equal(H, bf16_to_f64(Rs)), "W = 0: H = R"
        Y, H, _, rstd = o.gemm_postnorm_res(X, Z0, Rs, 1, eps, G)
        y2, _, r2 = o.norm_rows(Rs, 1, eps, G)
        assert np.array_equal(Y, y2) and np.array_equal(rstd, r2), "W = 0: RMSNorm(R)"
        R0 = bf16_round(np.zeros((M, N)))
        Y, H, mean, rstd = o.gemm_postnorm_res(X, W, R0, 0, eps, G, B)
        y2, m2, r2 = o.gemm_postnorm_ln(X, W, eps, G, B)
        assert np.array_equal(Y, y2) and np.array_equal(mean, m2) and np.array_equal(rstd, r2), \
            "R = 0: post-LN"
        assert np.array_equal(H, o.gemm_plain(X, W)), "R = 0: H = X W"
        Y, H, _, rstd = o.gemm_postnorm_res(X, W, R0, 1, eps, G)
        y2, r2 = o.gemm_postnorm_rms(X, W, eps, G)
        assert np.array_equal(Y, y2) and np.array_equal(rstd, r2), "R = 0: post-RMS"
        rows = np.array([M - 1, 0, M // 2, 1], np.int64)
        for kind in (0, 1):
            Yf, Hf, _, rf = o.gemm_postnorm_res(X, W, Rs, kind, eps, G, B)
            Ys, Hs, _, rs = o.gemm_postnorm_res(X, W, Rs, kind, eps, G, B, rows=rows)
            assert np.array_equal(Ys, Yf[rows]) and np.array_equal(Hs, Hf[rows]) and \
                np.array_equal(rs, rf[rows]), "row list"
        # R on a 1/64 grid in [-2, 2] and a small integer c_i added to row i:
        # both exact in bf16 (at most 9 significant bits).  H moves by c_i and
        # LayerNorm, blind to a constant shift of its row, does not move.
        rng = np.random.default_rng(M + N)
        Rq = bf16_round(rng.integers(-128, 129, size=(M, N)) / 64.0)
        c = np.arange(M, dtype=np.float64) % 5 - 2.0
        Rc = bf16_round(bf16_to_f64(Rq) + c[:, None])
        assert np.array_equal(bf16_to_f64(Rc), bf16_to_f64(Rq) + c[:, None])
        Y1, H1, _, _ = o.gemm_postnorm_res(X, W, Rq, 0, eps)
        Y2, H2, _, _ = o.gemm_postnorm_res(X, W, Rc, 0, eps)
        assert np.allclose(H2 - H1, c[:, None], rtol=0, atol=1e-12), "H moves with R"
        assert np.max(np.abs(Y2 - Y1)) <= 1e-10, "LN is shift invariant in R"


# ---------------------------------------------------------------- FlashNormAttention forward
def _fna_case(B, Lq, Lkv, H, D, seed, scale_kv=0.15):
    g = np.random.default_rng(seed)
    Q = bf16_round(g.standard_normal((B, Lq, H, D)) * 1.3 + 0.2)
    K = bf16_round(g.standard_normal((B, Lkv, H, D)) * scale_kv)
    V = bf16_round(g.standard_normal((B, Lkv, H, D)) * scale_kv)
    return Q, K, V


def _fna_torch(Q, K, V, act, eps1, eps2):
    """The blog §4 pseudocode as torch float64 ops, every intermediate kept in
    float64 (the pseudocode rounds nothing)."""
    import torch
    import torch.nn.functional as F
    B, Lq, H, D = Q.shape
    q = torch.from_numpy(bf16_to_f64(Q)).reshape(B, Lq, H * D)
    k = torch.from_numpy(bf16_to_f64(K))
    v = torch.from_numpy(bf16_to_f64(V))
    ln = F.layer_norm(q, (H * D,), eps=eps1).reshape(B, Lq, H, D)
    s = torch.einsum("bthd,bjhd->bhtj", ln, k)
    p = {0: s, 1: F.gelu(s, approximate="tanh"), 2: F.silu(s)}[act]
    o = torch.einsum("bhtj,bjhd->bthd", p, v) + ln
    out = F.rms_norm(o.reshape(B, Lq, H * D), (H * D,), eps=eps2) + q
    return out.reshape(B, Lq, H, D).numpy()


def pin_fna_torch(o):
    for (B, Lq, Lkv, H, D, act) in [(2, 5, 8, 3, 16, 1), (1, 4, 128, 2, 32, 2), (3, 2, 16, 1, 8, 0)]:
        Q, K, V = _fna_case(B, Lq, Lkv, H, D, seed=B * 7 + H)
        got = o.flashnorm_attn_fwd(Q, K, V, act, 1e-5, 1e-6)
        want = _fna_torch(Q, K, V, act, 1e-5, 1e-6)
        err = np.max(np.abs(got - want))
        assert err <= 1e-9, f"FlashNormAttention vs torch (act {act}): max err {err}"


def pin_fna_bruteforce(o):
    """Plain Python loops over a tiny case (math.tanh / math.exp)."""
    import math
    B, Lq, Lkv, H, D = 1, 2, 3, 2, 4
    Q, K, V = _fna_case(B, Lq, Lkv, H, D, seed=3, scale_kv=0.8)
    q, k, v = bf16_to_f64(Q), bf16_to_f64(K), bf16_to_f64(V)
    for act in (0, 1, 2):
        got = o.flashnorm_attn_fwd(Q, K, V, act, 1e-3, 1e-2)
        for t in range(Lq):
            x = [q[0, t, h, d] for h in range(H) for d in range(D)]
            n = len(x)
            mu = sum(x) / n
            var = sum((xi - mu) ** 2 for xi in x) / n
            ln = [(xi - mu) / math.sqrt(var + 1e-3) for xi in x]
            out_o = []
            for h in range(H):
                ps = []
                for j in range(Lkv):
                    sj = sum(ln[h * D + d] * k[0, j, h, d] for d in range(D))
                    if act == 1:
                        sj = 0.5 * sj * (1 + math.tanh(math.sqrt(2 / math.pi) * (sj + 0.044715 * sj ** 3)))
                    elif act == 2:
                        sj = sj / (1 + math.exp(-sj))
                    ps.append(sj)
                for d in range(D):
                    out_o.append(ln[h * D + d] + sum(ps[j] * v[0, j, h, d] for j in range(Lkv)))
            r = 1 / math.sqrt(sum(z * z for z in out_o) / n + 1e-2)
            want = [out_o[i] * r + x[i] for i in range(n)]
            err = max(abs(got[0, t].reshape(-1)[i] - want[i]) for i in range(n))
            assert err <= 1e-12, f"FlashNormAttention brute force (act {act}): {err}"


def pin_fna_reductions(o):
    """V = 0 leaves the two norms and residuals: out = RMSNorm(LayerNorm(q)) + q,
    with both norms over all heads; permuting the heads of Q, K and V permutes
    the output's heads; a jagged batch leaves rows past its length unwritten
    and gives the dense result on the others."""
    B, Lq, Lkv, H, D = 2, 6, 16, 4, 8
    Q, K, V = _fna_case(B, Lq, Lkv, H, D, seed=11)
    Z = bf16_round(np.zeros_like(bf16_to_f64(V)))
    got = o.flashnorm_attn_fwd(Q, K, Z, 1, 1e-5, 1e-6)
    rows = Q.reshape(B * Lq, H * D)
    ln = o.norm_rows(rows, 0, 1e-5)[0]                     # LayerNorm over H*D (pinned above)
    rms = ln / np.sqrt((ln * ln).mean(-1, keepdims=True) + 1e-6)
    want = (rms + bf16_to_f64(rows)).reshape(B, Lq, H, D)
    assert np.max(np.abs(got - want)) <= 1e-12, "V = 0"
    perm = np.array([2, 0, 3, 1])
    base = o.flashnorm_attn_fwd(Q, K, V, 2, 1e-5, 1e-6)
    pq = np.ascontiguousarray(Q[:, :, perm, :])
    pk = np.ascontiguousarray(K[:, :, perm, :])
    pv = np.ascontiguousarray(V[:, :, perm, :])
    assert np.max(np.abs(o.flashnorm_attn_fwd(pq, pk, pv, 2, 1e-5, 1e-6) - base[:, :, perm, :])) <= 1e-12, \
        "head permutation"
    jag = o.flashnorm_attn_fwd(Q, K, V, 2, 1e-5, 1e-6, q_len=[6, 2])
    assert np.array_equal(jag[0], base[0]) and np.array_equal(jag[1, :2], base[1, :2])
    assert np.isnan(jag[1, 2:]).all(), "rows past q_len are not written"


PINS = [pin_bruteforce_plain, pin_bruteforce_prenorm, pin_bruteforce_postnorm,
        pin_bruteforce_norm_rows, pin_torch_f64, pin_lazy_identity, pin_invariants,
        pin_reductions, pin_power_of_two_scale, pin_row_subset, pin_closed_forms,
        pin_bruteforce_norm_bwd, pin_torch_autograd_bwd, pin_norm_bwd_invariants,
        pin_norm_bwd_reductions, pin_prenorm_bwd_bruteforce, pin_prenorm_bwd_autograd,
        pin_prenorm_bwd_reductions, pin_residual_torch, pin_residual_reductions, pin_fna_torch,
        pin_fna_bruteforce, pin_fna_reductions]


def run_all(o):
    """Run every pin; return a list of (name, passed, message)."""
    out = []
    for pin in PINS:
        try:
            pin(o)
            out.append((pin.__name__, True, ""))
        except Exception as e:  # a mutant may also raise or return garbage
            out.append((pin.__name__, False, f"{type(e).__name__}: {e}"[:300]))
    return out


if __name__ == "__main__":
    import oracle
    res = run_all(oracle.Oracle(sys.argv[1]))
    print(json.dumps(res))
