"""CTA pairs (tcgen05 cta_group::2) for the plain and Lazy Pre-Norm GEMMs:
two CTAs of a cluster along M compute a 256 x 256 tile, each loading its own
128 rows of X and half of W's columns.  Parity with the fp64 oracle through
the C ABI on ragged shapes (an odd number of 128-row tiles leaves the last
pair's second CTA without rows), several tiles per cluster (accumulator
reuse across the pair) and the full 8192 x 4096 x 4096 workload; repeated
calls give the same bits."""
import numpy as np
import pytest

import nf_inputs
import normalization_gemm_gb300 as nf
from gpu_util import assert_close, require_gpu, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    d = require_gpu()
    from normalization_gemm_gb300 import _build
    _build.build()
    nf.clear_device_status()
    nf.set_wait_timeout_ns(250_000_000)
    nf.set_gemm_pair(2)
    yield d
    nf.set_gemm_pair(0)
    import torch
    torch.cuda.synchronize()
    status, detail = nf.device_status()
    assert status == nf.NF_OK, f"device status word set: {detail}"


@pytest.fixture(scope="module")
def orc():
    import oracle
    return oracle.get()


# (M, K, N): ragged M / K / N, odd tile counts, several pair tiles per cluster
PAIR_SHAPES = [(300, 200, 320), (256, 64, 256), (513, 520, 264), (257, 64, 456), (1024, 1024, 1024),
               (8192, 256, 2048), (2000, 1000, 600)]


@pytest.mark.parametrize("M,K,N", PAIR_SHAPES)
def test_pair_plain(dev, orc, M, K, N):
    import torch
    assert nf.plan_gemm(0, M, N, K, 148)["cluster"] == 2
    inp = nf_inputs.make_inputs(M, K, N, seed=M + 3 * K + N)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    y = nf.gemm_plain(X, W)
    y2 = nf.gemm_plain(X, W)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    assert_close(to_f64(y), orc.gemm_plain(inp["X"], inp["W"]), f"pair plain {M}x{K}x{N}")


@pytest.mark.parametrize("M,K,N", PAIR_SHAPES)
@pytest.mark.parametrize("x_dist", ["normal", "row_scaled"])
def test_pair_prenorm_rms(dev, orc, M, K, N, x_dist):
    import torch
    assert nf.plan_gemm(1, M, N, K, 148)["cluster"] == 2
    inp = nf_inputs.make_inputs(M, K, N, seed=2 * M + K + N, x_dist=x_dist)
    rstd = torch.full((M,), -1.0, dtype=torch.float32, device=dev)
    y = nf.gemm_prenorm_rms(to_dev(inp["X"], dev), to_dev(inp["W"], dev), 1e-6, rstd_out=rstd)
    ref, rref = orc.gemm_prenorm_rms(inp["X"], inp["W"], 1e-6)
    assert_close(to_f64(y), ref, f"pair pre {M}x{K}x{N} {x_dist}")
    np.testing.assert_allclose(rstd.cpu().numpy(), rref, rtol=1e-4)


def test_pair_full_size_llm(dev, orc):
    """8192 x 4096 x 4096, both ops, sampled rows against the oracle."""
    import torch
    w = nf_inputs.WORKLOADS["llm_8192x4096x4096"]
    inp = nf_inputs.workload_inputs(w)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    rows = nf_inputs.sample_rows(w.M, 128, seed=4)
    idx = torch.from_numpy(rows).to(dev)
    y = nf.gemm_prenorm_rms(X, W, w.eps)
    assert_close(to_f64(y[idx]), orc.gemm_prenorm_rms(inp["X"], inp["W"], w.eps, rows=rows)[0], "pair pre llm")
    yp = nf.gemm_plain(X, W)
    assert_close(to_f64(yp[idx]), orc.gemm_plain(inp["X"], inp["W"], rows=rows), "pair plain llm")


def test_pair_matches_single_cta_tiles(dev):
    """The pair computes the same products in the same order as one CTA per
    tile: identical bits on a shape with tensor-bound tiles."""
    import torch
    M, K, N = 1024, 2048, 1024
    inp = nf_inputs.make_inputs(M, K, N, seed=17)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    a = nf.gemm_prenorm_rms(X, W, 1e-6)
    nf.set_gemm_pair(1)
    try:
        b = nf.gemm_prenorm_rms(X, W, 1e-6)
    finally:
        nf.set_gemm_pair(2)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# Post-norm rows exchanged through L2 (K >= 512, N > 512), computed by CTA
# pairs: ragged M (an odd number of row tiles), ragged N, gamma / beta.
POST_PAIR_SHAPES = [(1000, 512, 1024), (513, 640, 4096), (2000, 1024, 2048), (300, 520, 1032)]


@pytest.mark.parametrize("M,K,N", POST_PAIR_SHAPES)
@pytest.mark.parametrize("kind", ["ln", "rms"])
def test_pair_postnorm(dev, orc, M, K, N, kind):
    import torch
    op = 2 if kind == "ln" else 3
    p = nf.plan_gemm(op, M, N, K, 148)
    assert p["cluster"] == 2 and p["exchange"] == nf.XCH_GLOBAL
    inp = nf_inputs.make_inputs(M, K, N, seed=M + K + 5 * N, gamma=True, beta=True)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    G, B = to_dev(inp["gamma"], dev), to_dev(inp["beta"], dev)
    rstd = torch.full((M,), -1.0, dtype=torch.float32, device=dev)
    if kind == "ln":
        mean = torch.full((M,), 7.0, dtype=torch.float32, device=dev)
        y = nf.gemm_postnorm_ln(X, W, 1e-5, G, B, mean_out=mean, rstd_out=rstd)
        y2 = nf.gemm_postnorm_ln(X, W, 1e-5, G, B)
        ref, mref, rref = orc.gemm_postnorm_ln(inp["X"], inp["W"], 1e-5, inp["gamma"], inp["beta"])
        np.testing.assert_allclose(mean.cpu().numpy(), mref, rtol=1e-3, atol=1e-3)
    else:
        y = nf.gemm_postnorm_rms(X, W, 1e-5, G, rstd_out=rstd)
        y2 = nf.gemm_postnorm_rms(X, W, 1e-5, G)
        ref, rref = orc.gemm_postnorm_rms(inp["X"], inp["W"], 1e-5, inp["gamma"])
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    assert_close(to_f64(y), ref, f"pair post-{kind} {M}x{K}x{N}")
    np.testing.assert_allclose(rstd.cpu().numpy(), rref, rtol=1e-3)


def test_pair_postnorm_full_size_llm(dev, orc):
    """8192 x 4096 x 4096 post-LN through CTA pairs and the L2 exchange,
    sampled rows against the oracle, every row's moments; the no-alloc entry
    point gives the same bits."""
    import torch
    w = nf_inputs.WORKLOADS["llm_8192x4096x4096"]
    inp = nf_inputs.workload_inputs(w)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    y = nf.gemm_postnorm_ln(X, W, w.eps)
    y2 = nf.gemm_postnorm_ln_noalloc(X, W, w.eps)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    rows = nf_inputs.sample_rows(w.M, 128, seed=8)
    ref = orc.gemm_postnorm_ln(inp["X"], inp["W"], w.eps, rows=rows)[0]
    assert_close(to_f64(y[torch.from_numpy(rows).to(dev)]), ref, "pair post-LN llm")
    yf = y.float()
    assert float(yf.mean(-1).abs().max()) < 2e-2 and float(((yf * yf).mean(-1) - 1).abs().max()) < 2e-2
