"""Parity of the residual-add post-norm (H = X W + R, Y = norm(H), H written
back as the updated residual) through the C ABI with the fp64 oracle, and of
the unfused residual-add row norm.  CUDA book chapter "Element-wise 与算子融合"
§8.4 / §8.5.1; the norm over the GEMM output as in blog "Towards Free
Normalization" §3."""
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
    yield d
    import torch
    torch.cuda.synchronize()
    status, detail = nf.device_status()
    assert status == nf.NF_OK, f"device status word set: {detail}"


@pytest.fixture(scope="module")
def orc():
    import oracle
    return oracle.get()


@pytest.fixture(params=[0, nf.XCH_GLOBAL, nf.XCH_CLUSTER], ids=["auto", "global", "cluster"])
def res_mode(request):
    """Rows wider than 256 columns: the automatic exchange, through L2, or in
    a cluster of 256-column CTAs."""
    nf.set_postnorm_exchange(request.param)
    yield request.param
    nf.set_postnorm_exchange(0)


def _problem(M, K, N, seed):
    inp = nf_inputs.make_inputs(M, K, N, seed=seed, gamma=True, beta=True)
    Rs = nf_inputs.make_inputs(M, N, 8, seed=seed + 1)["X"]
    return inp["X"], inp["W"], Rs, inp["gamma"], inp["beta"]


# (M, K, N): one CTA per row (N <= 256), a cluster of two (N <= 512), wider
# rows over the exchanges; ragged M, K and N; K >= 512 for the automatic L2
# exchange.
RES_SHAPES = [(300, 64, 8), (300, 136, 64), (257, 64, 120), (384, 128, 128), (129, 72, 200),
              (300, 64, 264), (200, 136, 576), (130, 64, 2048), (64, 64, 4088), (300, 520, 1032)]


@pytest.mark.parametrize("M,K,N", RES_SHAPES)
@pytest.mark.parametrize("kind", [0, 1], ids=["ln", "rms"])
@pytest.mark.parametrize("affine", [False, True])
def test_residual_postnorm(dev, orc, res_mode, M, K, N, kind, affine):
    import torch
    X, W, Rs, G, B = _problem(M, K, N, seed=7 * M + K + N)
    g = G if affine else None
    b = B if (affine and kind == 0) else None
    x, w, r = to_dev(X, dev), to_dev(W, dev), to_dev(Rs, dev)
    h = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    mean = torch.zeros(M, dtype=torch.float32, device=dev)
    rstd = torch.zeros(M, dtype=torch.float32, device=dev)
    gd = None if g is None else to_dev(g, dev)
    if kind == 0:
        y = nf.gemm_postnorm_ln_res(x, w, r, 1e-5, gd, None if b is None else to_dev(b, dev), h_out=h,
                                    mean_out=mean, rstd_out=rstd)
    else:
        y = nf.gemm_postnorm_rms_res(x, w, r, 1e-5, gd, h_out=h, rstd_out=rstd)
    torch.cuda.synchronize()
    Y, H, mref, rref = orc.gemm_postnorm_res(X, W, Rs, kind, 1e-5, g, b)
    what = f"residual {'ln' if kind == 0 else 'rms'} {M}x{K}x{N} affine={affine}"
    assert_close(to_f64(y), Y, what)
    assert_close(to_f64(h), H, what + " H")
    np.testing.assert_allclose(rstd.cpu().numpy(), rref, rtol=1e-3)
    if kind == 0:
        np.testing.assert_allclose(mean.cpu().numpy(), mref, atol=1e-3 / rref.min(), rtol=1e-3)


@pytest.mark.parametrize("M,K,N", [(300, 136, 64), (200, 136, 576), (130, 64, 2048), (300, 520, 1032)])
def test_residual_in_place_and_without_h(dev, orc, res_mode, M, K, N):
    """H written over R itself (the residual stream updated in place), and no
    H at all: the same Y."""
    import torch
    X, W, Rs, G, B = _problem(M, K, N, seed=M + 3 * N)
    x, w = to_dev(X, dev), to_dev(W, dev)
    r = to_dev(Rs, dev)
    y0 = nf.gemm_postnorm_ln_res(x, w, r, 1e-5, to_dev(G, dev), to_dev(B, dev))
    y1 = nf.gemm_postnorm_ln_res(x, w, r, 1e-5, to_dev(G, dev), to_dev(B, dev), h_out=r)
    torch.cuda.synchronize()
    Y, H, _, _ = orc.gemm_postnorm_res(X, W, Rs, 0, 1e-5, G, B)
    assert torch.equal(y0, y1)
    assert_close(to_f64(y1), Y, f"in place {M}x{K}x{N}")
    assert_close(to_f64(r), H, f"in place H {M}x{K}x{N}")
    r2 = to_dev(Rs, dev)
    y2 = nf.gemm_postnorm_rms_res(x, w, r2, 1e-5, to_dev(G, dev), h_out=r2)
    torch.cuda.synchronize()
    Y, H, _, _ = orc.gemm_postnorm_res(X, W, Rs, 1, 1e-5, G)
    assert_close(to_f64(y2), Y, f"in place rms {M}x{K}x{N}")
    assert_close(to_f64(r2), H, f"in place rms H {M}x{K}x{N}")


def test_residual_zero_is_the_plain_postnorm(dev):
    """R = 0: bit for bit the post-norm kernel without a residual (same
    exchange), and H = bf16(X W)."""
    import torch
    M, K, N = 1000, 256, 1024
    X, W, _, G, B = _problem(M, K, N, seed=41)
    x, w, g, b = to_dev(X, dev), to_dev(W, dev), to_dev(G, dev), to_dev(B, dev)
    zero = torch.zeros((M, N), dtype=torch.bfloat16, device=dev)
    h = torch.empty_like(zero)
    nf.set_postnorm_tile_n(256)
    try:
        y0 = nf.gemm_postnorm_ln(x, w, 1e-5, g, b)
        y1 = nf.gemm_postnorm_ln_res(x, w, zero, 1e-5, g, b, h_out=h)
        z = nf.gemm_plain(x, w)
    finally:
        nf.set_postnorm_tile_n(0)
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
    assert torch.equal(h, z)


@pytest.mark.parametrize("rows,cols", [(300, 8), (1000, 64), (257, 136), (129, 512), (33, 2048), (5, 16384)])
@pytest.mark.parametrize("kind", [0, 1], ids=["ln", "rms"])
def test_norm_rows_res(dev, orc, rows, cols, kind):
    """The unfused residual-add norm: out = norm(in + R), H = bf16(in + R)."""
    import torch
    inp = nf_inputs.make_inputs(rows, cols, cols, seed=rows + cols, gamma=True, beta=True)
    A = inp["X"]
    Rs = nf_inputs.make_inputs(rows, cols, 8, seed=rows + cols + 1)["X"]
    a, r = to_dev(A, dev), to_dev(Rs, dev)
    G = nf_inputs.make_inputs(8, 8, cols, seed=cols, gamma=True, beta=True)
    g, b = G["gamma"], (G["beta"] if kind == 0 else None)
    h = torch.empty_like(a)
    y = nf.norm_rows_res(a, r, kind, 1e-5, to_dev(g, dev), None if b is None else to_dev(b, dev), h_out=h)
    torch.cuda.synchronize()
    eye = nf_inputs.bf16_round(np.eye(cols))
    Y, H, _, _ = orc.gemm_postnorm_res(A, eye, Rs, kind, 1e-5, g, b)
    assert_close(to_f64(y), Y, f"norm_rows_res {rows}x{cols}")
    assert_close(to_f64(h), H, f"norm_rows_res H {rows}x{cols}")


def test_unfused_residual_pair(dev, orc):
    """The unfused baseline of the residual post-norm: the plain GEMM, then the
    residual-add row norm; against the oracle (bf16 intermediate)."""
    import torch
    M, K, N = 1000, 512, 1024
    X, W, Rs, G, B = _problem(M, K, N, seed=77)
    x, w, r = to_dev(X, dev), to_dev(W, dev), to_dev(Rs, dev)
    z = nf.gemm_plain(x, w)
    h = torch.empty_like(z)
    y = nf.norm_rows_res(z, r, nf.NORM_LN, 1e-5, to_dev(G, dev), to_dev(B, dev), h_out=h)
    torch.cuda.synchronize()
    Y, H, _, _ = orc.gemm_postnorm_res(X, W, Rs, 0, 1e-5, G, B)
    assert_close(to_f64(y), Y, "unfused residual pair")
    assert_close(to_f64(h), H, "unfused residual pair H")


@pytest.mark.parametrize("name", ["post_ln_65536x128x128", "post_affine_16384x1024x2048", "llm_8192x4096x4096"])
def test_residual_full_size(dev, orc, name):
    """The benchmark's post-norm shapes with a residual, on sampled rows."""
    import torch
    w = nf_inputs.WORKLOADS[name]
    inp = nf_inputs.workload_inputs(w)
    Rs = nf_inputs.make_inputs(w.M, w.N, 8, seed=11)["X"]
    X, W, R = to_dev(inp["X"], dev), to_dev(inp["W"], dev), to_dev(Rs, dev)
    G = to_dev(inp["gamma"], dev) if w.gamma else None
    B = to_dev(inp["beta"], dev) if w.beta else None
    h = torch.empty_like(R)
    y = nf.gemm_postnorm_ln_res(X, W, R, w.eps, G, B, h_out=h)
    torch.cuda.synchronize()
    rows = nf_inputs.sample_rows(w.M, 128)
    Y, H, _, _ = orc.gemm_postnorm_res(inp["X"], inp["W"], Rs, 0, w.eps, inp.get("gamma"), inp.get("beta"),
                                       rows=rows)
    idx = torch.from_numpy(rows).to(dev)
    assert bool(torch.isfinite(y.float()).all())
    assert_close(to_f64(y[idx]), Y, f"{name} residual")
    assert_close(to_f64(h[idx]), H, f"{name} residual H")
