"""Parity of the normalization backward (through the C ABI) with the fp64
oracle: the fused GEMM + norm-backward epilogue (blog "Towards Free
Normalization", §3 "What about backward? Fusion regrouping") and the unfused
row kernel, on small shapes compared element by element over the whole output
and on the full-size post-norm shapes on sampled rows."""
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
def bwd_mode(request):
    nf.set_postnorm_exchange(request.param)
    yield request.param
    nf.set_postnorm_exchange(0)


def _problem(M, K, N, seed, kind, eps=1e-5):
    """A (M x K), B (K x N), gamma, Z (M x N, mean 0.3, std 1.5) and Z's own
    row statistics rounded to fp32, as a forward pass would have saved them."""
    import oracle
    inp = nf_inputs.make_inputs(M, K, N, seed=seed, gamma=True)
    z = nf_inputs.make_inputs(M, N, 8, seed=seed + 7)["X"]
    Z = nf_inputs.bf16_round(nf_inputs.bf16_to_f64(z) * 1.5 + 0.3)
    _, mean, rstd = oracle.get().norm_rows(Z, kind, eps)
    mean32 = None if kind == 1 else mean.astype(np.float32)
    return inp["X"], inp["W"], Z, inp["gamma"], mean32, rstd.astype(np.float32)


def _f32(a, dev):
    import torch
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


def _f64(a):
    return None if a is None else a.astype(np.float64)


def _run_fused(kind, A, B, Z, mean, rstd, gamma, dev, rows=None):
    a, b, z = to_dev(A, dev), to_dev(B, dev), to_dev(Z, dev)
    g = None if gamma is None else to_dev(gamma, dev)
    if kind == 0:
        return nf.gemm_postnorm_ln_bwd(a, b, z, _f32(mean, dev), _f32(rstd, dev), g)
    return nf.gemm_postnorm_rms_bwd(a, b, z, _f32(rstd, dev), g)


# Shapes (M, K, N): one CTA per row (64/128/256 columns, ragged), and rows
# over 2, 3, 4, 8 and 16 tiles (the last ragged), with short and long K.
BWD_SHAPES = [(300, 64, 8), (300, 136, 64), (257, 64, 120), (129, 72, 200), (300, 64, 256),
              (300, 600, 264), (200, 136, 576), (256, 512, 1024), (130, 64, 2048), (129, 520, 4096),
              (64, 64, 4088)]


@pytest.mark.parametrize("M,K,N", BWD_SHAPES)
@pytest.mark.parametrize("kind", [0, 1], ids=["ln", "rms"])
@pytest.mark.parametrize("affine", [False, True])
def test_postnorm_bwd(dev, orc, bwd_mode, M, K, N, kind, affine):
    A, B, Z, G, mean, rstd = _problem(M, K, N, seed=11 * M + K + N, kind=kind)
    G = G if affine else None
    got = _run_fused(kind, A, B, Z, mean, rstd, G, dev)
    want = orc.gemm_postnorm_bwd(A, B, Z, kind, _f64(mean), _f64(rstd), G)
    assert_close(to_f64(got), want, f"bwd kind={kind} {M}x{K}x{N} affine={affine}")


@pytest.mark.parametrize("rows,cols", [(300, 8), (1000, 64), (65, 128), (257, 136), (129, 512),
                                       (33, 2048), (17, 4096), (5, 16384), (3, 1032)])
@pytest.mark.parametrize("kind", [0, 1], ids=["ln", "rms"])
def test_norm_rows_bwd(dev, orc, rows, cols, kind):
    A, _, Z, G, mean, rstd = _problem(rows, cols, cols, seed=rows + cols, kind=kind)
    got = nf.norm_rows_bwd(to_dev(A, dev), to_dev(Z, dev), kind, _f32(mean, dev), _f32(rstd, dev),
                           to_dev(G, dev))
    want = orc.norm_rows_bwd(A, Z, kind, _f64(mean), _f64(rstd), G)
    assert_close(to_f64(got), want, f"norm_rows_bwd kind={kind} {rows}x{cols}")


@pytest.mark.parametrize("kind", [0, 1], ids=["ln", "rms"])
def test_unfused_bwd_pair_matches_fused(dev, orc, kind):
    """Blog §1 baseline for the backward: the plain GEMM writes dY in bf16, the
    row kernel reads it back; both it and the fused kernel meet the bound
    against the oracle's unrounded dY."""
    import torch
    M, K, N = 1000, 512, 768
    A, B, Z, G, mean, rstd = _problem(M, K, N, seed=5, kind=kind)
    want = orc.gemm_postnorm_bwd(A, B, Z, kind, _f64(mean), _f64(rstd), G)
    fused = _run_fused(kind, A, B, Z, mean, rstd, G, dev)
    dy = nf.gemm_plain(to_dev(A, dev), to_dev(B, dev))
    unfused = nf.norm_rows_bwd(dy, to_dev(Z, dev), kind, _f32(mean, dev), _f32(rstd, dev), to_dev(G, dev))
    torch.cuda.synchronize()
    assert_close(to_f64(fused), want, "fused backward")
    assert_close(to_f64(unfused), want, "unfused backward pair")


@pytest.mark.parametrize("M,K,N", [(65536, 128, 128), (16384, 1024, 2048), (8192, 4096, 4096)],
                         ids=["ads_65536x128x128", "affine_16384x1024x2048", "llm_8192x4096x4096"])
@pytest.mark.parametrize("kind", [0, 1], ids=["ln", "rms"])
def test_postnorm_bwd_full_size(dev, orc, M, K, N, kind):
    """The post-norm workloads' shapes, in the benchmark's launch
    configuration; sampled rows against the oracle, and on every row the LN
    gradient's row sum (0 for Z's own statistics, up to rounding)."""
    import torch
    A, B, Z, G, mean, rstd = _problem(M, K, N, seed=M + N, kind=kind)
    got = _run_fused(kind, A, B, Z, mean, rstd, None, dev)
    assert bool(torch.isfinite(got.float()).all())
    rows = nf_inputs.sample_rows(M, 128 if K * N >= 4096 * 4096 else 384, seed=3)
    want = orc.gemm_postnorm_bwd(A, B, Z, kind, _f64(mean), _f64(rstd), None, rows=rows)
    assert_close(to_f64(got)[rows], want, f"bwd full size kind={kind} {M}x{K}x{N}")
    if kind == 0:
        g = got.float()
        rel = (g.sum(-1).abs() / g.abs().sum(-1).clamp_min(1e-30)).max().item()
        assert rel < 2e-2, f"LN backward rows should sum to ~0 (max relative row sum {rel})"
