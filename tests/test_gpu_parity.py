"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Small shapes span several tiles and ragged tails on every dimension and are
compared element by element over the whole output; the five full-size
workloads run in the benchmark's launch configuration and are compared on
sampled rows (the oracle computes rows independently), with whole-output
properties (finite values, per-row moments) checked on every row.
"""
import numpy as np
import pytest

import nf_inputs
import normalization_gemm_gb300 as nf
from gpu_util import ATOL, RTOL, assert_close, require_gpu, to_dev, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    d = require_gpu()
    from normalization_gemm_gb300 import _build
    _build.build()
    nf.clear_device_status()
    # Every kernel here finishes in milliseconds: a pipeline wait that needs
    # more than 250 ms is a bug, reported as NF_ERR_TIMEOUT instead of a stall.
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


def _inputs(M, K, N, seed, **kw):
    return nf_inputs.make_inputs(M, K, N, seed=seed, **kw)


# Shapes: (M, K, N).  Ragged M (not a multiple of 128), K (not of 64) and N
# (not of the tile), single rows, the smallest legal K and N, several tiles.
GEMM_SHAPES = [(256, 64, 64), (300, 200, 320), (1, 8, 8), (129, 72, 136), (513, 520, 264),
               (130, 1032, 8), (384, 128, 128), (257, 64, 456)]


@pytest.mark.parametrize("M,K,N", GEMM_SHAPES)
def test_plain(dev, orc, M, K, N):
    inp = _inputs(M, K, N, seed=M + K + N)
    y = nf.gemm_plain(to_dev(inp["X"], dev), to_dev(inp["W"], dev))
    assert_close(to_f64(y), orc.gemm_plain(inp["X"], inp["W"]), f"plain {M}x{K}x{N}")


@pytest.mark.parametrize("M,K,N", GEMM_SHAPES)
@pytest.mark.parametrize("x_dist", ["normal", "row_scaled"])
def test_prenorm_rms(dev, orc, M, K, N, x_dist):
    import torch
    inp = _inputs(M, K, N, seed=2 * M + K + N, x_dist=x_dist)
    rstd = torch.full((M,), -1.0, dtype=torch.float32, device=dev)
    y = nf.gemm_prenorm_rms(to_dev(inp["X"], dev), to_dev(inp["W"], dev), 1e-6, rstd_out=rstd)
    ref, rref = orc.gemm_prenorm_rms(inp["X"], inp["W"], 1e-6)
    assert_close(to_f64(y), ref, f"pre {M}x{K}x{N} {x_dist}")
    np.testing.assert_allclose(rstd.cpu().numpy(), rref, rtol=1e-4)


# Post-norm shapes: N covers one CTA (64/128/256 tiles, ragged) and clusters
# of 2, 3, 4, 8 and 16 CTAs (the last with a ragged CTA).
POST_SHAPES = [(300, 64, 8), (300, 136, 64), (257, 64, 120), (384, 128, 128), (129, 72, 200),
               (300, 64, 256), (300, 64, 264), (200, 136, 576), (256, 128, 1024),
               (130, 64, 2048), (129, 64, 4096), (64, 64, 4088)]


@pytest.fixture(params=[(0, 0), (nf.XCH_GLOBAL, 0), (nf.XCH_CLUSTER, 512), (nf.XCH_CLUSTER, 256)],
                ids=["auto", "global", "cluster512", "cluster256"])
def post_mode(request):
    """How rows wider than 256 columns exchange statistics: the automatic
    choice, through L2 between 256-column tiles, or inside a thread-block
    cluster of 512-column CTAs (<= 8) or of 256-column CTAs (<= 16)."""
    xch, tile = request.param
    nf.set_postnorm_exchange(xch)
    nf.set_postnorm_tile_n(tile)
    yield request.param
    nf.set_postnorm_exchange(0)
    nf.set_postnorm_tile_n(0)


@pytest.mark.parametrize("M,K,N", POST_SHAPES)
@pytest.mark.parametrize("affine", [False, True])
def test_postnorm_ln(dev, orc, post_mode, M, K, N, affine):
    import torch
    inp = _inputs(M, K, N, seed=3 * M + K + N, gamma=True, beta=True)
    g = inp["gamma"] if affine else None
    b = inp["beta"] if affine else None
    mean = torch.zeros(M, dtype=torch.float32, device=dev)
    rstd = torch.zeros(M, dtype=torch.float32, device=dev)
    y = nf.gemm_postnorm_ln(to_dev(inp["X"], dev), to_dev(inp["W"], dev), 1e-5,
                            None if g is None else to_dev(g, dev), None if b is None else to_dev(b, dev),
                            mean_out=mean, rstd_out=rstd)
    ref, mref, rref = orc.gemm_postnorm_ln(inp["X"], inp["W"], 1e-5, g, b)
    assert_close(to_f64(y), ref, f"post-ln {M}x{K}x{N} affine={affine}")
    np.testing.assert_allclose(rstd.cpu().numpy(), rref, rtol=1e-3)
    np.testing.assert_allclose(mean.cpu().numpy(), mref, atol=1e-3 / rref.min(), rtol=1e-3)


@pytest.mark.parametrize("M,K,N", POST_SHAPES)
@pytest.mark.parametrize("affine", [False, True])
def test_postnorm_rms(dev, orc, post_mode, M, K, N, affine):
    import torch
    inp = _inputs(M, K, N, seed=5 * M + K + N, gamma=True)
    g = inp["gamma"] if affine else None
    rstd = torch.zeros(M, dtype=torch.float32, device=dev)
    y = nf.gemm_postnorm_rms(to_dev(inp["X"], dev), to_dev(inp["W"], dev), 1e-5,
                             None if g is None else to_dev(g, dev), rstd_out=rstd)
    ref, rref = orc.gemm_postnorm_rms(inp["X"], inp["W"], 1e-5, g)
    assert_close(to_f64(y), ref, f"post-rms {M}x{K}x{N} affine={affine}")
    np.testing.assert_allclose(rstd.cpu().numpy(), rref, rtol=1e-3)


@pytest.mark.parametrize("rows,cols", [(300, 8), (1000, 64), (65, 128), (257, 136), (129, 512),
                                       (33, 2048), (17, 4096), (5, 16384), (3, 1032)])
@pytest.mark.parametrize("kind", [0, 1])
def test_norm_rows(dev, orc, rows, cols, kind):
    import torch
    inp = _inputs(rows, cols, cols, seed=rows + cols + kind, gamma=True, beta=True, w_var=1.0)
    X = inp["X"]
    G = inp["gamma"]
    B = inp["beta"] if kind == 0 else None
    mean = torch.zeros(rows, dtype=torch.float32, device=dev)
    rstd = torch.zeros(rows, dtype=torch.float32, device=dev)
    y = nf.norm_rows(to_dev(X, dev), kind, 1e-5, to_dev(G, dev), None if B is None else to_dev(B, dev),
                     mean_out=mean, rstd_out=rstd)
    ref, mref, rref = orc.norm_rows(X, kind, 1e-5, G, B)
    assert_close(to_f64(y), ref, f"norm_rows {rows}x{cols} kind={kind}")
    np.testing.assert_allclose(rstd.cpu().numpy(), rref, rtol=1e-4)
    if kind == 0:
        np.testing.assert_allclose(mean.cpu().numpy(), mref, atol=1e-5, rtol=1e-4)


# ------------------------------------------------------------ persistence
def test_many_tiles_per_cta(dev, orc):
    """Several tiles per persistent CTA: both TMEM buffers and every ring stage
    are reused many times (M = 3 waves of 128-row tiles per SM plus a tail)."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    M = 128 * sms * 3 + 77
    inp = _inputs(M, 192, 64, seed=17)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    rows = nf_inputs.sample_rows(M, 400, seed=3)
    y = to_f64(nf.gemm_prenorm_rms(X, W, 1e-6))[rows]
    assert_close(y, orc.gemm_prenorm_rms(inp["X"], inp["W"], 1e-6, rows=rows)[0], "pre persistent")
    y = to_f64(nf.gemm_postnorm_ln(X, W, 1e-5))[rows]
    assert_close(y, orc.gemm_postnorm_ln(inp["X"], inp["W"], 1e-5, rows=rows)[0], "post-ln persistent")
    y = to_f64(nf.gemm_plain(X, W))[rows]
    assert_close(y, orc.gemm_plain(inp["X"], inp["W"], rows=rows), "plain persistent")


def test_cluster_many_tiles_per_cluster(dev, orc, post_mode):
    """Row tiles many times the resident CTAs: cluster exchange barriers and
    both receive buffers cycle through many phases; global-exchange counters
    go up and back to zero many times within one launch."""
    M = 128 * 64 + 5
    inp = _inputs(M, 64, 4096, seed=19, gamma=True, beta=True)
    rows = nf_inputs.sample_rows(M, 160, seed=4)
    y = nf.gemm_postnorm_ln(to_dev(inp["X"], dev), to_dev(inp["W"], dev), 1e-6,
                            to_dev(inp["gamma"], dev), to_dev(inp["beta"], dev))
    ref = orc.gemm_postnorm_ln(inp["X"], inp["W"], 1e-6, inp["gamma"], inp["beta"], rows=rows)[0]
    assert_close(to_f64(y)[rows], ref, f"post-ln {post_mode}, many row tiles")


# ------------------------------------------------------------ full-size workloads
def _row_moments(y):
    import torch
    yf = y.float()
    return yf.mean(-1), (yf * yf).mean(-1)


@pytest.mark.parametrize("name", nf_inputs.WORKLOAD_ORDER)
def test_full_size_workloads(dev, orc, name):
    import torch
    w = nf_inputs.WORKLOADS[name]
    inp = nf_inputs.workload_inputs(w)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    G = to_dev(inp["gamma"], dev) if w.gamma else None
    B = to_dev(inp["beta"], dev) if w.beta else None
    rows = nf_inputs.sample_rows(w.M, 128 if w.K * w.N >= 4096 * 4096 else 512)
    for op in w.ops:
        if op == "pre_rms":
            y = nf.gemm_prenorm_rms(X, W, w.eps)
            ref = orc.gemm_prenorm_rms(inp["X"], inp["W"], w.eps, rows=rows)[0]
        elif op == "post_ln":
            y = nf.gemm_postnorm_ln(X, W, w.eps, G, B)
            ref = orc.gemm_postnorm_ln(inp["X"], inp["W"], w.eps, inp.get("gamma"), inp.get("beta"),
                                       rows=rows)[0]
        else:
            y = nf.gemm_postnorm_rms(X, W, w.eps, G)
            ref = orc.gemm_postnorm_rms(inp["X"], inp["W"], w.eps, inp.get("gamma"), rows=rows)[0]
        assert bool(torch.isfinite(y.float()).all()), f"{name} {op}: non-finite output"
        assert_close(to_f64(y[torch.from_numpy(rows).to(dev)]), ref, f"{name} {op}")
        if op in ("post_ln", "post_rms") and G is None:
            # every row of a no-affine post-norm: mean 0 (LN) and mean square
            # var/(var+eps) ~ 1 up to bf16 rounding
            mu, ms = _row_moments(y)
            if op == "post_ln":
                assert float(mu.abs().max()) < 2e-2, f"{name}: LN row mean"
            assert float((ms - 1).abs().max()) < 2e-2, f"{name}: row mean square"


@pytest.mark.parametrize("tile_n", [256, 512], ids=["cluster16x256", "cluster8x512"])
def test_llm_post_ln_row_cluster_full_shape(dev, orc, tile_n):
    """The 8192 x 4096 x 4096 post-LN with the blog §3 layout: a thread-block
    cluster spans the 4096-column row (16 CTAs of 256 columns, or 8 of 512),
    partial statistics through DSMEM, at the full shape: sampled rows against
    the oracle, every row's moments, and the same bits as a second call."""
    import torch
    w = nf_inputs.WORKLOADS["llm_8192x4096x4096"]
    inp = nf_inputs.workload_inputs(w)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    nf.set_postnorm_exchange(nf.XCH_CLUSTER)
    nf.set_postnorm_tile_n(tile_n)
    try:
        y = nf.gemm_postnorm_ln(X, W, w.eps)
        y2 = nf.gemm_postnorm_ln(X, W, w.eps)
        torch.cuda.synchronize()
    finally:
        nf.set_postnorm_exchange(0)
        nf.set_postnorm_tile_n(0)
    assert torch.equal(y, y2)
    rows = nf_inputs.sample_rows(w.M, 128, seed=9)
    ref = orc.gemm_postnorm_ln(inp["X"], inp["W"], w.eps, rows=rows)[0]
    assert_close(to_f64(y[torch.from_numpy(rows).to(dev)]), ref, f"llm post-LN cluster of {tile_n}-column CTAs")
    mu, ms = _row_moments(y)
    assert float(mu.abs().max()) < 2e-2 and float((ms - 1).abs().max()) < 2e-2


def test_unfused_pair_matches_fused(dev, orc):
    """Blog §1 baseline pair (GEMM + separate norm kernel) against the fused
    kernels, both against the oracle, on the same inputs."""
    import torch
    M, K, N = 1000, 512, 512
    inp = _inputs(M, K, N, seed=23, x_dist="row_scaled", gamma=True, beta=True)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    G, B = to_dev(inp["gamma"], dev), to_dev(inp["beta"], dev)
    # pre-norm: RMSNorm(X) materialised in bf16, then the GEMM
    xn = nf.norm_rows(X, nf.NORM_RMS, 1e-6)
    unf = to_f64(nf.gemm_plain(xn, W))
    fused = to_f64(nf.gemm_prenorm_rms(X, W, 1e-6))
    ref = orc.gemm_prenorm_rms(inp["X"], inp["W"], 1e-6)[0]
    assert_close(unf, ref, "unfused pre")
    assert_close(fused, ref, "fused pre")
    # post-norm: GEMM materialised in bf16, then LayerNorm
    z = nf.gemm_plain(X, W)
    unf = to_f64(nf.norm_rows(z, nf.NORM_LN, 1e-5, G, B))
    fused = to_f64(nf.gemm_postnorm_ln(X, W, 1e-5, G, B))
    ref = orc.gemm_postnorm_ln(inp["X"], inp["W"], 1e-5, inp["gamma"], inp["beta"])[0]
    assert_close(unf, ref, "unfused post")
    assert_close(fused, ref, "fused post")


# ------------------------------------------------------------ edge cases
def test_degenerate_rows(dev, orc):
    """Zero rows (RMS: output 0, rstd = 1/sqrt(eps)) and constant-output rows
    (LN: output beta)."""
    import torch
    M, K, N = 200, 64, 576
    inp = _inputs(M, K, N, seed=29, gamma=True, beta=True)
    X = inp["X"].copy()
    X[3] = 0
    X[130] = 0
    W = inp["W"].copy()
    Wc = W.copy()
    Wc[:] = nf_inputs.bf16_round(np.ones((K, N)) * 0.25)   # every column equal: Z rows constant
    for Wm in (W, Wc):
        for fn in ("ln", "rms"):
            if fn == "ln":
                y = nf.gemm_postnorm_ln(to_dev(X, dev), to_dev(Wm, dev), 1e-5,
                                        to_dev(inp["gamma"], dev), to_dev(inp["beta"], dev))
                ref = orc.gemm_postnorm_ln(X, Wm, 1e-5, inp["gamma"], inp["beta"])[0]
            else:
                y = nf.gemm_postnorm_rms(to_dev(X, dev), to_dev(Wm, dev), 1e-5, to_dev(inp["gamma"], dev))
                ref = orc.gemm_postnorm_rms(X, Wm, 1e-5, inp["gamma"])[0]
            assert_close(to_f64(y), ref, f"degenerate post-{fn}")
    rstd = torch.zeros(M, dtype=torch.float32, device=dev)
    y = nf.gemm_prenorm_rms(to_dev(X, dev), to_dev(W, dev), 1e-6, rstd_out=rstd)
    assert float(y[3].float().abs().max()) == 0.0
    assert abs(float(rstd[3]) - 1e3) < 1.0


def test_empty_m_leaves_output_untouched(dev):
    import torch
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device=dev)
    w = torch.zeros((64, 64), dtype=torch.bfloat16, device=dev)
    y = torch.full((0, 64), 1.0, dtype=torch.bfloat16, device=dev)
    nf.gemm_postnorm_ln(x, w, 1e-5, out=y)
    nf.gemm_prenorm_rms(x, w, 1e-5, out=y)
    nf.norm_rows(x, 0, 1e-5, out=torch.empty((0, 64), dtype=torch.bfloat16, device=dev))


@pytest.mark.parametrize("op", ["plain", "pre", "post_ln"])
def test_guard_band_around_output(dev, op):
    """Stores are clipped to M x N: canary rows before and after Y survive."""
    import torch
    M, K, N = 201, 64, 264
    inp = _inputs(M, K, N, seed=31)
    buf = torch.full(((M + 4) * N,), 7.0, dtype=torch.bfloat16, device=dev)
    y = buf[2 * N:(M + 2) * N].view(M, N)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    if op == "plain":
        nf.gemm_plain(X, W, out=y)
    elif op == "pre":
        nf.gemm_prenorm_rms(X, W, 1e-6, out=y)
    else:
        nf.gemm_postnorm_ln(X, W, 1e-5, out=y)
    torch.cuda.synchronize()
    assert bool((buf[:2 * N] == 7.0).all()) and bool((buf[(M + 2) * N:] == 7.0).all())


def test_repeated_calls_are_deterministic(dev):
    import torch
    inp = _inputs(1000, 256, 2048, seed=37, gamma=True, beta=True)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    G, B = to_dev(inp["gamma"], dev), to_dev(inp["beta"], dev)
    a = nf.gemm_postnorm_ln(X, W, 1e-5, G, B)
    b = nf.gemm_postnorm_ln(X, W, 1e-5, G, B)
    assert torch.equal(a, b)
    a = nf.gemm_prenorm_rms(X, W, 1e-6)
    b = nf.gemm_prenorm_rms(X, W, 1e-6)
    assert torch.equal(a, b)


def test_wait_timeout_is_reported_not_hung(dev):
    """A barrier nobody arrives on: the bounded wait gives up after 5 ms and
    records NF_ERR_TIMEOUT; the context stays usable."""
    import torch
    torch.cuda.synchronize()
    nf.clear_device_status()
    nf.selftest_wait_timeout(5_000_000)
    status, detail = nf.device_status()
    assert status == 5 and detail[1] == 9, (status, detail)
    nf.clear_device_status()
    assert nf.device_status()[0] == nf.NF_OK
    # the device still computes correctly afterwards
    inp = _inputs(128, 64, 64, seed=41)
    y = nf.gemm_plain(to_dev(inp["X"], dev), to_dev(inp["W"], dev))
    torch.cuda.synchronize()
    assert bool(torch.isfinite(y.float()).all())


def test_launch_overlap_keeps_dependent_chains_exact(dev):
    """Programmatic dependent launch: each kernel below reads the previous one's
    output.  With the overlap on, every result must be bit-identical to the
    serialized run (griddepcontrol.wait precedes every global access)."""
    import torch
    inp = _inputs(4096, 256, 256, seed=43, gamma=True, beta=True)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    G, B = to_dev(inp["gamma"], dev), to_dev(inp["beta"], dev)

    def chain():
        outs = []
        y = X
        for i in range(6):
            y = nf.gemm_postnorm_ln(y, W, 1e-5, G, B) if i % 3 == 0 else (
                nf.gemm_prenorm_rms(y, W, 1e-6) if i % 3 == 1 else nf.norm_rows(nf.gemm_plain(y, W), 0, 1e-5))
            outs.append(y)
        torch.cuda.synchronize()
        return outs

    try:
        nf.set_launch_overlap(False)
        ref = chain()
        nf.set_launch_overlap(True)
        for _ in range(3):
            got = chain()
            for a, b in zip(ref, got):
                assert torch.equal(a, b)
    finally:
        nf.set_launch_overlap(True)


@pytest.mark.parametrize("op", ["plain", "pre", "post_ln", "post_rms"])
def test_split_last_wave_whole_output(dev, orc, op):
    """Short-K shapes whose last wave holds few tiles run them as 64-row halves:
    two extra tiles here, the last with 72 rows (its second half has 8)."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    M, K, N = 128 * sms * 2 + 128 + 72, 64, 128
    inp = _inputs(M, K, N, seed=47, gamma=True, beta=True)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    stats = torch.full((M,), -7.0, dtype=torch.float32, device=dev)
    if op == "plain":
        got, want = nf.gemm_plain(X, W), orc.gemm_plain(inp["X"], inp["W"])
    elif op == "pre":
        got = nf.gemm_prenorm_rms(X, W, 1e-6, rstd_out=stats)
        want, wstat = orc.gemm_prenorm_rms(inp["X"], inp["W"], 1e-6)
    elif op == "post_ln":
        got = nf.gemm_postnorm_ln(X, W, 1e-5, to_dev(inp["gamma"], dev), to_dev(inp["beta"], dev),
                                  rstd_out=stats)
        want, _, wstat = orc.gemm_postnorm_ln(inp["X"], inp["W"], 1e-5, inp["gamma"], inp["beta"])
    else:
        got = nf.gemm_postnorm_rms(X, W, 1e-5, to_dev(inp["gamma"], dev), rstd_out=stats)
        want, wstat = orc.gemm_postnorm_rms(inp["X"], inp["W"], 1e-5, inp["gamma"])
    assert_close(to_f64(got), want, f"split last wave {op}")
    if op != "plain":
        np.testing.assert_allclose(stats.cpu().numpy(), wstat, rtol=1e-3)


# ------------------------------------------------------------ global exchange
@pytest.fixture
def force_global():
    nf.set_postnorm_exchange(nf.XCH_GLOBAL)
    yield
    nf.set_postnorm_exchange(0)


def test_global_exchange_across_launches_and_graph_replays(dev, orc, force_global):
    """The exchange counters live in scratch memory that each launch must
    leave at zero: back-to-back launches and replays of a captured graph all
    give the first launch's bits."""
    import torch
    M, K, N = 128 * 40 + 3, 64, 4096
    inp = _inputs(M, K, N, seed=53, gamma=True, beta=True)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    G, B = to_dev(inp["gamma"], dev), to_dev(inp["beta"], dev)
    assert nf.plan_gemm(2, M, N, K, 148)["exchange"] == nf.XCH_GLOBAL
    ys = [nf.gemm_postnorm_ln(X, W, 1e-5, G, B) for _ in range(5)]
    torch.cuda.synchronize()
    for y in ys[1:]:
        assert torch.equal(y, ys[0])
    rows = nf_inputs.sample_rows(M, 200, seed=6)
    ref = orc.gemm_postnorm_ln(inp["X"], inp["W"], 1e-5, inp["gamma"], inp["beta"], rows=rows)[0]
    assert_close(to_f64(ys[0])[rows], ref, "global exchange, first launch")

    s = torch.cuda.Stream()
    out = torch.empty_like(ys[0])
    with torch.cuda.stream(s):  # sets up the stream's scratch before capture
        nf.gemm_postnorm_ln(X, W, 1e-5, G, B, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        nf.gemm_postnorm_ln(X, W, 1e-5, G, B, out=out)
        nf.gemm_postnorm_ln(X, W, 1e-5, G, B, out=out)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ys[0])
    assert nf.device_status()[0] == nf.NF_OK


def test_global_exchange_unaligned_affine(dev, orc, force_global):
    """gamma / beta only 2-byte aligned: the epilogue falls back to scalar
    loads of the affine parameters (ragged N: the last tile holds 8 columns)."""
    import torch
    M, K, N = 300, 64, 1032
    inp = _inputs(M, K, N, seed=59, gamma=True, beta=True)
    gbuf = torch.zeros(N + 1, dtype=torch.bfloat16, device=dev)
    bbuf = torch.zeros(N + 1, dtype=torch.bfloat16, device=dev)
    gbuf[1:] = to_dev(inp["gamma"], dev)
    bbuf[1:] = to_dev(inp["beta"], dev)
    g, b = gbuf[1:], bbuf[1:]
    assert g.data_ptr() % 16 != 0
    y = nf.gemm_postnorm_ln(to_dev(inp["X"], dev), to_dev(inp["W"], dev), 1e-5, g, b)
    ref = orc.gemm_postnorm_ln(inp["X"], inp["W"], 1e-5, inp["gamma"], inp["beta"])[0]
    assert_close(to_f64(y), ref, "global exchange, unaligned gamma/beta")
    y = nf.gemm_postnorm_rms(to_dev(inp["X"], dev), to_dev(inp["W"], dev), 1e-5, g)
    ref = orc.gemm_postnorm_rms(inp["X"], inp["W"], 1e-5, inp["gamma"])[0]
    assert_close(to_f64(y), ref, "global exchange rms, unaligned gamma")


def test_global_exchange_on_two_streams(dev, force_global):
    """Each stream has its own scratch: launches on two streams may overlap and
    still give the single-stream bits."""
    import torch
    a = _inputs(1024, 256, 2048, seed=61, gamma=True, beta=True)
    b = _inputs(777, 128, 4096, seed=67, gamma=True)
    XA, WA = to_dev(a["X"], dev), to_dev(a["W"], dev)
    GA, BA = to_dev(a["gamma"], dev), to_dev(a["beta"], dev)
    XB, WB, GB = to_dev(b["X"], dev), to_dev(b["W"], dev), to_dev(b["gamma"], dev)
    ref_a = nf.gemm_postnorm_ln(XA, WA, 1e-5, GA, BA)
    ref_b = nf.gemm_postnorm_rms(XB, WB, 1e-6, GB)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        with torch.cuda.stream(s1):
            ya = [nf.gemm_postnorm_ln(XA, WA, 1e-5, GA, BA) for _ in range(4)]
        with torch.cuda.stream(s2):
            yb = [nf.gemm_postnorm_rms(XB, WB, 1e-6, GB) for _ in range(4)]
        torch.cuda.synchronize()
        for y in ya:
            assert torch.equal(y, ref_a)
        for y in yb:
            assert torch.equal(y, ref_b)


def test_global_exchange_shape_sequence_on_one_stream(dev, orc, force_global):
    """Shapes with different row-tile counts share one stream's scratch: a
    launch with more row tiles must find zero counters where an earlier launch
    with fewer row tiles (and more column tiles) wrote statistics; the last
    shape grows the buffer."""
    import torch
    for i, (M, K, N) in enumerate([(128 * 65 + 5, 64, 4096), (128 * 300, 64, 512), (128 * 65 + 5, 64, 4096),
                                   (128 * 1100, 64, 1024)]):
        inp = _inputs(M, K, N, seed=71 + i, gamma=True, beta=True)
        y = nf.gemm_postnorm_ln(to_dev(inp["X"], dev), to_dev(inp["W"], dev), 1e-5, to_dev(inp["gamma"], dev),
                                to_dev(inp["beta"], dev))
        rows = nf_inputs.sample_rows(M, 256, seed=i)
        ref = orc.gemm_postnorm_ln(inp["X"], inp["W"], 1e-5, inp["gamma"], inp["beta"], rows=rows)[0]
        assert_close(to_f64(y)[rows], ref, f"global exchange sequence {M}x{K}x{N}")
        torch.cuda.synchronize()
        assert nf.device_status()[0] == nf.NF_OK


@pytest.mark.parametrize("op,M,K,N", [("pre_rms", 24320, 512, 512), ("plain", 24320, 512, 512),
                                      ("post_ln", 27136, 320, 256), ("post_rms", 27136 + 40, 1024, 200)])
def test_split_last_wave_long_k(dev, orc, op, M, K, N):
    """Memory-bound tiles with K > 256 whose last partial wave holds at most
    half a wave: those tiles run as two 64-row units (each still a 128-row MMA,
    storing its own half).  Rows of the split tail and of full tiles against
    the oracle."""
    import torch
    inp = _inputs(M, K, N, seed=M + K, gamma=True, beta=True)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    rng = np.random.default_rng(M)
    rows = np.unique(np.concatenate([rng.integers(0, M, 64), rng.integers(max(0, M - 9000), M, 128),
                                     np.arange(M - 70, M)])).astype(np.int64)
    if op == "pre_rms":
        y = nf.gemm_prenorm_rms(X, W, 1e-6)
        ref = orc.gemm_prenorm_rms(inp["X"], inp["W"], 1e-6, rows=rows)[0]
    elif op == "plain":
        y = nf.gemm_plain(X, W)
        ref = orc.gemm_plain(inp["X"], inp["W"], rows=rows)
    elif op == "post_ln":
        y = nf.gemm_postnorm_ln(X, W, 1e-5, to_dev(inp["gamma"], dev), to_dev(inp["beta"], dev))
        ref = orc.gemm_postnorm_ln(inp["X"], inp["W"], 1e-5, inp["gamma"], inp["beta"], rows=rows)[0]
    else:
        y = nf.gemm_postnorm_rms(X, W, 1e-5, to_dev(inp["gamma"], dev))
        ref = orc.gemm_postnorm_rms(inp["X"], inp["W"], 1e-5, inp["gamma"], rows=rows)[0]
    torch.cuda.synchronize()
    assert bool(torch.isfinite(y.float()).all())
    assert_close(to_f64(y[torch.from_numpy(rows).to(dev)]), ref, f"split tail {op} {M}x{K}x{N}")
