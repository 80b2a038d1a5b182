"""Parity of the Lazy Pre-Norm backward (blog "Towards Free Normalization",
§2, limitation 3) and of the transposed plain GEMMs its unfused baseline uses,
through the C ABI, with the fp64 oracle."""
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


def _problem(M, K, N, seed, eps=1e-6):
    """A (M x K), B (K x N), dC (M x N) and A's own rstd in fp32, as the
    forward would have saved it."""
    import oracle
    inp = nf_inputs.make_inputs(M, K, N, seed=seed)
    dC = nf_inputs.make_inputs(M, N, 8, seed=seed + 3)["X"]
    _, rstd = oracle.get().gemm_prenorm_rms(inp["X"], inp["W"], eps)
    return inp["X"], inp["W"], dC, rstd.astype(np.float32)


def _abs_bf16(a):
    """|a| of a bf16 bit pattern (clears the sign bit)."""
    return (a & np.uint16(0x7FFF)).astype(np.uint16)


def _assert_db(orc, got, A, r64, dC, what, krows=None):
    """dB's MMA consumes bf16(xhat) = bf16(A rstd): besides the forward bound,
    each product may carry a 2^-9 relative rounding, so the result may differ
    from the exact one by up to 2^-9 sum_i |xhat_ik dC_in| (bounded here by
    2^-8 times that magnitude sum, which the oracle computes on |A| and |dC|)."""
    from gpu_util import ATOL, RTOL
    want = orc.prenorm_rms_bwd_db(A, r64, dC, krows=krows)
    mag = orc.prenorm_rms_bwd_db(_abs_bf16(A), r64, _abs_bf16(dC), krows=krows)
    err = np.abs(got - want)
    bound = ATOL + RTOL * np.abs(want) + 2.0 ** -8 * mag
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{bad.size} out of bound; max err {err.max():.3e}, "
                           f"max err / bound {(err / bound).max():.3f}")


def _f32(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


# (M, K, N): ragged K and N, M a multiple of 8 (A is read transposed for dB),
# several tiles in every direction, K over 1-16 column tiles of dA.
# The last two have a long contraction for dB over few output tiles, which
# the library splits over the contraction (16 and 8 slices on 152 SMs).
SHAPES = [(256, 64, 64), (264, 200, 136), (128, 520, 72), (1000, 136, 264), (512, 1024, 512), (136, 4096, 64),
          (64, 2056, 8), (8192, 64, 64), (4096, 200, 136)]


def _assert_xhat(got, A, rstd, what):
    """The side output xhat = bf16(A * rstd): the fp32 product rounded to
    bf16 is within 2^-8 of the exact product, relative."""
    want = nf_inputs.bf16_to_f64(A) * rstd.astype(np.float64)[:, None]
    err = np.abs(got - want)
    bad = err > 2.0 ** -8 * np.abs(want)
    assert not bad.any(), f"{what}: {int(bad.sum())}/{bad.size} off; max err {err.max():.3e}"


@pytest.mark.parametrize("M,K,N", SHAPES)
@pytest.mark.parametrize("use_xhat", [True, False], ids=["xhat", "rowscale"])
def test_prenorm_bwd(dev, orc, M, K, N, use_xhat):
    import torch
    A, B, dC, rstd = _problem(M, K, N, seed=M + K + N)
    xh = torch.full((M, K), float("nan"), dtype=torch.bfloat16, device=dev) if use_xhat else None
    da, db = nf.gemm_prenorm_rms_bwd(to_dev(A, dev), to_dev(B, dev), _f32(rstd, dev), to_dev(dC, dev), xhat=xh,
                                     use_xhat=use_xhat)
    torch.cuda.synchronize()
    r64 = rstd.astype(np.float64)
    assert_close(to_f64(da), orc.prenorm_rms_bwd_da(A, B, r64, dC), f"pre-norm bwd dA {M}x{K}x{N}")
    _assert_db(orc, to_f64(db), A, r64, dC, f"pre-norm bwd dB {M}x{K}x{N}")
    if use_xhat:
        _assert_xhat(to_f64(xh), A, rstd, f"xhat {M}x{K}x{N}")


def test_prenorm_bwd_one_output_only(dev, orc):
    import torch
    M, K, N = 264, 200, 136
    A, B, dC, rstd = _problem(M, K, N, seed=9)
    da, db = nf.gemm_prenorm_rms_bwd(to_dev(A, dev), to_dev(B, dev), _f32(rstd, dev), to_dev(dC, dev), want_db=False)
    assert db is None
    torch.cuda.synchronize()
    assert_close(to_f64(da), orc.prenorm_rms_bwd_da(A, B, rstd.astype(np.float64), dC), "dA alone")
    da, db = nf.gemm_prenorm_rms_bwd(to_dev(A, dev), to_dev(B, dev), _f32(rstd, dev), to_dev(dC, dev), want_da=False)
    assert da is None
    torch.cuda.synchronize()
    _assert_db(orc, to_f64(db), A, rstd.astype(np.float64), dC, "dB alone")


@pytest.mark.parametrize("M,K,N", [(256, 64, 64), (264, 200, 136), (520, 72, 1032), (8, 8, 8)])
@pytest.mark.parametrize("flags", [nf.TRANS_X, nf.TRANS_W], ids=["trans_x", "trans_w"])
def test_plain_transposed(dev, orc, M, K, N, flags):
    inp = nf_inputs.make_inputs(M, K, N, seed=M * 3 + N)
    X, W = inp["X"], inp["W"]
    xs = np.ascontiguousarray(X.T) if flags & nf.TRANS_X else X
    ws = np.ascontiguousarray(W.T) if flags & nf.TRANS_W else W
    y = nf.gemm_plain_t(to_dev(xs, dev), to_dev(ws, dev), flags)
    assert_close(to_f64(y), orc.gemm_plain(X, W), f"plain transposed flags={flags} {M}x{K}x{N}")


def test_unfused_prenorm_bwd_pair(dev, orc):
    """The unfused baseline: xhat = rmsnorm(A) materialized by the row kernel,
    dB = xhat^T dC and dXhat = dC B^T by the transposed plain GEMMs, dA by the
    row backward kernel; against the oracle (bf16 intermediates)."""
    import torch
    M, K, N = 1000, 512, 768
    A, B, dC, rstd = _problem(M, K, N, seed=13)
    a, b, dc = to_dev(A, dev), to_dev(B, dev), to_dev(dC, dev)
    xhat = nf.norm_rows(a, nf.NORM_RMS, 1e-6)
    db = nf.gemm_plain_t(xhat, dc, nf.TRANS_X)
    dxhat = nf.gemm_plain_t(dc, b, nf.TRANS_W)
    da = nf.norm_rows_bwd(dxhat, a, nf.NORM_RMS, None, _f32(rstd, dev))
    torch.cuda.synchronize()
    r64 = rstd.astype(np.float64)
    assert_close(to_f64(da), orc.prenorm_rms_bwd_da(A, B, r64, dC), "unfused dA")
    _assert_db(orc, to_f64(db), A, r64, dC, "unfused dB")


@pytest.mark.parametrize("M,K,N", [(32768, 512, 512), (8192, 4096, 4096)],
                         ids=["rowscale_32768x512x512", "llm_8192x4096x4096"])
@pytest.mark.parametrize("use_xhat", [True, False], ids=["xhat", "rowscale"])
def test_prenorm_bwd_full_size(dev, orc, M, K, N, use_xhat):
    import torch
    A, B, dC, rstd = _problem(M, K, N, seed=M + N)
    da, db = nf.gemm_prenorm_rms_bwd(to_dev(A, dev), to_dev(B, dev), _f32(rstd, dev), to_dev(dC, dev),
                                     use_xhat=use_xhat)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(da.float()).all()) and bool(torch.isfinite(db.float()).all())
    r64 = rstd.astype(np.float64)
    rows = nf_inputs.sample_rows(M, 96, seed=5)
    assert_close(to_f64(da)[rows], orc.prenorm_rms_bwd_da(A, B, r64, dC, rows=rows), f"dA full {M}x{K}x{N}")
    krows = nf_inputs.sample_rows(K, 24, seed=6)
    _assert_db(orc, to_f64(db)[krows], A, r64, dC, f"dB full {M}x{K}x{N}", krows=krows)


# Plain GEMMs with few output tiles over a long contraction: split over the
# contraction (fp32 partials, a second kernel adds them in a fixed order).
SPLIT_SHAPES = [(128, 4096, 64), (200, 2056, 136), (512, 32768, 512), (8, 1024, 8)]


@pytest.mark.parametrize("M,K,N", SPLIT_SHAPES)
@pytest.mark.parametrize("flags", [0, nf.TRANS_X, nf.TRANS_W], ids=["plain", "trans_x", "trans_w"])
def test_plain_splitk(dev, orc, M, K, N, flags):
    import torch
    p = nf.plan_gemm(0, M, N, K, torch.cuda.get_device_properties(dev).multi_processor_count)
    assert p["splitk"] > 1, "shape chosen to be split"
    inp = nf_inputs.make_inputs(M, K, N, seed=M + 7 * K + N)
    X, W = inp["X"], inp["W"]
    xs = np.ascontiguousarray(X.T) if flags & nf.TRANS_X else X
    ws = np.ascontiguousarray(W.T) if flags & nf.TRANS_W else W
    x, w = to_dev(xs, dev), to_dev(ws, dev)
    y = nf.gemm_plain_t(x, w, flags) if flags else nf.gemm_plain(x, w)
    y2 = nf.gemm_plain_t(x, w, flags) if flags else nf.gemm_plain(x, w)
    torch.cuda.synchronize()
    # the slices are added in a fixed order: the result does not depend on timing
    assert torch.equal(y, y2)
    assert_close(to_f64(y), orc.gemm_plain(X, W), f"split-K flags={flags} {M}x{K}x{N}")
    try:
        nf.set_gemm_splitk(1)
        y1 = nf.gemm_plain_t(x, w, flags) if flags else nf.gemm_plain(x, w)
    finally:
        nf.set_gemm_splitk(0)
    torch.cuda.synchronize()
    assert_close(to_f64(y1), orc.gemm_plain(X, W), f"unsplit flags={flags} {M}x{K}x{N}")


def test_splitk_graph_replay(dev, orc):
    """A split GEMM captured into a CUDA graph (after its first call on the
    stream set up the workspace) and replayed on new inputs."""
    import torch
    M, K, N = 256, 8192, 256
    s = torch.cuda.Stream()
    xs, ws, ys = [], [], []
    with torch.cuda.stream(s):
        for seed in (1, 2):
            inp = nf_inputs.make_inputs(M, K, N, seed=seed)
            xs.append(inp)
        x = to_dev(xs[0]["X"], dev)
        w = to_dev(xs[0]["W"], dev)
        y = nf.gemm_plain(x, w, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            nf.gemm_plain(x, w, out=y, stream=s)
        x.copy_(to_dev(xs[1]["X"], dev))
        w.copy_(to_dev(xs[1]["W"], dev))
        g.replay()
    s.synchronize()
    assert_close(to_f64(y), orc.gemm_plain(xs[1]["X"], xs[1]["W"]), "split-K graph replay")


@pytest.mark.parametrize("M,K,N", [(4096, 2688, 8192), (1000, 2688, 8200)])
def test_every_tile_computed_once(dev, M, K, N):
    """A GEMM of hundreds of tiles over several waves (ragged in M and N).
    With one-hot rows of X (row i picks row i mod K of W) every output row is a
    row of W, exactly: a tile computed twice, never, or at the wrong place
    shows up bit for bit."""
    import torch
    idx = torch.arange(M, device=dev) % K
    x = torch.zeros((M, K), dtype=torch.bfloat16, device=dev)
    x[torch.arange(M, device=dev), idx] = 1.0
    g = torch.Generator(device="cpu").manual_seed(M + N)
    w = (torch.randn((K, N), generator=g) * 4).to(torch.bfloat16).to(dev)
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    nf.gemm_plain(x, w, out=y)
    torch.cuda.synchronize()
    assert torch.equal(y, w[idx])


@pytest.mark.parametrize("flags", [0, nf.TRANS_X, nf.TRANS_W], ids=["plain", "trans_x", "trans_w"])
def test_plain_tail_splitk(dev, orc, flags):
    """A tensor-bound GEMM whose last wave is at most half full: its tiles are
    split over the contraction (whole tiles before them).  Rows of the split
    tiles and of whole tiles against the oracle; repeated calls give the same
    bits."""
    import torch
    M, K, N = 3840, 1024, 4096
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    nf.set_gemm_pair(1)  # the plain GEMM would take CTA pairs instead of the split (transposed forms never do)
    try:
        _tail_splitk(orc, dev, flags, M, K, N, sms)
    finally:
        nf.set_gemm_pair(0)


def _tail_splitk(orc, dev, flags, M, K, N, sms):
    import torch
    p = nf.plan_gemm(0, M, N, K, sms)
    tiles = p["tiles"]
    if tiles % sms == 0 or 2 * (tiles % sms) > sms:
        pytest.skip("shape does not leave a half-empty last wave on this device")
    assert p["splitk"] > 1 and p["split_tiles"] == tiles % sms
    inp = nf_inputs.make_inputs(M, K, N, seed=41)
    X, W = inp["X"], inp["W"]
    xs = np.ascontiguousarray(X.T) if flags & nf.TRANS_X else X
    ws = np.ascontiguousarray(W.T) if flags & nf.TRANS_W else W
    x, w = to_dev(xs, dev), to_dev(ws, dev)
    run = (lambda: nf.gemm_plain_t(x, w, flags)) if flags else (lambda: nf.gemm_plain(x, w))
    y, y2 = run(), run()
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    first_split_row = (tiles - p["split_tiles"]) // (N // 256) * 128
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([rng.integers(0, M, 24), rng.integers(first_split_row, M, 40),
                                     np.array([M - 1, first_split_row])])).astype(np.int64)
    assert_close(to_f64(y)[rows], orc.gemm_plain(X, W, rows=rows), f"tail split-K flags={flags}")
