"""Lazy Pre-Norm with the row sums of squares split over a row's tiles (blog
"Towards Free Normalization", §2, with the redundant per-CTA sums shared):
tile n of a row tile sums the squares of 1/n_tiles of its rows over the whole
contraction and the row tile's tiles gather the sums through L2 before the
epilogue scales the accumulator.  Parity with the fp64 oracle through the C
ABI for one CTA per tile and for CTA pairs, on ragged shapes whose last tile
holds fewer rows (R = ceil(128 / n_tiles)), 2..32 tiles a row, an odd number
of row tiles (a pair's second CTA past M), repeated launches, graph replays,
two streams, and launch sequences that share one stream's counters with the
post-norm exchange."""
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
    nf.set_prenorm_split(0)
    nf.set_gemm_pair(0)
    import torch
    torch.cuda.synchronize()
    status, detail = nf.device_status()
    assert status == nf.NF_OK, f"device status word set: {detail}"


@pytest.fixture(scope="module")
def orc():
    import oracle
    return oracle.get()


@pytest.fixture(params=[1, 2], ids=["one_cta", "pairs"])
def pair_mode(request):
    nf.set_prenorm_split(2)
    nf.set_gemm_pair(request.param)
    yield request.param
    nf.set_gemm_pair(0)
    nf.set_prenorm_split(0)


# (M, K, N): 2, 3, 8, 9 and 32 tiles a row (R = 64, 43, 16, 15, 4 rows a
# tile, the last tile of 3 and 9 holding fewer), ragged K and N, one row,
# an odd number of row tiles.
SPLIT_SHAPES = [(300, 200, 320), (513, 520, 264), (257, 64, 456), (700, 256, 768), (300, 136, 1800),
                (1000, 1032, 2056), (129, 72, 8192), (1, 64, 512), (640, 2048, 1024)]


@pytest.mark.parametrize("M,K,N", SPLIT_SHAPES)
@pytest.mark.parametrize("x_dist", ["normal", "row_scaled"])
def test_split_prenorm_rms(dev, orc, pair_mode, M, K, N, x_dist):
    import torch
    p = nf.plan_gemm(1, M, N, K, 148)
    assert p["exchange"] == nf.XCH_GLOBAL
    assert (p["cluster"] == 2) == (pair_mode == 2 and M > 128)
    inp = nf_inputs.make_inputs(M, K, N, seed=5 * M + K + N, x_dist=x_dist)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    rstd = torch.full((M,), -1.0, dtype=torch.float32, device=dev)
    y = nf.gemm_prenorm_rms(X, W, 1e-6, rstd_out=rstd)
    y2 = nf.gemm_prenorm_rms(X, W, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    ref, rref = orc.gemm_prenorm_rms(inp["X"], inp["W"], 1e-6)
    assert_close(to_f64(y), ref, f"split pre {M}x{K}x{N} {x_dist}")
    np.testing.assert_allclose(rstd.cpu().numpy(), rref, rtol=1e-4)


def test_split_matches_unsplit_within_rounding(dev):
    """The split changes only the fp32 order of each row's sum of squares:
    outputs agree with every tile summing every row to within bf16 rounding,
    and rstd to the fp32 rounding of a 4096-term sum (typically sqrt(K)
    ulps, halved by the square root: a few 1e-6)."""
    import torch
    M, K, N = 1024, 4096, 2048
    inp = nf_inputs.make_inputs(M, K, N, seed=23, x_dist="row_scaled")
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    ra = torch.empty(M, dtype=torch.float32, device=dev)
    rb = torch.empty(M, dtype=torch.float32, device=dev)
    try:
        nf.set_prenorm_split(2)
        a = nf.gemm_prenorm_rms(X, W, 1e-6, rstd_out=ra)
        nf.set_prenorm_split(1)
        b = nf.gemm_prenorm_rms(X, W, 1e-6, rstd_out=rb)
    finally:
        nf.set_prenorm_split(0)
    torch.cuda.synchronize()
    np.testing.assert_allclose(ra.cpu().numpy(), rb.cpu().numpy(), rtol=2e-5)
    d = (a.float() - b.float()).abs()
    assert float(d.max()) <= float(2.0 ** -7 * b.float().abs().max())


def test_split_full_size_llm_one_cta(dev, orc):
    """8192 x 4096 x 4096 with one CTA per tile (the CTA-pair form is the
    default, covered by the pair tests): sampled rows against the oracle."""
    import torch
    w = nf_inputs.WORKLOADS["llm_8192x4096x4096"]
    inp = nf_inputs.workload_inputs(w)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    try:
        nf.set_gemm_pair(1)
        assert nf.plan_gemm(1, w.M, w.N, w.K, 148)["exchange"] == nf.XCH_GLOBAL
        y = nf.gemm_prenorm_rms(X, W, w.eps)
    finally:
        nf.set_gemm_pair(0)
    rows = nf_inputs.sample_rows(w.M, 128, seed=12)
    ref = orc.gemm_prenorm_rms(inp["X"], inp["W"], w.eps, rows=rows)[0]
    assert_close(to_f64(y[torch.from_numpy(rows).to(dev)]), ref, "split pre llm one CTA")


def test_split_graph_replays_and_two_streams(dev, pair_mode):
    """The gather's counters and sums live in each stream's scratch: replays
    of a captured graph and launches overlapping on two streams give the
    bits of a lone launch."""
    import torch
    a = nf_inputs.make_inputs(1152, 1024, 2048, seed=29)
    b = nf_inputs.make_inputs(777, 2048, 4096, seed=31, x_dist="row_scaled")
    XA, WA = to_dev(a["X"], dev), to_dev(a["W"], dev)
    XB, WB = to_dev(b["X"], dev), to_dev(b["W"], dev)
    ref_a = nf.gemm_prenorm_rms(XA, WA, 1e-6)
    ref_b = nf.gemm_prenorm_rms(XB, WB, 1e-5)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        with torch.cuda.stream(s1):
            ya = [nf.gemm_prenorm_rms(XA, WA, 1e-6) for _ in range(4)]
        with torch.cuda.stream(s2):
            yb = [nf.gemm_prenorm_rms(XB, WB, 1e-5) for _ in range(4)]
        torch.cuda.synchronize()
        for y in ya:
            assert torch.equal(y, ref_a)
        for y in yb:
            assert torch.equal(y, ref_b)
    out = torch.empty_like(ref_a)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s1):  # s1's scratch was set up above
        nf.gemm_prenorm_rms(XA, WA, 1e-6, out=out)
        nf.gemm_prenorm_rms(XA, WA, 1e-6, out=out)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_a)
    assert nf.device_status()[0] == nf.NF_OK


def test_exchange_sequence_with_odd_row_tiles(dev, orc):
    """One stream's counters shared by launches of different row-tile counts,
    in CTA pairs: an odd number of row tiles leaves the last pair's second CTA
    past M, which must leave no count behind (the launch after next reuses the
    bank and clears only the row tiles of the launch before it).  Post-LN and
    split pre-RMS, interleaved; every launch against the oracle."""
    import torch
    s = torch.cuda.Stream()
    seq = [("post", 600, 512, 4096), ("post", 600, 512, 4096), ("post", 2048, 512, 4096),
           ("pre", 600, 2048, 4096), ("post", 600, 512, 4096), ("pre", 2048, 2048, 4096),
           ("pre", 2048, 2048, 4096)]
    try:
        nf.set_gemm_pair(2)
        nf.set_postnorm_exchange(nf.XCH_GLOBAL)
        for i, (op, M, K, N) in enumerate(seq):
            inp = nf_inputs.make_inputs(M, K, N, seed=101 + i, gamma=True, beta=True)
            X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
            p = nf.plan_gemm(1 if op == "pre" else 2, M, N, K, 148)
            assert p["cluster"] == 2 and p["exchange"] == nf.XCH_GLOBAL
            with torch.cuda.stream(s):
                if op == "pre":
                    y = nf.gemm_prenorm_rms(X, W, 1e-6)
                else:
                    y = nf.gemm_postnorm_ln(X, W, 1e-5, to_dev(inp["gamma"], dev), to_dev(inp["beta"], dev))
            s.synchronize()
            # row tiles 4..6 (the odd launches' last real row tile and the one
            # past M) whole, and a sample of the rest
            rows = np.unique(np.concatenate([np.arange(512, min(M, 896)),
                                             nf_inputs.sample_rows(M, 64, seed=i)])).astype(np.int64)
            if op == "pre":
                ref = orc.gemm_prenorm_rms(inp["X"], inp["W"], 1e-6, rows=rows)[0]
            else:
                ref = orc.gemm_postnorm_ln(inp["X"], inp["W"], 1e-5, inp["gamma"], inp["beta"], rows=rows)[0]
            assert_close(to_f64(y)[rows], ref, f"sequence {i}: {op} {M}x{K}x{N}")
    finally:
        nf.set_gemm_pair(0)
        nf.set_postnorm_exchange(0)
    assert nf.device_status()[0] == nf.NF_OK
