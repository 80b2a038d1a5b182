"""Scratch memory of the compute calls (the post-norm L2 exchange buffer and
the split-K workspace, one of each per stream): no compute call synchronizes
the host with the device, not even the one that sets a buffer up or enlarges
it, and nf_reserve_scratch sizes both so that calls within its sizes can be
captured into a graph without any earlier call."""
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


# Post-norm shapes that exchange through L2 (K >= 512, N > 512), growing in
# M x ceil(N / 256), then a plain GEMM that splits over the contraction.
GROWING = [(256, 512, 1024), (1024, 512, 1024), (2304, 512, 2048)]
SPLITK = (256, 8192, 256)


def _post_inputs(dev, M, K, N, seed):
    inp = nf_inputs.make_inputs(M, K, N, seed=seed)
    return inp, to_dev(inp["X"], dev), to_dev(inp["W"], dev)


def test_compute_calls_never_synchronize(dev, orc):
    """A fresh stream is kept busy by a long spin; post-norm calls that first
    set up and then twice enlarge its exchange buffer, and a split GEMM that
    sets up its workspace, all return while the spin still runs (an event
    recorded after them is still pending).  The results then match the
    oracle."""
    import torch
    s = torch.cuda.Stream()
    assert nf.plan_gemm(2, 256, 1024, 512, 148)["exchange"] == nf.XCH_GLOBAL
    assert nf.plan_gemm(0, *SPLITK[:1], SPLITK[2], SPLITK[1], 148)["splitk"] > 1
    cases = [_post_inputs(dev, M, K, N, seed=M + N) for (M, K, N) in GROWING]
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for (M, K, N) in GROWING]
    sk = nf_inputs.make_inputs(SPLITK[0], SPLITK[1], SPLITK[2], seed=5)
    skx, skw = to_dev(sk["X"], dev), to_dev(sk["W"], dev)
    sky = torch.empty((SPLITK[0], SPLITK[2]), dtype=torch.bfloat16, device=dev)
    # Load and set up the kernels first, on the default stream (the first use
    # of a kernel loads its code, which is not what this test is about); the
    # fresh stream's scratch is untouched.
    for (inp, X, W), y in zip(cases, ys):
        nf.gemm_postnorm_ln(X, W, 1e-5, out=y)
    nf.gemm_plain(skx, skw, out=sky)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        torch.cuda._sleep(400_000_000)  # about 0.2 s of spinning at 2 GHz
        for (inp, X, W), y in zip(cases, ys):
            nf.gemm_postnorm_ln(X, W, 1e-5, out=y, stream=s)
        nf.gemm_plain(skx, skw, out=sky, stream=s)
        ev = torch.cuda.Event()
        ev.record(s)
    assert not ev.query(), "a compute call waited for the stream"
    torch.cuda.synchronize()
    for (inp, X, W), y, (M, K, N) in zip(cases, ys, GROWING):
        rows = nf_inputs.sample_rows(M, 96, seed=M)
        ref = orc.gemm_postnorm_ln(inp["X"], inp["W"], 1e-5, rows=rows)[0]
        assert_close(to_f64(y)[rows], ref, f"post-LN {M}x{K}x{N} on a busy stream")
    assert_close(to_f64(sky), orc.gemm_plain(sk["X"], sk["W"]), "split-K plain on a busy stream")


def test_reserve_then_capture(dev, orc):
    """nf_reserve_scratch on a fresh stream, then a graph of calls within its
    sizes captured with no earlier call on that stream: its replays give the
    bits of the same calls made eagerly on another stream."""
    import torch
    M, K, N = 2048, 512, 2048
    inp, X, W = _post_inputs(dev, M, K, N, seed=77)
    sk = nf_inputs.make_inputs(SPLITK[0], SPLITK[1], SPLITK[2], seed=6)
    skx, skw = to_dev(sk["X"], dev), to_dev(sk["W"], dev)
    want_y = nf.gemm_postnorm_ln(X, W, 1e-5)
    want_sk = nf.gemm_plain(skx, skw)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    nf.reserve_scratch(M, N, stream=s)
    y = torch.empty_like(want_y)
    y2 = torch.empty_like(want_sk)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        nf.gemm_postnorm_ln(X, W, 1e-5, out=y, stream=s)
        nf.gemm_plain(skx, skw, out=y2, stream=s)
    for _ in range(2):
        y.zero_()
        y2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, want_y)
        assert torch.equal(y2, want_sk)
    rows = nf_inputs.sample_rows(M, 64, seed=3)
    assert_close(to_f64(y)[rows], orc.gemm_postnorm_ln(inp["X"], inp["W"], 1e-5, rows=rows)[0], "reserved + graph")


def test_prenorm_split_scratch_on_a_busy_stream_and_reserved(dev, orc):
    """The Lazy Pre-Norm with split sums of squares keeps its gathered sums in
    the same per-stream exchange scratch: its first call on a fresh, busy
    stream sets the scratch up without waiting for the stream, and after
    nf_reserve_scratch (rows only; any N) a graph of split calls captures and
    replays to the eager bits."""
    import torch
    M, K, N = 1152, 2048, 2048
    assert nf.plan_gemm(1, M, N, K, 148)["exchange"] == nf.XCH_GLOBAL
    inp = nf_inputs.make_inputs(M, K, N, seed=88, x_dist="row_scaled")
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    want = nf.gemm_prenorm_rms(X, W, 1e-6)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    y = torch.empty_like(want)
    with torch.cuda.stream(s):
        torch.cuda._sleep(400_000_000)
        nf.gemm_prenorm_rms(X, W, 1e-6, out=y, stream=s)
        ev = torch.cuda.Event()
        ev.record(s)
    assert not ev.query(), "the split pre-norm call waited for the stream"
    torch.cuda.synchronize()
    assert torch.equal(y, want)
    rows = nf_inputs.sample_rows(M, 64, seed=9)
    assert_close(to_f64(y)[rows], orc.gemm_prenorm_rms(inp["X"], inp["W"], 1e-6, rows=rows)[0],
                 "split pre-RMS on a busy stream")
    s2 = torch.cuda.Stream()
    nf.reserve_scratch(M, 8, stream=s2)
    y2 = torch.empty_like(want)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s2):
        nf.gemm_prenorm_rms(X, W, 1e-6, out=y2, stream=s2)
    for _ in range(2):
        y2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y2, want)
