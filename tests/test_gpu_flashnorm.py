"""Parity of the FlashNormAttention forward (blog "Towards Free Normalization",
§4: LayerNorm over all heads, per-head act(ln_q K^T) V with two residuals,
RMSNorm over all heads) through the C ABI with the fp64 oracle.

The oracle keeps ln_q and p unrounded, as the pseudocode does; the kernel's
tensor cores take both as bf16.  Each comparison therefore adds the bound
derived in fna_bound.py for those two roundings (and the hardware tanh) to the
common 2e-2 + 1.6e-2 |ref|."""
import numpy as np
import pytest

import nf_inputs
import normalization_gemm_gb300 as nf
from fna_bound import operand_bound
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


def _dev4(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def _run(dev, inp, act, jagged, sentinel=None):
    import torch
    q, k, v = _dev4(inp["Q"], dev), _dev4(inp["K"], dev), _dev4(inp["V"], dev)
    ql = torch.from_numpy(inp["q_len"]).to(dev) if jagged else None
    out = torch.full_like(q, float("nan") if sentinel is None else sentinel)
    nf.flashnorm_attn_fwd(q, k, v, act=act, eps1=1e-5, eps2=1e-6, q_len=ql, out=out)
    torch.cuda.synchronize()
    return out


def _valid_rows(got, want, q_len, extra=None):
    B, Lq, H, D = want.shape
    rows = [(b, t) for b in range(B) for t in range(int(q_len[b]))]
    if not rows:
        z = np.zeros((0, H * D))
        return (z, z) if extra is None else (z, z, z)
    bi, ti = np.array(rows).T
    out = (got[bi, ti].reshape(len(rows), H * D), want[bi, ti].reshape(len(rows), H * D))
    if extra is not None:
        out += (extra[bi, ti].reshape(len(rows), H * D),)
    return out


def _check(got, want, inp, act, q_len, what):
    """Valid rows of got against the oracle's want, with the operand bound."""
    ex = operand_bound(inp["Q"], inp["K"], inp["V"], act, 1e-5, 1e-6, q_len)
    g, w, e = _valid_rows(got, want, q_len, ex)
    return assert_close(g, w, what, extra=e)


@pytest.mark.parametrize("B,Lq,H", [(1, 128, 1), (2, 256, 2), (3, 128, 4), (2, 384, 8), (4, 256, 3)])
@pytest.mark.parametrize("act", [nf.ACT_GELU_TANH, nf.ACT_SILU, nf.ACT_IDENTITY], ids=["gelu", "silu", "identity"])
@pytest.mark.parametrize("jagged", [False, True], ids=["dense", "jagged"])
def test_flashnorm_fwd(dev, orc, B, Lq, H, act, jagged):
    inp = nf_inputs.fna_inputs(B, Lq, 128, H, 128, seed=B * 100 + Lq + H, jagged=jagged)
    out = _run(dev, inp, act, jagged)
    want = orc.flashnorm_attn_fwd(inp["Q"], inp["K"], inp["V"], act, 1e-5, 1e-6,
                                  q_len=inp["q_len"] if jagged else None)
    got = to_f64(out.reshape(B * Lq, H * 128)).reshape(B, Lq, H, 128)
    ql = inp["q_len"] if jagged else np.full(B, Lq)
    _check(got, want, inp, act, ql, f"FlashNormAttention B={B} Lq={Lq} H={H} act={act} jagged={jagged}")


def test_flashnorm_padding_rows(dev, orc):
    """Rows past q_len: those in the last 32-row group that holds a valid row
    are written as zero, later ones keep the caller's content."""
    import torch
    B, Lq, H = 4, 256, 2
    inp = nf_inputs.fna_inputs(B, Lq, 128, H, 128, seed=7)
    inp["q_len"] = np.array([0, 1, 40, 256], np.int32)
    out = _run(dev, inp, nf.ACT_GELU_TANH, True, sentinel=3.0)
    o = out.float().cpu().numpy()
    for b, n in enumerate(inp["q_len"]):
        end = min(Lq, -(-int(n) // 32) * 32)
        assert np.all(o[b, n:end] == 0.0), f"batch {b}: padded rows of the last group"
        assert np.all(o[b, end:] == 3.0), f"batch {b}: rows past the last group untouched"
    want = orc.flashnorm_attn_fwd(inp["Q"], inp["K"], inp["V"], 1, 1e-5, 1e-6, q_len=inp["q_len"])
    got = to_f64(out.reshape(B * Lq, H * 128)).reshape(B, Lq, H, 128)
    _check(got, want, inp, 1, inp["q_len"], "FlashNormAttention padding case")
    assert torch.isfinite(out).all()


def test_flashnorm_many_clusters(dev, orc):
    """More clusters than fit at once (a batch per cluster of 4 CTAs), jagged,
    on sampled batches against the oracle; repeated calls give the same bits."""
    import torch
    B, Lq, H = 160, 512, 4
    inp = nf_inputs.fna_inputs(B, Lq, 128, H, 128, seed=3)
    a = _run(dev, inp, nf.ACT_GELU_TANH, True)
    b2 = _run(dev, inp, nf.ACT_GELU_TANH, True)
    assert torch.equal(torch.nan_to_num(a, nan=7.0), torch.nan_to_num(b2, nan=7.0))
    pick = np.array([0, 1, 57, 100, 159])
    sub = {k: np.ascontiguousarray(inp[k][pick]) for k in ("Q", "K", "V", "q_len")}
    want = orc.flashnorm_attn_fwd(sub["Q"], sub["K"], sub["V"], 1, 1e-5, 1e-6, q_len=sub["q_len"])
    got = to_f64(a[torch.from_numpy(pick).to(dev)].reshape(len(pick) * Lq, H * 128)).reshape(len(pick), Lq, H, 128)
    _check(got, want, sub, 1, sub["q_len"], "FlashNormAttention many clusters")


@pytest.mark.parametrize("H", [2, 6], ids=["two_groups", "one_group"])
def test_flashnorm_persistent_batch_mix(dev, orc, H):
    """Many more batches than resident clusters with many empty and one-tile
    batches (a group with no tile in a batch, K/V reloads between one-tile
    batches), three launches in a row on one stream (the batch counter is
    reset by each launch): identical bits each time and oracle parity on a
    sample that includes every length class."""
    import torch
    B, Lq = 400, 384
    inp = nf_inputs.fna_inputs(B, Lq, 128, H, 128, seed=11 + H)
    classes = np.array([0, 1, 0, 127, 128, 129, 0, 255, 256, 384, 1, 0], np.int32)
    inp["q_len"] = classes[np.arange(B) % len(classes)]
    runs = [_run(dev, inp, nf.ACT_SILU, True) for _ in range(3)]
    for r in runs[1:]:
        assert torch.equal(torch.nan_to_num(runs[0], nan=7.0), torch.nan_to_num(r, nan=7.0))
    pick = np.array([0, 1, 3, 4, 5, 7, 8, 9, 10, 200, 397, 399])
    sub = {k: np.ascontiguousarray(inp[k][pick]) for k in ("Q", "K", "V", "q_len")}
    want = orc.flashnorm_attn_fwd(sub["Q"], sub["K"], sub["V"], nf.ACT_SILU, 1e-5, 1e-6, q_len=sub["q_len"])
    got = to_f64(runs[0][torch.from_numpy(pick).to(dev)].reshape(len(pick) * Lq, H * 128)).reshape(len(pick), Lq, H, 128)
    _check(got, want, sub, nf.ACT_SILU, sub["q_len"], f"FlashNormAttention batch mix H={H}")


def test_flashnorm_two_streams(dev):
    """Two independent problems launched on two streams at once (each stream
    has its own batch counter) give the same bits as when run one after the
    other."""
    import torch
    H, Lq = 4, 512
    ia = nf_inputs.fna_inputs(96, Lq, 128, H, 128, seed=21)
    ib = nf_inputs.fna_inputs(80, Lq, 128, H, 128, seed=22)
    ref_a = _run(dev, ia, nf.ACT_GELU_TANH, True)
    ref_b = _run(dev, ib, nf.ACT_GELU_TANH, True)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for inp, s in ((ia, s1), (ib, s2)):
        q, k, v = _dev4(inp["Q"], dev), _dev4(inp["K"], dev), _dev4(inp["V"], dev)
        ql = torch.from_numpy(inp["q_len"]).to(dev)
        out = torch.full_like(q, float("nan"))
        torch.cuda.synchronize()
        outs.append((q, k, v, ql, out, s))
    for q, k, v, ql, out, s in outs:
        nf.flashnorm_attn_fwd(q, k, v, act=nf.ACT_GELU_TANH, eps1=1e-5, eps2=1e-6, q_len=ql, out=out, stream=s)
    torch.cuda.synchronize()
    assert torch.equal(torch.nan_to_num(outs[0][4], nan=7.0), torch.nan_to_num(ref_a, nan=7.0))
    assert torch.equal(torch.nan_to_num(outs[1][4], nan=7.0), torch.nan_to_num(ref_b, nan=7.0))


def test_flashnorm_all_batches_empty(dev):
    """Every q_len is 0: no K/V is loaded, no row is written, the call succeeds."""
    import torch
    inp = nf_inputs.fna_inputs(5, 256, 128, 4, 128, seed=31)
    inp["q_len"] = np.zeros(5, np.int32)
    out = _run(dev, inp, nf.ACT_GELU_TANH, True, sentinel=3.0)
    assert torch.all(out == 3.0)


def test_flashnorm_full_length(dev, orc):
    """Dense batches of the benchmark's maximum length (8 tiles each, so both
    compute groups cycle through all four q buffers twice), every row against
    the oracle."""
    B, Lq, H = 2, 1024, 4
    inp = nf_inputs.fna_inputs(B, Lq, 128, H, 128, seed=33, jagged=False)
    out = _run(dev, inp, nf.ACT_GELU_TANH, False)
    want = orc.flashnorm_attn_fwd(inp["Q"], inp["K"], inp["V"], nf.ACT_GELU_TANH, 1e-5, 1e-6)
    got = to_f64(out.reshape(B * Lq, H * 128)).reshape(B, Lq, H, 128)
    _check(got, want, inp, nf.ACT_GELU_TANH, np.full(B, Lq), "FlashNormAttention full length")
