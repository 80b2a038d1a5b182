"""The FlashNormAttention operand bound (fna_bound.py) covers what it is
derived for: an fp64 emulation of the kernel's two bf16 operand roundings,
bf16(ln_q) into S = ln_q K^T and bf16(act(s)) into O = p V, stays within the
bound of the unrounded oracle on every element, for each activation.  CPU
only."""
import numpy as np
import pytest

import nf_inputs
from fna_bound import _act, operand_bound


def _rounded_operands(Q, K, V, act, eps1, eps2):
    q = nf_inputs.bf16_to_f64(Q)
    k = nf_inputs.bf16_to_f64(K)
    v = nf_inputs.bf16_to_f64(V)
    B, Lq, H, D = q.shape
    x = q.reshape(B, Lq, H * D)
    mu = x.mean(-1, keepdims=True)
    ln = ((x - mu) / np.sqrt(((x - mu) ** 2).mean(-1, keepdims=True) + eps1)).reshape(B, Lq, H, D)
    lnr = nf_inputs.bf16_to_f64(nf_inputs.bf16_round(ln))
    s = np.einsum("bthd,bjhd->bthj", lnr, k)
    p = nf_inputs.bf16_to_f64(nf_inputs.bf16_round(_act(s, act)))
    o = (np.einsum("bthj,bjhd->bthd", p, v) + ln).reshape(B, Lq, H * D)
    y = o / np.sqrt((o * o).mean(-1, keepdims=True) + eps2) + x
    return y.reshape(B, Lq, H, D)


@pytest.mark.parametrize("act", [0, 1, 2], ids=["identity", "gelu", "silu"])
def test_bound_covers_bf16_operands(act):
    import oracle
    orc = oracle.get()
    inp = nf_inputs.fna_inputs(2, 64, 128, 3, 128, seed=5 + act, jagged=False)
    want = orc.flashnorm_attn_fwd(inp["Q"], inp["K"], inp["V"], act, 1e-5, 1e-6)
    emul = _rounded_operands(inp["Q"], inp["K"], inp["V"], act, 1e-5, 1e-6)
    bound = operand_bound(inp["Q"], inp["K"], inp["V"], act, 1e-5, 1e-6)
    err = np.abs(emul - want)
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3f}"
    # the roundings are visible (the oracle does not round), and the bound is
    # not vacuous: the emulated errors reach a tenth of it somewhere, and on
    # average it stays near the common tolerance's absolute term (2e-2)
    assert err.max() > 1e-6
    assert np.max(err / bound) > 0.1
    assert bound.mean() < 5e-2
