"""nf_gemm_postnorm_ln_noalloc: the post-norm entry point whose L2 exchange
scratch is a fixed device array, against nf_gemm_postnorm_ln (collected last:
it shares the device array with nothing else in the suite)."""
import pytest

import nf_inputs
import normalization_gemm_gb300 as nf
from gpu_util import require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    d = require_gpu()  # fails, like every GPU module, when no device is present
    from normalization_gemm_gb300 import _build
    _build.build()
    return d


def _inputs(M, K, N, seed):
    w = nf_inputs.Workload("t", M, K, N, 1e-5, ("post_ln",), gamma=True, beta=True)
    return nf_inputs.workload_inputs(w, seed=seed)


@pytest.mark.parametrize("M,K,N", [(1000, 1024, 2048), (128 * 40 + 3, 512, 4096), (300, 64, 1032), (257, 64, 200)])
def test_noalloc_matches_the_allocating_entry_point_on_two_calls(dev, M, K, N):
    import torch
    inp = _inputs(M, K, N, seed=M + N)
    X, W = to_dev(inp["X"], dev), to_dev(inp["W"], dev)
    G, B = to_dev(inp["gamma"], dev), to_dev(inp["beta"], dev)
    for _ in range(2):
        mean_a = torch.zeros(M, dtype=torch.float32, device=dev)
        rstd_a = torch.zeros(M, dtype=torch.float32, device=dev)
        mean_b = torch.zeros(M, dtype=torch.float32, device=dev)
        rstd_b = torch.zeros(M, dtype=torch.float32, device=dev)
        ref = nf.gemm_postnorm_ln(X, W, 1e-5, G, B, mean_out=mean_a, rstd_out=rstd_a)
        got = nf.gemm_postnorm_ln_noalloc(X, W, 1e-5, G, B, mean_out=mean_b, rstd_out=rstd_b)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
        assert torch.equal(mean_a, mean_b) and torch.equal(rstd_a, rstd_b)
    assert nf.device_status()[0] == nf.NF_OK


def test_noalloc_rejects_shapes_beyond_its_array(dev):
    import torch
    # 65536 x 4096 with K >= 512 uses the L2 exchange: 512 x 16 tiles > 4096
    X = torch.empty(65536, 512, dtype=torch.bfloat16, device=dev)
    W = torch.empty(512, 4096, dtype=torch.bfloat16, device=dev)
    Y = torch.empty(65536, 4096, dtype=torch.bfloat16, device=dev)
    assert nf.plan_gemm(2, 65536, 4096, 512, 148)["exchange"] == nf.XCH_GLOBAL
    with pytest.raises(nf.NFError) as e:
        nf.gemm_postnorm_ln_noalloc(X, W, 1e-5, out=Y)
    assert e.value.status == 3  # NF_ERR_UNSUPPORTED_SHAPE
