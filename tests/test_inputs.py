"""The seeded input generator: bf16 rounding and determinism.  CPU only."""
import numpy as np
import pytest
import torch

import nf_inputs
from nf_inputs import bf16_round, bf16_to_f64


def test_bf16_round_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    v = rng.standard_normal(100000) * 10.0 ** rng.integers(-20, 20, 100000)
    v32 = v.astype(np.float32)
    want = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(bf16_round(v32.astype(np.float64)), want)


def test_bf16_round_ties_and_double_rounding():
    one = 1.0
    cases = {
        one + 2.0 ** -8: one,                          # tie -> even (1.0)
        one + 3 * 2.0 ** -8: one + 2.0 ** -6,          # tie -> even
        one + 2.0 ** -8 + 2.0 ** -30: one + 2.0 ** -7, # just above the tie: a float32 detour would give 1.0
        -(one + 2.0 ** -8 + 2.0 ** -30): -(one + 2.0 ** -7),
        0.0: 0.0,
    }
    for x, want in cases.items():
        got = bf16_to_f64(bf16_round(np.array([x])))[0]
        assert got == want, (x, got, want)


def test_inputs_are_seeded_and_independent_per_tensor():
    a = nf_inputs.make_inputs(16, 32, 24, seed=0, gamma=True, beta=True)
    b = nf_inputs.make_inputs(16, 32, 24, seed=0, gamma=True, beta=True)
    c = nf_inputs.make_inputs(16, 32, 48, seed=0, gamma=True, beta=True)
    for k in a:
        assert np.array_equal(a[k], b[k])
    # X does not depend on the shape of W (one stream per tensor)
    assert np.array_equal(a["X"], c["X"])
    x = bf16_to_f64(nf_inputs.make_inputs(4096, 64, 8, seed=1)["X"])
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    w = bf16_to_f64(nf_inputs.make_inputs(8, 512, 512, seed=1)["W"])
    assert abs(w.std() - 512 ** -0.5) < 0.002


def test_row_scaled_rows_are_z_times_lognormal():
    inp = nf_inputs.make_inputs(2048, 64, 8, seed=0, x_dist="row_scaled")
    x = bf16_to_f64(inp["X"])
    rms = np.sqrt((x * x).mean(-1))
    logs = np.log(rms)
    assert abs(logs.mean()) < 0.1 and abs(logs.std() - 1.0) < 0.1


def test_workloads_match_the_five_configurations():
    w = nf_inputs.WORKLOADS
    assert [w[n].M for n in nf_inputs.WORKLOAD_ORDER] == [256, 65536, 32768, 16384, 8192]
    assert [w[n].K for n in nf_inputs.WORKLOAD_ORDER] == [64, 128, 512, 1024, 4096]
    assert [w[n].N for n in nf_inputs.WORKLOAD_ORDER] == [64, 128, 512, 2048, 4096]
    assert [w[n].eps for n in nf_inputs.WORKLOAD_ORDER] == [1e-6, 1e-5, 1e-6, 1e-5, 1e-6]


def test_sample_rows_cover_edges():
    r = nf_inputs.sample_rows(65536, 64)
    assert r[0] == 0 and r[-1] == 65535 and 127 in r and 128 in r and np.all(np.diff(r) > 0)


@pytest.mark.parametrize("x_dist", ["normal", "row_scaled"])
@pytest.mark.parametrize("world", [1, 2, 3])
def test_shards_concatenate_to_the_global_problem(world, x_dist):
    """Rank r's shard is rows shard_rows(world * M, world, r) of exactly the X
    make_inputs draws for world * M rows; W, gamma and beta are the same."""
    w = nf_inputs.Workload("t", 150, 72, 40, 1e-5, ("post_ln",), x_dist=x_dist, gamma=True, beta=True)
    g = nf_inputs.make_inputs(world * w.M, w.K, w.N, seed=3, x_dist=x_dist, gamma=True, beta=True)
    xs = []
    for r in range(world):
        sh = nf_inputs.workload_shard(w, world, r, seed=3, chunk_rows=64)
        assert sh["rows"] == nf_inputs.shard_rows(world * w.M, world, r)
        for k in ("W", "gamma", "beta"):
            assert np.array_equal(sh[k], g[k])
        xs.append(sh["X"])
    assert np.array_equal(np.concatenate(xs), g["X"])
