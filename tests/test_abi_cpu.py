"""The C ABI on the CPU: the library loads, exports every symbol include/nf.h
declares, rejects bad arguments before touching a device, and plans tiles as
documented.  No compute call is made."""
import ctypes

import pytest

import normalization_gemm_gb300 as nf
from normalization_gemm_gb300 import _build

OK, INVALID, ALIGN, SHAPE = 0, 1, 2, 3
P = 1 << 20          # a 16-byte aligned fake device address (never dereferenced)


@pytest.fixture(scope="module")
def L():
    _build.build()
    return nf.lib()


def test_exports_every_declared_symbol(L):
    names = nf.header_symbols()
    assert "nf_gemm_prenorm_rms" in names and "nf_norm_rows" in names
    for name in names:
        assert hasattr(L, name), f"{name} declared in nf.h but not exported"
    assert L.nf_abi_version() == 3


def test_status_strings(L):
    for code in range(7):
        assert L.nf_status_string(code)
    assert L.nf_status_string(5) == b"device wait timed out"


def test_null_and_negative_arguments(L):
    assert L.nf_gemm_plain(None, P, P, 128, 64, 64, None) == INVALID
    assert L.nf_gemm_plain(P, P, P, -1, 64, 64, None) == INVALID
    assert L.nf_gemm_plain(P, P, P, 128, 0, 64, None) == INVALID
    assert L.nf_gemm_plain(P, P, P, 128, 64, 0, None) == INVALID
    assert b"non-null" in L.nf_last_error() or b"M >= 0" in L.nf_last_error()
    assert L.nf_norm_rows(P, P, None, None, 4, 64, 7, 1e-5, None, None, None) == INVALID


def test_residual_argument_checks(L):
    # R is required; an H without R; misaligned R / H; empty M is a no-op
    assert L.nf_gemm_postnorm_ln_res(P, P, None, None, None, P, None, 128, 64, 64, 1e-5, None, None, None) == INVALID
    assert L.nf_gemm_postnorm_rms_res(P, P, None, None, P, P, 128, 64, 64, 1e-5, None, None) == INVALID
    assert L.nf_gemm_postnorm_ln_res(P, P, P + 8, None, None, P, None, 128, 64, 64, 1e-5, None, None, None) == ALIGN
    assert L.nf_gemm_postnorm_ln_res(P, P, P, None, None, P, P + 2, 128, 64, 64, 1e-5, None, None, None) == ALIGN
    assert L.nf_gemm_postnorm_rms_res(P, P, P, None, P, None, 0, 64, 64, 1e-5, None, None) == OK
    assert L.nf_gemm_postnorm_ln_res(P, P, P, None, None, P, None, 128, 4104, 64, 1e-5, None, None, None) == SHAPE
    assert L.nf_norm_rows_res(P, None, P, None, None, None, 4, 64, 0, 1e-5, None, None, None) == INVALID
    assert L.nf_norm_rows_res(P, P + 8, P, None, None, None, 4, 64, 0, 1e-5, None, None, None) == ALIGN
    assert L.nf_norm_rows_res(P, P, P, P + 8, None, None, 4, 64, 1, 1e-5, None, None, None) == ALIGN
    assert L.nf_norm_rows_res(P, None, P, None, None, None, 0, 64, 0, 1e-5, None, None, None) == OK


def test_flashnorm_argument_checks(L):
    fn = L.nf_flashnorm_attn_fwd
    # shapes outside the kernel: D, Lkv, H, Lq; activation and eps; empty batch; alignment
    assert fn(P, P, P, None, P, 2, 256, 128, 4, 64, 1, 1e-5, 1e-6, None) == SHAPE
    assert fn(P, P, P, None, P, 2, 256, 64, 4, 128, 1, 1e-5, 1e-6, None) == SHAPE
    assert fn(P, P, P, None, P, 2, 256, 128, 9, 128, 1, 1e-5, 1e-6, None) == SHAPE
    assert fn(P, P, P, None, P, 2, 200, 128, 4, 128, 1, 1e-5, 1e-6, None) == SHAPE
    assert fn(P, P, P, None, P, 2, 256, 128, 4, 128, 3, 1e-5, 1e-6, None) == INVALID
    assert fn(P, P, P, None, P, 2, 256, 128, 4, 128, 1, -1.0, 1e-6, None) == INVALID
    assert fn(P, P, P, None, P, 2, 256, 128, 0, 128, 1, 1e-5, 1e-6, None) == INVALID
    assert fn(P, P, P, None, P, 0, 256, 128, 4, 128, 1, 1e-5, 1e-6, None) == OK
    assert fn(P + 8, P, P, None, P, 2, 256, 128, 4, 128, 1, 1e-5, 1e-6, None) == ALIGN
    assert fn(P, P, P, P + 2, P, 2, 256, 128, 4, 128, 1, 1e-5, 1e-6, None) == ALIGN
    assert fn(None, P, P, None, P, 2, 256, 128, 4, 128, 1, 1e-5, 1e-6, None) == INVALID


def test_eps_must_be_finite_and_nonnegative(L):
    for eps in (float("nan"), float("inf"), -1e-6):
        assert L.nf_gemm_prenorm_rms(P, P, P, 128, 64, 64, eps, None, None) == INVALID
        assert L.nf_gemm_postnorm_ln(P, P, None, None, P, 128, 64, 64, eps, None, None, None) == INVALID
        assert L.nf_norm_rows(P, P, None, None, 4, 64, 0, eps, None, None, None) == INVALID


def test_alignment_rules(L):
    assert L.nf_gemm_plain(P + 8, P, P, 128, 64, 64, None) == ALIGN
    assert L.nf_gemm_plain(P, P, P + 2, 128, 64, 64, None) == ALIGN
    assert L.nf_gemm_plain(P, P, P, 128, 64, 60, None) == ALIGN      # K % 8
    assert L.nf_gemm_plain(P, P, P, 128, 36, 64, None) == ALIGN      # N % 8
    assert L.nf_gemm_postnorm_ln(P, P, P + 1, None, P, 128, 64, 64, 1e-5, None, None, None) == ALIGN
    assert L.nf_gemm_prenorm_rms(P, P, P, 128, 64, 64, 1e-5, P + 2, None) == ALIGN
    assert L.nf_norm_rows(P, P, None, None, 4, 12, 0, 1e-5, None, None, None) == ALIGN
    assert L.nf_norm_rows(P, P, P + 2, None, 4, 64, 0, 1e-5, None, None, None) == ALIGN


def test_unsupported_shapes(L):
    assert L.nf_gemm_postnorm_ln(P, P, None, None, P, 128, 4104, 64, 1e-5, None, None, None) == SHAPE
    assert L.nf_gemm_postnorm_rms(P, P, None, P, 128, 8192, 64, 1e-5, None, None) == SHAPE
    assert L.nf_gemm_plain(P, P, P, 1 << 31, 64, 64, None) == SHAPE
    assert L.nf_norm_rows(P, P, None, None, 4, 16392, 0, 1e-5, None, None, None) == SHAPE


def test_empty_m_is_a_noop(L):
    # M == 0 returns before any device call, so this is safe without a GPU.
    assert L.nf_gemm_plain(P, P, P, 0, 64, 64, None) == OK
    assert L.nf_gemm_postnorm_ln(P, P, None, None, P, 0, 4096, 64, 1e-5, None, None, None) == OK
    assert L.nf_norm_rows(P, P, None, None, 0, 64, 1, 1e-5, None, None, None) == OK


def test_timeout_setting_range(L):
    assert L.nf_set_wait_timeout_ns(10) == INVALID
    assert L.nf_set_wait_timeout_ns(2_000_000_000) == OK


@pytest.mark.parametrize("op,M,N,K,tile_n,cluster,xch", [
    (0, 256, 64, 64, 64, 1, 0), (1, 256, 64, 64, 64, 1, 0), (1, 32768, 512, 512, 256, 1, 0),
    (2, 65536, 128, 128, 128, 1, 0), (2, 16384, 2048, 1024, 256, 1, 2), (3, 16384, 2048, 1024, 256, 1, 2),
    (2, 8192, 4096, 4096, 256, 1, 2), (2, 300, 264, 72, 512, 1, 0), (2, 5, 8, 8, 64, 1, 0),
    (0, 100, 200, 8, 256, 1, 0), (1, 100, 120, 8, 128, 1, 0), (3, 64, 4088, 64, 512, 8, 1),
    (2, 1000, 256, 64, 256, 1, 0), (2, 16384, 2048, 256, 256, 8, 1), (2, 16384, 512, 1024, 512, 1, 0),
    (3, 16384, 1024, 512, 256, 1, 2), (2, 16384, 1024, 448, 256, 4, 1),
])
def test_plans(L, op, M, N, K, tile_n, cluster, xch):
    if xch == 2 and K >= 2048:
        cluster = 2  # rows exchanged through L2 are computed by CTA pairs (long contractions)
    p = nf.plan_gemm(op, M, N, K, 148)
    assert p["tile_m"] == 128 and p["tile_k"] == (32 if tile_n == 512 else 64)
    assert p["tile_n"] == tile_n and p["cluster"] == cluster and p["exchange"] == xch
    assert p["smem_bytes"] <= 232448 and p["stages"] >= 2
    # four accumulators for tiles of <= 128 columns without a row exchange, else two
    assert p["tmem_cols"] == min((4 if (tile_n <= 128 and xch == 0) else 2) * tile_n, 512)
    assert p["threads"] == (448 if op == 1 else 320)
    m_tiles = -(-M // 128)
    n_tiles = 1 if (op >= 2 and xch != 2) else -(-N // tile_n)
    assert p["tiles"] == m_tiles * n_tiles
    assert 0 < p["grid"] <= 148 and p["grid"] % cluster == 0
    assert cluster <= 8  # automatic plans stay within the portable cluster size
    # 1 CTA per SM whenever the kernel takes all 512 TMEM columns
    if p["tmem_cols"] == 512:
        assert p["smem_bytes"] > 232448 // 2


def global_exchange_schedule(tiles, G):
    """Tiles of each CTA, in order, as the L2-exchange kernel walks them: tile t
    on CTA t mod G (host plan and kernel tile schedule)."""
    return [list(range(b, tiles, G)) for b in range(G)]


@pytest.mark.parametrize("M,N,K,sms", [
    (8192, 4096, 4096, 148), (16384, 2048, 1024, 148), (300, 264, 72, 148), (64, 4088, 64, 148),
    (128 * 9, 4096, 64, 8), (128 * 3, 2048, 64, 152), (65536, 4096, 64, 152), (1, 264, 8, 1),
    (8192, 3072, 4096, 152), (12345, 1800, 512, 152), (8192, 4096, 4096, 20),
])
def test_global_exchange_schedule_is_deadlock_free(L, M, N, K, sms):
    """Tiles i and i+2 of a CTA share a TMEM buffer, so the later one waits for
    the earlier one's row exchange: that wait must always point at an earlier
    row tile, and every tile must run exactly once."""
    try:
        nf.set_postnorm_exchange(nf.XCH_GLOBAL)
        p = nf.plan_gemm(2, M, N, K, sms)
    finally:
        nf.set_postnorm_exchange(0)
    assert p["exchange"] == 2
    n_tiles, G = -(-N // 256), p["grid"]
    assert p["tiles"] == -(-M // 128) * n_tiles and G == min(p["tiles"], sms)
    sched = global_exchange_schedule(p["tiles"], G)
    assert sorted(t for mine in sched for t in mine) == list(range(p["tiles"]))
    for mine in sched:
        assert mine == sorted(mine)
        for a, b in zip(mine, mine[2:]):
            assert a // n_tiles < b // n_tiles


def test_too_few_sms_for_the_global_exchange_use_a_cluster(L):
    try:
        nf.set_postnorm_exchange(nf.XCH_GLOBAL)
        p = nf.plan_gemm(2, 128 * 9, 4096, 64, 7)
    finally:
        nf.set_postnorm_exchange(0)
    assert p["exchange"] == 1 and p["cluster"] == 8


def test_cluster_exchange_plans(L):
    try:
        nf.set_postnorm_exchange(nf.XCH_CLUSTER)
        p = nf.plan_gemm(2, 8192, 4096, 4096, 148)
        assert (p["tile_n"], p["cluster"], p["tile_k"], p["exchange"]) == (512, 8, 32, 1)
        assert p["grid"] % 8 == 0
        p = nf.plan_gemm(3, 16384, 2048, 1024, 148)
        assert (p["tile_n"], p["cluster"], p["exchange"]) == (512, 4, 1)
        p = nf.plan_gemm(2, 300, 264, 72, 148)  # one 512-column CTA covers the row
        assert (p["tile_n"], p["cluster"], p["exchange"]) == (512, 1, 0)
        nf.set_postnorm_tile_n(256)
        p = nf.plan_gemm(2, 8192, 4096, 4096, 148)
        assert (p["tile_n"], p["cluster"], p["tile_k"], p["exchange"]) == (256, 16, 64, 1)
        p = nf.plan_gemm(3, 16384, 2048, 1024, 148)
        assert (p["tile_n"], p["cluster"]) == (256, 8)
    finally:
        nf.set_postnorm_tile_n(0)
        nf.set_postnorm_exchange(0)
    assert L.nf_set_postnorm_tile_n(384) == INVALID
    assert L.nf_set_postnorm_exchange(3) == INVALID


def test_python_binding_rejects_cpu_tensors():
    import torch
    x = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        nf.gemm_plain(x, x.t().contiguous())


def test_empty_m_accepts_null_bases(L):
    # empty torch tensors report a null data pointer
    assert L.nf_gemm_plain(None, P, None, 0, 64, 64, None) == OK
    assert L.nf_gemm_prenorm_rms(None, P, None, 0, 64, 64, 1e-6, None, None) == OK
    assert L.nf_norm_rows(None, None, None, None, 0, 64, 0, 1e-5, None, None, None) == OK
    assert L.nf_gemm_plain(None, P, None, 1, 64, 64, None) == INVALID


@pytest.mark.parametrize("op,M,N,K,tile_n,cluster,xch", [
    (4, 16384, 2048, 1024, 256, 1, 2), (5, 8192, 4096, 4096, 256, 1, 2), (4, 130, 2048, 64, 256, 8, 1),
    (5, 64, 4088, 64, 256, 16, 1), (4, 300, 200, 64, 256, 1, 0), (5, 300, 120, 512, 128, 1, 0),
    (4, 65536, 128, 128, 128, 1, 0),
    # rows of two tiles: a cluster of 2 (co-resident on every SM) whatever K
    (5, 32768, 512, 512, 256, 2, 1), (4, 1000, 512, 1024, 256, 2, 1), (5, 1000, 520, 4096, 256, 1, 2),
])
def test_backward_plans(L, op, M, N, K, tile_n, cluster, xch):
    """The norm backward (ops 4, 5) takes 256-column CTAs past 256 columns: the
    L2 exchange for K >= 512 and N > 512, else a cluster of ceil(N / 256) (<= 16)."""
    p = nf.plan_gemm(op, M, N, K, 148)
    assert (p["tile_n"], p["cluster"], p["exchange"], p["tile_k"]) == (tile_n, cluster, xch, 64)
    assert p["threads"] == 320 and p["tmem_cols"] == (4 if (tile_n <= 128 and xch == 0) else 2) * tile_n


def test_backward_argument_checks(L):
    # null Z / stats, misaligned Z, N beyond the post-norm limit
    assert L.nf_gemm_postnorm_ln_bwd(P, P, None, None, P, P, P, 128, 64, 64, None) == INVALID
    assert L.nf_gemm_postnorm_ln_bwd(P, P, P, None, None, P, P, 128, 64, 64, None) == INVALID
    assert L.nf_gemm_postnorm_rms_bwd(P, P, P, None, None, P, 128, 64, 64, None) == INVALID
    assert L.nf_gemm_postnorm_rms_bwd(P, P, P + 8, None, P, P, 128, 64, 64, None) in (2, 6)
    assert L.nf_gemm_postnorm_ln_bwd(P, P, P, None, P, P, P, 128, 4104, 64, None) == 3
    assert L.nf_norm_rows_bwd(P, P, None, None, P, P, 4, 64, 0, None) == INVALID
    assert L.nf_norm_rows_bwd(P, P, None, None, P, P, 0, 64, 0, None) == OK


def test_transposed_and_prenorm_backward_checks(L):
    # both operands transposed; an unknown flag; a transposed X needs M % 8 == 0
    assert L.nf_gemm_plain_t(P, P, P, 64, 64, 64, 5, None) == SHAPE
    assert L.nf_gemm_plain_t(P, P, P, 64, 64, 64, 2, None) == INVALID
    assert L.nf_gemm_plain_t(P, P, P, 60, 64, 64, 1, None) == ALIGN
    assert L.nf_gemm_plain_t(P, P, P, 0, 64, 64, 1, None) == OK
    # pre-norm backward: null inputs; dB needs M % 8 == 0; dA needs K <= 4096; nothing asked
    assert L.nf_gemm_prenorm_rms_bwd(P, P, None, P, P, P, None, 64, 64, 64, None) == INVALID
    assert L.nf_gemm_prenorm_rms_bwd(P, P, P, P, None, P, None, 60, 64, 64, None) == ALIGN
    assert L.nf_gemm_prenorm_rms_bwd(P, P, P, P, P, None, None, 64, 64, 4104, None) == SHAPE
    assert L.nf_gemm_prenorm_rms_bwd(P, P, P, P, None, None, None, 64, 64, 64, None) == OK
    # the xhat side buffer is written with 16-byte stores
    assert L.nf_gemm_prenorm_rms_bwd(P, P, P, P, P, P, P + 2, 64, 64, 64, None) == ALIGN


def splitk_slices(k_tiles, splitk):
    """K-tile range of each contraction slice, as the kernel's tile schedule
    assigns them: slice s covers [s k_tiles / splitk, (s+1) k_tiles / splitk)."""
    return [(s * k_tiles // splitk, (s + 1) * k_tiles // splitk) for s in range(splitk)]


@pytest.mark.parametrize("M,N,K,sms,splitk", [
    (512, 512, 32768, 152, 19),    # the weight gradient of the Lazy Pre-Norm backward, 32768 x 512 x 512
    (512, 512, 32768, 148, 18),
    (128, 64, 4096, 152, 8),       # one tile: slices of 8 K-tiles
    (4096, 4096, 8192, 152, 2),    # 512 tiles, tensor-bound: the last wave's 56 tiles in 2 slices
    (512, 512, 512, 152, 1),       # 8 K-tiles: no split
    (8192, 4096, 4096, 152, 1),    # 1024 tiles: last wave of 112 tiles, more than half the SMs
    (4096, 4096, 256, 152, 1),     # last wave of 56 tiles but 4 K-tiles: too short to split
    (9728, 256, 4096, 152, 2),     # 76 tiles = half the SMs, 64 K-tiles: 2 slices
    (100, 200, 2048, 152, 4),      # one tile, 32 K-tiles: slices of 8
])
def test_splitk_plans(L, M, N, K, sms, splitk):
    nf.set_gemm_pair(1)  # the split-K rules alone (CTA pairs take tensor-bound shapes by default)
    try:
        p = nf.plan_gemm(0, M, N, K, sms)
    finally:
        nf.set_gemm_pair(0)
    tiles = p["tiles"]
    assert p["splitk"] == splitk
    assert p["grid"] <= sms
    k_tiles = -(-K // 64)
    if splitk > 1 and 2 * tiles > sms:
        # only the last, partial wave is split: whole waves, then <= one split unit per SM
        rest = tiles % sms
        assert p["split_tiles"] == rest and 0 < 2 * rest <= sms and rest * splitk <= sms
        assert p["grid"] == sms
        return
    assert p["grid"] == (tiles * splitk if splitk > 1 else min(tiles, sms))
    if splitk > 1:
        assert p["split_tiles"] == tiles
        assert 2 * tiles <= sms
        sl = splitk_slices(k_tiles, splitk)
        assert sl[0][0] == 0 and sl[-1][1] == k_tiles
        assert all(a[1] == b[0] for a, b in zip(sl, sl[1:]))
        assert all(hi - lo >= 8 for lo, hi in sl)
        # a split workspace of splitk x M x N fp32 fits the per-stream buffer (SMs x 128 x 256)
        assert splitk * M * N <= sms * 128 * 256
    # the normalizing epilogues never split the contraction
    for op in (1, 2, 3):
        if N <= 4096:
            assert nf.plan_gemm(op, M, N, K, sms)["splitk"] == 1


def test_splitk_can_be_switched_off(L):
    try:
        nf.set_gemm_splitk(1)
        assert nf.plan_gemm(0, 512, 512, 32768, 152)["splitk"] == 1
    finally:
        nf.set_gemm_splitk(0)
    assert nf.plan_gemm(0, 512, 512, 32768, 152)["splitk"] == 19
    assert L.nf_set_gemm_splitk(2) == INVALID


def test_reserve_scratch_argument_checks(L):
    """Sizes are validated before any device work."""
    assert L.nf_reserve_scratch(-1, 0, None) == INVALID
    assert L.nf_reserve_scratch(0, -8, None) == INVALID
    assert L.nf_reserve_scratch(1024, 4104, None) == SHAPE


@pytest.mark.parametrize("op,M,N,K,pair", [
    (0, 8192, 4096, 4096, True),    # tensor-bound 256-column tiles
    (1, 8192, 4096, 4096, True),    # pre-norm GEMMs whose sums of squares are split over a row's tiles
    (1, 8192, 256, 4096, False),    # ... but not a row of one tile (every tile sums its own rows)
    (0, 4096, 4096, 8192, True),    # pairs instead of splitting the last wave
    (0, 512, 512, 32768, False),    # 8 tiles: every tile split over the contraction instead
    (1, 32768, 512, 512, False),    # memory-bound tiles
    (0, 100, 200, 2048, False),     # a single 128-row tile
    (0, 4096, 128, 4096, False),    # 128-column tiles
    (2, 8192, 4096, 4096, True),    # post-norm rows exchanged through L2
    (3, 16384, 2048, 1024, False),  # ... but not with a short contraction (epilogue-bound tiles)
    (2, 16384, 2048, 256, False),   # post-norm rows in a DSMEM cluster (K < 512)
    (2, 65536, 128, 128, False),    # one CTA holds whole rows
])
def test_pair_plans(L, op, M, N, K, pair):
    p = nf.plan_gemm(op, M, N, K, 148)
    assert (p["cluster"] == 2 and p["exchange"] in (0, 2)) == pair
    if pair:
        assert p["tile_n"] == 256 and p["splitk"] == 1 and p["grid"] % 2 == 0
        pair_tiles = -(-M // 256) * -(-N // 256)
        assert p["grid"] == 2 * min(pair_tiles, 148 // 2)
    nf.set_gemm_pair(1)
    try:
        assert nf.plan_gemm(op, M, N, K, 148)["cluster"] != 2 or nf.plan_gemm(op, M, N, K, 148)["exchange"] == 1
    finally:
        nf.set_gemm_pair(0)
    assert L.nf_set_gemm_pair(3) == INVALID


@pytest.mark.parametrize("M,N,K,split", [
    (8192, 4096, 4096, (2, 0, 2)),    # tensor-bound tiles, 16 a row: split by default
    (16384, 2048, 2048, (2, 0, 2)),   # 8 a row
    (16384, 2048, 1024, (0, 0, 2)),   # ... but a contraction shorter than 2048: only on request
    (32768, 512, 512, (0, 0, 2)),     # memory-bound tiles: only on request
    (8192, 256, 4096, (0, 0, 0)),     # one tile a row: nothing to share
    (1024, 8448, 4096, (0, 0, 0)),    # 33 tiles a row: beyond the gather's limit
    (100, 4096, 4096, (2, 0, 2)),     # a single row tile
])
def test_prenorm_split_plans(L, M, N, K, split):
    """Lazy Pre-Norm with the row sums of squares split over a row's tiles:
    exchange 2 (the L2 gather) for modes 0 (automatic), 1 (never), 2 (always)."""
    try:
        for mode, want in zip((0, 1, 2), split):
            nf.set_prenorm_split(mode)
            p = nf.plan_gemm(1, M, N, K, 148)
            assert p["exchange"] == want, (mode, p)
            if want:
                assert p["tile_n"] == 256 and p["splitk"] == 1
    finally:
        nf.set_prenorm_split(0)
    assert L.nf_set_prenorm_split(3) == INVALID
    assert L.nf_set_prenorm_split(-1) == INVALID
