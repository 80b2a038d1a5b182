"""Seeded synthetic inputs for the normalization-fused GEMM.

This module is shared by the CPU oracle's tests and by the CUDA path's tests
and benchmark.  It draws random samples and rounds them to bfloat16; it holds
none of the method's arithmetic (no matmul, no norm).

Recipe (one independent PCG64 stream per tensor, spawned from one seed):
  * samples are drawn in float64 with numpy's ``Generator(PCG64)``;
  * each sample is rounded once to bfloat16, round-to-nearest-even, by exact
    float64 operations (``frexp`` / ``rint`` / ``ldexp``), never through an
    intermediate float32 (which could double-round);
  * ``N(mu, v)`` names a normal distribution with mean ``mu`` and VARIANCE
    ``v``; ``LogNormal(0, 1)`` is ``exp`` of a standard normal.

The five workloads follow the shapes and distributions of the blog "Towards
Free Normalization: Fusing Normalization into GEMM and Attention Kernels"
(ads shapes of §1/§3 with M large and K, N of a few hundred; LLM-sized
K = N = 4096 of §3).  The blog's own ads data is proprietary, so these
synthetic tensors stand in for it.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np

# Stream order inside one seed; fixed so that every consumer draws the same
# numbers for the same tensor.
_STREAMS = ("X", "W", "gamma", "beta", "scale")


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round float64 values to bfloat16 (round-to-nearest-even); return bits.

    The result is a ``uint16`` array holding the upper 16 bits of the
    float32 encoding of the rounded value.  Values whose magnitude is below
    the smallest normal float32 are flushed to a signed zero; the generators
    here never produce one in practice (probability < 1e-30).
    """
    a = np.asarray(a, dtype=np.float64)
    if not np.all(np.isfinite(a)):
        raise ValueError("bf16_round: non-finite input")
    mant, expo = np.frexp(a)              # a = mant * 2**expo, |mant| in [0.5, 1)
    q = np.rint(mant * 256.0)             # 8 significant bits, ties to even
    r = np.ldexp(q / 256.0, expo)         # exact in float64
    tiny = np.abs(r) < np.ldexp(1.0, -126)
    r = np.where(tiny, np.copysign(0.0, a), r)
    if np.any(np.abs(r) > 3.3895313892515355e38):
        raise ValueError("bf16_round: overflow")
    bits = r.astype(np.float32).view(np.uint32)   # exact: r has 8 significant bits
    return (bits >> 16).astype(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float64 exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def _streams(seed: int) -> Dict[str, np.random.Generator]:
    children = np.random.SeedSequence(seed).spawn(len(_STREAMS))
    return {name: np.random.Generator(np.random.PCG64(c))
            for name, c in zip(_STREAMS, children)}


def _normal(g: np.random.Generator, shape, mean: float, var: float) -> np.ndarray:
    return g.normal(loc=mean, scale=np.sqrt(var), size=shape)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic problem: shapes, distributions and which ops run on it."""
    name: str
    M: int
    K: int
    N: int
    eps: float
    ops: tuple                      # subset of ("pre_rms", "post_ln", "post_rms")
    x_dist: str = "normal"          # "normal" or "row_scaled"
    gamma: bool = False             # post-norm gain gamma ~ N(1, 0.1)
    beta: bool = False              # post-LN bias beta ~ N(0, 0.1)
    description: str = ""

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


# The five workloads: a tiny pre-norm case, the ads-shaped post-LayerNorm
# case, a pre-norm case with widely varying row scales, a post-norm case
# with affine parameters and a row that spans an 8-CTA cluster, and an
# LLM-sized case whose post-norm row spans a 16-CTA cluster.
WORKLOADS: Dict[str, Workload] = {w.name: w for w in (
    Workload("pre_rms_256x64x64", 256, 64, 64, 1e-6, ("pre_rms",),
             description="Lazy pre-RMSNorm GEMM, no affine, X~N(0,1), W~N(0,1/64)"),
    Workload("post_ln_65536x128x128", 65536, 128, 128, 1e-5, ("post_ln",),
             description="ads-shaped post-LayerNorm GEMM, no affine"),
    Workload("pre_rms_rowscale_32768x512x512", 32768, 512, 512, 1e-6, ("pre_rms",),
             x_dist="row_scaled",
             description="pre-RMSNorm GEMM, X row i = z_i*s_i, s_i~LogNormal(0,1)"),
    Workload("post_affine_16384x1024x2048", 16384, 1024, 2048, 1e-5,
             ("post_ln", "post_rms"), gamma=True, beta=True,
             description="post-LN (gamma, beta) and post-RMS (gamma) over N=2048"),
    Workload("llm_8192x4096x4096", 8192, 4096, 4096, 1e-6, ("pre_rms", "post_ln"),
             description="LLM-shaped pre-RMS and post-LN GEMM, no affine"),
)}

# Order used by the five configurations of the benchmark definition.
WORKLOAD_ORDER = ("pre_rms_256x64x64", "post_ln_65536x128x128",
                  "pre_rms_rowscale_32768x512x512", "post_affine_16384x1024x2048",
                  "llm_8192x4096x4096")


def make_inputs(M: int, K: int, N: int, seed: int = 0, x_dist: str = "normal",
                gamma: bool = False, beta: bool = False,
                w_var: Optional[float] = None) -> Dict[str, np.ndarray]:
    """Draw X (M x K), W (K x N) and optional gamma / beta (N) as bf16 bits.

    X ~ N(0, 1) (or z_i * s_i with s_i ~ LogNormal(0, 1) per row when
    ``x_dist == "row_scaled"``, the product formed in float64 and rounded
    once), W ~ N(0, 1/K) unless ``w_var`` is given, gamma ~ N(1, 0.1),
    beta ~ N(0, 0.1).  Row-major, C-contiguous.
    """
    g = _streams(seed)
    if x_dist == "normal":
        x = _normal(g["X"], (M, K), 0.0, 1.0)
    elif x_dist == "row_scaled":
        z = _normal(g["X"], (M, K), 0.0, 1.0)
        s = np.exp(g["scale"].normal(0.0, 1.0, size=(M, 1)))
        x = z * s
    else:
        raise ValueError(f"unknown x_dist {x_dist!r}")
    out = {
        "X": bf16_round(x),
        "W": bf16_round(_normal(g["W"], (K, N), 0.0,
                                (1.0 / K) if w_var is None else w_var)),
    }
    if gamma:
        out["gamma"] = bf16_round(_normal(g["gamma"], (N,), 1.0, 0.1))
    if beta:
        out["beta"] = bf16_round(_normal(g["beta"], (N,), 0.0, 0.1))
    return out


def workload_inputs(w: Workload, seed: int = 0) -> Dict[str, np.ndarray]:
    return make_inputs(w.M, w.K, w.N, seed=seed, x_dist=w.x_dist,
                       gamma=w.gamma, beta=w.beta)


def shard_rows(total_rows: int, world: int, rank: int):
    """Contiguous row range [lo, hi) of `rank` when rows split over `world`
    processes (sizes differ by at most one)."""
    base, extra = divmod(total_rows, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def workload_shard(w: Workload, world: int, rank: int, seed: int = 0,
                   chunk_rows: int = 4096) -> Dict[str, np.ndarray]:
    """Rows shard_rows(world * w.M, world, rank) of the global problem with
    world * w.M rows (X drawn exactly as make_inputs would draw it for that
    many rows: the same streams in the same order, generated in chunks and
    only the shard kept), with the full W, gamma and beta.  world == 1 gives
    workload_inputs(w)."""
    total = world * w.M
    lo, hi = shard_rows(total, world, rank)
    g = _streams(seed)
    parts = []
    scale = None
    if w.x_dist == "row_scaled":  # the row scales have a stream of their own
        scale = np.exp(g["scale"].normal(0.0, 1.0, size=(total, 1)))[lo:hi]
    elif w.x_dist != "normal":
        raise ValueError(f"unknown x_dist {w.x_dist!r}")
    for r0 in range(0, hi, chunk_rows):
        r1 = min(hi, r0 + chunk_rows)
        z = _normal(g["X"], (r1 - r0, w.K), 0.0, 1.0)
        if r1 > lo:
            parts.append(z[max(lo, r0) - r0:])
    x = np.concatenate(parts) if parts else np.zeros((0, w.K))
    if scale is not None:
        x = x * scale
    out = {"X": bf16_round(x),
           "W": bf16_round(_normal(g["W"], (w.K, w.N), 0.0, 1.0 / w.K))}
    if w.gamma:
        out["gamma"] = bf16_round(_normal(g["gamma"], (w.N,), 1.0, 0.1))
    if w.beta:
        out["beta"] = bf16_round(_normal(g["beta"], (w.N,), 0.0, 0.1))
    out["rows"] = (lo, hi)
    return out


def sample_rows(M: int, count: int, seed: int = 1, tile_m: int = 128) -> np.ndarray:
    """Rows to check at full size: both ends, every tile edge near them and a
    seeded spread in between (sorted, unique, int64)."""
    edges = [0, 1, M - 1, M - 2]
    for t in (1, 2, (M // tile_m) // 2, M // tile_m - 1):
        for d in (-1, 0):
            edges.append(t * tile_m + d)
    rng = np.random.Generator(np.random.PCG64(seed))
    extra = rng.integers(0, M, size=max(0, count - len(edges)))
    rows = np.unique(np.clip(np.array(edges + list(extra), dtype=np.int64), 0, M - 1))
    return rows


# ---------------------------------------------------------------- attention inputs
# FlashNormAttention (blog §4): Q [B, Lq, H, D] with jagged lengths, dense K / V
# [B, Lkv, H, D].  The pages give the structure (K/V length exactly 128, head
# dimension 128, batch 768, Q of average sparsity 0.5 and varied maximum
# length) but no value distributions: Q ~ N(0, 1); K with variance 1/D and V
# with variance 1/Lkv, so that scores and the attention output stay of order
# one; q_len[b] uniform on [0, Lq] (half the positions empty on average).
def fna_inputs(B: int, Lq: int, Lkv: int, H: int, D: int, seed: int = 0, jagged: bool = True):
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0xF7A])))
    Q = bf16_round(_normal(g, (B, Lq, H, D), 0.0, 1.0))
    K = bf16_round(_normal(g, (B, Lkv, H, D), 0.0, 1.0 / D))
    V = bf16_round(_normal(g, (B, Lkv, H, D), 0.0, 1.0 / Lkv))
    q_len = (g.integers(0, Lq + 1, size=B) if jagged else np.full(B, Lq)).astype(np.int32)
    return {"Q": Q, "K": K, "V": V, "q_len": q_len}


# The attention workload of the blog's §4 benchmark shapes: batch 768, K/V
# length 128, head dimension 128, 4 heads (H*D = 512), maximum query length 1024.
FNA_WORKLOAD = {"name": "fna_768x1024x4x128", "B": 768, "Lq": 1024, "Lkv": 128, "H": 4, "D": 128,
                "act": 1, "eps1": 1e-5, "eps2": 1e-6}
