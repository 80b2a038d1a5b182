"""Benchmark of the fused norm-GEMM on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {nf,reference}]

Workload of the headline line: the LLM-shaped configuration, X 8192 x 4096 and
W 4096 x 4096 (bf16, fp32 accumulation, eps 1e-6, no affine; X ~ N(0, 1),
W ~ N(0, 1/4096)), on which the two fused operations run: the Lazy Pre-Norm
GEMM Y1 = RMSNorm(X) @ W and the Multi-CTA post-norm GEMM Y2 = LayerNorm(X @ W)
over the 4096-column row.  One step = both calls (nf_gemm_prenorm_rms, then
nf_gemm_postnorm_ln) on one batch, i.e. one pass of the whole hot path:
2 * 2MNK flops.

Prints ONE JSON line (rank 0):
  value        TFLOP/s of the whole job (all ranks' steps), inputs resident in
               HBM, timed with CUDA events on the launching stream over exactly
               K steps replayed from one CUDA graph.  Successive steps rotate
               over buffer sets whose footprint exceeds 3x L2.
  roofline     the dominant kernel of the step (the one with the larger mean
               duration, each timed alone: short bursts of back-to-back launches
               from CUDA graphs, the step's kernels interleaved over five rounds,
               median) against the burst bf16 tensor peak of MEASURED_PEAKS.json
               (2MNK per launch over its mean duration); traffic (DRAM read +
               write bytes per launch) from the committed ncu summary of that
               kernel when its source hash matches, else null.
  norm_hidden_pct  100 * (sum of T_plain + T_norm - sum of T_fused) / sum of
               T_norm over the step's two operations, against this library's
               own unfused pairs (nf_gemm_plain + nf_norm_rows), every kernel
               timed the same way (CUDA graphs of back-to-back launches).
  e2e          the same metric through the Python API with host buffers: each
               step copies X and W from pinned host memory, runs both calls and
               reads both outputs back (pipelined over copy and compute streams).
  cpu_baseline the fp64 oracle on the host cores (a bounded sample of rows).
  configs      compact per-workload figures for every other configuration, the
               backward and residual variants and the FlashNormAttention
               forward: [fused us, plain us, norm us, fraction of roofline,
               % of the norm hidden] (context, not the headline).
--impl reference times the fp64 oracle itself as the reference arm.
Under torchrun (N > 1) the global problem has N * 8192 rows of one seeded X;
each rank takes its contiguous shard of rows (shard_rows), W is replicated,
and no collective touches the data path (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import nf_inputs  # noqa: E402

WORKLOAD = "llm_8192x4096x4096"
GRAPH_CHUNK = 1000
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------- helpers
def algorithmic_bytes(M, N, K, gamma=False, beta=False, stats=0):
    """Each tensor moved once: X and W read, Y written (+ gamma/beta, + stats)."""
    return 2 * M * K + 2 * K * N + 2 * M * N + 2 * N * (int(gamma) + int(beta)) + 4 * M * stats


def norm_bytes(rows, cols, affine=0):
    return 4 * rows * cols + 2 * cols * affine


shard_rows = nf_inputs.shard_rows


def max_over_ranks(x: float, dist) -> float:
    """Max of a per-rank float over the process group (identity without one)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    import torch
    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def kernel_source_hash() -> str:
    """Hash of the sources the fused GEMM kernels are built from (not the
    attention kernel's), which a profile's counters are tied to."""
    from normalization_gemm_gb300 import _build
    return _build.source_hash(_build.GEMM_SOURCES)


KERNEL_OF_OP = {"pre_rms": "nf_gemm_prenorm_rms", "post_ln": "nf_gemm_postnorm_ln",
                "post_rms": "nf_gemm_postnorm_rms", "plain": "nf_gemm_plain"}


OPCODE = {"plain": 0, "pre_rms": 1, "post_ln": 2, "post_rms": 3}


def profiled_traffic(workload: str, op: str, cta_pair: bool = False):
    """Per-launch DRAM bytes (read + write) of the op's fused kernel from the
    committed ncu summary, or None when the summary is missing, gives no
    write bytes, was taken of the other form (CTA pair or single CTA) than
    the one the bench ran, or the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{KERNEL_OF_OP[op]}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith(("traffic_bytes_per_launch", "kernel_source_hash",
                                                    "traffic_includes_writes", "traffic_cta_pair")):
            k, v = line.strip().split(":", 1)
            vals[k.strip()] = (v.split() or [""])[0].strip("`")
    if vals.get("kernel_source_hash") != kernel_source_hash() or vals.get("traffic_includes_writes") != "yes":
        return None
    if vals.get("traffic_cta_pair", "no") != ("yes" if cta_pair else "no"):
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while a region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t_start = time.time()

        def reader():
            for line in self.proc.stdout:
                self.lines.append((time.time(), line.strip()))
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self):
        self.t_stop = time.time()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self, window: str):
        rows = []
        for _, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[4:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": window}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, _, flags in rows:
            for name, flag in zip(names, flags[1:5]):
                if flag.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows), "window": window}


# ---------------------------------------------------------------- device timing
def _to_dev(a, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def _l2_bytes(dev):
    import torch
    return int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2 ** 20))


def make_sets(tensors, set_bytes, dev, min_sets=2):
    """Copies of the input/output tensors so that cycling through them touches
    more than 3x L2 between two uses of the same set."""
    n = max(min_sets, -(-3 * _l2_bytes(dev) // max(1, set_bytes)))
    return [[t.clone() for t in tensors] for _ in range(n)], n


def graph_of(fn, count, stream):
    """Capture `count` calls fn(i) (i = 0..count-1) into one CUDA graph."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(count):
            fn(i)
    return g


def time_steps(fn, steps, warmup, stream, dist=None, chunk=GRAPH_CHUNK, sampler=None, eager=False):
    """Run `warmup` untimed steps, then time exactly `steps` calls of fn(i) from
    CUDA graphs (or eagerly) with events on `stream`; returns seconds (max over
    ranks)."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(warmup):
            fn(i)
    torch.cuda.synchronize()
    if eager:
        if dist is not None and dist.is_initialized():
            dist.barrier()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for i in range(steps):
                fn(i)
            t1.record(stream)
        torch.cuda.synchronize()
        return max_over_ranks(t0.elapsed_time(t1) / 1e3, dist)
    full = min(chunk, steps)
    g_full = graph_of(fn, full, stream) if full > 0 else None
    rem = steps - (steps // full) * full if full else 0
    g_rem = graph_of(fn, rem, stream) if rem else None
    torch.cuda.synchronize()
    if dist is not None and dist.is_initialized():
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.start()
    with torch.cuda.stream(stream):
        t0.record(stream)
        for _ in range(steps // full if full else 0):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.stop()
    if dist is not None and dist.is_initialized():
        dist.barrier()
    sec = t0.elapsed_time(t1) / 1e3
    return max_over_ranks(sec, dist)


# ---------------------------------------------------------------- workloads
def run_op(nf, op, X, W, Y, G, B, eps, stream):
    if op == "pre_rms":
        nf.gemm_prenorm_rms(X, W, eps, out=Y, stream=stream)
    elif op == "post_ln":
        nf.gemm_postnorm_ln(X, W, eps, G, B, out=Y, stream=stream)
    elif op == "post_rms":
        nf.gemm_postnorm_rms(X, W, eps, G, out=Y, stream=stream)
    else:
        nf.gemm_plain(X, W, out=Y, stream=stream)


def measure_workload(nf, w, op, dev, stream, steps, warmup, seed=0, dist=None, sampler=None,
                     unfused=True, eager=False, rounds=1):
    """Fused, plain-GEMM and norm-kernel time per launch for one workload/op.

    rounds > 1: the three kernels are timed in `rounds` interleaved bursts of
    `steps` launches each and the medians kept -- on a power-capped part a
    long loop of one kernel heats the chip for the next one, which then runs
    at a lower clock than the first."""
    import torch
    inp = nf_inputs.workload_inputs(w, seed=seed)
    X0, W0 = _to_dev(inp["X"], dev), _to_dev(inp["W"], dev)
    G = _to_dev(inp["gamma"], dev) if w.gamma else None
    B = _to_dev(inp["beta"], dev) if (w.beta and op == "post_ln") else None
    Y0 = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
    set_bytes = X0.numel() * 2 + Y0.numel() * 2
    sets, nsets = make_sets([X0, Y0], set_bytes, dev)
    fused = lambda i: run_op(nf, op, sets[i % nsets][0], W0, sets[i % nsets][1], G, B, w.eps, stream)  # noqa: E731
    if rounds == 1:
        t_fused = time_steps(fused, steps, warmup, stream, dist, sampler=sampler, eager=eager)
        out = {"t_fused": t_fused / steps, "sets": nsets, "set_bytes": set_bytes, "fused_fn": fused}
    else:
        out = {"sets": nsets, "set_bytes": set_bytes, "fused_fn": fused}
    if not unfused:
        if rounds > 1:
            out["t_fused"] = statistics.median(time_steps(fused, steps, warmup, stream, dist, eager=eager) / steps
                                               for _ in range(rounds))
        return out
    # unfused pair of the blog's §1 baseline
    plain = lambda i: nf.gemm_plain(sets[i % nsets][0], W0, out=sets[i % nsets][1], stream=stream)  # noqa: E731
    ksteps = max(1, min(steps, 2000))
    if rounds == 1:
        out["t_plain"] = time_steps(plain, ksteps, min(warmup, 10), stream, dist, eager=eager) / ksteps
    if op == "pre_rms":
        rows, cols, src = w.M, w.K, 0   # norm on X (M x K) into a scratch copy
        scratch = [torch.empty_like(s[0]) for s in sets]
        norm = lambda i: nf.norm_rows(sets[i % nsets][0], nf.NORM_RMS, w.eps, out=scratch[i % nsets],  # noqa: E731
                                      stream=stream)
    else:
        rows, cols = w.M, w.N
        scratch = [torch.empty_like(s[1]) for s in sets]
        kind = nf.NORM_LN if op == "post_ln" else nf.NORM_RMS
        norm = lambda i: nf.norm_rows(sets[i % nsets][1], kind, w.eps, G, B, out=scratch[i % nsets],  # noqa: E731
                                      stream=stream)
    if rounds == 1:
        out["t_norm"] = time_steps(norm, ksteps, min(warmup, 10), stream, dist, eager=eager) / ksteps
    else:
        times = {"t_fused": [], "t_plain": [], "t_norm": []}
        for _ in range(rounds):
            for key, fn in (("t_fused", fused), ("t_plain", plain), ("t_norm", norm)):
                times[key].append(time_steps(fn, steps, warmup, stream, dist, eager=eager) / steps)
        out.update({key: statistics.median(v) for key, v in times.items()})
    out["norm_cols"] = cols
    out["norm_rows"] = rows
    del scratch
    torch.cuda.empty_cache()
    return out


def measure_residual(nf, w, kind, dev, stream, steps, warmup, seed=0, eager=False, unfused=True):
    """Residual-add post-norm (H = X W + R, Y = norm(H), H written back) and
    its unfused pair: the plain GEMM, then the residual-add row norm."""
    import torch
    inp = nf_inputs.workload_inputs(w, seed=seed)
    R0 = _to_dev(nf_inputs.make_inputs(w.M, w.N, 8, seed=seed + 11)["X"], dev)
    X0, W0 = _to_dev(inp["X"], dev), _to_dev(inp["W"], dev)
    G = _to_dev(inp["gamma"], dev) if w.gamma else None
    B = _to_dev(inp["beta"], dev) if (w.beta and kind == 0) else None
    Y0 = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
    H0 = torch.empty_like(Y0)
    set_bytes = 2 * (X0.numel() + 3 * Y0.numel())
    sets, nsets = make_sets([X0, R0, Y0, H0], set_bytes, dev)

    def fused(i):
        x, r, y, h = sets[i % nsets]
        if kind == 0:
            nf.gemm_postnorm_ln_res(x, W0, r, w.eps, G, B, out=y, h_out=h, stream=stream)
        else:
            nf.gemm_postnorm_rms_res(x, W0, r, w.eps, G, out=y, h_out=h, stream=stream)

    out = {"t_fused": time_steps(fused, steps, warmup, stream, eager=eager) / steps}
    if not unfused:
        del sets
        torch.cuda.empty_cache()
        return out
    zs = [torch.empty_like(Y0) for _ in range(nsets)]

    def plain(i):
        nf.gemm_plain(sets[i % nsets][0], W0, out=zs[i % nsets], stream=stream)

    def norm(i):
        x, r, y, h = sets[i % nsets]
        nf.norm_rows_res(zs[i % nsets], r, kind, w.eps, G, B, out=y, h_out=h, stream=stream)

    ksteps = max(1, min(steps, 2000))
    out["t_plain"] = time_steps(plain, ksteps, min(warmup, 10), stream) / ksteps
    out["t_norm"] = time_steps(norm, ksteps, min(warmup, 10), stream) / ksteps
    del sets, zs
    torch.cuda.empty_cache()
    return out


def measure_flashnorm(nf, dev, stream, steps, warmup, seed=0, eager=False, unfused=True, batch=None):
    """FlashNormAttention forward on the blog §4 benchmark shapes (batch 768, K/V
    length 128, head dimension 128, 4 heads, query length up to 1024 with
    jagged lengths of average sparsity 0.5).  Returns times and the algorithmic
    figures: each valid query row read once and written once, K and V read
    once; flops of the two matmuls over the valid rows.  The comparison is the
    same computation as torch eager ops (layer_norm, two bf16 einsums, the
    activation, adds, rms_norm), dense over the padded rows."""
    import torch
    import torch.nn.functional as F
    fw = nf_inputs.FNA_WORKLOAD
    B, Lq, Lkv, H, D = fw["B"], fw["Lq"], fw["Lkv"], fw["H"], fw["D"]
    B = batch or B
    inp = nf_inputs.fna_inputs(B, Lq, Lkv, H, D, seed=seed)
    dev4 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    q0, k, v = dev4(inp["Q"]), dev4(inp["K"]), dev4(inp["V"])
    ql = torch.from_numpy(inp["q_len"]).to(dev)
    rows = int(inp["q_len"].sum())
    out0 = torch.empty_like(q0)
    sets, nsets = make_sets([q0, out0], 4 * q0.numel(), dev)

    def fused(i):
        q, o = sets[i % nsets]
        nf.flashnorm_attn_fwd(q, k, v, act=fw["act"], eps1=fw["eps1"], eps2=fw["eps2"], q_len=ql, out=o,
                              stream=stream)

    res = {"t_fused": time_steps(fused, steps, warmup, stream, eager=eager) / steps,
           "bytes": 2 * rows * H * D * 2 + 2 * B * Lkv * H * D * 2,
           "flops": 4 * rows * Lkv * D * H, "rows": rows}
    if unfused:
        def torch_step(i):
            q, o = sets[i % nsets]
            x = q.view(B, Lq, H * D)
            ln = F.layer_norm(x.float(), (H * D,), eps=fw["eps1"]).to(torch.bfloat16).view(B, Lq, H, D)
            s = torch.einsum("bthd,bjhd->bhtj", ln, k)
            p = F.gelu(s.float(), approximate="tanh").to(torch.bfloat16)
            h = torch.einsum("bhtj,bjhd->bthd", p, v).float() + ln.float()
            y = F.rms_norm(h.reshape(B, Lq, H * D), (H * D,), eps=fw["eps2"]) + x.float()
            o.copy_(y.view(B, Lq, H, D))
        n = max(3, min(steps, 20))
        res["t_torch"] = time_steps(torch_step, n, 3, stream, eager=True) / n
    del sets
    torch.cuda.empty_cache()
    return res


def residual_bytes(w, kind):
    """Each tensor moved once: X, W and R read, Y and H written (+ gamma, beta)."""
    return (2 * w.M * w.K + 2 * w.K * w.N + 6 * w.M * w.N + (2 * w.N if w.gamma else 0)
            + (2 * w.N if (w.beta and kind == 0) else 0))


def backward_inputs(w, seed=0):
    """Inputs of the normalization backward on workload w's shapes: A = X
    (M x K, the incoming gradient dOut), B = W (K x N, standing in for the next
    linear's transposed weight), Z (M x N, the forward's norm input: mean 0.3,
    std 1.5) and Z's own row statistics (fp32), as the forward would save them."""
    inp = nf_inputs.workload_inputs(w, seed=seed)
    z = nf_inputs.make_inputs(w.M, w.N, 8, seed=seed + 7)["X"]
    Z = nf_inputs.bf16_round(nf_inputs.bf16_to_f64(z) * 1.5 + 0.3)
    zf = nf_inputs.bf16_to_f64(Z)
    mean = zf.mean(-1)
    var = ((zf - mean[:, None]) ** 2).mean(-1)
    ms = (zf * zf).mean(-1)
    return inp, Z, mean.astype(np.float32), var, ms


def measure_backward(nf, w, kind, dev, stream, steps, warmup, seed=0, eager=False, unfused=True):
    """Fused GEMM + norm-backward epilogue, and the unfused pair (plain GEMM
    writing dY, then the row backward kernel), time per launch."""
    import torch
    inp, Z, mean, var, ms = backward_inputs(w, seed)
    rstd = (1.0 / np.sqrt((var if kind == 0 else ms) + w.eps)).astype(np.float32)
    A0, B0, Z0 = _to_dev(inp["X"], dev), _to_dev(inp["W"], dev), _to_dev(Z, dev)
    G = _to_dev(inp["gamma"], dev) if w.gamma else None
    mean_d = torch.from_numpy(mean).to(dev) if kind == 0 else None
    rstd_d = torch.from_numpy(rstd).to(dev)
    D0 = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
    set_bytes = A0.numel() * 2 + Z0.numel() * 2 + D0.numel() * 2
    sets, nsets = make_sets([A0, Z0, D0], set_bytes, dev)

    def fused(i):
        a, z, d = sets[i % nsets]
        if kind == 0:
            nf.gemm_postnorm_ln_bwd(a, B0, z, mean_d, rstd_d, G, out=d, stream=stream)
        else:
            nf.gemm_postnorm_rms_bwd(a, B0, z, rstd_d, G, out=d, stream=stream)

    out = {"t_fused": time_steps(fused, steps, warmup, stream, eager=eager) / steps}
    if not unfused:
        del sets
        torch.cuda.empty_cache()
        return out
    dys = [torch.empty_like(D0) for _ in range(nsets)]
    plain = lambda i: nf.gemm_plain(sets[i % nsets][0], B0, out=dys[i % nsets], stream=stream)  # noqa: E731
    norm = lambda i: nf.norm_rows_bwd(dys[i % nsets], sets[i % nsets][1], kind, mean_d, rstd_d, G,  # noqa: E731
                                      out=sets[i % nsets][2], stream=stream)
    ksteps = max(1, min(steps, 2000))
    out["t_plain"] = time_steps(plain, ksteps, min(warmup, 10), stream) / ksteps
    out["t_norm"] = time_steps(norm, ksteps, min(warmup, 10), stream) / ksteps
    del sets, dys
    torch.cuda.empty_cache()
    return out


def measure_prenorm_backward(nf, w, dev, stream, steps, warmup, seed=0, eager=False, unfused=True):
    """Lazy Pre-Norm backward: the fused pair of kernels (dA with the RMS-backward
    epilogue, which also writes rmsnorm(A) as a side output; dB a GEMM over it)
    against the unfused sequence: rmsnorm(A) materialized, dB = xhat^T dC and
    dXhat = dC B^T by the transposed plain GEMMs, dA by the row backward kernel."""
    import torch
    inp = nf_inputs.workload_inputs(w, seed=seed)
    dC = nf_inputs.make_inputs(w.M, w.N, 8, seed=seed + 3)["X"]
    a = nf_inputs.bf16_to_f64(inp["X"])
    rstd = (1.0 / np.sqrt((a * a).mean(-1) + w.eps)).astype(np.float32)
    A0, B0, C0 = _to_dev(inp["X"], dev), _to_dev(inp["W"], dev), _to_dev(dC, dev)
    r = torch.from_numpy(rstd).to(dev)
    dA0 = torch.empty_like(A0)
    dB0 = torch.empty((w.K, w.N), dtype=torch.bfloat16, device=dev)
    XH0 = torch.empty_like(A0)
    set_bytes = 2 * (3 * A0.numel() + C0.numel()) + dB0.numel() * 2
    sets, nsets = make_sets([A0, C0, dA0, dB0, XH0], set_bytes, dev)

    def fused(i):
        x, c, da, db, xhat = sets[i % nsets]
        nf.gemm_prenorm_rms_bwd(x, B0, r, c, da=da, db=db, xhat=xhat, stream=stream)

    out = {"t_fused": time_steps(fused, steps, warmup, stream, eager=eager) / steps}
    if not unfused:
        del sets
        torch.cuda.empty_cache()
        return out
    xh = [torch.empty_like(A0) for _ in range(nsets)]
    dxh = [torch.empty_like(A0) for _ in range(nsets)]

    def gemms(i):
        x, c, da, db, _ = sets[i % nsets]
        nf.gemm_plain_t(xh[i % nsets], c, nf.TRANS_X, out=db, stream=stream)
        nf.gemm_plain_t(c, B0, nf.TRANS_W, out=dxh[i % nsets], stream=stream)

    def norms(i):
        x, c, da, db, _ = sets[i % nsets]
        nf.norm_rows(x, nf.NORM_RMS, w.eps, out=xh[i % nsets], stream=stream)
        nf.norm_rows_bwd(dxh[i % nsets], x, nf.NORM_RMS, None, r, out=da, stream=stream)

    ksteps = max(1, min(steps, 2000))
    out["t_plain"] = time_steps(gemms, ksteps, min(warmup, 10), stream) / ksteps
    out["t_norm"] = time_steps(norms, ksteps, min(warmup, 10), stream) / ksteps
    del sets, xh, dxh
    torch.cuda.empty_cache()
    return out


def backward_bytes(w, kind):
    """Each tensor moved once: A, B and Z read, dZ written, the saved
    statistics (and gamma) read."""
    return (2 * w.M * w.K + 2 * w.K * w.N + 4 * w.M * w.N + 4 * w.M * (2 if kind == 0 else 1)
            + (2 * w.N if w.gamma else 0))


def roofline_time(w, op, hbm_gbs, tflops):
    nbytes = algorithmic_bytes(w.M, w.N, w.K, gamma=w.gamma and op != "pre_rms",
                               beta=w.beta and op == "post_ln")
    return max(w.flops / (tflops * 1e12), nbytes / (hbm_gbs * 1e9)), nbytes


def call_op(nf, op, X, W, Y, G, B, eps, stream):
    """One fused call of the step (the public Python API)."""
    run_op(nf, op, X, W, Y, G, B, eps, stream)


def measure_step(nf, w, ops, X0, W0, G, B, dev, stream, steps, warmup, dist=None, sampler=None):
    """The timed region of the headline: exactly `steps` steps, each one call
    per op in `ops` on one buffer set (rotating sets > 3x L2), replayed from
    a CUDA graph of the `steps` steps on `stream` (programmatic dependent
    launch between the kernels stays on), CUDA events before and after.
    Returns (seconds (max over ranks), buffer sets, set bytes, step fn)."""
    import torch
    Ys = [torch.empty((X0.shape[0], w.N), dtype=torch.bfloat16, device=dev) for _ in ops]
    set_bytes = X0.numel() * 2 + sum(y.numel() * 2 for y in Ys)
    sets, nsets = make_sets([X0, *Ys], set_bytes, dev)

    def step(i):
        x, *ys = sets[i % nsets]
        for op, y in zip(ops, ys):
            call_op(nf, op, x, W0, y, G, B, w.eps, stream)

    sec = time_steps(step, steps, warmup, stream, dist, chunk=steps, sampler=sampler)
    return sec, nsets, set_bytes, step, sets


KERNEL_ROUNDS, KERNEL_LAUNCHES = 5, 30
KERNEL_TIMING = (f"median of {KERNEL_ROUNDS} rounds, the step's kernels interleaved, of {KERNEL_LAUNCHES} "
                 f"back-to-back launches from a CUDA graph each, rotating buffers, CUDA events")


def measure_kernel_alone(nf, w, op, X0, W0, G, B, dev, stream, launches=200, warmup=10):
    """Mean duration of one op's fused kernel timed alone: `launches`
    back-to-back calls from a CUDA graph over rotating buffer sets, CUDA
    events on the launching stream."""
    import torch
    Y0 = torch.empty((X0.shape[0], w.N), dtype=torch.bfloat16, device=dev)
    sets, nsets = make_sets([X0, Y0], X0.numel() * 2 + Y0.numel() * 2, dev)
    fn = lambda i: call_op(nf, op, sets[i % nsets][0], W0, sets[i % nsets][1], G, B, w.eps, stream)  # noqa: E731
    t = time_steps(fn, launches, warmup, stream) / launches
    del sets
    torch.cuda.empty_cache()
    return t


def e2e_measure(nf, w, ops, inp, dev, stream, steps):
    """Public API with host buffers: every step copies its X and W from pinned
    host memory to the device, runs the step's fused calls and copies their
    outputs back.  Steps are pipelined over three streams and two buffer sets
    (the copy of step i+1's inputs and of step i-1's outputs overlap step i's
    kernels; host-to-device and device-to-host copies use separate copy
    engines); every copy of every step is inside the timed region."""
    import torch
    Xh = torch.from_numpy(inp["X"].view(np.int16)).view(torch.bfloat16).pin_memory()
    Wh = torch.from_numpy(inp["W"].view(np.int16)).view(torch.bfloat16).pin_memory()
    M = Xh.shape[0]
    Yh = [[torch.empty((M, w.N), dtype=torch.bfloat16).pin_memory() for _ in ops] for _ in range(2)]
    Xd = [torch.empty_like(Xh, device=dev) for _ in range(2)]
    Wd = [torch.empty_like(Wh, device=dev) for _ in range(2)]
    Yd = [[torch.empty((M, w.N), dtype=torch.bfloat16, device=dev) for _ in ops] for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    read_done = [ev(), ev()]   # the kernels of the last step on buffer b have read Xd[b], Wd[b]
    out_done = [ev(), ev()]    # Yd[b] has been copied out
    for b in range(2):
        read_done[b].record(stream)
        out_done[b].record(s_out)

    def step(i):
        b = i & 1
        in_ready, y_ready = ev(), ev()
        with torch.cuda.stream(s_in):
            s_in.wait_event(read_done[b])
            Xd[b].copy_(Xh, non_blocking=True)
            Wd[b].copy_(Wh, non_blocking=True)
            in_ready.record(s_in)
        with torch.cuda.stream(stream):
            stream.wait_event(in_ready)
            stream.wait_event(out_done[b])
            for op, y in zip(ops, Yd[b]):
                call_op(nf, op, Xd[b], Wd[b], y, None, None, w.eps, stream)
            read_done[b].record(stream)
            y_ready.record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(y_ready)
            for yh, yd in zip(Yh[b], Yd[b]):
                yh.copy_(yd, non_blocking=True)
            out_done[b].record(s_out)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for i in range(steps):
        step(i)
    for b in range(2):
        s_out.wait_event(out_done[b])
    t1.record(s_out)
    torch.cuda.synchronize()
    sec = t0.elapsed_time(t1) / 1e3
    return sec, Xh.numel() * 2 + Wh.numel() * 2, sum(y.numel() * 2 for y in Yh[0])


# ---------------------------------------------------------------- CPU oracle
def oracle_rows(orc, inp, w, op, rows):
    if op == "post_ln":
        orc.gemm_postnorm_ln(inp["X"], inp["W"], w.eps, inp.get("gamma"), inp.get("beta"), rows=rows)
    elif op == "post_rms":
        orc.gemm_postnorm_rms(inp["X"], inp["W"], w.eps, inp.get("gamma"), rows=rows)
    else:
        orc.gemm_prenorm_rms(inp["X"], inp["W"], w.eps, rows=rows)


def oracle_sample(w, ops, inp, budget_s, rows_cap):
    """Time the fp64 oracle on whole-row samples of the step (every op on the
    same rows) for about budget_s seconds; returns (flops_done, seconds,
    rows_per_pass, threads)."""
    import oracle
    orc = oracle.get()
    M = inp["X"].shape[0]
    rows_per_pass = max(1, min(M, rows_cap))
    rows = np.arange(rows_per_pass, dtype=np.int64)
    done = 0
    t0 = time.perf_counter()
    while True:
        for op in ops:
            oracle_rows(orc, inp, w, op, rows)
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    sec = time.perf_counter() - t0
    return done * len(ops) * 2 * rows_per_pass * w.N * w.K, sec, rows_per_pass, orc.max_threads()


def workload_config(w, ops, world, rows_per_gpu):
    """The `config` keys that name the workload; both arms print them alike."""
    return {"workload": w.name, "ops": list(ops), "M": w.M, "K": w.K, "N": w.N, "eps": w.eps,
            "gamma": bool(w.gamma), "beta": bool(w.beta),
            "step": " + ".join(KERNEL_OF_OP[o] for o in ops) + " on one batch",
            "per_gpu_rows": rows_per_gpu,
            "parallelism": f"rows x{world} (shard of one seeded problem), no collective"}


def reference_arm(args):
    """--impl reference: the fp64 CPU oracle on the headline's step (every op
    of the workload on the same rows), timed as the reference arm."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    w = nf_inputs.WORKLOADS[args.workload]
    ops = tuple(args.op.split(",")) if args.op else w.ops
    orc = oracle.get()
    inp = nf_inputs.workload_inputs(w)
    # calibrate seconds per row of a step, then size each step so the run
    # stays near 60 s
    cal_rows = np.arange(min(w.M, 32), dtype=np.int64)
    t0 = time.perf_counter()
    for op in ops:
        oracle_rows(orc, inp, w, op, cal_rows)
    per_row = (time.perf_counter() - t0) / len(cal_rows)
    total = args.steps + args.warmup
    rows_per_step = int(max(1, min(w.M, 60.0 / max(1, total) / max(per_row, 1e-9))))
    rows = np.arange(rows_per_step, dtype=np.int64)
    for _ in range(args.warmup):
        for op in ops:
            oracle_rows(orc, inp, w, op, rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for op in ops:
            oracle_rows(orc, inp, w, op, rows)
    sec = time.perf_counter() - t0
    flops = args.steps * len(ops) * 2 * rows_per_step * w.N * w.K
    value = flops / sec / 1e12
    line = {
        "impl": "reference", "metric": "fused norm-GEMM TFLOP/s", "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, ops, args.gpus, w.M),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": orc.max_threads(), "kind": "oracle",
                         "sample": f"{rows_per_step} of {w.M} rows per step, every op of the step on them "
                                   f"(whole rows, fp64 oracle)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- configs
WL_SHORT = {"pre_rms_256x64x64": "C1", "post_ln_65536x128x128": "C2", "pre_rms_rowscale_32768x512x512": "C3",
            "post_affine_16384x1024x2048": "C4", "llm_8192x4096x4096": "C5"}


def _r(x, nd=3):
    """Round to nd significant digits (compact JSON)."""
    if x is None or x == 0 or not np.isfinite(x):
        return x
    return float(f"{x:.{nd}g}")


def _row(t_fused, t_plain, t_norm, frac):
    hid = None if t_norm is None else 100.0 * (t_plain + t_norm - t_fused) / t_norm
    return [_r(t_fused * 1e6), _r(t_plain * 1e6) if t_plain is not None else None,
            _r(t_norm * 1e6) if t_norm is not None else None, _r(frac, 2), _r(hid, 3)]


def config_table(nf, dev, stream, hbm_gbs, bf16_tf):
    """Every configuration's forward ops, the DSMEM cluster layouts of the
    wide post-norm rows, the backward and residual variants, and the
    FlashNormAttention forward: name -> [fused us, plain us, norm us,
    roofline fraction, % norm hidden]."""
    import torch
    rows = {}

    def roof(flops, nbytes, t):
        return max(flops / (bf16_tf * 1e12), nbytes / (hbm_gbs * 1e9)) / t

    for name in nf_inputs.WORKLOAD_ORDER:
        cw = nf_inputs.WORKLOADS[name]
        c = WL_SHORT[name]
        big = cw.flops > 5e10
        for cop in cw.ops:
            if big:  # interleaved bursts: fused, plain and norm see the same clock
                r = measure_workload(nf, cw, cop, dev, stream, KERNEL_LAUNCHES, 3, rounds=KERNEL_ROUNDS)
            else:
                r = measure_workload(nf, cw, cop, dev, stream, 1000, 10)
            tr, _ = roofline_time(cw, cop, hbm_gbs, bf16_tf)
            rows[f"{c} {cop}"] = _row(r["t_fused"], r["t_plain"], r["t_norm"], tr / r["t_fused"])
            if cop == "post_ln" and cw.N > 512:
                # the blog's §3 layout: a thread-block cluster of 256-column
                # CTAs spans the row, partials through DSMEM
                nf.set_postnorm_exchange(nf.XCH_CLUSTER)
                nf.set_postnorm_tile_n(256)
                try:
                    rc = (measure_workload(nf, cw, cop, dev, stream, KERNEL_LAUNCHES, 3, unfused=False,
                                           rounds=KERNEL_ROUNDS) if big else
                          measure_workload(nf, cw, cop, dev, stream, 1000, 10, unfused=False))
                finally:
                    nf.set_postnorm_exchange(0)
                    nf.set_postnorm_tile_n(0)
                rows[f"{c} {cop} cluster{cw.N // 256}x256"] = _row(rc["t_fused"], r["t_plain"], r["t_norm"],
                                                                    tr / rc["t_fused"])
            del r
            torch.cuda.empty_cache()
        if "pre_rms" in cw.ops:
            r = measure_prenorm_backward(nf, cw, dev, stream, 100 if big else 500, 10)
            nb = 6 * cw.M * cw.K + 4 * cw.M * cw.N + 4 * cw.K * cw.N + 8 * cw.M
            rows[f"{c} pre_rms_bwd"] = _row(r["t_fused"], r["t_plain"], r["t_norm"],
                                            roof(2 * cw.flops, nb, r["t_fused"]))
            del r
        for cop in cw.ops:
            if cop not in ("post_ln", "post_rms"):
                continue
            kind = 0 if cop == "post_ln" else 1
            r = measure_backward(nf, cw, kind, dev, stream, 200 if big else 1000, 10)
            rows[f"{c} {cop}_bwd"] = _row(r["t_fused"], r["t_plain"], r["t_norm"],
                                          roof(cw.flops, backward_bytes(cw, kind), r["t_fused"]))
            r = measure_residual(nf, cw, kind, dev, stream, 200 if big else 1000, 10)
            rows[f"{c} {cop}_res"] = _row(r["t_fused"], r["t_plain"], r["t_norm"],
                                          roof(cw.flops, residual_bytes(cw, kind), r["t_fused"]))
            del r
        torch.cuda.empty_cache()
    r = measure_flashnorm(nf, dev, stream, 50, 5)
    rows["FNA fwd"] = [_r(r["t_fused"] * 1e6), None, None,
                       _r(roof(r["flops"], r["bytes"], r["t_fused"]), 2), None, _r(r["t_torch"] * 1e6)]
    del r
    torch.cuda.empty_cache()
    return rows


# ---------------------------------------------------------------- main
def build_parser() -> argparse.ArgumentParser:
    """The command line (also used to check the commands quoted in profiles/)."""
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["nf", "reference"], default="nf")
    ap.add_argument("--workload", default=WORKLOAD, choices=list(nf_inputs.WORKLOAD_ORDER),
                    help="workload of the headline line (default: the LLM-shaped configuration)")
    ap.add_argument("--op", default=None,
                    help="comma-separated ops of a step: pre_rms, post_ln, post_rms (default: the workload's)")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload table")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end figure")
    ap.add_argument("--no-unfused", action="store_true", help="skip timing the unfused pairs")
    ap.add_argument("--no-soak", action="store_true", help="never add a clock-sampling soak")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--backward", choices=["post_ln", "post_rms", "pre_rms"], default=None,
                    help="time only this op's backward on the workload's shapes and print its figures "
                         "(a profiling aid; not the benchmark line)")
    ap.add_argument("--flashnorm", action="store_true",
                    help="time only the FlashNormAttention forward on its benchmark shapes and print its figures "
                         "(a profiling aid; not the benchmark line)")
    ap.add_argument("--fna-batch", type=int, default=None,
                    help="with --flashnorm: batch size in place of the benchmark's 768 (small profiling cases)")
    ap.add_argument("--residual", choices=["post_ln", "post_rms"], default=None,
                    help="time only this op with a residual add on the workload's shapes and print its "
                         "figures (a profiling aid; not the benchmark line)")
    ap.add_argument("--single", default=None, choices=["pre_rms", "post_ln", "post_rms", "plain", "norm"],
                    help="time only this kernel on the workload's shapes, back to back from CUDA graphs, and "
                         "print its figures (a profiling aid; not the benchmark line)")
    ap.add_argument("--exchange", default=None, choices=["cluster", "global"],
                    help="with --single: force the post-norm exchange (cluster: 256-column CTAs)")
    ap.add_argument("--gemm-pair", default="auto", choices=["auto", "never"],
                    help="never: no CTA pairs (nf_set_gemm_pair(1)); for profilers that cannot re-issue a "
                         "cooperative launch of clusters")
    return ap


def main(argv=None):
    ap = build_parser()
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    import torch.distributed as dist_mod
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    import normalization_gemm_gb300 as nf
    from normalization_gemm_gb300 import _build
    _build.build()
    nf.clear_device_status()
    if args.gemm_pair == "never":
        nf.set_gemm_pair(1)
    stream = torch.cuda.Stream(device=dev)
    hbm_gbs, bf16_tf, bf16_sus, peak_src = measured_peaks()
    w = nf_inputs.WORKLOADS[args.workload]
    if args.backward:
        if args.backward == "pre_rms":
            r = measure_prenorm_backward(nf, w, dev, stream, args.steps, args.warmup, unfused=not args.no_unfused)
        else:
            r = measure_backward(nf, w, 0 if args.backward == "post_ln" else 1, dev, stream, args.steps,
                                 args.warmup, unfused=not args.no_unfused)
        print(json.dumps({"backward": args.backward, "workload": w.name,
                          **{k: v * 1e6 for k, v in r.items() if k.startswith("t_")}}), flush=True)
        return 0
    if args.flashnorm:
        r = measure_flashnorm(nf, dev, stream, args.steps, args.warmup, unfused=not args.no_unfused,
                              batch=args.fna_batch)
        print(json.dumps({"flashnorm": nf_inputs.FNA_WORKLOAD["name"],
                          **{k: (v * 1e6 if k.startswith("t_") else v) for k, v in r.items()}}), flush=True)
        return 0
    if args.residual:
        r = measure_residual(nf, w, 0 if args.residual == "post_ln" else 1, dev, stream, args.steps,
                             args.warmup, unfused=not args.no_unfused)
        print(json.dumps({"residual": args.residual, "workload": w.name,
                          **{k: v * 1e6 for k, v in r.items() if k.startswith("t_")}}), flush=True)
        return 0
    if args.single:
        if args.exchange:
            nf.set_postnorm_exchange(nf.XCH_CLUSTER if args.exchange == "cluster" else nf.XCH_GLOBAL)
            if args.exchange == "cluster":
                nf.set_postnorm_tile_n(256)
        op = args.single
        kop = op if op in ("pre_rms", "post_ln", "post_rms") else (w.ops[-1] if op == "norm" else "plain")
        r = measure_workload(nf, w, kop, dev, stream, args.steps, args.warmup, unfused=op in ("plain", "norm"))
        key = {"plain": "t_plain", "norm": "t_norm"}.get(op, "t_fused")
        print(json.dumps({"single": op, "workload": w.name, "us": r[key] * 1e6}), flush=True)
        return 0

    ops = tuple(args.op.split(",")) if args.op else w.ops
    for op in ops:
        if op not in ("pre_rms", "post_ln", "post_rms"):
            ap.error(f"--op: unknown op {op}")
    # rows shard_rows(world * M, world, rank) of one seeded global problem
    inp = nf_inputs.workload_shard(w, world, rank)
    lo, hi = inp["rows"]
    rows_here = hi - lo
    X0, W0 = _to_dev(inp["X"], dev), _to_dev(inp["W"], dev)
    G = _to_dev(inp["gamma"], dev) if w.gamma else None
    B = _to_dev(inp["beta"], dev) if w.beta else None
    flops_step = len(ops) * 2 * rows_here * w.N * w.K
    sampler = ClockSampler(local_rank)
    sec, nsets, set_bytes, step_fn, sets = measure_step(nf, w, ops, X0, W0, G, B, dev, stream, args.steps,
                                                        args.warmup, dist=dist, sampler=sampler)
    t_step = sec / args.steps
    value = world * flops_step / t_step / 1e12
    clocks = sampler.summary("timed")
    if clocks["samples"] < 3 and not args.no_soak:
        # The timed region was shorter than three sampling periods: replay the
        # same steps for ~1.5 s right after it and sample that instead.
        soak = ClockSampler(local_rank)
        reps = max(args.steps, int(1.5 / max(t_step, 1e-7)))
        time_steps(step_fn, reps, 3, stream, None, chunk=min(reps, 200), sampler=soak)
        clocks = soak.summary("soak right after the timed region (the timed region was shorter than "
                              "three 50 ms sampling periods)")
    del sets
    torch.cuda.empty_cache()

    # each kernel of the step timed alone; the dominant one against its roofline
    # Short bursts, the step's kernels interleaved over five rounds (median):
    # a long loop of one kernel on a power-capped part runs at a lower clock
    # than the burst peak it is compared with, and whichever kernel went
    # second would pay for the first one's heat.
    rounds = {op: [] for op in ops}
    for _ in range(KERNEL_ROUNDS):
        for op in ops:
            rounds[op].append(measure_kernel_alone(nf, w, op, X0, W0, G, B, dev, stream,
                                                   launches=KERNEL_LAUNCHES, warmup=3))
    per_op = {op: statistics.median(v) for op, v in rounds.items()}
    dom = max(ops, key=lambda o: per_op[o])
    kflops = 2 * rows_here * w.N * w.K
    kbytes = algorithmic_bytes(rows_here, w.N, w.K, gamma=w.gamma and dom != "pre_rms",
                               beta=w.beta and dom == "post_ln")
    t_dom = per_op[dom]
    plan = nf.plan_gemm(OPCODE[dom], rows_here, w.N, w.K, torch.cuda.get_device_properties(dev).multi_processor_count)
    dom_pair = plan["cluster"] == 2 and (dom in ("plain", "pre_rms") or plan["exchange"] == 2)
    traffic = profiled_traffic(w.name, dom, dom_pair)
    if kflops / (bf16_tf * 1e12) > kbytes / (hbm_gbs * 1e9):
        achieved = kflops / t_dom / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": bf16_tf, "unit": "TFLOP/s",
                "frac": achieved / bf16_tf, "traffic": traffic, "cta_pair": dom_pair,
                "kernel": KERNEL_OF_OP[dom], "peak_source": f"{peak_src} bf16_tflops (burst: the kernel "
                                                            f"timed alone; of measured)",
                "algorithmic_flops_per_launch": kflops, "mean_launch_us": t_dom * 1e6,
                "timing": KERNEL_TIMING}
    else:
        achieved = kbytes / t_dom / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved / hbm_gbs, "traffic": traffic, "cta_pair": dom_pair,
                "kernel": KERNEL_OF_OP[dom], "peak_source": f"{peak_src} hbm_gbs (of measured)",
                "algorithmic_bytes_per_launch": kbytes, "mean_launch_us": t_dom * 1e6,
                "timing": KERNEL_TIMING}
    status, detail = nf.device_status()

    line = {
        "metric": "fused norm-GEMM TFLOP/s", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {**workload_config(w, ops, world, rows_here),
                   "l2": f"rotating {nsets} buffer sets of {set_bytes / 2**20:.0f} MiB (> 3x L2 between reuses)",
                   "launch": f"one CUDA graph of the {args.steps} steps",
                   **({"gemm_pair": "never"} if args.gemm_pair == "never" else {})},
        "gpu_launches": args.steps * len(ops),
        "roofline": roof,
        "kernel_us": {KERNEL_OF_OP[o]: per_op[o] * 1e6 for o in ops},
        "clocks": clocks,
        "device_status": int(status),
    }
    if status != 0:
        line["device_status_detail"] = detail

    if rank == 0:
        if not args.no_unfused:
            tf = tp = tn = 0.0
            unf = {}
            for op in ops:
                m = measure_workload(nf, w, op, dev, stream, KERNEL_LAUNCHES, 3, rounds=KERNEL_ROUNDS)
                tf, tp, tn = tf + m["t_fused"], tp + m["t_plain"], tn + m["t_norm"]
                unf[op] = {"fused_us": m["t_fused"] * 1e6, "plain_us": m["t_plain"] * 1e6,
                           "norm_us": m["t_norm"] * 1e6}
                del m
                torch.cuda.empty_cache()
            line["norm_hidden_pct"] = 100.0 * (tp + tn - tf) / tn
            line["unfused"] = unf
        if not args.no_e2e:
            e2e_steps = max(1, min(args.e2e_steps, args.steps))
            full = inp if world == 1 else nf_inputs.workload_inputs(w)
            sec_e, hb, db = e2e_measure(nf, w, ops, full, dev, stream, e2e_steps)
            line["e2e"] = {"value": world * flops_step * e2e_steps / sec_e / 1e12, "unit": "TFLOP/s",
                           "h2d_bytes_per_step": hb, "d2h_bytes_per_step": db, "steps": e2e_steps}
        if not args.no_cpu and world == 1:
            cap = max(1, int(2e10 // (len(ops) * 2 * w.N * w.K)))   # about 20 GFLOP per pass
            flops, sec_c, rpp, thr = oracle_sample(w, ops, inp, budget_s=10.0, rows_cap=cap)
            line["cpu_baseline"] = {"value": flops / sec_c / 1e12, "unit": "TFLOP/s", "cores": thr,
                                    "kind": "oracle",
                                    "sample": f"rows 0..{rpp - 1} of {w.M} x {w.K} x {w.N}, every op of the "
                                              f"step, repeated for {sec_c:.1f} s (fp64, OpenMP over rows)"}
        if not args.no_configs:
            line["configs_legend"] = {"C1": "pre_rms_256x64x64", "C2": "post_ln_65536x128x128",
                                      "C3": "pre_rms_rowscale_32768x512x512",
                                      "C4": "post_affine_16384x1024x2048", "C5": "llm_8192x4096x4096",
                                      "row": ["fused_us", "plain_us", "norm_us", "roofline_frac",
                                              "norm_hidden_pct"],
                                      "FNA fwd": "FlashNormAttention forward, batch 768, Lq <= 1024, 4 heads: "
                                                 "[fused_us, -, -, roofline_frac, -, torch_eager_us]"}
            line["configs"] = config_table(nf, dev, stream, hbm_gbs, bf16_tf)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
