"""Builds libnf.so (the CUDA kernels and the C ABI) in-tree with nvcc.

Each .cu translation unit compiles in parallel to an object file under
``_build/``; the objects link into ``libnf.so`` next to this file.  A stamp of
the sources, headers and flags skips the work when nothing changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libnf.so")

SOURCES = ["nf_api.cu", "nf_norm.cu", "nf_gemm_plain.cu", "nf_gemm_pre.cu",
           "nf_gemm_post_ln.cu", "nf_gemm_post_rms.cu", "nf_gemm_bwd_ln.cu", "nf_gemm_bwd_rms.cu",
           "nf_gemm_trans_plain.cu", "nf_gemm_trans_bwd.cu", "nf_splitk.cu",
           "nf_gemm_res_ln.cu", "nf_gemm_res_rms.cu", "nf_flashnorm.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-ffp-contract=off", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return exe


def _stamp(extra_flags, names=None) -> str:
    h = hashlib.sha256()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            if name.endswith((".cu", ".cuh", ".h")) and (names is None or name in names):
                with open(os.path.join(d, name), "rb") as fh:
                    h.update(name.encode() + fh.read())
    # flags without the machine-specific include paths
    flags = [f for f in NVCC_FLAGS + list(extra_flags) if not os.path.isabs(f)]
    h.update(" ".join(flags).encode())
    return h.hexdigest()


def source_hash(names=None) -> str:
    """Short hash of the CUDA sources, headers and flags (path independent);
    with `names`, of those files only (the sources one kernel is built from)."""
    return _stamp((), names)[:16]


# The files the fused GEMM kernels and their launch plans are built from: a
# profile of one of them stays valid while these are unchanged.
GEMM_SOURCES = ("nf_api.cu", "nf_gemm_post_ln.cu", "nf_gemm_post_rms.cu", "nf_gemm_pre.cu", "nf_gemm_plain.cu",
                "nf_gemm_kernel.cuh", "nf_gemm_wide.cuh", "nf_internal.h", "nf_ptx.cuh", "nf.h")
# ... and of the backward, residual and transposed-operand GEMMs (their
# profiles), the row-norm kernels, and the FlashNormAttention kernel.
GEMM_EXTRA_SOURCES = GEMM_SOURCES + ("nf_gemm_bwd_ln.cu", "nf_gemm_bwd_rms.cu", "nf_gemm_res_ln.cu",
                                     "nf_gemm_res_rms.cu", "nf_gemm_trans_plain.cu", "nf_gemm_trans_bwd.cu",
                                     "nf_splitk.cu")
NORM_SOURCES = ("nf_api.cu", "nf_norm.cu", "nf_internal.h", "nf_ptx.cuh", "nf.h")
FNA_SOURCES = ("nf_api.cu", "nf_flashnorm.cu", "nf_internal.h", "nf_ptx.cuh", "nf.h")


def build(force: bool = False, extra_flags=(), verbose: bool = False) -> str:
    """Compile and link libnf.so; return its path."""
    stamp = _stamp(extra_flags)
    stamp_file = LIB + ".stamp"
    if (not force and os.path.exists(LIB) and os.path.exists(stamp_file)
            and open(stamp_file).read() == stamp):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [exe, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{p.stderr}")
        return obj, p.stderr

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for obj, err in results:
            if err.strip():
                print(f"--- {os.path.basename(obj)}\n{err}")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [exe, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stderr}")
    os.replace(tmp, LIB)
    with open(stamp_file, "w") as fh:
        fh.write(stamp)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else ()))
