"""Python handle on the fp64 CPU oracle (``oracle/nfo.c``).

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package.  The CUDA
product path never imports it.

The oracle computes the plain definitions of the fused operations (blog
"Towards Free Normalization: Fusing Normalization into GEMM and Attention
Kernels", §2 Lazy Pre-Norm and §3 Multi-CTA Norm) in double precision on
bf16 inputs widened exactly.  Arrays cross the boundary as numpy arrays:
bf16 tensors as ``uint16`` bit patterns, results as ``float64``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nfo.c")
_HDR = os.path.join(_HERE, "nfo.h")
LIB_PATH = os.path.join(_HERE, "libnfo.so")

NORM_LN = 0
ACT_IDENTITY, ACT_GELU_TANH, ACT_SILU = 0, 1, 2
NORM_RMS = 1

# -ffp-contract=off keeps every multiply and add separately rounded, so the
# oracle gives the same bits on x86-64 and on aarch64 (where GCC would
# otherwise fuse into FMAs).
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off"]


def build(src: str = _SRC, out: str = LIB_PATH, force: bool = False) -> str:
    """Compile the oracle with gcc into a shared library; return its path."""
    newest = max(os.path.getmtime(src), os.path.getmtime(_HDR))
    if not force and os.path.exists(out) and os.path.getmtime(out) >= newest:
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", *CFLAGS, "-I", _HERE, src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


_P_U16 = ctypes.POINTER(ctypes.c_uint16)
_P_F64 = ctypes.POINTER(ctypes.c_double)
_P_I64 = ctypes.POINTER(ctypes.c_int64)
_I64 = ctypes.c_int64


def _u16(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.dtype == np.uint16 and a.flags.c_contiguous
    return a.ctypes.data_as(_P_U16)


def _f64(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(_P_F64)


class Oracle:
    """ctypes wrapper over one build of the oracle library."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        lib.nfo_gemm_plain.argtypes = [_P_U16, _P_U16, _I64, _I64, _I64, _P_I64, _I64, _P_F64]
        lib.nfo_gemm_prenorm_rms.argtypes = [_P_U16, _P_U16, _I64, _I64, _I64, ctypes.c_double,
                                             _P_I64, _I64, _P_F64, _P_F64]
        lib.nfo_gemm_postnorm_ln.argtypes = [_P_U16, _P_U16, _P_U16, _P_U16, _I64, _I64, _I64,
                                             ctypes.c_double, _P_I64, _I64, _P_F64, _P_F64, _P_F64]
        lib.nfo_gemm_postnorm_rms.argtypes = [_P_U16, _P_U16, _P_U16, _I64, _I64, _I64,
                                              ctypes.c_double, _P_I64, _I64, _P_F64, _P_F64]
        lib.nfo_gemm_postnorm_res.argtypes = [_P_U16, _P_U16, _P_U16, _P_U16, _P_U16, _I64, _I64, _I64,
                                              ctypes.c_int, ctypes.c_double, _P_I64, _I64, _P_F64, _P_F64,
                                              _P_F64, _P_F64]
        lib.nfo_flashnorm_attn_fwd.argtypes = [_P_U16, _P_U16, _P_U16, ctypes.POINTER(ctypes.c_int32), _I64, _I64,
                                               _I64, _I64, _I64, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                               _P_F64]
        lib.nfo_norm_rows.argtypes = [_P_U16, _P_U16, _P_U16, _I64, _I64, ctypes.c_int,
                                      ctypes.c_double, _P_I64, _I64, _P_F64, _P_F64, _P_F64]
        lib.nfo_gemm_postnorm_bwd.argtypes = [_P_U16, _P_U16, _P_U16, _P_U16, _P_F64, _P_F64, _I64,
                                              _I64, _I64, ctypes.c_int, _P_I64, _I64, _P_F64]
        lib.nfo_norm_rows_bwd.argtypes = [_P_U16, _P_U16, _P_U16, _P_F64, _P_F64, _I64, _I64,
                                          ctypes.c_int, _P_I64, _I64, _P_F64]
        lib.nfo_prenorm_rms_bwd_da.argtypes = [_P_U16, _P_U16, _P_F64, _P_U16, _I64, _I64, _I64,
                                               _P_I64, _I64, _P_F64]
        lib.nfo_prenorm_rms_bwd_db.argtypes = [_P_U16, _P_F64, _P_U16, _I64, _I64, _I64, _P_I64, _I64,
                                               _P_F64]
        for f in ("nfo_gemm_plain", "nfo_gemm_prenorm_rms", "nfo_gemm_postnorm_ln",
                  "nfo_gemm_postnorm_rms", "nfo_norm_rows", "nfo_gemm_postnorm_bwd",
                  "nfo_norm_rows_bwd", "nfo_prenorm_rms_bwd_da", "nfo_prenorm_rms_bwd_db",
                  "nfo_gemm_postnorm_res", "nfo_flashnorm_attn_fwd",
                  "nfo_max_threads"):
            getattr(lib, f).restype = ctypes.c_int
        lib.nfo_set_threads.argtypes = [ctypes.c_int]
        lib.nfo_set_threads.restype = None
        self.lib = lib

    # -- helpers -----------------------------------------------------------
    @staticmethod
    def _rows(rows, M):
        if rows is None:
            return None, M, None
        r = np.ascontiguousarray(rows, dtype=np.int64)
        return r, len(r), r.ctypes.data_as(_P_I64)

    @staticmethod
    def _check(rc, name):
        if rc != 0:
            raise ValueError(f"{name}: invalid argument (rc={rc})")

    def max_threads(self) -> int:
        return int(self.lib.nfo_max_threads())

    def set_threads(self, n: int) -> None:
        self.lib.nfo_set_threads(int(n))

    # -- operations --------------------------------------------------------
    def gemm_plain(self, X, W, rows=None):
        M, K = X.shape
        N = W.shape[1]
        r, R, rp = self._rows(rows, M)
        Y = np.empty((R, N), np.float64)
        self._check(self.lib.nfo_gemm_plain(_u16(X), _u16(W), M, N, K, rp, R, _f64(Y)),
                    "gemm_plain")
        return Y

    def gemm_prenorm_rms(self, X, W, eps, rows=None):
        M, K = X.shape
        N = W.shape[1]
        r, R, rp = self._rows(rows, M)
        Y = np.empty((R, N), np.float64)
        rstd = np.empty(R, np.float64)
        self._check(self.lib.nfo_gemm_prenorm_rms(_u16(X), _u16(W), M, N, K, eps, rp, R,
                                                  _f64(Y), _f64(rstd)), "gemm_prenorm_rms")
        return Y, rstd

    def gemm_postnorm_ln(self, X, W, eps, gamma=None, beta=None, rows=None):
        M, K = X.shape
        N = W.shape[1]
        r, R, rp = self._rows(rows, M)
        Y = np.empty((R, N), np.float64)
        mean = np.empty(R, np.float64)
        rstd = np.empty(R, np.float64)
        self._check(self.lib.nfo_gemm_postnorm_ln(_u16(X), _u16(W), _u16(gamma), _u16(beta),
                                                  M, N, K, eps, rp, R, _f64(Y), _f64(mean),
                                                  _f64(rstd)), "gemm_postnorm_ln")
        return Y, mean, rstd

    def gemm_postnorm_rms(self, X, W, eps, gamma=None, rows=None):
        M, K = X.shape
        N = W.shape[1]
        r, R, rp = self._rows(rows, M)
        Y = np.empty((R, N), np.float64)
        rstd = np.empty(R, np.float64)
        self._check(self.lib.nfo_gemm_postnorm_rms(_u16(X), _u16(W), _u16(gamma), M, N, K, eps,
                                                   rp, R, _f64(Y), _f64(rstd)),
                    "gemm_postnorm_rms")
        return Y, rstd

    def gemm_postnorm_res(self, X, W, Rs, kind, eps, gamma=None, beta=None, rows=None):
        """H = X @ W + Rs; Y = norm(H) (LN: kind 0, RMS: kind 1).  Returns
        (Y, H, mean or None, rstd)."""
        M, K = X.shape
        N = W.shape[1]
        assert Rs.shape == (M, N)
        r, R, rp = self._rows(rows, M)
        Y = np.empty((R, N), np.float64)
        H = np.empty((R, N), np.float64)
        mean = np.full(R, np.nan, np.float64)
        rstd = np.empty(R, np.float64)
        self._check(self.lib.nfo_gemm_postnorm_res(_u16(X), _u16(W), _u16(Rs), _u16(gamma), _u16(beta), M, N,
                                                   K, int(kind), eps, rp, R, _f64(Y), _f64(H), _f64(mean),
                                                   _f64(rstd)), "gemm_postnorm_res")
        return Y, H, (mean if kind == NORM_LN else None), rstd

    def flashnorm_attn_fwd(self, Q, K, V, act, eps1, eps2, q_len=None):
        """FlashNormAttention forward.  Q: [B, Lq, H, D], K / V: [B, Lkv, H, D]
        (bf16 bit patterns); q_len: B ints or None.  Returns Out [B, Lq, H, D]
        fp64 with rows t >= q_len[b] left NaN."""
        Bn, Lq, H, D = Q.shape
        Lkv = K.shape[1]
        assert K.shape == (Bn, Lkv, H, D) and V.shape == K.shape
        out = np.full((Bn, Lq, H, D), np.nan, np.float64)
        ql = None
        if q_len is not None:
            ql = np.ascontiguousarray(q_len, dtype=np.int32)
            assert ql.shape == (Bn,)
        self._check(self.lib.nfo_flashnorm_attn_fwd(
            _u16(Q), _u16(K), _u16(V), None if ql is None else ql.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
            Bn, Lq, Lkv, H, D, int(act), float(eps1), float(eps2), _f64(out)), "flashnorm_attn_fwd")
        return out

    def norm_rows(self, A, kind, eps, gamma=None, beta=None, rows=None):
        Rr, C = A.shape
        r, R, rp = self._rows(rows, Rr)
        out = np.empty((R, C), np.float64)
        mean = np.full(R, np.nan, np.float64)
        rstd = np.empty(R, np.float64)
        self._check(self.lib.nfo_norm_rows(_u16(A), _u16(gamma), _u16(beta), Rr, C, int(kind),
                                           eps, rp, R, _f64(out), _f64(mean), _f64(rstd)),
                    "norm_rows")
        return out, (mean if kind == NORM_LN else None), rstd

    @staticmethod
    def _stats(a, M):
        if a is None:
            return None, None
        v = np.ascontiguousarray(a, dtype=np.float64)
        assert v.shape == (M,)
        return v, v.ctypes.data_as(_P_F64)

    def gemm_postnorm_bwd(self, A, B, Z, kind, mean, rstd, gamma=None, rows=None):
        """dZ = norm_bwd(A @ B; Z, mean, rstd, gamma) (mean: None for RMS)."""
        M, K = A.shape
        N = B.shape[1]
        assert Z.shape == (M, N)
        r, R, rp = self._rows(rows, M)
        m, mp = self._stats(mean, M)
        s, sp = self._stats(rstd, M)
        dZ = np.empty((R, N), np.float64)
        self._check(self.lib.nfo_gemm_postnorm_bwd(_u16(A), _u16(B), _u16(Z), _u16(gamma), mp, sp,
                                                   M, N, K, int(kind), rp, R, _f64(dZ)),
                    "gemm_postnorm_bwd")
        return dZ

    def norm_rows_bwd(self, dY, Z, kind, mean, rstd, gamma=None, rows=None):
        """dZ = norm_bwd(dY; Z, mean, rstd, gamma) row by row (mean: None for RMS)."""
        Rr, C = dY.shape
        assert Z.shape == (Rr, C)
        r, R, rp = self._rows(rows, Rr)
        m, mp = self._stats(mean, Rr)
        s, sp = self._stats(rstd, Rr)
        dZ = np.empty((R, C), np.float64)
        self._check(self.lib.nfo_norm_rows_bwd(_u16(dY), _u16(Z), _u16(gamma), mp, sp, Rr, C,
                                               int(kind), rp, R, _f64(dZ)), "norm_rows_bwd")
        return dZ

    def prenorm_rms_bwd_da(self, A, B, rstd, dC, rows=None):
        """dA of C = rmsnorm(A) @ B from dC and the saved rstd (rows of dA)."""
        M, K = A.shape
        N = B.shape[1]
        assert dC.shape == (M, N)
        r, R, rp = self._rows(rows, M)
        s, sp = self._stats(rstd, M)
        dA = np.empty((R, K), np.float64)
        self._check(self.lib.nfo_prenorm_rms_bwd_da(_u16(A), _u16(B), sp, _u16(dC), M, N, K, rp, R,
                                                    _f64(dA)), "prenorm_rms_bwd_da")
        return dA

    def prenorm_rms_bwd_db(self, A, rstd, dC, krows=None):
        """dB of C = rmsnorm(A) @ B from dC and the saved rstd (rows of dB, over K)."""
        M, K = A.shape
        N = dC.shape[1]
        r, R, rp = self._rows(krows, K)
        s, sp = self._stats(rstd, M)
        dB = np.empty((R, N), np.float64)
        self._check(self.lib.nfo_prenorm_rms_bwd_db(_u16(A), sp, _u16(dC), M, N, K, rp, R, _f64(dB)),
                    "prenorm_rms_bwd_db")
        return dB


_DEFAULT: Optional[Oracle] = None


def get() -> Oracle:
    """The oracle built from ``oracle/nfo.c`` (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle(build())
    return _DEFAULT
