"""Python binding of libnf.so, the normalization-fused bf16 GEMM for GB300.

Argument marshalling only: every step of every operation runs in the CUDA
kernels behind the C ABI of ``include/nf.h``.  Tensors are PyTorch CUDA
tensors (device memory and streams); nothing here computes on them.  There is
no fallback: if the library is missing or the device is not sm_103 the calls
raise.

Operations (blog "Towards Free Normalization: Fusing Normalization into GEMM
and Attention Kernels"):
  gemm_plain          Y = X @ W                                  (§1 baseline)
  gemm_prenorm_rms    Y = RMSNorm(X) @ W, Lazy Pre-Norm          (§2)
  gemm_postnorm_ln    Y = LayerNorm(X @ W) * gamma + beta        (§3)
  gemm_postnorm_rms   Y = RMSNorm(X @ W) * gamma                 (§3)
  norm_rows           standalone LayerNorm / RMSNorm of rows     (§1 baseline)
  gemm_postnorm_ln_bwd / gemm_postnorm_rms_bwd
                      dZ = norm backward of (A @ B) from saved   (§3 backward,
                      row statistics, fused in the GEMM epilogue   fusion regrouping)
  norm_rows_bwd       their backward from saved row statistics   (§3 backward baseline)
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "libnf.so")
HEADER = os.path.join(ROOT, "include", "nf.h")

NF_OK = 0
NORM_LN = 0
NORM_RMS = 1
POSTNORM_MAX_N = 4096
XCH_CLUSTER = 1
XCH_GLOBAL = 2

STATUS_NAMES = {0: "NF_OK", 1: "NF_ERR_INVALID_ARG", 2: "NF_ERR_ALIGNMENT",
                3: "NF_ERR_UNSUPPORTED_SHAPE", 4: "NF_ERR_CUDA", 5: "NF_ERR_TIMEOUT",
                6: "NF_ERR_NO_DEVICE"}


class NFError(RuntimeError):
    """A non-zero nf_status from the library."""

    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}"
                         + (f" ({detail})" if detail else ""))


class NFPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "tile_m", "tile_n", "tile_k", "stages", "cluster", "grid", "threads", "smem_bytes",
        "tmem_cols", "tiles", "exchange", "splitk", "split_tiles")]


_lib: Optional[ctypes.CDLL] = None

_VP = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SIGS = {
    "nf_gemm_plain": [_VP, _VP, _VP, _I64, _I64, _I64, _VP],
    "nf_gemm_prenorm_rms": [_VP, _VP, _VP, _I64, _I64, _I64, _F, _VP, _VP],
    "nf_gemm_postnorm_ln": [_VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _F, _VP, _VP, _VP],
    "nf_gemm_postnorm_ln_noalloc": [_VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _F, _VP, _VP, _VP],
    "nf_gemm_postnorm_rms": [_VP, _VP, _VP, _VP, _I64, _I64, _I64, _F, _VP, _VP],
    "nf_gemm_postnorm_ln_res": [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _F, _VP, _VP, _VP],
    "nf_gemm_postnorm_rms_res": [_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _F, _VP, _VP],
    "nf_flashnorm_attn_fwd": [_VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _I64, _I64, ctypes.c_int, _F, _F, _VP],
    "nf_norm_rows_res": [_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, ctypes.c_int, _F, _VP, _VP, _VP],
    "nf_norm_rows": [_VP, _VP, _VP, _VP, _I64, _I64, ctypes.c_int, _F, _VP, _VP, _VP],
    "nf_norm_rows_bwd": [_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, ctypes.c_int, _VP],
    "nf_gemm_plain_t": [_VP, _VP, _VP, _I64, _I64, _I64, ctypes.c_int, _VP],
    "nf_gemm_prenorm_rms_bwd": [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _VP],
    "nf_gemm_postnorm_ln_bwd": [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _VP],
    "nf_gemm_postnorm_rms_bwd": [_VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _VP],
    "nf_get_device_status": [_VP],
    "nf_clear_device_status": [],
    "nf_set_wait_timeout_ns": [ctypes.c_uint64],
    "nf_set_launch_overlap": [ctypes.c_int],
    "nf_set_postnorm_tile_n": [ctypes.c_int],
    "nf_set_gemm_tile_n": [ctypes.c_int],
    "nf_set_gemm_pair": [ctypes.c_int],
    "nf_set_postnorm_exchange": [ctypes.c_int],
    "nf_set_prenorm_split": [ctypes.c_int],
    "nf_set_gemm_splitk": [ctypes.c_int],
    "nf_reserve_scratch": [_I64, _I64, _VP],
    "nf_selftest_wait_timeout": [ctypes.c_uint64, _VP],
    "nf_plan_gemm": [ctypes.c_int, _I64, _I64, _I64, ctypes.c_int, ctypes.POINTER(NFPlan)],
    "nf_abi_version": [],
}


def header_symbols() -> list:
    """Names of the functions include/nf.h declares."""
    with open(HEADER) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nf_[a-z_0-9]+)\s*\(", text)))


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, argtypes in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = argtypes
            f.restype = ctypes.c_int
        L.nf_status_string.argtypes = [ctypes.c_int]
        L.nf_status_string.restype = ctypes.c_char_p
        L.nf_last_error.argtypes = []
        L.nf_last_error.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _check(status: int, where: str) -> None:
    if status != NF_OK:
        raise NFError(status, where, lib().nf_last_error().decode(errors="replace"))


# ------------------------------------------------------------- tensor helpers
def _torch():
    import torch
    return torch


def _mat(t, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D tensor")
    return t.data_ptr()


def _vec(t, name, n, dtype):
    if t is None:
        return None
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != dtype:
        raise TypeError(f"{name} must be a CUDA {dtype} tensor")
    if t.dim() != 1 or t.numel() != n or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous vector of {n}")
    return t.data_ptr()


def _stream(stream):
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _out(out, M, N, like):
    torch = _torch()
    if out is None:
        return torch.empty((M, N), dtype=torch.bfloat16, device=like.device)
    if tuple(out.shape) != (M, N):
        raise ValueError(f"out must have shape {(M, N)}")
    return out


def _shapes(x, w):
    M, K = x.shape
    K2, N = w.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: X is {tuple(x.shape)}, W is {tuple(w.shape)}")
    return M, N, K


# ------------------------------------------------------------- operations
def gemm_plain(x, w, out=None, stream=None):
    """Y = X @ W (bf16 in and out, fp32 accumulation)."""
    M, N, K = _shapes(x, w)
    y = _out(out, M, N, x)
    _check(lib().nf_gemm_plain(_mat(x, "x"), _mat(w, "w"), _mat(y, "out"), M, N, K,
                               _stream(stream)), "nf_gemm_plain")
    return y


TRANS_X = 1
TRANS_W = 4


def gemm_plain_t(x, w, flags, out=None, stream=None):
    """Y = op(x) op(w): TRANS_X -- x holds X^T (K x M); TRANS_W -- w holds W^T (N x K)."""
    if flags & TRANS_X:
        K, M = x.shape
    else:
        M, K = x.shape
    if flags & TRANS_W:
        N, K2 = w.shape
    else:
        K2, N = w.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: {tuple(x.shape)} and {tuple(w.shape)} with flags {flags}")
    y = _out(out, M, N, x)
    _check(lib().nf_gemm_plain_t(_mat(x, "x"), _mat(w, "w"), _mat(y, "out"), M, N, K, int(flags), _stream(stream)),
           "nf_gemm_plain_t")
    return y


def gemm_prenorm_rms_bwd(a, b, rstd, dc, da=None, db=None, want_da=True, want_db=True, xhat=None,
                         use_xhat=True, stream=None):
    """Backward of C = rmsnorm(a) @ b from the saved rstd (fp32 [M]): returns (dA, dB).

    With both gradients wanted and ``use_xhat`` (default), the dA kernel also
    writes rmsnorm(a) (bf16 [M, K], into ``xhat`` if given, else a temporary)
    and dB is a plain GEMM over it; ``use_xhat=False`` rebuilds it in shared
    memory inside the dB GEMM instead (no extra memory)."""
    torch = _torch()
    M, N, K = _shapes(a, b)
    if tuple(dc.shape) != (M, N):
        raise ValueError(f"dc must have shape {(M, N)}")
    da = (_out(da, M, K, a) if want_da else None)
    db = (_out(db, K, N, a) if want_db else None)
    if want_da and want_db and use_xhat:
        xhat = _out(xhat, M, K, a)
    else:
        xhat = None
    _check(lib().nf_gemm_prenorm_rms_bwd(_mat(a, "a"), _mat(b, "b"), _vec(rstd, "rstd", M, torch.float32),
                                         _mat(dc, "dc"), None if da is None else _mat(da, "da"),
                                         None if db is None else _mat(db, "db"),
                                         None if xhat is None else _mat(xhat, "xhat"), M, N, K,
                                         _stream(stream)),
           "nf_gemm_prenorm_rms_bwd")
    return da, db


def gemm_prenorm_rms(x, w, eps, out=None, rstd_out=None, stream=None):
    """Y = RMSNorm(X) @ W, no affine (Lazy Pre-Norm).  rstd_out: optional fp32 [M]."""
    torch = _torch()
    M, N, K = _shapes(x, w)
    y = _out(out, M, N, x)
    _check(lib().nf_gemm_prenorm_rms(_mat(x, "x"), _mat(w, "w"), _mat(y, "out"), M, N, K,
                                     float(eps), _vec(rstd_out, "rstd_out", M, torch.float32),
                                     _stream(stream)), "nf_gemm_prenorm_rms")
    return y


def gemm_postnorm_ln(x, w, eps, gamma=None, beta=None, out=None, mean_out=None, rstd_out=None,
                     stream=None):
    """Y = LayerNorm(X @ W) over N, optional gamma / beta (bf16 [N])."""
    torch = _torch()
    M, N, K = _shapes(x, w)
    y = _out(out, M, N, x)
    _check(lib().nf_gemm_postnorm_ln(_mat(x, "x"), _mat(w, "w"),
                                     _vec(gamma, "gamma", N, torch.bfloat16),
                                     _vec(beta, "beta", N, torch.bfloat16), _mat(y, "out"),
                                     M, N, K, float(eps),
                                     _vec(mean_out, "mean_out", M, torch.float32),
                                     _vec(rstd_out, "rstd_out", M, torch.float32),
                                     _stream(stream)), "nf_gemm_postnorm_ln")
    return y


def gemm_postnorm_ln_noalloc(x, w, eps, gamma=None, beta=None, out=None, mean_out=None, rstd_out=None,
                             stream=None):
    """gemm_postnorm_ln whose L2 exchange uses the library's fixed per-device
    scratch array (no allocation; calls that may overlap must be serialized)."""
    torch = _torch()
    M, N, K = _shapes(x, w)
    y = _out(out, M, N, x)
    _check(lib().nf_gemm_postnorm_ln_noalloc(_mat(x, "x"), _mat(w, "w"),
                                             _vec(gamma, "gamma", N, torch.bfloat16),
                                             _vec(beta, "beta", N, torch.bfloat16), _mat(y, "out"),
                                             M, N, K, float(eps),
                                             _vec(mean_out, "mean_out", M, torch.float32),
                                             _vec(rstd_out, "rstd_out", M, torch.float32),
                                             _stream(stream)), "nf_gemm_postnorm_ln_noalloc")
    return y


def gemm_postnorm_rms(x, w, eps, gamma=None, out=None, rstd_out=None, stream=None):
    """Y = RMSNorm(X @ W) * gamma over N."""
    torch = _torch()
    M, N, K = _shapes(x, w)
    y = _out(out, M, N, x)
    _check(lib().nf_gemm_postnorm_rms(_mat(x, "x"), _mat(w, "w"),
                                      _vec(gamma, "gamma", N, torch.bfloat16), _mat(y, "out"),
                                      M, N, K, float(eps),
                                      _vec(rstd_out, "rstd_out", M, torch.float32),
                                      _stream(stream)), "nf_gemm_postnorm_rms")
    return y


def _res(r, M, N, name="r"):
    if tuple(r.shape) != (M, N):
        raise ValueError(f"{name} must have shape {(M, N)}")
    return _mat(r, name)


def gemm_postnorm_ln_res(x, w, r, eps, gamma=None, beta=None, out=None, h_out=None, mean_out=None,
                         rstd_out=None, stream=None):
    """H = X @ W + R; Y = LayerNorm(H) * gamma + beta over N.  h_out (optional,
    may be r itself): bf16(H), the updated residual.  Returns Y."""
    torch = _torch()
    M, N, K = _shapes(x, w)
    y = _out(out, M, N, x)
    _check(lib().nf_gemm_postnorm_ln_res(_mat(x, "x"), _mat(w, "w"), _res(r, M, N),
                                         _vec(gamma, "gamma", N, torch.bfloat16),
                                         _vec(beta, "beta", N, torch.bfloat16), _mat(y, "out"),
                                         None if h_out is None else _res(h_out, M, N, "h_out"), M, N, K,
                                         float(eps), _vec(mean_out, "mean_out", M, torch.float32),
                                         _vec(rstd_out, "rstd_out", M, torch.float32), _stream(stream)),
           "nf_gemm_postnorm_ln_res")
    return y


def gemm_postnorm_rms_res(x, w, r, eps, gamma=None, out=None, h_out=None, rstd_out=None, stream=None):
    """H = X @ W + R; Y = RMSNorm(H) * gamma over N.  h_out as gemm_postnorm_ln_res."""
    torch = _torch()
    M, N, K = _shapes(x, w)
    y = _out(out, M, N, x)
    _check(lib().nf_gemm_postnorm_rms_res(_mat(x, "x"), _mat(w, "w"), _res(r, M, N),
                                          _vec(gamma, "gamma", N, torch.bfloat16), _mat(y, "out"),
                                          None if h_out is None else _res(h_out, M, N, "h_out"), M, N, K,
                                          float(eps), _vec(rstd_out, "rstd_out", M, torch.float32),
                                          _stream(stream)), "nf_gemm_postnorm_rms_res")
    return y


ACT_IDENTITY, ACT_GELU_TANH, ACT_SILU = 0, 1, 2


def flashnorm_attn_fwd(q, k, v, act=ACT_GELU_TANH, eps1=1e-5, eps2=1e-6, q_len=None, out=None, stream=None):
    """FlashNormAttention forward: q [B, Lq, H, D], k / v [B, Lkv, H, D] (bf16
    CUDA tensors, D = Lkv = 128, H <= 8, Lq % 128 == 0); q_len: int32 CUDA
    tensor [B] or None.  Returns out [B, Lq, H, D]."""
    torch = _torch()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k and v must be 4-D [B, L, H, D]")
    B, Lq, H, D = q.shape
    Lkv = k.shape[1]
    if tuple(k.shape) != (B, Lkv, H, D) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, Lkv, H, D] with q's B, H, D")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous bf16 CUDA tensor")
    if out is None:
        out = torch.empty_like(q)
    elif tuple(out.shape) != tuple(q.shape) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like q")
    ql = None
    if q_len is not None:
        if not q_len.is_cuda or q_len.dtype != torch.int32 or q_len.numel() != B or not q_len.is_contiguous():
            raise TypeError("q_len must be a contiguous int32 CUDA tensor of B entries")
        ql = q_len.data_ptr()
    _check(lib().nf_flashnorm_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), ql, out.data_ptr(), B, Lq,
                                       Lkv, H, D, int(act), float(eps1), float(eps2), _stream(stream)),
           "nf_flashnorm_attn_fwd")
    return out


def norm_rows_res(x, r, kind, eps, gamma=None, beta=None, out=None, h_out=None, mean_out=None,
                  rstd_out=None, stream=None):
    """The unfused residual-add norm: H = x + r, out = norm(H) (kind 0 LN, 1 RMS);
    h_out (optional, may be r): bf16(H)."""
    torch = _torch()
    R = x.shape[0] if x.dim() == 2 else -1
    C = x.shape[1] if x.dim() == 2 else -1
    y = _out(out, R, C, x)
    _check(lib().nf_norm_rows_res(_mat(x, "x"), _res(r, R, C), _mat(y, "out"),
                                  None if h_out is None else _res(h_out, R, C, "h_out"),
                                  _vec(gamma, "gamma", C, torch.bfloat16), _vec(beta, "beta", C, torch.bfloat16),
                                  R, C, int(kind), float(eps), _vec(mean_out, "mean_out", R, torch.float32),
                                  _vec(rstd_out, "rstd_out", R, torch.float32), _stream(stream)),
           "nf_norm_rows_res")
    return y


def norm_rows(x, kind, eps, gamma=None, beta=None, out=None, mean_out=None, rstd_out=None,
              stream=None):
    """LayerNorm (kind 0) or RMSNorm (kind 1) of each row of x (the unfused norm kernel)."""
    torch = _torch()
    R = x.shape[0] if x.dim() == 2 else -1
    C = x.shape[1] if x.dim() == 2 else -1
    y = _out(out, R, C, x)
    _check(lib().nf_norm_rows(_mat(x, "x"), _mat(y, "out"), _vec(gamma, "gamma", C, torch.bfloat16),
                              _vec(beta, "beta", C, torch.bfloat16), R, C, int(kind), float(eps),
                              _vec(mean_out, "mean_out", R, torch.float32),
                              _vec(rstd_out, "rstd_out", R, torch.float32), _stream(stream)),
           "nf_norm_rows")
    return y


def gemm_postnorm_ln_bwd(a, b, z, mean, rstd, gamma=None, out=None, stream=None):
    """dZ = LayerNorm backward of dY = a @ b (fused), from the saved row mean / rstd (fp32 [M])."""
    torch = _torch()
    M, N, K = _shapes(a, b)
    if tuple(z.shape) != (M, N):
        raise ValueError(f"z must have shape {(M, N)}")
    y = _out(out, M, N, a)
    _check(lib().nf_gemm_postnorm_ln_bwd(_mat(a, "a"), _mat(b, "b"), _mat(z, "z"),
                                         _vec(gamma, "gamma", N, torch.bfloat16),
                                         _vec(mean, "mean", M, torch.float32), _vec(rstd, "rstd", M, torch.float32),
                                         _mat(y, "out"), M, N, K, _stream(stream)), "nf_gemm_postnorm_ln_bwd")
    return y


def gemm_postnorm_rms_bwd(a, b, z, rstd, gamma=None, out=None, stream=None):
    """dZ = RMSNorm backward of dY = a @ b (fused), from the saved row rstd (fp32 [M])."""
    torch = _torch()
    M, N, K = _shapes(a, b)
    if tuple(z.shape) != (M, N):
        raise ValueError(f"z must have shape {(M, N)}")
    y = _out(out, M, N, a)
    _check(lib().nf_gemm_postnorm_rms_bwd(_mat(a, "a"), _mat(b, "b"), _mat(z, "z"),
                                          _vec(gamma, "gamma", N, torch.bfloat16),
                                          _vec(rstd, "rstd", M, torch.float32), _mat(y, "out"), M, N, K,
                                          _stream(stream)), "nf_gemm_postnorm_rms_bwd")
    return y


def norm_rows_bwd(dy, z, kind, mean, rstd, gamma=None, out=None, stream=None):
    """Backward of LayerNorm (kind 0) / RMSNorm (kind 1) of each row from the saved
    statistics (mean: fp32 [rows], None for RMS; rstd: fp32 [rows]); returns dZ."""
    torch = _torch()
    R = dy.shape[0] if dy.dim() == 2 else -1
    C = dy.shape[1] if dy.dim() == 2 else -1
    if tuple(z.shape) != (R, C):
        raise ValueError(f"z must have shape {(R, C)}")
    y = _out(out, R, C, dy)
    _check(lib().nf_norm_rows_bwd(_mat(dy, "dy"), _mat(z, "z"), _vec(gamma, "gamma", C, torch.bfloat16),
                                  _vec(mean, "mean", R, torch.float32), _vec(rstd, "rstd", R, torch.float32),
                                  _mat(y, "out"), R, C, int(kind), _stream(stream)), "nf_norm_rows_bwd")
    return y


# ------------------------------------------------------------- diagnostics
def device_status():
    """(status, [code, site, block, tile]) after synchronizing the device."""
    buf = (ctypes.c_uint32 * 4)()
    s = lib().nf_get_device_status(ctypes.cast(buf, ctypes.c_void_p))
    return s, list(buf)


def clear_device_status() -> None:
    _check(lib().nf_clear_device_status(), "nf_clear_device_status")


def set_wait_timeout_ns(ns: int) -> None:
    _check(lib().nf_set_wait_timeout_ns(int(ns)), "nf_set_wait_timeout_ns")


def set_launch_overlap(enable: bool) -> None:
    """Programmatic dependent launch on (default) or off."""
    _check(lib().nf_set_launch_overlap(1 if enable else 0), "nf_set_launch_overlap")


def set_postnorm_tile_n(tile_n: int) -> None:
    """Post-norm column tile per CTA: 0 automatic, 256 or 512 forced."""
    _check(lib().nf_set_postnorm_tile_n(int(tile_n)), "nf_set_postnorm_tile_n")


def set_gemm_tile_n(tile_n: int) -> None:
    """Column tile of plain and pre-norm GEMMs: 0 automatic, 64, 128 or 256 forced."""
    _check(lib().nf_set_gemm_tile_n(int(tile_n)), "nf_set_gemm_tile_n")


def set_gemm_pair(mode: int) -> None:
    """CTA pairs (cta_group::2) for plain / pre-norm GEMMs: 0 automatic, 1 never, 2 whenever possible."""
    _check(lib().nf_set_gemm_pair(int(mode)), "nf_set_gemm_pair")


def set_gemm_splitk(mode: int) -> None:
    """Split-K of plain GEMMs with few output tiles: 0 automatic (default), 1 never."""
    _check(lib().nf_set_gemm_splitk(int(mode)), "nf_set_gemm_splitk")


def set_prenorm_split(mode: int) -> None:
    """Lazy Pre-Norm row sums of squares split over a row's 256-column tiles and
    gathered through L2: 0 automatic (tensor-bound tiles, K >= 2048), 1 never,
    2 whenever a row has 2..32 tiles."""
    _check(lib().nf_set_prenorm_split(int(mode)), "nf_set_prenorm_split")


def set_postnorm_exchange(mode: int) -> None:
    """Post-norm rows wider than 256 columns: 0 automatic, XCH_CLUSTER (DSMEM in a
    thread-block cluster) or XCH_GLOBAL (L2 between tiles of a cooperative grid)."""
    _check(lib().nf_set_postnorm_exchange(int(mode)), "nf_set_postnorm_exchange")


def reserve_scratch(max_rows: int, max_cols: int, stream=None) -> None:
    """Size the stream's scratch (exchange buffer, split-K workspace) for
    post-norm shapes up to max_rows x max_cols and Lazy Pre-Norm calls of up to
    max_rows rows; later calls within it allocate nothing."""
    _check(lib().nf_reserve_scratch(int(max_rows), int(max_cols), _stream(stream)), "nf_reserve_scratch")


def selftest_wait_timeout(ns: int, stream=None) -> None:
    _check(lib().nf_selftest_wait_timeout(int(ns), _stream(stream)), "nf_selftest_wait_timeout")


def plan_gemm(op: int, M: int, N: int, K: int, sm_count: int) -> dict:
    """Launch plan for op 0 plain / 1 pre-RMS / 2 post-LN / 3 post-RMS / 4 LN bwd / 5 RMS bwd (host only)."""
    p = NFPlan()
    _check(lib().nf_plan_gemm(op, M, N, K, sm_count, ctypes.byref(p)), "nf_plan_gemm")
    return {f: getattr(p, f) for f, _ in NFPlan._fields_}
