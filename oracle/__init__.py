"""CPU fp64 oracle for RMSNorm (and LayerNorm) forward and backward.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` (``cpu_baseline`` and ``--impl reference``) may
import this package. The product path (the CUDA library and its Python
binding) never imports it and shares no code with it.

The arithmetic lives in ``rmsnorm_oracle.c`` (plain C, every step in
double); this module only marshals numpy arrays into it. The definitions
and the sources they follow are stated at the top of that file:
RMSNorm in llama mode with weight (offset + w), the optional fused residual
add, and the exact gradient dx = rstd (g - xhat c), dW = sum dy xhat, as
described by the Liger-Kernel page "perf(cutedsl): add Blackwell fast path
to RMSNorm" (Summary, section 2) and the FlyDSL page "[Perf] Optimize
RMSNorm backward with staged reduction and vec8 I/O" (Implementation).

The same library holds the E4M3 (fp8) output of the forward (``fwd_fp8``)
and LayerNorm forward and backward (``ln_fwd``, ``ln_bwd``), defined in the
C file's header.

Storage types: ``"bf16"`` arrays are numpy ``uint16`` bit patterns,
``"f16"`` arrays are ``float16``, ``"f32"`` arrays are ``float32``,
``"f64"`` arrays are ``float64`` (no rounding; used by the finite-difference
pins).

Every function here is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rmsnorm_oracle.c")
_LIB = os.path.join(_HERE, "librmsnorm_oracle.so")

_DTYPE_CODE = {"f32": 0, "bf16": 1, "f64": 2, "f16": 3}
_NP_STORAGE = {"f32": np.float32, "bf16": np.uint16, "f64": np.float64, "f16": np.float16}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction, so x86
    and Arm hosts produce identical doubles). Returns the library path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call([
            "gcc", "-O2", "-std=gnu99", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-o", tmp, _SRC, "-lm", "-lpthread",
        ])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # The mutation tests point this at deliberately broken copies of
            # the oracle to show that the pins catch them.
            override = os.environ.get("RMSNORM_ORACLE_LIB_OVERRIDE")
            lib = ctypes.CDLL(override if override else build())
            i64, dbl, vp, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
            lib.oracle_rmsnorm_fwd.restype = i32
            lib.oracle_rmsnorm_fwd.argtypes = [i32, i32, i64, i64, vp, vp, vp, dbl, dbl,
                                               vp, vp, vp, vp, vp, i32]
            lib.oracle_rmsnorm_bwd.restype = i32
            lib.oracle_rmsnorm_bwd.argtypes = [i32, i32, i64, i64, vp, vp, vp, vp, vp, dbl, dbl,
                                               vp, vp, vp, vp, vp, vp, vp, i32]
            lib.oracle_bf16_round_array.restype = i32
            lib.oracle_bf16_round_array.argtypes = [vp, i64, vp]
            lib.oracle_bf16_decode.restype = dbl
            lib.oracle_bf16_decode.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_round_array.restype = i32
            lib.oracle_f16_round_array.argtypes = [vp, i64, vp]
            lib.oracle_e4m3_round_array.restype = i32
            lib.oracle_e4m3_round_array.argtypes = [vp, i64, vp]
            lib.oracle_e4m3_decode_array.restype = None
            lib.oracle_e4m3_decode_array.argtypes = [vp, i64, vp]
            lib.oracle_layernorm_fwd.restype = i32
            lib.oracle_layernorm_fwd.argtypes = [i32, i32, i64, i64, vp, vp, vp, vp, dbl, dbl,
                                                 vp, vp, vp, vp, vp, vp, vp, i32]
            lib.oracle_layernorm_bwd.restype = i32
            lib.oracle_layernorm_bwd.argtypes = [i32, i32, i64, i64, vp, vp, vp, vp, vp, vp, dbl, dbl,
                                                 vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32]
            lib.oracle_rmsnorm_fwd_fp8.restype = i32
            lib.oracle_rmsnorm_fwd_fp8.argtypes = [i32, i32, i64, i64, vp, vp, vp, dbl, dbl, i32, dbl,
                                                   vp, vp, vp, vp, vp, vp, vp, vp, i32]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _as_storage(a, dtype, shape=None):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    want = _NP_STORAGE[dtype]
    if a.dtype != want:
        raise TypeError(f"oracle: {dtype} data must be numpy {np.dtype(want).name}, got {a.dtype}")
    if shape is not None and a.size != int(np.prod(shape)):
        raise ValueError(f"oracle: expected {shape} elements, got {a.shape}")
    return a


def bf16_round(v) -> np.ndarray:
    """Round float64 values to bf16 (ties to even) in one step; returns bit patterns."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_bf16_round_array(_ptr(v), v.size, _ptr(out))
    return out


def bf16_decode(b) -> np.ndarray:
    """Exact value of bf16 bit patterns as float64 (bf16 is the top half of binary32)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f16_round(v) -> np.ndarray:
    """Round float64 values to binary16 (ties to even) in one step; returns float16."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_f16_round_array(_ptr(v), v.size, _ptr(out))
    return out.view(np.float16)


def e4m3_round(v) -> np.ndarray:
    """Round float64 values to E4M3 codes (nearest-even, saturating at +-448) in one step."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().oracle_e4m3_round_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_decode(b) -> np.ndarray:
    """Exact values of E4M3 codes as float64 (NaN for the two NaN codes)."""
    b = np.ascontiguousarray(b, dtype=np.uint8)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_e4m3_decode_array(_ptr(b), b.size, _ptr(out))
    return out


def to_f64(a, dtype) -> np.ndarray:
    """Decode storage-type data to float64 exactly."""
    if dtype == "bf16":
        return bf16_decode(a)
    return np.asarray(a, dtype=np.float64)


def fwd(x, w, *, dtype, eps, offset, residual=None, nthreads=1, wdtype=None):
    """RMSNorm forward (optionally with the fused residual add) on an M x N block.
    ``w`` None is non-affine RMSNorm (weight factor 1, offset unused);
    ``wdtype`` is the weight's storage type (default: ``dtype``).

    Returns a dict with
      ``y``       R(y) in the storage type, shape (M, N)
      ``y64``     unrounded y (float64)
      ``h``       R(x + residual) in the storage type (fused only; else None)
      ``rstd64``  rstd in double, shape (M,)
      ``rstd32``  rstd rounded to float32
    """
    wdtype = wdtype or dtype
    x = _as_storage(x, dtype)
    M, N = x.shape
    w = _as_storage(w, wdtype, (N,))   # None: non-affine (weight factor 1)
    residual = _as_storage(residual, dtype, (M, N))
    st = _NP_STORAGE[dtype]
    y = np.empty((M, N), dtype=st)
    y64 = np.empty((M, N), dtype=np.float64)
    h = np.empty((M, N), dtype=st) if residual is not None else None
    r64 = np.empty((M,), dtype=np.float64)
    r32 = np.empty((M,), dtype=np.float32)
    bad = _load().oracle_rmsnorm_fwd(_DTYPE_CODE[dtype], _DTYPE_CODE[wdtype], M, N, _ptr(x), _ptr(residual), _ptr(w),
                                     float(eps), float(offset), _ptr(y), _ptr(y64), _ptr(h),
                                     _ptr(r64), _ptr(r32), int(nthreads))
    if bad:
        raise FloatingPointError(f"oracle fwd: {bad} non-finite or overflowing stores")
    return {"y": y, "y64": y64, "h": h, "rstd64": r64, "rstd32": r32}


def fwd_fp8(x, w, *, dtype, eps, offset, scaling, scale=None, residual=None, nthreads=1, wdtype=None):
    """RMSNorm forward with E4M3 output: yq = E4M3(y * s).

    ``scaling`` "tensor": ``s = scale`` (given); "row": s_i = 448 / max_j |y_ij|
    (1 for an all-zero row). Returns a dict with ``yq`` (uint8 codes),
    ``y64`` (unrounded y), ``scaled64`` (y * s before rounding), ``amax_row``
    (max_j |y_ij|), ``amax`` (max over the block), ``scale_inv`` (1 / s per
    row), ``h`` (fused only), ``rstd64``, ``rstd32``.
    """
    wdtype = wdtype or dtype
    mode = {"tensor": 0, "row": 1}[scaling]
    if mode == 0 and scale is None:
        raise ValueError("oracle fwd_fp8: per-tensor scaling needs a scale")
    x = _as_storage(x, dtype)
    M, N = x.shape
    w = _as_storage(w, wdtype, (N,))
    residual = _as_storage(residual, dtype, (M, N))
    yq = np.empty((M, N), dtype=np.uint8)
    y64 = np.empty((M, N), dtype=np.float64)
    sc64 = np.empty((M, N), dtype=np.float64)
    amax_row = np.empty((M,), dtype=np.float64)
    sinv = np.empty((M,), dtype=np.float64)
    h = np.empty((M, N), dtype=_NP_STORAGE[dtype]) if residual is not None else None
    r64 = np.empty((M,), dtype=np.float64)
    r32 = np.empty((M,), dtype=np.float32)
    bad = _load().oracle_rmsnorm_fwd_fp8(_DTYPE_CODE[dtype], _DTYPE_CODE[wdtype], M, N, _ptr(x), _ptr(residual),
                                         _ptr(w), float(eps), float(offset), mode,
                                         float(scale) if scale is not None else 1.0,
                                         _ptr(yq), _ptr(y64), _ptr(sc64), _ptr(amax_row), _ptr(sinv), _ptr(h),
                                         _ptr(r64), _ptr(r32), int(nthreads))
    if bad:
        raise FloatingPointError(f"oracle fwd_fp8: {bad} non-finite values")
    return {"yq": yq, "y64": y64, "scaled64": sc64, "amax_row": amax_row,
            "amax": float(amax_row.max()) if M else 0.0, "scale_inv": sinv, "h": h,
            "rstd64": r64, "rstd32": r32}


def bwd(dy, h, w, *, dtype, eps, offset, rstd=None, dres=None, want_dx=True, nthreads=1, wdtype=None):
    """RMSNorm backward on an M x N block.

    ``h`` is the normalised input (x, or residual_out of the fused forward).
    ``w`` None is non-affine RMSNorm (weight factor 1; the dW outputs are
    then the sums of dy xhat, which a non-affine layer does not use).
    ``rstd`` None recomputes rstd in double from h; otherwise the given
    float32 values are used. ``dres`` is the fused variant's incoming
    residual-stream gradient. With ``want_dx=False`` only the dW sums are
    produced (no M x N outputs).

    Returns a dict with ``dx`` (storage type), ``dx64``, ``dx_scale``
    (rstd (|g| + |xhat c|) [+ |dres|]), ``dx_cscale`` (rstd |xhat| (1/N)
    sum |g xhat|, the sensitivity of dx to rounding in the sum behind c),
    ``dw64``, ``dw_abs`` (sum |dy xhat|) and ``dw`` (the weight's storage
    type, ``wdtype``, default ``dtype``).
    """
    wdtype = wdtype or dtype
    dy = _as_storage(dy, dtype)
    M, N = dy.shape
    h = _as_storage(h, dtype, (M, N))
    w = _as_storage(w, wdtype, (N,))   # None: non-affine (g = dy; dW is not a result)
    dres = _as_storage(dres, dtype, (M, N))
    if rstd is not None:
        rstd = np.ascontiguousarray(rstd, dtype=np.float32)
        if rstd.size != M:
            raise ValueError("oracle bwd: rstd must have M entries")
    st = _NP_STORAGE[dtype]
    dx = np.empty((M, N), dtype=st) if want_dx else None
    dx64 = np.empty((M, N), dtype=np.float64) if want_dx else None
    dxs = np.empty((M, N), dtype=np.float64) if want_dx else None
    dxc = np.empty((M, N), dtype=np.float64) if want_dx else None
    dw64 = np.empty((N,), dtype=np.float64)
    dwa = np.empty((N,), dtype=np.float64)
    dw = np.empty((N,), dtype=_NP_STORAGE[wdtype])
    bad = _load().oracle_rmsnorm_bwd(_DTYPE_CODE[dtype], _DTYPE_CODE[wdtype], M, N, _ptr(dy), _ptr(h), _ptr(w),
                                     _ptr(rstd), _ptr(dres), float(eps), float(offset),
                                     _ptr(dx), _ptr(dx64), _ptr(dxs), _ptr(dxc), _ptr(dw64), _ptr(dwa),
                                     _ptr(dw), int(nthreads))
    if bad:
        raise FloatingPointError(f"oracle bwd: {bad} non-finite or overflowing stores")
    return {"dx": dx, "dx64": dx64, "dx_scale": dxs, "dx_cscale": dxc, "dw64": dw64, "dw_abs": dwa, "dw": dw}


# ------------------------------------------------------------- LayerNorm --

def ln_fwd(x, gamma, beta, *, dtype, eps, offset, residual=None, nthreads=1, wdtype=None):
    """LayerNorm forward (y = (h - mean) rstd (offset + gamma) + beta, biased
    variance, h = x or R(x + residual)); gamma None: factor 1; beta None: no
    bias. Returns ``y``, ``y64``, ``h`` (fused only), ``mean64``, ``mean32``,
    ``rstd64``, ``rstd32``."""
    wdtype = wdtype or dtype
    x = _as_storage(x, dtype)
    M, N = x.shape
    gamma = _as_storage(gamma, wdtype, (N,))
    beta = _as_storage(beta, wdtype, (N,))
    residual = _as_storage(residual, dtype, (M, N))
    st = _NP_STORAGE[dtype]
    y = np.empty((M, N), dtype=st)
    y64 = np.empty((M, N), dtype=np.float64)
    h = np.empty((M, N), dtype=st) if residual is not None else None
    m64, r64 = np.empty((M,), dtype=np.float64), np.empty((M,), dtype=np.float64)
    m32, r32 = np.empty((M,), dtype=np.float32), np.empty((M,), dtype=np.float32)
    bad = _load().oracle_layernorm_fwd(_DTYPE_CODE[dtype], _DTYPE_CODE[wdtype], M, N, _ptr(x), _ptr(residual),
                                       _ptr(gamma), _ptr(beta), float(eps), float(offset), _ptr(y), _ptr(y64),
                                       _ptr(h), _ptr(m64), _ptr(m32), _ptr(r64), _ptr(r32), int(nthreads))
    if bad:
        raise FloatingPointError(f"oracle ln_fwd: {bad} non-finite or overflowing stores")
    return {"y": y, "y64": y64, "h": h, "mean64": m64, "mean32": m32, "rstd64": r64, "rstd32": r32}


def ln_bwd(dy, h, gamma, *, dtype, eps, offset, mean=None, rstd=None, dres=None, want_dx=True, nthreads=1,
           wdtype=None):
    """LayerNorm backward. ``mean``/``rstd`` None: recomputed in double from
    h; otherwise the forward's float32 values. Returns ``dx``, ``dx64``,
    ``dx_scale``, ``dx_cscale``, ``dg64``, ``dg_abs``, ``dg`` (dgamma in
    the weight type), ``db64``, ``db_abs``, ``db`` (dbeta)."""
    wdtype = wdtype or dtype
    dy = _as_storage(dy, dtype)
    M, N = dy.shape
    h = _as_storage(h, dtype, (M, N))
    gamma = _as_storage(gamma, wdtype, (N,))
    dres = _as_storage(dres, dtype, (M, N))
    if (mean is None) != (rstd is None):
        raise ValueError("oracle ln_bwd: give both mean and rstd, or neither")
    if rstd is not None:
        mean = np.ascontiguousarray(mean, dtype=np.float32)
        rstd = np.ascontiguousarray(rstd, dtype=np.float32)
        if mean.size != M or rstd.size != M:
            raise ValueError("oracle ln_bwd: mean and rstd must have M entries")
    st = _NP_STORAGE[dtype]
    dx = np.empty((M, N), dtype=st) if want_dx else None
    dx64 = np.empty((M, N), dtype=np.float64) if want_dx else None
    dxs = np.empty((M, N), dtype=np.float64) if want_dx else None
    dxc = np.empty((M, N), dtype=np.float64) if want_dx else None
    dg64, dga = np.empty((N,), dtype=np.float64), np.empty((N,), dtype=np.float64)
    db64, dba = np.empty((N,), dtype=np.float64), np.empty((N,), dtype=np.float64)
    dg = np.empty((N,), dtype=_NP_STORAGE[wdtype])
    db = np.empty((N,), dtype=_NP_STORAGE[wdtype])
    bad = _load().oracle_layernorm_bwd(_DTYPE_CODE[dtype], _DTYPE_CODE[wdtype], M, N, _ptr(dy), _ptr(h),
                                       _ptr(gamma), _ptr(mean), _ptr(rstd), _ptr(dres), float(eps), float(offset),
                                       _ptr(dx), _ptr(dx64), _ptr(dxs), _ptr(dxc), _ptr(dg64), _ptr(dga), _ptr(dg),
                                       _ptr(db64), _ptr(dba), _ptr(db), int(nthreads))
    if bad:
        raise FloatingPointError(f"oracle ln_bwd: {bad} non-finite or overflowing stores")
    return {"dx": dx, "dx64": dx64, "dx_scale": dxs, "dx_cscale": dxc, "dg64": dg64, "dg_abs": dga, "dg": dg,
            "db64": db64, "db_abs": dba, "db": db}
