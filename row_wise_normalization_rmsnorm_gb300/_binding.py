"""ctypes binding of librmsnorm_gb300.so (declared in include/rmsnorm.h).

Argument marshalling only: every step of RMSNorm runs in the library's CUDA
kernels. PyTorch supplies device memory and the current stream. There is no
CPU fallback: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librmsnorm_gb300.so")

RMSNORM_F32, RMSNORM_BF16, RMSNORM_F16 = 0, 1, 2
RMSNORM_WEIGHT_F32 = 0x100  # OR'ed into a 16-bit type: w and dw are fp32
RMSNORM_OUT_BF16 = 0x200    # forward of fp32 activations: y in bf16
RMSNORM_OUT_F16 = 0x400     # ... or in fp16
STATUS = {0: "SUCCESS", 1: "ERR_INVALID_ARG", 2: "ERR_UNSUPPORTED", 3: "ERR_WORKSPACE", 4: "ERR_CUDA"}
PATH_NAMES = {0: "vector", 1: "staged", 2: "generic"}
OP_FWD, OP_BWD, OP_LN_BWD = 0, 1, 2
TORCH_DTYPE = {torch.float32: RMSNORM_F32, torch.bfloat16: RMSNORM_BF16, torch.float16: RMSNORM_F16}


class RMSNormError(RuntimeError):
    def __init__(self, status: int, what: str, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = f"{what}: {STATUS.get(status, status)}"
        if status == 4:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)


class Plan(ctypes.Structure):
    _fields_ = [
        ("path", ctypes.c_int32),
        ("plan_id", ctypes.c_int32),
        ("threads_per_row", ctypes.c_int32),
        ("chunks_per_thread", ctypes.c_int32),
        ("rows_per_cta", ctypes.c_int32),
        ("cta_threads", ctypes.c_int32),
        ("packed", ctypes.c_int32),
        ("ctas", ctypes.c_int32),
        ("ctas_per_sm", ctypes.c_int32),
        ("smem_bytes", ctypes.c_int32),
        ("cluster_size", ctypes.c_int32),
        ("ws_rows", ctypes.c_int32),
        ("workspace_bytes", ctypes.c_int64),
        ("peel", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        d = {f: getattr(self, f) for f, _ in self._fields_}
        d["path_name"] = PATH_NAMES.get(self.path, "?")
        return d


_lock = threading.Lock()
_lib = None

# name -> (restype, argtypes)
_vp, _i64, _f, _i, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_size_t
_PPlan = ctypes.POINTER(Plan)
SIGNATURES = {
    "rmsnorm_fwd": (_i, [_vp, _vp, _vp, _vp, _i64, _i64, _i, _f, _f, _vp]),
    "rmsnorm_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64, _i, _f, _f, _vp]),
    "rmsnorm_add_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i, _f, _f, _vp]),
    "rmsnorm_add_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64, _i, _f, _f, _vp]),
    "rmsnorm_bwd_workspace_bytes": (_sz, [_i64, _i64, _i]),
    "rmsnorm_bwd_call_workspace_bytes": (_sz, [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i, _i]),
    "rmsnorm_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i, _f, _f, _vp]),
    "rmsnorm_plan_query": (_i, [_i, _i64, _i64, _i, _i, _i, _i, _i, _i, _PPlan]),
    "rmsnorm_plan_count": (_i, []),
    "rmsnorm_plan_id_at": (_i, [_i]),
    "rmsnorm_fwd_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _i64, _i64, _i, _f, _f, _vp]),
    "rmsnorm_fwd_fp8_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _vp, _vp, _i64, _i64, _i, _f, _f, _vp,
                                _i, _PPlan]),
    "layernorm_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i, _f, _f, _vp]),
    "layernorm_fwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i, _f, _f, _vp, _i, _PPlan]),
    "layernorm_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64, _i, _f, _f, _vp]),
    "layernorm_bwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64, _i, _f, _f, _vp,
                              _i, _i, _PPlan]),
    "layernorm_bwd_workspace_bytes": (_sz, [_i64, _i64, _i]),
    "rmsnorm_fwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i, _f, _f, _vp, _i, _PPlan]),
    "rmsnorm_bwd_ex": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i64, _i64, _i, _f, _f, _vp,
                            _i, _i, _i, _i, _vp, _PPlan]),
    "rmsnorm_status_string": (ctypes.c_char_p, [_i]),
    "rmsnorm_last_cuda_error": (_i, []),
    "rmsnorm_self_check": (_i, []),
    "rmsnorm_device_status": (_i, [_i]),
    "rmsnorm_set_generic_note": (None, [_i]),
}


def lib() -> ctypes.CDLL:
    """The loaded library with every entry point's signature declared."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built; run `python -m row_wise_normalization_rmsnorm_gb300.build` "
                    "(or __graft_entry__.build()). There is no CPU fallback.")
            h = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
    return _lib


def _raise(status: int, what: str) -> None:
    if status != 0:
        raise RMSNormError(status, what, lib().rmsnorm_last_cuda_error() if status == 4 else 0)


def _stream_handle(stream, device) -> int:
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_code(t: torch.Tensor) -> int:
    try:
        return TORCH_DTYPE[t.dtype]
    except KeyError:
        raise TypeError(f"unsupported dtype {t.dtype}; use torch.float32, torch.bfloat16 or torch.float16") from None


def _dtype_code_w(x: torch.Tensor, w) -> int:
    """Type code for activations x and weight w: w in x's type, or fp32
    beside 16-bit activations (RMSNORM_WEIGHT_F32)."""
    code = _dtype_code(x)
    if w is None or w.dtype == x.dtype:
        return code
    if w.dtype == torch.float32:
        return code | RMSNORM_WEIGHT_F32
    raise ValueError(f"w must be {x.dtype} or torch.float32, is {w.dtype}")


def _param_dtype(x: torch.Tensor, *params) -> torch.dtype:
    """The storage type shared by LayerNorm's gamma / beta (and their
    gradients) among the given tensors (None entries skipped): x's type, or
    fp32 beside 16-bit activations; x's type when none is given."""
    for t in params:
        if t is not None and t.device != x.device:
            raise ValueError("gamma, beta and their gradients must be on the input's device")
    types = {t.dtype for t in params if t is not None}
    if len(types) > 1:
        raise ValueError(f"gamma, beta and their gradients must share one type, have {sorted(map(str, types))}")
    dt = types.pop() if types else x.dtype
    if dt != x.dtype and not (dt == torch.float32 and x.dtype in (torch.bfloat16, torch.float16)):
        raise ValueError(f"gamma / beta must be {x.dtype} or (beside 16-bit x) torch.float32, are {dt}")
    return dt


def _param_code(x: torch.Tensor, dt: torch.dtype) -> int:
    return _dtype_code(x) | (RMSNORM_WEIGHT_F32 if dt != x.dtype else 0)


def _out_flag(x: torch.Tensor, y: torch.Tensor) -> int:
    """The forward's output-type flag: 0 when y has x's type; fp32 x may
    write y in bf16 (RMSNORM_OUT_BF16) or fp16 (RMSNORM_OUT_F16)."""
    if y.dtype == x.dtype:
        return 0
    if x.dtype == torch.float32 and y.dtype in (torch.bfloat16, torch.float16):
        return RMSNORM_OUT_BF16 if y.dtype == torch.bfloat16 else RMSNORM_OUT_F16
    raise ValueError(f"y must be {x.dtype} (or, for float32 x, bfloat16 / float16), is {y.dtype}")


def _new_y(x: torch.Tensor, y, out_dtype):
    if y is not None:
        return y
    return torch.empty(x.shape, dtype=out_dtype or x.dtype, device=x.device)


def _check_w(w, name: str, x: torch.Tensor, N: int):
    _check(w, name, numel=N)
    if w.device != x.device:
        raise ValueError(f"{name} must be on the input's device")
    if w.dtype not in (x.dtype, torch.float32):
        raise ValueError(f"{name} must be {x.dtype} or torch.float32, is {w.dtype}")


def _check(t: torch.Tensor, name: str, like: torch.Tensor | None = None, numel: int | None = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if like is not None and (t.dtype != like.dtype or t.device != like.device):
        raise ValueError(f"{name} must match dtype/device of the input")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, has {t.numel()}")


def _rows(x: torch.Tensor):
    N = x.shape[-1]
    M = x.numel() // N if N else 0
    return M, N


def _ptr(t):
    return None if t is None else t.data_ptr()


def _ws(workspace):
    if workspace is None:
        return None, 0
    _check(workspace, "workspace")
    return workspace.data_ptr(), workspace.numel() * workspace.element_size()


def rmsnorm_fwd(x, w, *, eps: float = 1e-6, offset: float = 0.0, y=None, rstd=None, out_dtype=None, stream=None):
    """y, rstd = RMSNorm(x) over the last dimension (llama mode); w None is
    non-affine RMSNorm (y = x * rstd). For float32 x, y may be bfloat16 or
    float16 (``out_dtype``, or a given ``y`` of that type)."""
    M, N = _rows(x)
    _check(x, "x")
    if w is not None:
        _check_w(w, "w", x, N)
    y = _new_y(x, y, out_dtype)
    rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device) if rstd is None else rstd
    _check(y, "y", numel=x.numel())
    _check(rstd, "rstd", numel=M)
    st = lib().rmsnorm_fwd(x.data_ptr(), _ptr(w), y.data_ptr(), rstd.data_ptr(), M, N,
                           _dtype_code_w(x, w) | _out_flag(x, y), eps, offset, _stream_handle(stream, x.device))
    _raise(st, "rmsnorm_fwd")
    return y, rstd


def rmsnorm_add_fwd(x, residual, w, *, eps: float = 1e-6, offset: float = 0.0, y=None, residual_out=None,
                    rstd=None, out_dtype=None, stream=None):
    """h = x + residual (rounded), y = RMSNorm(h); returns y, h, rstd. For
    float32 x, y may be bfloat16 or float16 (h stays float32)."""
    M, N = _rows(x)
    _check(x, "x")
    _check(residual, "residual", like=x, numel=x.numel())
    if w is not None:
        _check_w(w, "w", x, N)
    y = _new_y(x, y, out_dtype)
    residual_out = torch.empty_like(x) if residual_out is None else residual_out
    rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device) if rstd is None else rstd
    _check(y, "y", numel=x.numel())
    _check(residual_out, "residual_out", like=x, numel=x.numel())
    _check(rstd, "rstd", numel=M)
    st = lib().rmsnorm_add_fwd(x.data_ptr(), residual.data_ptr(), _ptr(w), y.data_ptr(),
                               residual_out.data_ptr(), rstd.data_ptr(), M, N, _dtype_code_w(x, w) | _out_flag(x, y),
                               eps, offset, _stream_handle(stream, x.device))
    _raise(st, "rmsnorm_add_fwd")
    return y, residual_out, rstd


FP8_SCALING = {"tensor": 0, "row": 1}


def rmsnorm_fwd_fp8(x, w, *, scaling="row", scale=None, residual=None, eps: float = 1e-6, offset: float = 0.0,
                    y=None, residual_out=None, rstd=None, scale_inv=None, amax=False, force_plan=-1,
                    stream=None):
    """RMSNorm forward with an E4M3 output: y = E4M3(y' * s), y' the fp32 forward.

    scaling "row": s_i = 448 / max_j |y'_ij|; "tensor": s = scale (a CUDA
    fp32 tensor of one element). Returns a dict with ``y`` (torch.uint8
    codes, view as torch.float8_e4m3fn to compute), ``residual_out`` (fused
    only), ``rstd``, ``scale_inv`` (per row, or one value) and ``amax`` (one
    fp32, when requested), plus ``plan``.
    """
    M, N = _rows(x)
    _check(x, "x")
    if w is not None:
        _check_w(w, "w", x, N)
    mode = FP8_SCALING[scaling]
    if mode == 0:
        if scale is None:
            raise ValueError("per-tensor scaling needs `scale`")
        _check(scale, "scale", numel=1)
        if scale.dtype != torch.float32:
            raise ValueError("scale must be float32")
    elif scale is not None:
        raise ValueError("per-row scaling derives its scales; pass no `scale`")
    y = torch.empty(x.shape, dtype=torch.uint8, device=x.device) if y is None else y
    _check(y, "y", numel=x.numel())
    if y.element_size() != 1:
        raise ValueError("y must have one-byte elements")
    if residual is not None:
        _check(residual, "residual", like=x, numel=x.numel())
        residual_out = torch.empty_like(x) if residual_out is None else residual_out
        _check(residual_out, "residual_out", like=x, numel=x.numel())
    rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device) if rstd is None else rstd
    _check(rstd, "rstd", numel=M)
    if scale_inv is None:
        scale_inv = torch.empty(x.shape[:-1] if mode == 1 else (1,), dtype=torch.float32, device=x.device)
    _check(scale_inv, "scale_inv", numel=M if mode == 1 else 1)
    amax_t = torch.empty(1, dtype=torch.float32, device=x.device) if amax is True else (amax or None)
    if amax_t is not None:
        _check(amax_t, "amax", numel=1)
    p = Plan()
    st = lib().rmsnorm_fwd_fp8_ex(x.data_ptr(), _ptr(residual), _ptr(w), y.data_ptr(), _ptr(residual_out),
                                  rstd.data_ptr(), mode, _ptr(scale), scale_inv.data_ptr(), _ptr(amax_t), M, N,
                                  _dtype_code_w(x, w), eps, offset, _stream_handle(stream, x.device), force_plan,
                                  ctypes.byref(p))
    _raise(st, "rmsnorm_fwd_fp8")
    return {"y": y, "residual_out": residual_out, "rstd": rstd, "scale_inv": scale_inv, "amax": amax_t,
            "plan": p.as_dict()}


def rmsnorm_bwd(dy, x, w, rstd, *, eps: float = 1e-6, offset: float = 0.0, dx=None, dw=None, workspace=None,
                stream=None):
    """dx, dw of RMSNorm given the forward's rstd; w None is non-affine (dw None)."""
    M, N = _rows(x)
    for t, n in ((dy, "dy"), (x, "x")):
        _check(t, n, like=x, numel=x.numel())
    _check(rstd, "rstd", numel=M)
    dx = torch.empty_like(x) if dx is None else dx
    _check(dx, "dx", like=x, numel=x.numel())
    if w is not None:
        _check_w(w, "w", x, N)
        dw = torch.empty_like(w) if dw is None else dw
        _check(dw, "dw", like=w, numel=N)
    else:
        dw = None
    wp, wb = _ws(workspace)
    st = lib().rmsnorm_bwd(dy.data_ptr(), x.data_ptr(), _ptr(w), rstd.data_ptr(), dx.data_ptr(),
                           _ptr(dw), wp, wb, M, N, _dtype_code_w(x, w), eps, offset,
                           _stream_handle(stream, x.device))
    _raise(st, "rmsnorm_bwd")
    return dx, dw


def rmsnorm_add_bwd(dy, dresidual_out, h, w, rstd, *, eps: float = 1e-6, offset: float = 0.0, dx=None, dw=None,
                    workspace=None, stream=None):
    """dx (= dresidual) and dw of the fused residual-add RMSNorm; h is the forward's residual_out."""
    M, N = _rows(h)
    _check(dy, "dy", like=h, numel=h.numel())
    _check(h, "h", like=h, numel=h.numel())
    if dresidual_out is not None:
        _check(dresidual_out, "dresidual_out", like=h, numel=h.numel())
    _check(rstd, "rstd", numel=M)
    dx = torch.empty_like(h) if dx is None else dx
    _check(dx, "dx", like=h, numel=h.numel())
    if w is not None:
        _check_w(w, "w", h, N)
        dw = torch.empty_like(w) if dw is None else dw
        _check(dw, "dw", like=w, numel=N)
    else:
        dw = None
    wp, wb = _ws(workspace)
    st = lib().rmsnorm_add_bwd(dy.data_ptr(), _ptr(dresidual_out), h.data_ptr(), _ptr(w), rstd.data_ptr(),
                               dx.data_ptr(), _ptr(dw), wp, wb, M, N, _dtype_code_w(h, w), eps, offset,
                               _stream_handle(stream, h.device))
    _raise(st, "rmsnorm_add_bwd")
    return dx, dw


def rmsnorm_bwd_workspace_bytes(M: int, N: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else TORCH_DTYPE[dtype]
    return int(lib().rmsnorm_bwd_workspace_bytes(M, N, code))


def plan_query(op: int, M: int, N: int, dtype: int, *, aligned: bool = True, num_sms: int = 152,
               ctas_per_sm: int = 0, force_plan: int = -1, force_ctas: int = 0) -> dict:
    """Host-only plan selection (no GPU needed). aligned: True (1) 16-byte
    aligned rows, False (0) the generic kernels, 1 + k rows at a common offset
    of k elements past a 16-byte boundary."""
    p = Plan()
    st = lib().rmsnorm_plan_query(op, M, N, dtype, int(aligned), num_sms, ctas_per_sm, force_plan, force_ctas,
                                  ctypes.byref(p))
    _raise(st, "rmsnorm_plan_query")
    return p.as_dict()


def rmsnorm_fwd_ex(x, w, *, residual=None, eps=1e-6, offset=0.0, y=None, residual_out=None, rstd=None,
                   force_plan=-1, out_dtype=None, stream=None):
    """Forward with a forced plan; returns (y, residual_out or None, rstd, plan dict)."""
    M, N = _rows(x)
    y = _new_y(x, y, out_dtype)
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(x)
    rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device) if rstd is None else rstd
    p = Plan()
    st = lib().rmsnorm_fwd_ex(_ptr(x), _ptr(residual), _ptr(w), _ptr(y), _ptr(residual_out), _ptr(rstd), M, N,
                              _dtype_code_w(x, w) | _out_flag(x, y), eps, offset, _stream_handle(stream, x.device),
                              force_plan, ctypes.byref(p))
    _raise(st, "rmsnorm_fwd_ex")
    return y, residual_out, rstd, p.as_dict()


def rmsnorm_bwd_ex(dy, x, w, rstd, *, dresidual_out=None, fused=False, eps=1e-6, offset=0.0, dx=None, dw=None,
                   workspace=None, force_plan=-1, force_ctas=0, force_packed=-1, event_after_main=None,
                   stream=None):
    """Backward with forced plan / CTA count / packed math; returns (dx, dw, plan dict)."""
    M, N = _rows(x)
    dx = torch.empty_like(x) if dx is None else dx
    if w is not None and dw is None:
        dw = torch.empty_like(w)
    wp, wb = _ws(workspace)
    ev = None if event_after_main is None else event_after_main.cuda_event
    p = Plan()
    st = lib().rmsnorm_bwd_ex(_ptr(dy), _ptr(dresidual_out), _ptr(x), _ptr(w), _ptr(rstd), _ptr(dx), _ptr(dw),
                              wp, wb, M, N, _dtype_code_w(x, w), eps, offset, _stream_handle(stream, x.device),
                              int(fused), force_plan, force_ctas, force_packed, ev, ctypes.byref(p))
    _raise(st, "rmsnorm_bwd_ex")
    return dx, dw, p.as_dict()


# ------------------------------------------------------------- LayerNorm --

def layernorm_fwd(x, gamma, beta, *, residual=None, eps: float = 1e-5, offset: float = 0.0, y=None,
                  residual_out=None, mean=None, rstd=None, force_plan=-1, stream=None):
    """LayerNorm over the last dimension: y = (h - mean) rstd (offset + gamma) + beta,
    h = x or x + residual (fused, h also returned). gamma / beta may be None.
    Returns a dict with y, residual_out (fused only), mean, rstd, plan."""
    M, N = _rows(x)
    _check(x, "x")
    pdt = _param_dtype(x, gamma, beta)
    for t, n in ((gamma, "gamma"), (beta, "beta")):
        if t is not None:
            _check(t, n, numel=N)
    y = torch.empty_like(x) if y is None else y
    _check(y, "y", like=x, numel=x.numel())
    if residual is not None:
        _check(residual, "residual", like=x, numel=x.numel())
        residual_out = torch.empty_like(x) if residual_out is None else residual_out
        _check(residual_out, "residual_out", like=x, numel=x.numel())
    mean = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device) if mean is None else mean
    rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device) if rstd is None else rstd
    _check(mean, "mean", numel=M)
    _check(rstd, "rstd", numel=M)
    p = Plan()
    st = lib().layernorm_fwd_ex(x.data_ptr(), _ptr(residual), _ptr(gamma), _ptr(beta), y.data_ptr(),
                                _ptr(residual_out), mean.data_ptr(), rstd.data_ptr(), M, N, _param_code(x, pdt),
                                eps, offset, _stream_handle(stream, x.device), force_plan, ctypes.byref(p))
    _raise(st, "layernorm_fwd")
    return {"y": y, "residual_out": residual_out, "mean": mean, "rstd": rstd, "plan": p.as_dict()}


def layernorm_bwd(dy, x, gamma, mean, rstd, *, dresidual_out=None, want_dgamma=True, want_dbeta=True,
                  eps: float = 1e-5, offset: float = 0.0, dx=None, dgamma=None, dbeta=None, workspace=None,
                  force_plan=-1, force_ctas=0, stream=None):
    """dx (plus dresidual_out, fused), dgamma and dbeta of LayerNorm given the
    forward's mean and rstd. dgamma is None without gamma or when not wanted;
    dbeta is None when not wanted. Returns a dict with dx, dgamma, dbeta, plan."""
    M, N = _rows(x)
    for t, n in ((dy, "dy"), (x, "x")):
        _check(t, n, like=x, numel=x.numel())
    _check(mean, "mean", numel=M)
    _check(rstd, "rstd", numel=M)
    if dresidual_out is not None:
        _check(dresidual_out, "dresidual_out", like=x, numel=x.numel())
    dx = torch.empty_like(x) if dx is None else dx
    _check(dx, "dx", like=x, numel=x.numel())
    # gamma, dgamma and dbeta share one type: x's, or fp32 beside 16-bit x
    pdt = _param_dtype(x, gamma, dgamma if want_dgamma else None, dbeta if want_dbeta else None)
    if gamma is not None:
        _check(gamma, "gamma", numel=N)
    if gamma is not None and want_dgamma:
        dgamma = torch.empty(N, dtype=pdt, device=x.device) if dgamma is None else dgamma
        _check(dgamma, "dgamma", numel=N)
    else:
        dgamma = None
    if want_dbeta:
        dbeta = torch.empty(N, dtype=pdt, device=x.device) if dbeta is None else dbeta
        _check(dbeta, "dbeta", numel=N)
    else:
        dbeta = None
    wp, wb = _ws(workspace)
    p = Plan()
    st = lib().layernorm_bwd_ex(dy.data_ptr(), _ptr(dresidual_out), x.data_ptr(), _ptr(gamma), mean.data_ptr(),
                                rstd.data_ptr(), dx.data_ptr(), _ptr(dgamma), _ptr(dbeta), wp, wb, M, N,
                                _param_code(x, pdt), eps, offset, _stream_handle(stream, x.device), force_plan,
                                force_ctas, ctypes.byref(p))
    _raise(st, "layernorm_bwd")
    return {"dx": dx, "dgamma": dgamma, "dbeta": dbeta, "plan": p.as_dict()}


def layernorm_bwd_workspace_bytes(M: int, N: int, dtype) -> int:
    code = dtype if isinstance(dtype, int) else TORCH_DTYPE[dtype]
    return int(lib().layernorm_bwd_workspace_bytes(M, N, code))
