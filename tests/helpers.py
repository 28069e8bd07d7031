"""Shared helpers for the GPU parity tests: device upload (optionally at a
non-16-byte-aligned offset), readback, and the tolerance checks.

Tolerances (the RMSNorm definition and bounds are restated in the oracle):
  y    bf16 / fp16: within 1 ulp of the correctly rounded oracle value
       (distance of the ordered bit patterns); fp32: |d| <= 1e-5 |ref| + 1e-6.
  dx   as y, or -- where the result comes from cancelling terms -- within
       8 * 2^-24 * rstd (|g| + |xhat c|) [+ |dres|], the fp32 rounding bound
       of the difference of the two terms, plus (N/256 + 48) * 2^-24 *
       rstd |xhat| (1/N) sum |g xhat|, the worst-case fp32 error of the sum
       behind c (at most N/256 terms added in sequence per thread, then a
       tree and at most 32 warp partials), which can itself cancel
       (counted and reported).
  dw   bf16: |d| <= 4e-3 |ref| + 2^-20 S; fp16: 1e-3 |ref| + 2^-20 S (its
       output rounding is 2^-11); fp32: |d| <= 1e-4 |ref| + 2^-20 S,
       with ref the unrounded double sum and S = sum_i |dy xhat| (the scale
       of the fp32 summation error).
  rstd relative 2e-6.
  E4M3 codes: equal (as values) to the oracle's nearest-even rounding of the
       exact y * s, except where the exact scaled value lies within
       2^-19 |v| of the midpoint between two adjacent codes: the kernel's
       fp32 y * s carries a relative error of a few 2^-24 (rstd, the three
       products, the scale), so there either neighbour is correct.
       Row scales 1/s and amax: relative 2^-19.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

FLOOR_ULPS = 8.0 * 2.0 ** -24


TORCH_DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}


def to_dev(a: np.ndarray, dtype: str, device="cuda", offset: int = 0) -> torch.Tensor:
    """Upload storage-typed numpy data. offset > 0 places the tensor `offset`
    elements past a 256-byte-aligned allocation (a contiguous tensor whose
    base is not 16-byte aligned)."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    elif dtype == "f16":
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float16))
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    if offset == 0:
        return t.to(device)
    buf = torch.empty(t.numel() + offset + 16, dtype=t.dtype, device=device)
    view = buf[offset:offset + t.numel()].view(t.shape)
    view.copy_(t.to(device))
    return view


def empty_dev(shape, dtype: str, device="cuda", offset: int = 0, fill=float("nan")) -> torch.Tensor:
    td = TORCH_DT[dtype]
    n = int(np.prod(shape))
    buf = torch.full((n + offset + 16,), fill, dtype=td, device=device)
    return buf[offset:offset + n].view(shape)


def to_host(t: torch.Tensor, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()   # float16 or float32


def decode(a: np.ndarray, dtype: str) -> np.ndarray:
    return oracle.to_f64(a, dtype)


def ulp16_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|ordered(a) - ordered(b)| for 16-bit sign-magnitude bit patterns (bf16
    or fp16, as uint16 or float16 arrays), mapped to a monotone integer line
    so +0 and -0 are 0 apart; 1 means adjacent representable values."""
    def ordered(x):
        x = np.ascontiguousarray(x).view(np.uint16).astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a) - ordered(b))


bf16_ulp_distance = ulp16_distance


def check_y(got: np.ndarray, ref: dict, dtype: str, key="y", key64="y64"):
    if dtype in ("bf16", "f16"):
        d = ulp16_distance(got, ref[key])
        assert d.max() <= 1, f"{key}: max {d.max()} ulp"
        return {"max_ulp": int(d.max())}
    r = ref[key64]
    err = np.abs(got.astype(np.float64) - r)
    bad = err > 1e-5 * np.abs(r) + 1e-6
    assert not bad.any(), f"{key}: {bad.sum()} elements off, worst {err.max()}"
    return {"max_abs": float(err.max())}


def check_rstd(got: np.ndarray, ref64: np.ndarray):
    rel = np.abs(got.astype(np.float64) - ref64) / ref64
    assert rel.max() <= 2e-6, f"rstd rel err {rel.max()}"
    return float(rel.max())


def reduction_ulps(N: int) -> float:
    return (N / 256.0 + 48.0) * 2.0 ** -24


# Elements that needed the cancellation floor, per dx check: (test id,
# elements checked, elements that needed it). The session summary prints
# them (tests/conftest.py).
FLOOR_USES: list = []

# Largest share of elements that may need the floor. A correct fp32
# evaluation of dx misses the 1-ulp check only where g and xhat c nearly
# cancel: fp32 emulations of the kernel's arithmetic in numpy measured 0.2
# to 0.5 elements per million with a pairwise row sum and 0.6 to 1.4 with a
# sequential one on the parity workloads (tests/test_floor_rate_cpu.py keeps
# the pairwise measurement and shows that a coarse row sum, relative error
# 2^-12, exceeds the cap by two orders of magnitude), so the cap allows
# four per million (plus two for small cases) and a kernel whose error is
# not a cancellation effect cannot hide behind the floor.
FLOOR_RATE_CAP = 4e-6


def floor_cap(elements: int) -> float:
    return 2 + FLOOR_RATE_CAP * elements


def check_dx(got: np.ndarray, ref: dict, dtype: str, floor_mult: float = 1.0, cap: bool = True):
    """Returns the number of elements that needed the cancellation floor.
    With `cap` (and rows of at least 64 elements: shorter rows cancel by
    construction, e.g. at N = 1 dx = rstd g eps / (x^2 + eps)), that number
    must stay within floor_cap()."""
    v = decode(got, dtype)
    N = got.shape[-1]
    floor = floor_mult * (FLOOR_ULPS * ref["dx_scale"] + reduction_ulps(N) * ref["dx_cscale"])
    near = np.abs(v - ref["dx64"]) <= floor
    if dtype in ("bf16", "f16"):
        ok = (ulp16_distance(got, ref["dx"]) <= 1)
    else:
        r = ref["dx64"]
        ok = np.abs(v - r) <= 1e-5 * np.abs(r) + 1e-6
    needed = int((~ok & near).sum())
    ok = ok | near
    if not ok.all():
        i = np.flatnonzero(~ok)[0]
        raise AssertionError(f"dx: {(~ok).sum()} elements off; first at flat index {i}: got {v.flat[i]!r} "
                             f"ref {ref['dx64'].flat[i]!r} scale {ref['dx_scale'].flat[i]!r} "
                             f"cscale {ref['dx_cscale'].flat[i]!r}")
    import os
    FLOOR_USES.append((os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], int(v.size), needed))
    if cap and N >= 64:
        assert needed <= floor_cap(v.size), f"dx: {needed} of {v.size} elements needed the cancellation floor"
    return needed


# Columns of a parameter gradient that needed the summation floor
# 2^-20 sum |dy xhat| beyond the relative bound: (test id, columns, count,
# worst error as a fraction of the relative bound alone).
DW_FLOOR_USES: list = []


def check_dw(got: np.ndarray, ref: dict, dtype: str):
    import os
    v = decode(got, dtype)
    rel = {"bf16": 4e-3, "f16": 1e-3, "f32": 1e-4}[dtype]
    err = np.abs(v - ref["dw64"])
    rtol = rel * np.abs(ref["dw64"])
    tol = rtol + 2.0 ** -20 * ref["dw_abs"]
    assert (err <= tol).all(), f"dw: {(err > tol).sum()} columns off, worst ratio {(err / tol).max()}"
    DW_FLOOR_USES.append((os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], int(v.size),
                          int((err > rtol).sum()), float((err / np.maximum(rtol, 1e-300)).max())))
    return float((err / np.maximum(tol, 1e-300)).max())


def cuda_bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    if a.dtype != b.dtype or a.shape != b.shape:
        return False
    iv = {1: torch.uint8, 2: torch.int16, 4: torch.int32, 8: torch.int64}[a.element_size()]
    return torch.equal(a.contiguous().view(iv), b.contiguous().view(iv))


FP8_TIE_REL = 2.0 ** -19


def check_fp8(got_codes: np.ndarray, ref: dict, rows=None):
    """E4M3 codes of the kernel against the oracle's (see the module
    docstring); returns the number of elements decided at a near-tie."""
    want = ref["yq"] if rows is None else ref["yq"][rows]
    v = ref["scaled64"] if rows is None else ref["scaled64"][rows]
    g, w = oracle.e4m3_decode(got_codes), oracle.e4m3_decode(want)
    diff = g != w
    if not diff.any():
        return 0
    gd, wd, vd = g[diff], w[diff], v[diff]
    gc, wc = got_codes[diff].astype(np.int32), want[diff].astype(np.int32)
    adjacent = ((gc >> 7) == (wc >> 7)) & (np.abs(gc - wc) == 1)
    tie = np.abs(vd - (gd + wd) / 2.0) <= FP8_TIE_REL * np.abs(vd)
    bad = ~(adjacent & tie)
    assert not bad.any(), (f"E4M3: {bad.sum()} codes off; first scaled value {vd[bad][0]!r}, "
                           f"kernel {gd[bad][0]!r}, oracle {wd[bad][0]!r}")
    return int(diff.sum())


def check_rel(got, ref, rel, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    assert np.all(err <= rel * np.abs(ref)), f"{what}: worst rel {(err / np.maximum(np.abs(ref), 1e-300)).max()}"


def check_ln_y(got: np.ndarray, ref: dict, dtype: str, h64: np.ndarray, factor: np.ndarray, bias: np.ndarray):
    """LayerNorm y: as check_y, or -- where y comes from cancelling terms
    (xhat (offset + gamma) against beta, or h against the mean) -- within
    2^-24 (8 (|xhat f| + |beta|) + (N/256 + 56) rstd |f| mean|h|): the fp32
    rounding of the two terms plus the fp32 error of the mean, carried
    through rstd and the weight factor. Returns the elements that needed it."""
    v = decode(got, dtype)
    N = got.shape[-1]
    xf = np.abs(ref["y64"] - bias[None, :])
    mh = np.abs(h64).mean(axis=1, keepdims=True)
    floor = 2.0 ** -24 * (8.0 * (xf + np.abs(bias)[None, :]) +
                          (N / 256.0 + 56.0) * ref["rstd64"][:, None] * np.abs(factor)[None, :] * mh)
    near = np.abs(v - ref["y64"]) <= floor
    if dtype in ("bf16", "f16"):
        ok = ulp16_distance(got, ref["y"]) <= 1
    else:
        r = ref["y64"]
        ok = np.abs(v - r) <= 1e-5 * np.abs(r) + 1e-6
    needed = int((~ok & near).sum())
    ok = ok | near
    assert ok.all(), f"y: {(~ok).sum()} elements off, first {v[~ok][0]!r} vs {ref['y64'][~ok][0]!r}"
    return needed


def check_ln_stats(mean: np.ndarray, rstd: np.ndarray, ref: dict, h64: np.ndarray):
    """mean within the fp32 summation error (N/256 + 48) 2^-24 mean|h|;
    rstd relative within (N/256 + 64) 2^-24 (the variance's summation error,
    halved by the root, plus rsqrt's own)."""
    N = h64.shape[-1]
    mh = np.abs(h64).mean(axis=1)
    tol = (N / 256.0 + 48.0) * 2.0 ** -24 * mh
    err = np.abs(mean.astype(np.float64) - ref["mean64"])
    assert np.all(err <= tol), f"mean: worst {(err / tol).max()} of tolerance"
    rel = np.abs(rstd.astype(np.float64) - ref["rstd64"]) / ref["rstd64"]
    assert rel.max() <= (N / 256.0 + 64.0) * 2.0 ** -24, f"rstd rel err {rel.max()}"


def check_param_grad(got: np.ndarray, ref64: np.ndarray, ref_abs: np.ndarray, dtype: str):
    return check_dw(got, {"dw64": ref64, "dw_abs": ref_abs}, dtype)
