"""Seeded synthetic inputs for RMSNorm workloads.

This module holds no RMSNorm arithmetic. It draws random numbers and rounds
them to a storage type, and it is the one module that both the CUDA path's
tests/benchmark and the CPU oracle read their inputs from, so that both
sides see identical bytes.

Recipe (numpy PCG64, ``default_rng([seed, stream])``):
  stream 0  x        ~ N(0, 1)
  stream 1  dy       ~ N(0, 1) * dy_scale
  stream 2  w        = 1 + 0.1 N(0, 1)  ("llama", offset 0)
                     = 0.1 N(0, 1)      ("gemma", offset 1)
  stream 3  residual ~ N(0, 1)
  stream 4  dres     ~ N(0, 1)           (incoming residual-stream gradient)
  stream 5  outlier columns: ceil(frac * N) columns chosen by a seeded
            permutation, whose x values are multiplied by 20
  stream 6  beta     ~ 0.1 N(0, 1)       (LayerNorm bias, on request)
  x_shift   added to every x draw before the outlier scaling (LayerNorm
            inputs with a non-zero row mean)
Draws are float32; bf16 values are the float32 draws rounded to nearest
(ties to even) on their bit patterns, fp16 values numpy's float32 -> float16
conversion (nearest, ties to even). bf16 arrays are numpy uint16 bit
patterns, fp16 arrays float16, fp32 arrays float32.

The shapes, scales and outlier structure follow the workloads of the
RMSNorm pages (llama/gemma weights, bf16 activations, 1% outlier channels
for the wide-row backward).
"""
from __future__ import annotations

import math

import numpy as np

STREAM_X, STREAM_DY, STREAM_W, STREAM_RES, STREAM_DRES, STREAM_OUTLIER, STREAM_BETA = range(7)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, nearest with ties to even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream)])


def _normal(seed, stream, shape, scale=1.0):
    a = _rng(seed, stream).standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        a *= np.float32(scale)
    return a


def to_storage(a_f32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return f32_to_bf16_bits(a_f32)
    if dtype == "f16":
        return np.ascontiguousarray(a_f32).astype(np.float16)   # nearest, ties to even
    if dtype == "f32":
        return np.ascontiguousarray(a_f32, dtype=np.float32)
    raise ValueError(f"unsupported storage dtype {dtype!r}")


def outlier_columns(N: int, seed: int, frac: float) -> np.ndarray:
    k = int(math.ceil(frac * N))
    perm = _rng(seed, STREAM_OUTLIER).permutation(N)
    return np.sort(perm[:k])


def make_inputs(M: int, N: int, dtype: str, seed: int, *, dy_scale: float = 1.0,
                w_mode: str = "llama", residual: bool = False, dres: bool = False,
                outlier_frac: float = 0.0, outlier_scale: float = 20.0, wdtype: str | None = None,
                beta: bool = False, x_shift: float = 0.0) -> dict:
    """Return a dict of storage-typed numpy arrays: x, dy, w and, on request,
    residual, dres and beta. ``w_mode`` "llama" pairs with offset 0, "gemma"
    with 1. ``wdtype`` is the weight's (and beta's) storage type (default
    ``dtype``)."""
    x = _normal(seed, STREAM_X, (M, N))
    if x_shift != 0.0:
        x += np.float32(x_shift)
    if outlier_frac > 0.0:
        cols = outlier_columns(N, seed, outlier_frac)
        x[:, cols] *= np.float32(outlier_scale)
    out = {"x": to_storage(x, dtype)}
    del x
    out["dy"] = to_storage(_normal(seed, STREAM_DY, (M, N), dy_scale), dtype)
    wn = _normal(seed, STREAM_W, (N,))
    if w_mode == "llama":
        w = np.float32(1.0) + np.float32(0.1) * wn
    elif w_mode == "gemma":
        w = np.float32(0.1) * wn
    else:
        raise ValueError(f"unknown w_mode {w_mode!r}")
    out["w"] = to_storage(w, wdtype or dtype)
    if residual:
        out["residual"] = to_storage(_normal(seed, STREAM_RES, (M, N)), dtype)
    if dres:
        out["dres"] = to_storage(_normal(seed, STREAM_DRES, (M, N)), dtype)
    if beta:
        out["beta"] = to_storage(_normal(seed, STREAM_BETA, (N,), 0.1), wdtype or dtype)
    return out


# Named workloads, after the RMSNorm pages' shapes. ``seed`` is 1000 + k.
WORKLOADS = {
    "small_f32": dict(M=64, N=256, dtype="f32", seed=1001, eps=1e-6, offset=0.0),
    "llama_bf16_4096x2048": dict(M=4096, N=2048, dtype="bf16", seed=1002, eps=1e-6,
                                 offset=0.0, dy_scale=0.01),
    "add_bf16_4096x4096": dict(M=4096, N=4096, dtype="bf16", seed=1003, eps=1e-6, offset=0.0,
                               residual=True, dres=True),
    "add_bf16_1024x8192": dict(M=1024, N=8192, dtype="bf16", seed=1003, eps=1e-6, offset=0.0,
                               residual=True, dres=True),
    "add_gemma_bf16_4096x4096": dict(M=4096, N=4096, dtype="bf16", seed=1003, eps=1e-6,
                                     offset=1.0, w_mode="gemma", residual=True, dres=True),
    "add_gemma_bf16_1024x8192": dict(M=1024, N=8192, dtype="bf16", seed=1003, eps=1e-6,
                                     offset=1.0, w_mode="gemma", residual=True, dres=True),
    "wide_bf16_16384x8192": dict(M=16384, N=8192, dtype="bf16", seed=1004, eps=1e-6,
                                 offset=0.0, outlier_frac=0.01),
    "wide_f32_16384x6144": dict(M=16384, N=6144, dtype="f32", seed=1004, eps=1e-6,
                                offset=0.0, outlier_frac=0.01),
}

SWEEP_N = (128, 2048, 4096, 7168, 8192, 16384)
SWEEP_M = (512, 4096, 16384)
SWEEP_SEED = 1005
PER_HEAD_M = 16384 * 32


def sweep_points(dtype: str):
    """(M, N) points of the shape sweep: N=128 is the per-head norm with
    16384*32 rows; every other N crosses M in {512, 4096, 16384}."""
    pts = []
    for N in SWEEP_N:
        if N == 128:
            pts.append((PER_HEAD_M, N))
        else:
            pts.extend((M, N) for M in SWEEP_M)
    return pts


def workload_inputs(name: str) -> tuple[dict, dict]:
    """Inputs and scalar parameters of a named workload."""
    cfg = dict(WORKLOADS[name])
    params = {k: cfg.pop(k) for k in ("M", "N", "dtype", "seed", "eps", "offset")}
    arrays = make_inputs(params["M"], params["N"], params["dtype"], params["seed"], **cfg)
    return arrays, params
