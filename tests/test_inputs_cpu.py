"""The seeded input recipe (shared by the CUDA path's tests and bench and by
the oracle): reproducible draws, storage rounding, outlier columns, weight
modes and the named workloads' shapes, checked on CPU."""
import math

import numpy as np
import pytest
import torch

from row_wise_normalization_rmsnorm_gb300 import inputs


def test_same_seed_same_bytes_and_streams_independent():
    a = inputs.make_inputs(64, 96, "bf16", 7, residual=True, dres=True, beta=True)
    b = inputs.make_inputs(64, 96, "bf16", 7, residual=True, dres=True, beta=True)
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    # each array has its own stream: no two activation arrays coincide
    assert not np.array_equal(a["x"], a["dy"])
    assert not np.array_equal(a["residual"], a["dres"])
    c = inputs.make_inputs(64, 96, "bf16", 8)
    assert not np.array_equal(a["x"], c["x"])
    # optional arrays draw from their own streams, so asking for them leaves x, dy, w alone
    d = inputs.make_inputs(64, 96, "bf16", 7)
    assert set(d) == {"x", "dy", "w"}
    for k in d:
        assert np.array_equal(a[k], d[k]), k


def test_bf16_rounding_matches_torch_nearest_even():
    rng = np.random.default_rng(5)
    a = (rng.standard_normal(100_000) * np.exp2(rng.integers(-30, 30, 100_000))).astype(np.float32)
    # exact ties (low 16 bits 0x8000) with even and odd upper halves, subnormal
    # and normal (from 1.0 up)
    hi = np.concatenate([np.arange(1, 2001, dtype=np.uint32), np.uint32(0x3F80) + np.arange(2000, dtype=np.uint32)])
    ties = (hi << np.uint32(16) | np.uint32(0x8000)).view(np.float32)
    a = np.concatenate([a, ties, -ties, np.float32([0.0, -0.0, 1.0, 65504.0, 3.0e38])])
    ours = inputs.f32_to_bf16_bits(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(inputs.bf16_bits_to_f32(ours), torch.from_numpy(a).to(torch.bfloat16).float().numpy())


def test_storage_types():
    for dt, np_dt in (("bf16", np.uint16), ("f16", np.float16), ("f32", np.float32)):
        d = inputs.make_inputs(3, 5, dt, 1)
        assert d["x"].dtype == np_dt and d["x"].shape == (3, 5) and d["w"].shape == (5,)
    d = inputs.make_inputs(3, 5, "bf16", 1, wdtype="f32", beta=True)
    assert d["w"].dtype == np.float32 and d["beta"].dtype == np.float32
    with pytest.raises(ValueError):
        inputs.make_inputs(3, 5, "f64", 1)


@pytest.mark.parametrize("N,frac", [(8192, 0.01), (100, 0.01), (7, 0.5), (64, 0.02)])
def test_outlier_columns_scale_x_by_20(N, frac):
    cols = inputs.outlier_columns(N, 11, frac)
    assert len(cols) == math.ceil(frac * N)
    assert np.all(np.diff(cols) > 0) and cols[0] >= 0 and cols[-1] < N
    base = inputs.make_inputs(4, N, "f32", 11)["x"]
    out = inputs.make_inputs(4, N, "f32", 11, outlier_frac=frac)["x"]
    assert np.array_equal(out[:, cols], base[:, cols] * np.float32(20.0))
    rest = np.setdiff1d(np.arange(N), cols)
    assert np.array_equal(out[:, rest], base[:, rest])


def test_weight_modes_and_shift():
    ll = inputs.make_inputs(2, 300, "f32", 3)
    gm = inputs.make_inputs(2, 300, "f32", 3, w_mode="gemma")
    # both come from the same N(0,1) draw: llama 1 + 0.1 z, gemma 0.1 z
    z = gm["w"] / np.float32(0.1)
    assert np.allclose(ll["w"], 1.0 + 0.1 * z, rtol=0, atol=1e-6)
    assert abs(float(np.mean(ll["w"])) - 1.0) < 0.03 and abs(float(np.mean(gm["w"]))) < 0.03
    sh = inputs.make_inputs(2, 300, "f32", 3, x_shift=0.5)
    assert np.array_equal(sh["x"], ll["x"] + np.float32(0.5))
    assert np.array_equal(sh["dy"], ll["dy"])
    with pytest.raises(ValueError):
        inputs.make_inputs(2, 3, "f32", 3, w_mode="other")


def test_draws_are_standard_normal():
    d = inputs.make_inputs(512, 512, "f32", 9, dy_scale=0.01, beta=True)
    x, dy = d["x"].astype(np.float64), d["dy"].astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert abs(dy.std() - 0.01) < 1e-4
    assert abs(d["beta"].astype(np.float64).std() - 0.1) < 0.02


def test_named_workloads_and_sweep_shapes():
    shapes = {k: (v["M"], v["N"], v["dtype"]) for k, v in inputs.WORKLOADS.items()}
    assert shapes["small_f32"] == (64, 256, "f32")
    assert shapes["wide_bf16_16384x8192"] == (16384, 8192, "bf16")
    assert shapes["wide_f32_16384x6144"] == (16384, 6144, "f32")
    for k, v in inputs.WORKLOADS.items():
        assert v["seed"] >= 1000 and (v["offset"] == 1.0) == (v.get("w_mode") == "gemma"), k
    pts = inputs.sweep_points("bf16")
    assert len(pts) == 1 + 3 * (len(inputs.SWEEP_N) - 1)
    assert (16384 * 32, 128) in pts and (16384, 16384) in pts and (512, 2048) in pts
    arrays, params = inputs.workload_inputs("small_f32")
    assert arrays["x"].shape == (64, 256) and params == {"M": 64, "N": 256, "dtype": "f32", "seed": 1001,
                                                         "eps": 1e-6, "offset": 0.0}
