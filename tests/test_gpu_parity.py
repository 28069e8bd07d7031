"""GPU parity: the CUDA path through the C ABI against the fp64 oracle,
element by element, on seeded inputs.

The backward is fed the oracle forward's own float32 rstd (an input of the
backward), so every oracle input is generator- or oracle-made; the
end-to-end test then runs forward and backward on the GPU against the exact
gradient. Shapes span several tiles, ragged row counts and every kernel
family: register-resident vector plans, sub-warp teams, multi-warp teams,
and the generic path for N not a multiple of the 16-byte chunk.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import check_dw, check_dx, check_rstd, check_y, cuda_bits_equal, empty_dev, to_dev, to_host
from row_wise_normalization_rmsnorm_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rn():
    from row_wise_normalization_rmsnorm_gb300 import build
    build.build()
    import row_wise_normalization_rmsnorm_gb300 as pkg
    return pkg


GENERIC_FWD, GENERIC_BWD = 16, 36   # plan ids of the generic kernels
# the streamed generic backward by row length: (plan id, longest row)
STREAM_PLANS = ((58, 256), (57, 1024), (56, 2048), (43, 4096), (37, 8192))


STREAM_FWD_PLANS = ((104, 256), (105, 1024), (106, 2048), (107, 4096), (108, 8192), (109, 16384))


def stream_plan_for(N, fwd=False):
    return next((pid for pid, nmax in (STREAM_FWD_PLANS if fwd else STREAM_PLANS) if N <= nmax), None)


def _fwd_bwd_check(rn, d, dt, eps, offset, fused=False, offset_elems=0, expect_path=None, wdt=None,
                   force_generic=False):
    """wdt: the weight's (and dW's) storage type, default the activations'.
    offset_elems: one element offset for every array, or a dict of offsets
    by array name (x, w, dy, y, residual, residual_out, h, dx, dw, dres;
    missing names: 0). force_generic: run the generic kernels whatever the
    layout."""
    wdt = wdt or dt
    M, N = d["x"].shape
    offs = offset_elems if isinstance(offset_elems, dict) else None

    def o(name):
        return offs.get(name, 0) if offs is not None else offset_elems
    x = to_dev(d["x"], dt, offset=o("x"))
    w = to_dev(d["w"], wdt, offset=o("w"))
    dy = to_dev(d["dy"], dt, offset=o("dy"))
    y = empty_dev((M, N), dt, offset=o("y"))
    rstd = torch.full((M,), float("nan"), device="cuda")
    res = to_dev(d["residual"], dt, offset=o("residual")) if fused else None
    hout = empty_dev((M, N), dt, offset=o("residual_out")) if fused else None
    _, _, _, fplan = rn.rmsnorm_fwd_ex(x, w, residual=res, residual_out=hout, y=y, rstd=rstd, eps=eps,
                                       offset=offset, force_plan=GENERIC_FWD if force_generic else -1)
    f = oracle.fwd(d["x"], d["w"], dtype=dt, eps=eps, offset=offset, residual=d.get("residual") if fused else None,
                   wdtype=wdt)
    torch.cuda.synchronize()
    check_y(to_host(y, dt), f, dt)
    check_rstd(rstd.cpu().numpy(), f["rstd64"])
    if fused:
        assert np.array_equal(to_host(hout, dt), f["h"]), "residual_out differs from R(x + residual)"
    h_np = f["h"] if fused else d["x"]

    # backward, fed the oracle's fp32 rstd
    r32 = torch.from_numpy(f["rstd32"]).cuda()
    hdev = to_dev(h_np, dt, offset=o("h"))
    dx = empty_dev((M, N), dt, offset=o("dx"))
    dw = empty_dev((N,), wdt, offset=o("dw"))
    dres_np = d.get("dres") if fused else None
    dres = to_dev(dres_np, dt, offset=o("dres")) if dres_np is not None else None
    _, _, bplan = rn.rmsnorm_bwd_ex(dy, hdev, w, r32, dresidual_out=dres, fused=fused, dx=dx, dw=dw, eps=eps,
                                    offset=offset, force_plan=GENERIC_BWD if force_generic else -1)
    b = oracle.bwd(d["dy"], h_np, d["w"], dtype=dt, eps=eps, offset=offset, rstd=f["rstd32"], dres=dres_np,
                   wdtype=wdt)
    torch.cuda.synchronize()
    needed = check_dx(to_host(dx, dt), b, dt)
    check_dw(to_host(dw, wdt), b, wdt)
    if expect_path is not None:
        # "vector": the fast paths (rows in registers; either direction may
        # instead stage rows in shared memory)
        fast = ("vector", "staged") if expect_path == "vector" else (expect_path,)
        assert fplan["path_name"] in fast and bplan["path_name"] in fast, (fplan, bplan)
    # (check_dx caps how many elements may need the cancellation floor)
    return fplan, bplan


def test_config_small_f32_64x256(rn):
    d, p = inputs.workload_inputs("small_f32")
    fp, bp = _fwd_bwd_check(rn, d, "f32", p["eps"], p["offset"])
    assert fp["path_name"] == "vector" and bp["path_name"] in ("vector", "staged")


def test_config_llama_bf16_4096x2048(rn):
    d, p = inputs.workload_inputs("llama_bf16_4096x2048")
    fp, bp = _fwd_bwd_check(rn, d, "bf16", p["eps"], p["offset"])
    assert fp["path_name"] == "vector" and bp["path_name"] in ("vector", "staged")


@pytest.mark.parametrize("name", ["add_bf16_1024x8192", "add_gemma_bf16_1024x8192",
                                  "add_bf16_4096x4096", "add_gemma_bf16_4096x4096"])
def test_config_fused_add(rn, name):
    d, p = inputs.workload_inputs(name)
    _fwd_bwd_check(rn, d, "bf16", p["eps"], p["offset"], fused=True, expect_path="vector")


def test_fused_add_without_dres(rn):
    d = inputs.make_inputs(300, 4096, "bf16", 41, residual=True)
    _fwd_bwd_check(rn, d, "bf16", 1e-6, 0.0, fused=True)


RAGGED = [
    # (dtype, M, N)  sub-warp, warp and multi-warp teams, ragged M, generic N
    ("bf16", 333, 8), ("bf16", 333, 64), ("bf16", 513, 128), ("bf16", 77, 256), ("bf16", 129, 1000),
    ("bf16", 300, 4096), ("bf16", 301, 5000), ("bf16", 130, 7168), ("bf16", 257, 8192),
    ("bf16", 97, 12288), ("bf16", 65, 16384), ("bf16", 33, 32768),
    ("bf16", 211, 4097), ("bf16", 101, 8191), ("bf16", 101, 8193), ("bf16", 9, 65536),
    ("bf16", 1, 2048), ("bf16", 3, 2048), ("bf16", 5, 1), ("bf16", 40, 3),
    ("f32", 333, 4), ("f32", 333, 32), ("f32", 513, 128), ("f32", 77, 256), ("f32", 301, 2048),
    ("f32", 130, 5000), ("f32", 257, 6144), ("f32", 97, 8192), ("f32", 65, 16384),
    ("f32", 211, 4097), ("f32", 101, 8191), ("f32", 1, 1), ("f32", 7, 3), ("f32", 9, 65536),
]


@pytest.mark.parametrize("dt,M,N", RAGGED)
def test_ragged_shapes(rn, dt, M, N):
    d = inputs.make_inputs(M, N, dt, 50 + N % 97)
    _fwd_bwd_check(rn, d, dt, 1e-6, 0.0)


@pytest.mark.parametrize("dt,M,N", [("bf16", 257, 8192), ("f32", 130, 5000), ("bf16", 77, 100)])
def test_fused_ragged_gemma(rn, dt, M, N):
    d = inputs.make_inputs(M, N, dt, 60, w_mode="gemma", residual=True, dres=True)
    _fwd_bwd_check(rn, d, dt, 1e-5, 1.0, fused=True)


@pytest.mark.parametrize("dt,M,N", [("bf16", 4096, 7168), ("f32", 4096, 2048)])
def test_misaligned_storage_offset(rn, dt, M, N):
    """All of x, w, y, dy, dx at +1 element from a 256-byte-aligned
    allocation (the sweep's misaligned case): the vectorised kernels with
    each row's head and tail joined into one chunk."""
    d = inputs.make_inputs(M, N, dt, inputs.SWEEP_SEED)
    fp, bp = _fwd_bwd_check(rn, d, dt, 1e-6, 0.0, offset_elems=1, expect_path="vector")
    assert fp["peel"] == 1 and bp["peel"] == 1, (fp, bp)


# Rows at a common offset past a 16-byte boundary, on every fast kernel
# family: sub-warp, warp and multi-warp register rows (one chunk a row
# included), staged rows (held and re-read schedules), cluster rows in both
# directions, the fused add with and without dres, gemma offset, fp16.
COMMON_OFFSET = [
    ("bf16", 257, 8, 3), ("bf16", 333, 64, 7), ("bf16", 129, 128, 1), ("bf16", 300, 2048, 5),
    ("bf16", 301, 4096, 2), ("bf16", 211, 7168, 1), ("bf16", 257, 8192, 7), ("bf16", 97, 16384, 4),
    ("bf16", 33, 32768, 1), ("bf16", 9, 65536, 3), ("f32", 333, 4, 1), ("f32", 129, 256, 3),
    ("f32", 300, 2048, 2), ("f32", 101, 6144, 1), ("f32", 65, 16384, 3), ("f16", 257, 8192, 5),
    ("f16", 77, 1024, 1),
]


@pytest.mark.parametrize("dt,M,N,k", COMMON_OFFSET)
def test_common_offset_rows_take_fast_kernels(rn, dt, M, N, k):
    d = inputs.make_inputs(M, N, dt, 360 + N % 17 + k)
    fp, bp = _fwd_bwd_check(rn, d, dt, 1e-6, 0.0, offset_elems=k, expect_path="vector")
    assert fp["peel"] == k and bp["peel"] == k, (fp, bp)


@pytest.mark.parametrize("dt,M,N,k", [("bf16", 257, 8192, 1), ("bf16", 65, 2048, 6), ("f32", 130, 5120, 2),
                                      ("bf16", 33, 32768, 5)])
@pytest.mark.parametrize("gemma", [False, True])
def test_common_offset_fused_add(rn, dt, M, N, k, gemma):
    d = inputs.make_inputs(M, N, dt, 370 + k, w_mode="gemma" if gemma else "llama", residual=True, dres=True)
    fp, bp = _fwd_bwd_check(rn, d, dt, 1e-6, 1.0 if gemma else 0.0, fused=True, offset_elems=k,
                            expect_path="vector")
    assert fp["peel"] == k and bp["peel"] == k, (fp, bp)


@pytest.mark.parametrize("dt,N,k", [("bf16", 7168, 1), ("bf16", 8192, 3), ("f32", 2048, 1), ("f32", 6144, 2)])
def test_common_offset_dw_equals_generic_at_same_ctas(rn, dt, N, k):
    """Rows at a common offset on the persistent staged backward (one row
    team a CTA) and on the generic kernel forced to the same CTA count: each
    CTA adds the same rows in the same order into its partial row, and one
    finalizer sums those in a fixed order, so dW agrees bit for bit."""
    M = 1000
    d = inputs.make_inputs(M, N, dt, 380 + k)
    x, w, dy = (to_dev(d[key], dt, offset=k) for key in ("x", "w", "dy"))
    _, rstd = rn.rmsnorm_fwd(x, w)
    dx_a = empty_dev((M, N), dt, offset=k)
    dx_b = empty_dev((M, N), dt, offset=k)
    dw_a = empty_dev((N,), dt)
    dw_b = empty_dev((N,), dt)
    _, _, pa = rn.rmsnorm_bwd_ex(dy, x, w, rstd, dx=dx_a, dw=dw_a)
    assert pa["path_name"] == "staged" and pa["peel"] == k and pa["rows_per_cta"] == 1 and pa["cluster_size"] == 1
    _, _, pb = rn.rmsnorm_bwd_ex(dy, x, w, rstd, dx=dx_b, dw=dw_b, force_plan=GENERIC_BWD, force_ctas=pa["ctas"])
    torch.cuda.synchronize()
    assert pb["path_name"] == "generic" and pb["ctas"] == pa["ctas"]
    assert cuda_bits_equal(dw_a, dw_b)


# Generic rows with 16-byte chunks between a scalar head and tail (the
# arrays share their address mod 16, the weight may not) and without them
# (the arrays do not share it): every combination against the oracle.
PEEL_CASES = [
    ("bf16", 301, 7168, {"x": 1, "w": 1, "dy": 1, "y": 1, "h": 1, "dx": 1, "dw": 1}),
    ("bf16", 300, 7171, {"x": 3, "w": 5, "dy": 3, "y": 3, "h": 3, "dx": 3, "dw": 2}),
    ("bf16", 64, 5, {"x": 3, "w": 1, "dy": 3, "y": 3, "h": 3, "dx": 3}),
    ("f16", 129, 4100, {"x": 2, "w": 2, "dy": 2, "y": 2, "h": 2, "dx": 2}),
    ("f32", 257, 2050, {"x": 1, "w": 3, "dy": 1, "y": 1, "h": 1, "dx": 1, "dw": 1}),
    ("bf16", 200, 4096, {"x": 1, "y": 0, "dy": 2, "h": 1, "dx": 0}),
    ("f32", 100, 1000, {"x": 0, "y": 1, "dy": 1, "h": 3, "dx": 1}),
]


@pytest.mark.parametrize("dt,M,N,offs", PEEL_CASES)
@pytest.mark.parametrize("fused", [False, True])
def test_generic_peeled_and_scalar_rows(rn, dt, M, N, offs, fused):
    """The generic kernels' own row split (forced: arrays at one common
    offset would otherwise take the vectorised kernels)."""
    d = inputs.make_inputs(M, N, dt, 300 + N % 11, residual=fused, dres=fused)
    if fused:
        offs = dict(offs, residual=offs.get("x", 0), residual_out=offs.get("x", 0), dres=offs.get("dy", 0))
    _fwd_bwd_check(rn, d, dt, 1e-6, 0.0, fused=fused, offset_elems=offs, expect_path="generic", force_generic=True)


# Rows no vectorised kernel takes (odd N, or arrays at different addresses
# mod 16): the streamed generic backward, which copies each row's 16-byte
# covers into shared memory at any offset. (dt, weight type, M, N, offsets)
STREAM_CASES = [
    ("bf16", None, 1000, 7169, {"x": 1, "dy": 2, "dx": 3, "h": 1, "dres": 5}),
    ("bf16", None, 700, 1500, {"x": 3, "dy": 2, "dx": 1, "h": 3, "dres": 7}),
    ("f16", "f32", 300, 3001, {"x": 1, "dy": 4, "dx": 5, "h": 1, "dres": 2}),
    ("f32", None, 2000, 250, {"x": 1, "dy": 2, "dx": 3, "h": 1, "dres": 1}),
    ("bf16", None, 3000, 257, {"x": 5, "dy": 2, "h": 5, "dres": 3}),
    ("bf16", None, 300, 7168, {"x": 1, "dy": 2, "dx": 0, "h": 1, "dres": 0}),
    ("f32", None, 300, 8191, {"x": 1, "dy": 3, "dx": 2, "h": 1, "dres": 1}),
    ("f32", None, 153, 8192, {"x": 1, "dy": 2, "h": 1, "dres": 3}),
    ("f16", None, 257, 1000, {"x": 3, "dy": 1, "h": 3, "dres": 6}),
    ("bf16", "f32", 513, 4100, {"x": 1, "dy": 5, "h": 1, "dres": 2}),
    ("f16", "f32", 129, 8192, {"x": 2, "dy": 1, "dx": 7, "h": 2, "dres": 4}),
    ("bf16", None, 64, 5, {"x": 3, "dy": 1, "h": 3, "dres": 1}),
    ("bf16", None, 2000, 1, {"x": 1, "h": 1}),
    ("bf16", None, 1, 8191, {"x": 1, "dy": 6, "h": 1, "dres": 7}),
]


@pytest.mark.parametrize("dt,wdt,M,N,offs", STREAM_CASES)
@pytest.mark.parametrize("fused", [False, True])
def test_streamed_generic_kernels(rn, dt, wdt, M, N, offs, fused):
    """The streamed generic forward and backward, element-wise against the
    oracle, on ragged M (fewer rows than SMs, one row, several rows a CTA),
    odd N down to 1, and every array at its own offset."""
    d = inputs.make_inputs(M, N, dt, 390 + N % 13, residual=fused, dres=fused, wdtype=wdt or dt)
    if fused:
        offs = dict(offs, residual=offs.get("x", 0), residual_out=offs.get("x", 0))
    fp, bp = _fwd_bwd_check(rn, d, dt, 1e-6, 0.0, fused=fused, offset_elems=offs, expect_path="generic", wdt=wdt)
    assert fp["plan_id"] == stream_plan_for(N, fwd=True), fp
    assert bp["plan_id"] == stream_plan_for(N), bp
    assert bp["ws_rows"] <= M and bp["ctas"] == bp["ws_rows"], bp
    if bp["plan_id"] == 37:  # one CTA an SM
        assert bp["ws_rows"] == min(M, torch.cuda.get_device_properties(0).multi_processor_count), bp


@pytest.mark.parametrize("dt,N,offs", [("bf16", 7169, (1, 2)), ("f32", 6000, (1, 3)), ("bf16", 4096, (3, 0)),
                                       ("bf16", 1999, (0, 0)), ("f16", 777, (2, 1)), ("f32", 100, (1, 0))])
def test_streamed_dw_equals_generic_at_same_ctas(rn, dt, N, offs):
    """The streamed kernel and the one-CTA-a-row kernel forced to the same
    CTA count: each CTA adds the same rows in the same order (one fp32
    fused multiply-add of dy xhat a row) into its partial row, and the same
    finalizer sums those in a fixed order, so dW agrees bit for bit."""
    M = 1000
    d = inputs.make_inputs(M, N, dt, 395)
    x = to_dev(d["x"], dt, offset=offs[0])
    dy = to_dev(d["dy"], dt, offset=offs[1])
    w = to_dev(d["w"], dt)
    _, rstd = rn.rmsnorm_fwd(x, w)
    _, dw_a, pa = rn.rmsnorm_bwd_ex(dy, x, w, rstd)
    _, dw_b, pb = rn.rmsnorm_bwd_ex(dy, x, w, rstd, force_plan=GENERIC_BWD, force_ctas=pa["ctas"])
    torch.cuda.synchronize()
    assert pa["plan_id"] == stream_plan_for(N) and pb["plan_id"] == GENERIC_BWD and pb["ctas"] == pa["ctas"]
    assert cuda_bits_equal(dw_a, dw_b)
    assert rn.lib().rmsnorm_device_status(1) == 0


def test_streamed_kernels_full_size_odd_row(rn):
    """bf16 4096 x 7169 with x and dy at different offsets (the odd-N point
    of the sweep): sampled rows of y, rstd and dx against the oracle, dW over
    every row."""
    M, N, dt = 4096, 7169, "bf16"
    d = inputs.make_inputs(M, N, dt, inputs.SWEEP_SEED)
    x, dy = to_dev(d["x"], dt, offset=1), to_dev(d["dy"], dt, offset=2)
    w = to_dev(d["w"], dt)
    y = empty_dev((M, N), dt, offset=3)
    _, _, rstd, fp = rn.rmsnorm_fwd_ex(x, w, y=y, eps=1e-6)
    assert fp["plan_id"] == stream_plan_for(N, fwd=True)
    r32 = _rstd32_all_rows(d["x"], d["w"], dt, 1e-6)
    dx, dw, p = rn.rmsnorm_bwd_ex(dy, x, w, torch.from_numpy(r32).cuda(), eps=1e-6)
    torch.cuda.synchronize()
    assert p["plan_id"] == stream_plan_for(N)
    assert rn.lib().rmsnorm_device_status(1) == 0
    rows = sampled_rows(M, seed=7)
    rows_t = torch.from_numpy(rows).cuda()
    f = oracle.fwd(d["x"][rows], d["w"], dtype=dt, eps=1e-6, offset=0.0)
    check_y(to_host(y[rows_t], dt), f, dt)
    check_rstd(rstd.cpu().numpy()[rows], f["rstd64"])
    b = oracle.bwd(d["dy"][rows], d["x"][rows], d["w"], dtype=dt, eps=1e-6, offset=0.0, rstd=r32[rows])
    check_dx(to_host(dx[rows_t], dt), b, dt)
    full = oracle.bwd(d["dy"], d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0, rstd=r32, want_dx=False, nthreads=8)
    check_dw(to_host(dw, dt), full, dt)


def test_generic_fused_residual_alone_misaligned(rn):
    """A residual at another address mod 16 than x turns the forward's peel
    off (element accesses); the result is the same arithmetic."""
    d = inputs.make_inputs(96, 4104, "bf16", 311, residual=True, dres=True)
    _fwd_bwd_check(rn, d, "bf16", 1e-6, 0.0, fused=True, expect_path="generic",
                   offset_elems={"x": 1, "y": 1, "residual": 2, "residual_out": 1, "dy": 1, "h": 1, "dx": 1,
                                 "dres": 3})


@pytest.mark.parametrize("dt,M,N", [("bf16", 160, 7169), ("bf16", 96, 10223), ("bf16", 96, 10247),
                                    ("f32", 130, 5111), ("f32", 64, 5121)])
@pytest.mark.parametrize("fused", [False, True])
def test_generic_backward_rows_around_40kb(rn, dt, M, N, fused):
    """Rows whose x and dy together come just under and just over 40 KB
    (where the LayerNorm generic backward stops caching them), on the
    generic backward the call selects (the streamed kernel up to 8192
    elements, with its stages in shared memory) and on the one-CTA-a-row
    kernel, which re-reads global memory at every length and takes no
    dynamic shared memory."""
    d = inputs.make_inputs(M, N, dt, 330 + N % 7, residual=fused, dres=fused)
    _, bplan = _fwd_bwd_check(rn, d, dt, 1e-6, 0.0, fused=fused, offset_elems=1, expect_path="generic")
    if N <= 8192:
        assert bplan["plan_id"] == stream_plan_for(N) and bplan["smem_bytes"] > 0, (N, bplan)
    else:
        assert bplan["plan_id"] == GENERIC_BWD and bplan["smem_bytes"] == 0, (N, bplan)
    _, bplan = _fwd_bwd_check(rn, d, dt, 1e-6, 0.0, fused=fused, offset_elems=1, expect_path="generic",
                              force_generic=True)
    assert bplan["plan_id"] == GENERIC_BWD and bplan["smem_bytes"] == 0, (N, bplan)


@pytest.mark.parametrize("eps", [0.0, 1e-2, 10.0])
def test_eps_values(rn, eps):
    d = inputs.make_inputs(200, 2048, "bf16", 71)
    _fwd_bwd_check(rn, d, "bf16", eps, 0.0)


def test_end_to_end_against_exact_gradient(rn):
    """GPU forward, then GPU backward on the GPU's rstd, against the oracle's
    exact gradient (rstd recomputed in double). The forward's rstd error
    (<= 2e-6 relative) enters dx three times over, hence 4x the floor."""
    for dt, M, N in (("bf16", 1024, 8192), ("f32", 512, 6144)):
        d = inputs.make_inputs(M, N, dt, 80, outlier_frac=0.01)
        x, w, dy = (to_dev(d[k], dt) for k in ("x", "w", "dy"))
        y, rstd = rn.rmsnorm_fwd(x, w, eps=1e-6)
        dx, dw = rn.rmsnorm_bwd(dy, x, w, rstd, eps=1e-6)
        b = oracle.bwd(d["dy"], d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0)
        torch.cuda.synchronize()
        check_dx(to_host(dx, dt), b, dt, floor_mult=4.0)
        check_dw(to_host(dw, dt), b, dt)


def _rstd32_all_rows(x, w, dt, eps, chunk=2048):
    out = np.empty(x.shape[0], dtype=np.float32)
    for r0 in range(0, x.shape[0], chunk):
        out[r0:r0 + chunk] = oracle.fwd(x[r0:r0 + chunk], w, dtype=dt, eps=eps, offset=0.0, nthreads=8)["rstd32"]
    return out


def sampled_rows(M, k=48, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(M, size=min(k, M), replace=False).tolist()) | {0, M - 1}
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", ["wide_bf16_16384x8192", "wide_f32_16384x6144"])
def test_full_size_wide_rows(rn, name):
    """The bench's workload sizes: sampled rows of y, rstd and dx against the
    oracle, dW over every row (the oracle's dW-only pass)."""
    d, p = inputs.workload_inputs(name)
    dt, eps = p["dtype"], p["eps"]
    M, N = d["x"].shape
    x, w, dy = (to_dev(d[k], dt) for k in ("x", "w", "dy"))
    y, rstd = rn.rmsnorm_fwd(x, w, eps=eps)
    r32 = _rstd32_all_rows(d["x"], d["w"], dt, eps)
    dx, dw = rn.rmsnorm_bwd(dy, x, w, torch.from_numpy(r32).cuda(), eps=eps)
    torch.cuda.synchronize()
    rows = sampled_rows(M)
    rows_t = torch.from_numpy(rows).cuda()
    f = oracle.fwd(d["x"][rows], d["w"], dtype=dt, eps=eps, offset=0.0)
    check_y(to_host(y[rows_t], dt), f, dt)
    check_rstd(rstd.cpu().numpy()[rows], f["rstd64"])
    b = oracle.bwd(d["dy"][rows], d["x"][rows], d["w"], dtype=dt, eps=eps, offset=0.0, rstd=r32[rows])
    check_dx(to_host(dx[rows_t], dt), b, dt)
    full = oracle.bwd(d["dy"], d["x"], d["w"], dtype=dt, eps=eps, offset=0.0, rstd=r32, want_dx=False, nthreads=8)
    check_dw(to_host(dw, dt), full, dt)
    # no bounded wait of the staged kernels gave up during these calls
    assert rn.lib().rmsnorm_device_status(1) == 0


@pytest.mark.parametrize("dt,M,N", [("bf16", 524288, 128), ("f32", 524288, 128), ("bf16", 16384, 16384),
                                    ("f32", 16384, 16384)])
def test_full_size_sweep_ends(rn, dt, M, N):
    """The sweep's extreme points at full size: the per-head norm (N = 128,
    M = 16384 * 32 rows: each persistent CTA adds thousands of rows into its
    fp32 dW partials) and the widest aligned row of the grid. Sampled rows of
    y, rstd and dx against the oracle, dW over every row."""
    d = inputs.make_inputs(M, N, dt, inputs.SWEEP_SEED)
    x, w, dy = (to_dev(d[k], dt) for k in ("x", "w", "dy"))
    y, rstd = rn.rmsnorm_fwd(x, w, eps=1e-6)
    r32 = _rstd32_all_rows(d["x"], d["w"], dt, 1e-6, chunk=max(1, (1 << 22) // N))
    dx, dw = rn.rmsnorm_bwd(dy, x, w, torch.from_numpy(r32).cuda(), eps=1e-6)
    torch.cuda.synchronize()
    assert rn.lib().rmsnorm_device_status(1) == 0
    rows = sampled_rows(M, k=256 if N <= 1024 else 48, seed=M % 97)
    rows_t = torch.from_numpy(rows).cuda()
    f = oracle.fwd(d["x"][rows], d["w"], dtype=dt, eps=1e-6, offset=0.0)
    check_y(to_host(y[rows_t], dt), f, dt)
    check_rstd(rstd.cpu().numpy()[rows], f["rstd64"])
    b = oracle.bwd(d["dy"][rows], d["x"][rows], d["w"], dtype=dt, eps=1e-6, offset=0.0, rstd=r32[rows])
    check_dx(to_host(dx[rows_t], dt), b, dt)
    full = oracle.bwd(d["dy"], d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0, rstd=r32, want_dx=False,
                      nthreads=8)
    check_dw(to_host(dw, dt), full, dt)


# ------------------------------------------------------------ non-affine --

@pytest.mark.parametrize("dt,M,N", [("bf16", 4096, 2048), ("f32", 300, 6144), ("bf16", 257, 16384),
                                    ("f32", 65, 16384), ("bf16", 211, 4097), ("bf16", 333, 128)])
@pytest.mark.parametrize("fused", [False, True])
def test_non_affine_matches_oracle(rn, dt, M, N, fused):
    """w absent: y = h rstd, dx = rstd (dy - xhat c), no dW."""
    d = inputs.make_inputs(M, N, dt, 110 + N % 7, residual=fused, dres=fused)
    x, dy = to_dev(d["x"], dt), to_dev(d["dy"], dt)
    if fused:
        y, h, rstd = rn.rmsnorm_add_fwd(x, to_dev(d["residual"], dt), None)
    else:
        y, rstd = rn.rmsnorm_fwd(x, None)
        h = x
    f = oracle.fwd(d["x"], None, dtype=dt, eps=1e-6, offset=0.0, residual=d.get("residual") if fused else None)
    torch.cuda.synchronize()
    check_y(to_host(y, dt), f, dt)
    check_rstd(rstd.cpu().numpy(), f["rstd64"])
    h_np = f["h"] if fused else d["x"]
    r32 = torch.from_numpy(f["rstd32"]).cuda()
    if fused:
        dx, dw = rn.rmsnorm_add_bwd(dy, to_dev(d["dres"], dt), to_dev(h_np, dt), None, r32)
    else:
        dx, dw = rn.rmsnorm_bwd(dy, h, None, r32)
    assert dw is None
    b = oracle.bwd(d["dy"], h_np, None, dtype=dt, eps=1e-6, offset=0.0, rstd=f["rstd32"],
                   dres=d.get("dres") if fused else None)
    torch.cuda.synchronize()
    check_dx(to_host(dx, dt), b, dt)



# ------------------------------------------------------------------ fp16 --

F16_SHAPES = [(333, 128), (4096, 2048), (300, 4096), (301, 5000), (257, 8192), (65, 16384), (33, 32768),
              (211, 4097), (9, 65536), (40, 3)]


@pytest.mark.parametrize("M,N", F16_SHAPES)
def test_f16_shapes(rn, M, N):
    d = inputs.make_inputs(M, N, "f16", 120 + N % 11)
    _fwd_bwd_check(rn, d, "f16", 1e-6, 0.0)


@pytest.mark.parametrize("M,N", [(4096, 4096), (1024, 8192)])
def test_f16_fused_add_gemma(rn, M, N):
    d = inputs.make_inputs(M, N, "f16", 121, w_mode="gemma", residual=True, dres=True)
    _fwd_bwd_check(rn, d, "f16", 1e-6, 1.0, fused=True)


def test_f16_misaligned(rn):
    d = inputs.make_inputs(1024, 7168, "f16", inputs.SWEEP_SEED)
    fp, bp = _fwd_bwd_check(rn, d, "f16", 1e-6, 0.0, offset_elems=1, expect_path="vector")
    assert fp["peel"] == 1 and bp["peel"] == 1
    _fwd_bwd_check(rn, d, "f16", 1e-6, 0.0, offset_elems=1, expect_path="generic", force_generic=True)


def test_f16_non_affine(rn):
    d = inputs.make_inputs(2048, 8192, "f16", 122)
    x, dy = to_dev(d["x"], "f16"), to_dev(d["dy"], "f16")
    y, rstd = rn.rmsnorm_fwd(x, None)
    f = oracle.fwd(d["x"], None, dtype="f16", eps=1e-6, offset=0.0)
    dx, dw = rn.rmsnorm_bwd(dy, x, None, torch.from_numpy(f["rstd32"]).cuda())
    b = oracle.bwd(d["dy"], d["x"], None, dtype="f16", eps=1e-6, offset=0.0, rstd=f["rstd32"])
    torch.cuda.synchronize()
    assert dw is None
    check_y(to_host(y, "f16"), f, "f16")
    check_dx(to_host(dx, "f16"), b, "f16")


# ---- fp32 weight beside 16-bit activations (w and dW stored in fp32) ----

@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("M,N", [(333, 64), (257, 1024), (300, 4096), (1031, 8192), (129, 12288), (65, 16384),
                                 (17, 65536), (101, 8193)])
def test_fp32_weight_shapes(rn, dt, M, N):
    d = inputs.make_inputs(M, N, dt, 140 + N % 13, wdtype="f32")
    exp = "generic" if N % 8 else "vector"
    _fwd_bwd_check(rn, d, dt, 1e-6, 0.0, wdt="f32", expect_path=exp)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_fp32_weight_fused_add_gemma(rn, dt):
    d = inputs.make_inputs(513, 4096, dt, 141, w_mode="gemma", residual=True, dres=True, wdtype="f32")
    _fwd_bwd_check(rn, d, dt, 1e-6, 1.0, fused=True, wdt="f32", expect_path="vector")


def test_fp32_weight_misaligned_takes_generic(rn):
    d = inputs.make_inputs(300, 2048, "bf16", 142, wdtype="f32")
    _fwd_bwd_check(rn, d, "bf16", 1e-6, 0.0, offset_elems=1, wdt="f32", expect_path="generic")


def test_fp32_weight_full_size(rn):
    """The bench's shape with an fp32 master weight, checked on sampled rows
    (y, dx) and on every column of dW against the oracle."""
    M, N = 16384, 8192
    d = inputs.make_inputs(M, N, "bf16", inputs.SWEEP_SEED, wdtype="f32", outlier_frac=0.01)
    x, dy = to_dev(d["x"], "bf16"), to_dev(d["dy"], "bf16")
    w = to_dev(d["w"], "f32")
    y, rstd = rn.rmsnorm_fwd(x, w)
    dx, dw = rn.rmsnorm_bwd(dy, x, w, rstd)
    assert dw.dtype == torch.float32
    torch.cuda.synchronize()
    rows = np.random.default_rng(7).choice(M, 256, replace=False)
    f = oracle.fwd(d["x"][rows], d["w"], dtype="bf16", eps=1e-6, offset=0.0, wdtype="f32")
    check_y(to_host(y, "bf16")[rows], f, "bf16")
    bs = oracle.bwd(d["dy"][rows], d["x"][rows], d["w"], dtype="bf16", eps=1e-6, offset=0.0,
                    rstd=rstd.cpu().numpy()[rows], wdtype="f32")
    check_dx(to_host(dx, "bf16")[rows], bs, "bf16")
    b = oracle.bwd(d["dy"], d["x"], d["w"], dtype="bf16", eps=1e-6, offset=0.0, rstd=rstd.cpu().numpy(),
                   want_dx=False, wdtype="f32")
    check_dw(to_host(dw, "f32"), b, "f32")


def test_fp32_weight_refuses_alternative_plans(rn):
    """Only the default plans are compiled with an fp32 weight: a forced
    alternative is refused before launch, the default runs."""
    d = inputs.make_inputs(64, 2048, "bf16", 143, wdtype="f32")
    x, w = to_dev(d["x"], "bf16"), to_dev(d["w"], "f32")
    default = rn.plan_query(rn.OP_FWD, 64, 2048, rn.RMSNORM_BF16)["plan_id"]
    defaults = {rn.plan_query(rn.OP_FWD, 64, n, t)["plan_id"] for n in range(8, 65537, 8) for t in (0, 1, 2)}
    alternatives = []
    for i in range(rn.lib().rmsnorm_plan_count()):
        pid = rn.lib().rmsnorm_plan_id_at(i)
        try:
            p = rn.plan_query(rn.OP_FWD, 64, 2048, rn.RMSNORM_BF16, force_plan=pid)
        except rn.RMSNormError:
            continue
        # (the register cluster plans stay table defaults, for the E4M3
        # outputs, and so are compiled for every pairing)
        if p["path_name"] == "vector" and p["cluster_size"] == 1 and pid not in defaults:
            alternatives.append(pid)
    assert alternatives
    for pid in alternatives:
        with pytest.raises(rn.RMSNormError):
            rn.rmsnorm_fwd_ex(x, w, force_plan=pid)
    y, _, _, plan = rn.rmsnorm_fwd_ex(x, w, force_plan=default)
    torch.cuda.synchronize()
    assert plan["plan_id"] == default


# ------------------------------------------- fp32 in, bf16 / fp16 out --

@pytest.mark.parametrize("odt", ["bf16", "f16"])
@pytest.mark.parametrize("M,N", [(333, 64), (257, 1024), (300, 4096), (129, 8192), (65, 16384), (33, 32768),
                                 (101, 4097), (40, 3)])
@pytest.mark.parametrize("fused", [False, True])
def test_fp32_in_narrow_out(rn, odt, M, N, fused):
    """fp32 activations and weight, y stored in bf16 or fp16 (rounded once
    from the fp32 result: within 1 ulp of the exact value rounded to the
    output type); rstd and the fp32 residual_out as for an fp32 forward.
    Register rows, staged cluster rows (N > 8192) and generic rows."""
    d = inputs.make_inputs(M, N, "f32", 420 + N % 13, residual=fused)
    x, w = to_dev(d["x"], "f32"), to_dev(d["w"], "f32")
    tdt = torch.bfloat16 if odt == "bf16" else torch.float16
    if fused:
        y, h, rstd, plan = rn.rmsnorm_fwd_ex(x, w, residual=to_dev(d["residual"], "f32"), out_dtype=tdt)
    else:
        y, _, rstd, plan = rn.rmsnorm_fwd_ex(x, w, out_dtype=tdt)
    f = oracle.fwd(d["x"], d["w"], dtype="f32", eps=1e-6, offset=0.0, residual=d.get("residual") if fused else None)
    torch.cuda.synchronize()
    assert y.dtype == tdt
    ref = {"y": oracle.bf16_round(f["y64"]) if odt == "bf16" else oracle.f16_round(f["y64"])}
    check_y(to_host(y, odt), ref, odt)
    check_rstd(rstd.cpu().numpy(), f["rstd64"])
    if fused:
        assert np.array_equal(to_host(h, "f32"), f["h"])
    expect = ("vector", "staged") if N % 4 == 0 else ("generic",)
    assert plan["path_name"] in expect, plan


def test_fp32_in_narrow_out_misaligned_and_refusals(rn):
    """y one element past an aligned allocation takes the generic kernel;
    the output flags are refused on 16-bit activations and by the backward."""
    d = inputs.make_inputs(200, 2048, "f32", 430)
    x, w = to_dev(d["x"], "f32"), to_dev(d["w"], "f32")
    y = empty_dev((200, 2048), "bf16", offset=1)
    _, _, rstd, plan = rn.rmsnorm_fwd_ex(x, w, y=y)
    f = oracle.fwd(d["x"], d["w"], dtype="f32", eps=1e-6, offset=0.0)
    torch.cuda.synchronize()
    assert plan["path_name"] == "generic"
    check_y(to_host(y, "bf16"), {"y": oracle.bf16_round(f["y64"])}, "bf16")
    L = rn.lib()
    xb = to_dev(d["x"], "bf16")
    assert L.rmsnorm_fwd(xb.data_ptr(), None, xb.data_ptr(), rstd.data_ptr(), 200, 2048,
                         rn.RMSNORM_BF16 | rn.RMSNORM_OUT_F16, 1e-6, 0.0, None) == 1
    assert L.rmsnorm_bwd(x.data_ptr(), x.data_ptr(), w.data_ptr(), rstd.data_ptr(), x.data_ptr(), w.data_ptr(),
                         None, 0, 200, 2048, rn.RMSNORM_F32 | rn.RMSNORM_OUT_BF16, 1e-6, 0.0, None) == 1
