"""GPU parity of LayerNorm forward and backward against the fp64 oracle.

The forward's y, mean and rstd are compared with the oracle's; the backward
is fed the oracle forward's fp32 mean and rstd (inputs of the backward), and
an end-to-end test runs both directions on the GPU against the exact
gradient. Shapes cover every LayerNorm plan family: sub-warp and multi-warp
teams, 512-thread rows, cluster rows, and the generic kernels.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import (check_dx, check_ln_stats, check_ln_y, check_param_grad, decode, empty_dev, to_dev,
                     to_host, cuda_bits_equal)
from row_wise_normalization_rmsnorm_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rn():
    from row_wise_normalization_rmsnorm_gb300 import build
    build.build()
    import row_wise_normalization_rmsnorm_gb300 as pkg
    return pkg


def _factor(d, dt, offset):
    return offset + oracle.to_f64(d["w"], dt) if d.get("w") is not None else np.ones(d["x"].shape[1])


def _ln_check(rn, d, dt, eps=1e-5, offset=0.0, fused=False, offset_elems=0, expect_path=None, gamma=True,
              beta=True, want_dgamma=True, want_dbeta=True, wdt=None):
    """offset_elems: one element offset for every array, or a dict of
    offsets by array name (x, gamma, beta, y, residual, residual_out, dy,
    dx, dgamma, dbeta, dres; missing names: 0). wdt: the storage type of
    gamma, beta and their gradients (default the activations')."""
    wdt = wdt or dt
    M, N = d["x"].shape
    offs = offset_elems if isinstance(offset_elems, dict) else None

    def o(name):
        return offs.get(name, 0) if offs is not None else offset_elems
    dg_np = d["w"] if gamma else None
    b_np = d.get("beta") if beta else None
    x = to_dev(d["x"], dt, offset=o("x"))
    g = to_dev(dg_np, wdt, offset=o("gamma")) if gamma else None
    b = to_dev(b_np, wdt, offset=o("beta")) if beta else None
    y = empty_dev((M, N), dt, offset=o("y"))
    res = to_dev(d["residual"], dt, offset=o("residual")) if fused else None
    hout = empty_dev((M, N), dt, offset=o("residual_out")) if fused else None
    out = rn.layernorm_fwd(x, g, b, residual=res, residual_out=hout, y=y, eps=eps, offset=offset)
    f = oracle.ln_fwd(d["x"], dg_np, b_np, dtype=dt, eps=eps, offset=offset,
                      residual=d.get("residual") if fused else None, wdtype=wdt)
    torch.cuda.synchronize()
    h_np = f["h"] if fused else d["x"]
    h64 = oracle.to_f64(h_np, dt)
    factor = (offset + oracle.to_f64(dg_np, wdt)) if gamma else np.ones(N)
    bias = oracle.to_f64(b_np, wdt) if beta else np.zeros(N)
    check_ln_y(to_host(y, dt), f, dt, h64, factor, bias)
    check_ln_stats(out["mean"].cpu().numpy(), out["rstd"].cpu().numpy(), f, h64)
    if fused:
        assert np.array_equal(to_host(hout, dt), f["h"])

    # backward, fed the oracle's fp32 statistics
    m32 = torch.from_numpy(f["mean32"]).cuda()
    r32 = torch.from_numpy(f["rstd32"]).cuda()
    hdev = to_dev(h_np, dt, offset=o("x"))
    dy = to_dev(d["dy"], dt, offset=o("dy"))
    dx = empty_dev((M, N), dt, offset=o("dx"))
    dgam = empty_dev((N,), wdt, offset=o("dgamma")) if (gamma and want_dgamma) else None
    dbet = empty_dev((N,), wdt, offset=o("dbeta")) if want_dbeta else None
    dres_np = d.get("dres") if fused else None
    dres = to_dev(dres_np, dt, offset=o("dres")) if dres_np is not None else None
    bo = rn.layernorm_bwd(dy, hdev, g, m32, r32, dresidual_out=dres, eps=eps, offset=offset, dx=dx, dgamma=dgam,
                          dbeta=dbet, want_dgamma=want_dgamma, want_dbeta=want_dbeta)
    r = oracle.ln_bwd(d["dy"], h_np, dg_np, dtype=dt, eps=eps, offset=offset, mean=f["mean32"],
                      rstd=f["rstd32"], dres=dres_np, wdtype=wdt)
    torch.cuda.synchronize()
    needed = check_dx(to_host(dx, dt), r, dt)
    if dgam is not None:
        check_param_grad(to_host(dgam, wdt), r["dg64"], r["dg_abs"], wdt)
    if dbet is not None:
        check_param_grad(to_host(dbet, wdt), r["db64"], r["db_abs"], wdt)
    if expect_path is not None:
        # "vector": the fast paths (the backward may stage rows in shared memory)
        fast = ("vector", "staged") if expect_path == "vector" else (expect_path,)
        assert out["plan"]["path_name"] in fast and bo["plan"]["path_name"] in fast
    return out, bo


SHAPES = [(333, 64), (257, 1024), (300, 4096), (129, 8192), (65, 16384), (101, 8193), (40, 3), (5, 1)]


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("M,N", SHAPES)
def test_ln_shapes(rn, dt, M, N):
    d = inputs.make_inputs(M, N, dt, 170 + N % 19, beta=True, x_shift=0.5)
    es = 4 if dt == "f32" else 2
    _ln_check(rn, d, dt, expect_path="vector" if (N * es) % 16 == 0 else "generic")


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("M,N", [(333, 64), (257, 1024), (300, 4096), (129, 8192), (65, 16384), (33, 32768),
                                 (101, 8193), (40, 3), (200, 12288), (77, 2048)])
@pytest.mark.parametrize("fused", [False, True])
def test_ln_fp32_params(rn, dt, M, N, fused):
    """gamma, beta, dgamma and dbeta in fp32 beside 16-bit activations, on
    register, staged (held and re-read schedules), cluster and generic rows."""
    d = inputs.make_inputs(M, N, dt, 175 + N % 23, beta=True, x_shift=0.5, wdtype="f32", residual=fused,
                           dres=fused)
    _ln_check(rn, d, dt, fused=fused, expect_path="vector" if (N * 2) % 16 == 0 else "generic", wdt="f32")


def test_ln_fp32_params_partial_outputs_and_alignment(rn):
    """No gamma (dbeta alone), dgamma without dbeta, and a misaligned x,
    which takes the generic kernels with fp32 parameters."""
    d = inputs.make_inputs(300, 4096, "bf16", 176, beta=True, wdtype="f32")
    _ln_check(rn, d, "bf16", gamma=False, wdt="f32")
    _ln_check(rn, d, "bf16", want_dbeta=False, wdt="f32")
    _ln_check(rn, d, "bf16", offset_elems={"x": 1, "y": 1, "dy": 1, "dx": 1}, expect_path="generic", wdt="f32")


@pytest.mark.parametrize("dt,N", [("bf16", 32768), ("bf16", 65536), ("f32", 16384), ("f32", 32768)])
def test_ln_cluster_rows(rn, dt, N):
    d = inputs.make_inputs(33, N, dt, 171, beta=True, x_shift=0.25)
    _, bo = _ln_check(rn, d, dt, expect_path="vector")
    assert bo["plan"]["cluster_size"] > 1


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
def test_ln_fused_add_gemma(rn, dt):
    d = inputs.make_inputs(513, 4096, dt, 172, w_mode="gemma", residual=True, dres=True, beta=True)
    _ln_check(rn, d, dt, offset=1.0, fused=True, expect_path="vector")


@pytest.mark.parametrize("gamma,beta,want_dgamma,want_dbeta", [(False, False, False, False), (True, False, True, True),
                                                                (False, True, False, True), (True, True, False, True),
                                                                (True, True, True, False), (True, True, False, False)])
def test_ln_optional_parameters(rn, gamma, beta, want_dgamma, want_dbeta):
    d = inputs.make_inputs(300, 2048, "bf16", 173, beta=True, x_shift=1.0)
    _ln_check(rn, d, "bf16", gamma=gamma, beta=beta, want_dgamma=want_dgamma, want_dbeta=want_dbeta,
              expect_path="vector")


@pytest.mark.parametrize("dt,M,N,k", [("bf16", 257, 2048, 1), ("bf16", 300, 7168, 3), ("bf16", 129, 8192, 7),
                                      ("bf16", 33, 32768, 2), ("f32", 200, 4096, 1), ("f16", 77, 128, 5)])
@pytest.mark.parametrize("fused", [False, True])
def test_ln_common_offset_takes_fast_kernels(rn, dt, M, N, k, fused):
    """Every array k elements past a 16-byte boundary: the vectorised
    LayerNorm kernels with each row's head and tail joined into one chunk."""
    d = inputs.make_inputs(M, N, dt, 174 + k, beta=True, x_shift=0.5, residual=fused, dres=fused)
    out, bo = _ln_check(rn, d, dt, fused=fused, offset_elems=k, expect_path="vector")
    assert out["plan"]["peel"] == k and bo["plan"]["peel"] == k


@pytest.mark.parametrize("dt,M,N", [("bf16", 160, 7169), ("bf16", 96, 10247), ("f32", 96, 5111)])
@pytest.mark.parametrize("fused", [False, True])
def test_ln_generic_backward_row_cache_both_sides_of_its_limit(rn, dt, M, N, fused):
    """x and dy of the row in shared memory where both fit 40 KB (slots of
    (N es + 31) // 16 * 16 bytes), global re-reads beyond; the oracle's
    result either way, and the plan reports the cache it took."""
    d = inputs.make_inputs(M, N, dt, 340 + N % 5, beta=True, residual=fused, dres=fused)
    _, bo = _ln_check(rn, d, dt, fused=fused, offset_elems=1, expect_path="generic")
    es = 4 if dt == "f32" else 2
    slot = (N * es + 31) // 16 * 16
    assert bo["plan"]["smem_bytes"] == (2 * slot if 2 * slot <= 40 * 1024 else 0), bo["plan"]


@pytest.mark.parametrize("dt,M,N,offs", [
    ("bf16", 129, 4099, {"x": 3, "gamma": 3, "beta": 1, "y": 3, "dy": 3, "dx": 3, "dgamma": 1}),
    ("f32", 100, 1030, {"x": 1, "gamma": 2, "beta": 1, "y": 1, "dy": 1, "dx": 1, "dbeta": 3}),
    ("bf16", 64, 6, {"x": 1, "gamma": 1, "beta": 1, "y": 1, "dy": 1, "dx": 1}),
    ("f16", 80, 2048, {"x": 1, "y": 2, "dy": 3, "dx": 0}),
])
@pytest.mark.parametrize("fused", [False, True])
def test_ln_generic_peeled_and_scalar_rows(rn, dt, M, N, offs, fused):
    """Generic LayerNorm rows split into a scalar head, 16-byte chunks and a
    scalar tail (the arrays share their address mod 16; gamma and beta may
    not) or not split (they do not share it), against the oracle."""
    d = inputs.make_inputs(M, N, dt, 320 + N % 13, beta=True, residual=fused, dres=fused)
    if fused:
        offs = dict(offs, residual=offs.get("x", 0), residual_out=offs.get("x", 0), dres=offs.get("dy", 0))
    _ln_check(rn, d, dt, fused=fused, offset_elems=offs, expect_path="generic")


def test_ln_large_mean_two_pass_variance(rn):
    # rows with mean 300 and unit spread: a one-pass E[x^2] - E[x]^2 in fp32
    # would lose most of the variance's bits
    d = inputs.make_inputs(256, 4096, "f32", 175, x_shift=300.0, beta=True)
    _ln_check(rn, d, "f32", expect_path="vector")


def test_ln_end_to_end_against_exact_gradient(rn):
    for dt, M, N in (("bf16", 1024, 8192), ("f32", 512, 4096)):
        d = inputs.make_inputs(M, N, dt, 176, beta=True, x_shift=0.5)
        x, g, b, dy = (to_dev(d[k], dt) for k in ("x", "w", "beta", "dy"))
        out = rn.layernorm_fwd(x, g, b)
        bo = rn.layernorm_bwd(dy, x, g, out["mean"], out["rstd"])
        torch.cuda.synchronize()
        r = oracle.ln_bwd(d["dy"], d["x"], d["w"], dtype=dt, eps=1e-5, offset=0.0)
        # the GPU's statistics carry fp32 error: the floor grows accordingly
        check_dx(to_host(bo["dx"], dt), r, dt, floor_mult=4.0)
        check_param_grad(to_host(bo["dgamma"], dt), r["dg64"], r["dg_abs"], dt)
        check_param_grad(to_host(bo["dbeta"], dt), r["db64"], r["db_abs"], dt)


def test_ln_full_size_sampled(rn):
    M, N = 16384, 8192
    d = inputs.make_inputs(M, N, "bf16", inputs.SWEEP_SEED, beta=True, x_shift=0.5, outlier_frac=0.01)
    x, g, b, dy = (to_dev(d[k], "bf16") for k in ("x", "w", "beta", "dy"))
    out = rn.layernorm_fwd(x, g, b)
    bo = rn.layernorm_bwd(dy, x, g, out["mean"], out["rstd"])
    torch.cuda.synchronize()
    rows = np.random.default_rng(11).choice(M, 256, replace=False)
    f = oracle.ln_fwd(d["x"][rows], d["w"], d["beta"], dtype="bf16", eps=1e-5, offset=0.0)
    h64 = oracle.to_f64(d["x"][rows], "bf16")
    check_ln_y(to_host(out["y"], "bf16")[rows], f, "bf16", h64, oracle.to_f64(d["w"], "bf16"),
               oracle.to_f64(d["beta"], "bf16"))
    check_ln_stats(out["mean"].cpu().numpy()[rows], out["rstd"].cpu().numpy()[rows], f, h64)
    m, r_ = out["mean"].cpu().numpy(), out["rstd"].cpu().numpy()
    rs = oracle.ln_bwd(d["dy"][rows], d["x"][rows], d["w"], dtype="bf16", eps=1e-5, offset=0.0, mean=m[rows],
                       rstd=r_[rows])
    check_dx(to_host(bo["dx"], "bf16")[rows], rs, "bf16")
    full = oracle.ln_bwd(d["dy"], d["x"], d["w"], dtype="bf16", eps=1e-5, offset=0.0, mean=m, rstd=r_,
                         want_dx=False, nthreads=8)
    check_param_grad(to_host(bo["dgamma"], "bf16"), full["dg64"], full["dg_abs"], "bf16")
    check_param_grad(to_host(bo["dbeta"], "bf16"), full["db64"], full["db_abs"], "bf16")
    assert bo["plan"]["path_name"] in ("vector", "staged")


def test_ln_dx_independent_of_cta_count(rn):
    d = inputs.make_inputs(2048, 2048, "bf16", 177, beta=True)
    x, g, dy = (to_dev(d[k], "bf16") for k in ("x", "w", "dy"))
    out = rn.layernorm_fwd(x, g, None)
    a = rn.layernorm_bwd(dy, x, g, out["mean"], out["rstd"], force_ctas=37)
    b = rn.layernorm_bwd(dy, x, g, out["mean"], out["rstd"], force_ctas=152)
    torch.cuda.synchronize()
    assert a["plan"]["ctas"] == 37 and b["plan"]["ctas"] == 152
    assert cuda_bits_equal(a["dx"], b["dx"])
    da, db = a["dgamma"].float(), b["dgamma"].float()
    assert torch.allclose(da, db, rtol=8e-3, atol=1e-3)


def test_ln_fused_forward_equals_plain_forward_on_rounded_sum(rn):
    d = inputs.make_inputs(300, 4096, "bf16", 178, residual=True, beta=True)
    x, r, g, b = (to_dev(d[k], "bf16") for k in ("x", "residual", "w", "beta"))
    fo = rn.layernorm_fwd(x, g, b, residual=r)
    po = rn.layernorm_fwd(fo["residual_out"].clone(), g, b)
    torch.cuda.synchronize()
    assert cuda_bits_equal(fo["y"], po["y"]) and cuda_bits_equal(fo["rstd"], po["rstd"])
    assert cuda_bits_equal(fo["mean"], po["mean"])


def test_ln_empty_batch_zeroes_parameter_grads(rn):
    x = torch.empty((0, 512), dtype=torch.bfloat16, device="cuda")
    g = torch.ones(512, dtype=torch.bfloat16, device="cuda")
    m = torch.empty(0, device="cuda")
    dg = torch.full((512,), 3.0, dtype=torch.bfloat16, device="cuda")
    db = torch.full((512,), 3.0, dtype=torch.bfloat16, device="cuda")
    rn.layernorm_bwd(x, x, g, m, m, dgamma=dg, dbeta=db)
    torch.cuda.synchronize()
    assert torch.all(dg == 0) and torch.all(db == 0)


@pytest.mark.parametrize("M,N,staged,vector", [(2049, 4096, 100, 82), (999, 8192, 99, 76), (300, 12288, 101, 86),
                                               (777, 8192, 112, 76)])
def test_ln_staged_backward_matches_register_backward(rn, M, N, staged, vector):
    """The staged LayerNorm backward does the register kernel's arithmetic:
    on the same chunk mapping dx is bit-identical (dgamma and dbeta differ
    only in how partial rows are grouped); on another mapping the row sums
    associate differently and the results agree to rounding."""
    d = inputs.make_inputs(M, N, "bf16", 195, beta=True, x_shift=0.5)
    x, g, b, dy = (to_dev(d[k], "bf16") for k in ("x", "w", "beta", "dy"))
    out = rn.layernorm_fwd(x, g, b)
    a = rn.layernorm_bwd(dy, x, g, out["mean"], out["rstd"], force_plan=staged)
    v = rn.layernorm_bwd(dy, x, g, out["mean"], out["rstd"], force_plan=vector)
    torch.cuda.synchronize()
    assert a["plan"]["path_name"] == "staged" and v["plan"]["path_name"] == "vector"
    same_mapping = (v["plan"]["cluster_size"] == 1 and
                    (a["plan"]["threads_per_row"], a["plan"]["chunks_per_thread"]) ==
                    (v["plan"]["threads_per_row"], v["plan"]["chunks_per_thread"]))
    if same_mapping:
        assert cuda_bits_equal(a["dx"], v["dx"])
    else:
        assert torch.allclose(a["dx"].float(), v["dx"].float(), rtol=1e-2, atol=1e-2)
    assert torch.allclose(a["dgamma"].float(), v["dgamma"].float(), rtol=1e-2, atol=1e-2)
    assert torch.allclose(a["dbeta"].float(), v["dbeta"].float(), rtol=1e-2, atol=1e-2)
    assert rn.lib().rmsnorm_device_status(1) == 0


@pytest.mark.parametrize("M,N,reread,held", [(1001, 16384, 116, 102), (300, 8192, 115, 102), (517, 12288, 122, 101),
                                             (777, 8192, 120, 99), (45, 6144, 120, 99)])
@pytest.mark.parametrize("fused", [False, True])
def test_ln_reread_staged_backward_matches_held_bitwise(rn, M, N, reread, held, fused):
    """The LayerNorm backward's re-read staged schedule (chunks read from
    the stage in each pass, so the two parameter-gradient accumulators fit
    in registers) gives the held schedule's dx, dgamma and dbeta bit for bit
    on the same geometry and number of partial rows."""
    d = inputs.make_inputs(M, N, "bf16", 240 + N % 7, beta=True, x_shift=0.5, residual=fused, dres=fused)
    x, g, b, dy = (to_dev(d[k], "bf16") for k in ("x", "w", "beta", "dy"))
    dres = to_dev(d["dres"], "bf16") if fused else None
    out = rn.layernorm_fwd(x, g, b)
    a = rn.layernorm_bwd(dy, x, g, out["mean"], out["rstd"], dresidual_out=dres, force_plan=reread,
                         force_ctas=100)
    v = rn.layernorm_bwd(dy, x, g, out["mean"], out["rstd"], dresidual_out=dres, force_plan=held,
                         force_ctas=100)
    torch.cuda.synchronize()
    assert a["plan"]["plan_id"] == reread and a["plan"]["path_name"] == "staged"
    assert a["plan"]["ctas"] == v["plan"]["ctas"] == min(100, M)
    for k in ("dx", "dgamma", "dbeta"):
        assert cuda_bits_equal(a[k], v[k]), k
    assert rn.lib().rmsnorm_device_status(1) == 0


@pytest.mark.parametrize("plan,N", [(115, 12288), (116, 16384), (117, 12288), (120, 8192), (122, 10240), (129, 20488),
                                    (130, 40968)])
def test_ln_forced_reread_plans_match_oracle(rn, plan, N):
    M, dt = 203, "bf16"
    d = inputs.make_inputs(M, N, dt, 250 + plan, beta=True, x_shift=0.5)
    x, g, b, dy = (to_dev(d[k], dt) for k in ("x", "w", "beta", "dy"))
    f = oracle.ln_fwd(d["x"], d["w"], d["beta"], dtype=dt, eps=1e-5, offset=0.0)
    mean = torch.from_numpy(f["mean32"]).cuda()
    rstd = torch.from_numpy(f["rstd32"]).cuda()
    o = rn.layernorm_bwd(dy, x, g, mean, rstd, force_plan=plan)
    assert o["plan"]["plan_id"] == plan
    r = oracle.ln_bwd(d["dy"], d["x"], d["w"], dtype=dt, eps=1e-5, offset=0.0, mean=f["mean32"], rstd=f["rstd32"])
    torch.cuda.synchronize()
    check_dx(to_host(o["dx"], dt), r, dt)
    check_param_grad(to_host(o["dgamma"], dt), r["dg64"], r["dg_abs"], dt)
    check_param_grad(to_host(o["dbeta"], dt), r["db64"], r["db_abs"], dt)


@pytest.mark.parametrize("M,N,cluster", [(301, 16384, 125), (90, 12288, 126), (50, 24, 126)])
@pytest.mark.parametrize("fused", [False, True])
def test_ln_cluster_staged_rows_independent_of_partial_rows(rn, M, N, cluster, fused):
    """The LayerNorm backward on a cluster of staged CTAs: dx keeps its bits
    over another number of partial rows, and dgamma, dbeta agree."""
    d = inputs.make_inputs(M, N, "bf16", 360 + N % 7, beta=True, x_shift=0.5, residual=fused, dres=fused)
    x, g, b, dy = (to_dev(d[k], "bf16") for k in ("x", "w", "beta", "dy"))
    dres = to_dev(d["dres"], "bf16") if fused else None
    out = rn.layernorm_fwd(x, g, b)
    a = rn.layernorm_bwd(dy, x, g, out["mean"], out["rstd"], dresidual_out=dres, force_plan=cluster, force_ctas=30)
    v = rn.layernorm_bwd(dy, x, g, out["mean"], out["rstd"], dresidual_out=dres, force_plan=cluster, force_ctas=7)
    torch.cuda.synchronize()
    assert a["plan"]["cluster_size"] > 1 and a["plan"]["ws_rows"] == 30 and v["plan"]["ws_rows"] == 7
    assert cuda_bits_equal(a["dx"], v["dx"])
    for k in ("dgamma", "dbeta"):
        assert torch.allclose(a[k].float(), v[k].float(), rtol=1e-2, atol=1e-2), k
    assert rn.lib().rmsnorm_device_status(1) == 0


@pytest.mark.parametrize("dt,M,N,plan", [("bf16", 101, 20488, 125), ("f32", 64, 16384, 125), ("bf16", 33, 40968, 126),
                                         ("bf16", 77, 8192, 125), ("f32", 29, 12, 126)])
@pytest.mark.parametrize("fused", [False, True])
def test_ln_cluster_staged_wide_rows_match_oracle(rn, dt, M, N, plan, fused):
    d = inputs.make_inputs(M, N, dt, 370 + N % 13, beta=True, x_shift=0.5, residual=fused, dres=fused)
    x, g, dy = (to_dev(d[k], dt) for k in ("x", "w", "dy"))
    dres = to_dev(d["dres"], dt) if fused else None
    f = oracle.ln_fwd(d["x"], d["w"], d["beta"], dtype=dt, eps=1e-5, offset=0.0)
    mean = torch.from_numpy(f["mean32"]).cuda()
    rstd = torch.from_numpy(f["rstd32"]).cuda()
    o = rn.layernorm_bwd(dy, x, g, mean, rstd, dresidual_out=dres, force_plan=plan)
    assert o["plan"]["plan_id"] == plan
    r = oracle.ln_bwd(d["dy"], d["x"], d["w"], dtype=dt, eps=1e-5, offset=0.0, mean=f["mean32"], rstd=f["rstd32"],
                      dres=d.get("dres") if fused else None)
    torch.cuda.synchronize()
    check_dx(to_host(o["dx"], dt), r, dt)
    check_param_grad(to_host(o["dgamma"], dt), r["dg64"], r["dg_abs"], dt)
    check_param_grad(to_host(o["dbeta"], dt), r["db64"], r["db_abs"], dt)
    assert rn.lib().rmsnorm_device_status(1) == 0



@pytest.mark.parametrize("dt,M,N,staged,vector", [("bf16", 97, 32768, 139, 17), ("bf16", 130, 20480, 139, 17),
                                                  ("bf16", 33, 65536, 143, 18), ("f32", 100, 8192, 138, 8),
                                                  ("f16", 64, 12288, 138, 8)])
@pytest.mark.parametrize("fused", [False, True])
def test_ln_staged_forward_matches_register_forward_bitwise(rn, dt, M, N, staged, vector, fused):
    """The staged LayerNorm forward (a sum, squared deviations, y, each a pass
    over the row's shared-memory stage) gives the register forward's y, mean
    and rstd bits for the same geometry."""
    d = inputs.make_inputs(M, N, dt, 400 + N % 7, beta=True, x_shift=0.5, residual=fused)
    x, g, b = (to_dev(d[k], dt) for k in ("x", "w", "beta"))
    res = to_dev(d["residual"], dt) if fused else None
    kw = dict(residual=res)
    a = rn.layernorm_fwd(x, g, b, residual_out=torch.empty_like(x) if fused else None, force_plan=staged, **kw)
    v = rn.layernorm_fwd(x, g, b, residual_out=torch.empty_like(x) if fused else None, force_plan=vector, **kw)
    torch.cuda.synchronize()
    assert a["plan"]["plan_id"] == staged and a["plan"]["path_name"] == "staged"
    for k in ("y", "mean", "rstd") + (("residual_out",) if fused else ()):
        assert cuda_bits_equal(a[k], v[k]), k
    assert rn.lib().rmsnorm_device_status(1) == 0


@pytest.mark.parametrize("dt,M,N,plan", [("bf16", 150, 20488, 141), ("bf16", 40, 40968, 145), ("f32", 9, 12, 143)])
@pytest.mark.parametrize("fused", [False, True])
def test_ln_staged_forward_matches_oracle(rn, dt, M, N, plan, fused):
    d = inputs.make_inputs(M, N, dt, 410 + N % 5, beta=True, x_shift=0.5, residual=fused)
    x, g, b = (to_dev(d[k], dt) for k in ("x", "w", "beta"))
    res = to_dev(d["residual"], dt) if fused else None
    out = rn.layernorm_fwd(x, g, b, residual=res, residual_out=torch.empty_like(x) if fused else None,
                           force_plan=plan)
    f = oracle.ln_fwd(d["x"], d["w"], d["beta"], dtype=dt, eps=1e-5, offset=0.0,
                      residual=d.get("residual") if fused else None)
    torch.cuda.synchronize()
    assert out["plan"]["plan_id"] == plan
    h64 = oracle.to_f64(f["h"] if fused else d["x"], dt)
    check_ln_y(to_host(out["y"], dt), f, dt, h64, oracle.to_f64(d["w"], dt), oracle.to_f64(d["beta"], dt))
    check_ln_stats(out["mean"].cpu().numpy(), out["rstd"].cpu().numpy(), f, h64)
    if fused:
        assert np.array_equal(to_host(out["residual_out"], dt), f["h"])
    assert rn.lib().rmsnorm_device_status(1) == 0


@pytest.mark.parametrize("dt,N", [("bf16", 8192), ("bf16", 16384), ("bf16", 32768), ("f32", 12288), ("bf16", 7169)])
def test_ln_in_place_aliasing(rn, dt, N):
    """y may be x, residual_out may be residual, dx may be dy (and
    dresidual_out): the in-place calls give the out-of-place bits on every
    path (register, staged, cluster staged, generic)."""
    M = 300
    d = inputs.make_inputs(M, N, dt, 430 + N % 11, beta=True, residual=True, dres=True)
    x, g, b, r, dy, dr = (to_dev(d[k], dt) for k in ("x", "w", "beta", "residual", "dy", "dres"))
    o = rn.layernorm_fwd(x, g, b)
    xa = x.clone()
    rn.layernorm_fwd(xa, g, b, y=xa)
    of = rn.layernorm_fwd(x, g, b, residual=r, residual_out=torch.empty_like(x))
    ra = r.clone()
    rn.layernorm_fwd(x, g, b, residual=ra, residual_out=ra)
    bo = rn.layernorm_bwd(dy, x, g, o["mean"], o["rstd"])
    dya = dy.clone()
    rn.layernorm_bwd(dya, x, g, o["mean"], o["rstd"], dx=dya)
    bf = rn.layernorm_bwd(dy, x, g, o["mean"], o["rstd"], dresidual_out=dr)
    dra = dr.clone()
    rn.layernorm_bwd(dy, x, g, o["mean"], o["rstd"], dresidual_out=dra, dx=dra)
    torch.cuda.synchronize()
    assert cuda_bits_equal(xa, o["y"]) and cuda_bits_equal(ra, of["residual_out"])
    assert cuda_bits_equal(dya, bo["dx"]) and cuda_bits_equal(dra, bf["dx"])

