"""GPU launch-variant tests: where two launches use the same association of
every sum, their results must be identical bit for bit (packed vs scalar
arithmetic, CUDA-graph replay vs direct launch, default vs side stream,
concurrent streams with their own workspaces, poisoned vs clean workspace,
different batch sizes and batch splits, fused add vs plain on the rounded
sum). Also: in-place aliasing, guard regions, M == 0 and status codes.
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


def dev_inputs(M, N, dt, seed, **kw):
    d = inputs.make_inputs(M, N, dt, seed, **kw)
    return d, {k: to_dev(v, dt) for k, v in d.items()}


@pytest.mark.parametrize("dt,M,N", [("bf16", 2048, 8192), ("f32", 1024, 6144), ("bf16", 999, 128),
                                    ("bf16", 500, 2048), ("f32", 300, 16), ("bf16", 300, 16384),
                                    ("f32", 200, 16384), ("f16", 1000, 8192), ("f16", 300, 16384)])
@pytest.mark.parametrize("fused", [False, True])
def test_packed_matches_scalar_bitwise(rn, dt, M, N, fused):
    _, t = dev_inputs(M, N, dt, 90, residual=fused, dres=fused)
    _, rstd = rn.rmsnorm_fwd(t["x"], t["w"])
    # the register kernel of the same geometry where the default is staged
    # (the staged kernel has the packed variant only)
    code = {"bf16": rn.RMSNORM_BF16, "f32": rn.RMSNORM_F32, "f16": rn.RMSNORM_F16}[dt]
    default = rn.plan_query(rn.OP_BWD, M, N, code)
    plan = {88: 27, 95: 26, 121: 42, 118: 45, 127: 46, 123: 46, 128: 47, 124: 47}.get(default["plan_id"], -1) if default["path_name"] == "staged" else -1
    kw = dict(dresidual_out=t.get("dres"), fused=fused, force_plan=plan)
    dx1, dw1, p1 = rn.rmsnorm_bwd_ex(t["dy"], t["x"], t["w"], rstd, force_packed=1, **kw)
    dx0, dw0, p0 = rn.rmsnorm_bwd_ex(t["dy"], t["x"], t["w"], rstd, force_packed=0, **kw)
    assert p1["path_name"] == "vector"
    assert p1["packed"] == 1 and p0["packed"] == 0 and p1["plan_id"] == p0["plan_id"]
    assert p1["ctas"] == p0["ctas"]
    assert cuda_bits_equal(dx1, dx0) and cuda_bits_equal(dw1, dw0)


@pytest.mark.parametrize("dt,M,N", [("bf16", 600, 8192), ("bf16", 400, 16384), ("f32", 500, 6144), ("f32", 300, 2048),
                                    ("bf16", 200, 32768), ("bf16", 300, 4096)])
@pytest.mark.parametrize("fused", [False, True])
def test_staged_packed_matches_scalar_bitwise(rn, dt, M, N, fused):
    """The staged backward's packed f32x2 arithmetic and its scalar variant
    (same pairing, same CTA count) give the same bits, on the held and
    re-read schedules and on cluster rows; fp16 refuses the scalar one."""
    _, t = dev_inputs(M, N, dt, 93, residual=fused, dres=fused)
    _, rstd = rn.rmsnorm_fwd(t["x"], t["w"])
    kw = dict(dresidual_out=t.get("dres"), fused=fused)
    dx1, dw1, p1 = rn.rmsnorm_bwd_ex(t["dy"], t["x"], t["w"], rstd, force_packed=1, **kw)
    dx0, dw0, p0 = rn.rmsnorm_bwd_ex(t["dy"], t["x"], t["w"], rstd, force_packed=0, **kw)
    torch.cuda.synchronize()
    assert p1["path_name"] == p0["path_name"] == "staged" and p1["plan_id"] == p0["plan_id"]
    assert p1["packed"] == 1 and p0["packed"] == 0 and p1["ctas"] == p0["ctas"]
    assert cuda_bits_equal(dx1, dx0) and cuda_bits_equal(dw1, dw0)
    _, h = dev_inputs(64, 8192, "f16", 94)
    _, r16 = rn.rmsnorm_fwd(h["x"], h["w"])
    with pytest.raises(rn.RMSNormError):
        rn.rmsnorm_bwd_ex(h["dy"], h["x"], h["w"], r16, force_packed=0)


def test_graph_replay_matches_direct(rn):
    _, t = dev_inputs(1000, 4096, "bf16", 91)
    ws = torch.empty(rn.rmsnorm_bwd_workspace_bytes(1000, 4096, torch.bfloat16), dtype=torch.uint8, device="cuda")
    y0, r0 = rn.rmsnorm_fwd(t["x"], t["w"])
    dx0, dw0 = rn.rmsnorm_bwd(t["dy"], t["x"], t["w"], r0, workspace=ws)
    y, r, dx, dw = (torch.empty_like(a) for a in (y0, r0, dx0, dw0))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            rn.rmsnorm_fwd(t["x"], t["w"], y=y, rstd=r)
            rn.rmsnorm_bwd(t["dy"], t["x"], t["w"], r, dx=dx, dw=dw, workspace=ws)
    for a in (y, r, dx, dw):
        a.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert cuda_bits_equal(y, y0) and cuda_bits_equal(r, r0)
    assert cuda_bits_equal(dx, dx0) and cuda_bits_equal(dw, dw0)


def test_side_streams_concurrent_match_serial(rn):
    M, N, dt = 4096, 2048, "bf16"
    _, a = dev_inputs(M, N, dt, 92)
    _, b = dev_inputs(M, N, dt, 93)
    ya, ra = rn.rmsnorm_fwd(a["x"], a["w"])
    yb, rb = rn.rmsnorm_fwd(b["x"], b["w"])
    dxa, dwa = rn.rmsnorm_bwd(a["dy"], a["x"], a["w"], ra)
    dxb, dwb = rn.rmsnorm_bwd(b["dy"], b["x"], b["w"], rb)
    nb = rn.rmsnorm_bwd_workspace_bytes(M, N, torch.bfloat16)
    wsa = torch.empty(nb, dtype=torch.uint8, device="cuda")
    wsb = torch.empty(nb, dtype=torch.uint8, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    out = {}
    for _ in range(3):
        with torch.cuda.stream(s1):
            out["ya"] = rn.rmsnorm_fwd(a["x"], a["w"])
            out["ga"] = rn.rmsnorm_bwd(a["dy"], a["x"], a["w"], ra, workspace=wsa)
        with torch.cuda.stream(s2):
            out["yb"] = rn.rmsnorm_fwd(b["x"], b["w"])
            out["gb"] = rn.rmsnorm_bwd(b["dy"], b["x"], b["w"], rb, workspace=wsb)
    torch.cuda.synchronize()
    assert cuda_bits_equal(out["ya"][0], ya) and cuda_bits_equal(out["yb"][0], yb)
    assert cuda_bits_equal(out["ga"][0], dxa) and cuda_bits_equal(out["ga"][1], dwa)
    assert cuda_bits_equal(out["gb"][0], dxb) and cuda_bits_equal(out["gb"][1], dwb)


@pytest.mark.parametrize("dt,N", [("bf16", 8192), ("f32", 4097), ("bf16", 128)])
def test_workspace_poisoned_clean_and_null(rn, dt, N):
    M = 1500
    _, t = dev_inputs(M, N, dt, 94)
    _, rstd = rn.rmsnorm_fwd(t["x"], t["w"])
    nb = rn.rmsnorm_bwd_workspace_bytes(M, N, t["x"].dtype)
    assert nb > 0
    nan_ws = torch.full((nb,), 0xFF, dtype=torch.uint8, device="cuda")   # every fp32 word a NaN
    zero_ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    dx1, dw1 = rn.rmsnorm_bwd(t["dy"], t["x"], t["w"], rstd, workspace=nan_ws)
    dx2, dw2 = rn.rmsnorm_bwd(t["dy"], t["x"], t["w"], rstd, workspace=zero_ws)
    dx3, dw3 = rn.rmsnorm_bwd(t["dy"], t["x"], t["w"], rstd)
    torch.cuda.synchronize()
    assert not torch.isnan(dw1.float()).any()
    assert cuda_bits_equal(dw1, dw2) and cuda_bits_equal(dw1, dw3)
    assert cuda_bits_equal(dx1, dx2) and cuda_bits_equal(dx1, dx3)


@pytest.mark.parametrize("dt,N", [("bf16", 8192), ("bf16", 128), ("f32", 5000), ("bf16", 4097),
                                  ("bf16", 16384), ("f32", 32768)])
def test_rows_independent_of_batch_and_split(rn, dt, N):
    M = 1234
    _, t = dev_inputs(M, N, dt, 95)
    y, r = rn.rmsnorm_fwd(t["x"], t["w"])
    dx, _ = rn.rmsnorm_bwd(t["dy"], t["x"], t["w"], r)
    cut = 517
    parts = []
    for lo, hi in ((0, cut), (cut, M)):
        yp, rp = rn.rmsnorm_fwd(t["x"][lo:hi], t["w"])
        dxp, _ = rn.rmsnorm_bwd(t["dy"][lo:hi], t["x"][lo:hi], t["w"], rp)
        parts.append((yp, rp, dxp))
    torch.cuda.synchronize()
    assert cuda_bits_equal(torch.cat([p[0] for p in parts]), y)
    assert cuda_bits_equal(torch.cat([p[1] for p in parts]), r)
    assert cuda_bits_equal(torch.cat([p[2] for p in parts]), dx)


@pytest.mark.parametrize("dt,N", [("bf16", 4096), ("f32", 2048), ("bf16", 5003)])
def test_fused_forward_equals_plain_on_rounded_sum(rn, dt, N):
    M = 700
    _, t = dev_inputs(M, N, dt, 96, residual=True)
    ya, h, ra = rn.rmsnorm_add_fwd(t["x"], t["residual"], t["w"])
    yp, rp = rn.rmsnorm_fwd(h.clone(), t["w"])
    torch.cuda.synchronize()
    assert cuda_bits_equal(ya, yp) and cuda_bits_equal(ra, rp)


def test_fused_backward_null_dres_equals_zero_buffer(rn):
    _, t = dev_inputs(800, 8192, "bf16", 97, residual=True)
    _, h, r = rn.rmsnorm_add_fwd(t["x"], t["residual"], t["w"])
    dx1, dw1 = rn.rmsnorm_add_bwd(t["dy"], None, h, t["w"], r)
    dx2, dw2 = rn.rmsnorm_add_bwd(t["dy"], torch.zeros_like(h), h, t["w"], r)
    dx3, dw3 = rn.rmsnorm_bwd(t["dy"], h, t["w"], r)
    torch.cuda.synchronize()
    assert cuda_bits_equal(dx1, dx2) and cuda_bits_equal(dw1, dw2)
    assert cuda_bits_equal(dx1, dx3) and cuda_bits_equal(dw1, dw3)


@pytest.mark.parametrize("dt,N", [("bf16", 8192), ("f32", 257), ("bf16", 64), ("bf16", 16384), ("f32", 12288),
                                  ("bf16", 32768), ("bf16", 7169)])
def test_in_place_aliasing(rn, dt, N):
    M = 640
    _, t = dev_inputs(M, N, dt, 98, residual=True, dres=True)
    y, r = rn.rmsnorm_fwd(t["x"], t["w"])
    dx, dw = rn.rmsnorm_bwd(t["dy"], t["x"], t["w"], r)
    xa = t["x"].clone()
    rn.rmsnorm_fwd(xa, t["w"], y=xa, rstd=torch.empty_like(r))          # y == x
    dya = t["dy"].clone()
    rn.rmsnorm_bwd(dya, t["x"], t["w"], r, dx=dya)                      # dx == dy
    ya, h, ra = rn.rmsnorm_add_fwd(t["x"], t["residual"], t["w"])
    res = t["residual"].clone()
    rn.rmsnorm_add_fwd(t["x"], res, t["w"], residual_out=res)           # residual_out == residual
    dxa, dwa = rn.rmsnorm_add_bwd(t["dy"], t["dres"], h, t["w"], ra)
    dr = t["dres"].clone()
    rn.rmsnorm_add_bwd(t["dy"], dr, h, t["w"], ra, dx=dr)               # dx == dresidual_out
    torch.cuda.synchronize()
    assert cuda_bits_equal(xa, y) and cuda_bits_equal(dya, dx)
    assert cuda_bits_equal(res, h) and cuda_bits_equal(dr, dxa)


@pytest.mark.parametrize("dt,N", [("bf16", 2048), ("bf16", 4097), ("f32", 130), ("bf16", 8192), ("f32", 6144)])
def test_guard_regions_untouched(rn, dt, N):
    M, G = 301, 4096
    d, t = dev_inputs(M, N, dt, 99)
    td = t["x"].dtype

    def guarded(n):
        buf = torch.full((G + n + G,), float("nan"), dtype=td, device="cuda")
        return buf, buf[G:G + n]

    ybuf, y = guarded(M * N)
    rbuf = torch.full((G + M + G,), float("nan"), device="cuda")
    r = rbuf[G:G + M]
    dxbuf, dx = guarded(M * N)
    dwbuf, dw = guarded(N)
    rn.rmsnorm_fwd(t["x"], t["w"], y=y.view(M, N), rstd=r)
    rn.rmsnorm_bwd(t["dy"], t["x"], t["w"], r, dx=dx.view(M, N), dw=dw)
    torch.cuda.synchronize()
    for buf, n in ((ybuf, M * N), (rbuf, M), (dxbuf, M * N), (dwbuf, N)):
        assert torch.isnan(buf[:G].float()).all() and torch.isnan(buf[G + n:].float()).all()
        assert not torch.isnan(buf[G:G + n].float()).any()


def test_zero_rows(rn):
    x = torch.empty((0, 1024), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(1024, dtype=torch.bfloat16, device="cuda")
    y, r = rn.rmsnorm_fwd(x, w)
    assert y.shape == (0, 1024) and r.shape == (0,)
    dw = torch.full((1024,), float("nan"), dtype=torch.bfloat16, device="cuda")
    rn.rmsnorm_bwd(x, x, w, r, dw=dw)
    torch.cuda.synchronize()
    assert (dw.float() == 0).all()          # the empty sum


def test_status_codes_on_device(rn):
    _, t = dev_inputs(64, 2048, "bf16", 100)
    _, r = rn.rmsnorm_fwd(t["x"], t["w"])
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(rn.RMSNormError) as e:
        rn.rmsnorm_bwd(t["dy"], t["x"], t["w"], r, workspace=small)
    assert e.value.status == 3
    with pytest.raises(rn.RMSNormError) as e:
        rn.rmsnorm_fwd_ex(t["x"], t["w"], force_plan=0)                 # plan too narrow for N
    assert e.value.status == 2


@pytest.mark.parametrize("plan", [7, 9, 10, 11, 12, 16, 17])
def test_forced_forward_plans_match_oracle(rn, plan):
    M, N, dt = 777, 8192, "bf16"
    d, t = dev_inputs(M, N, dt, 101)
    y, _, r, p = rn.rmsnorm_fwd_ex(t["x"], t["w"], force_plan=plan)
    assert p["plan_id"] == plan
    f = oracle.fwd(d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0)
    torch.cuda.synchronize()
    from helpers import check_rstd, check_y
    check_y(to_host(y, dt), f, dt)
    check_rstd(r.cpu().numpy(), f["rstd64"])


@pytest.mark.parametrize("plan", [27, 34, 35, 36, 37, 44, 45, 48, 49, 88, 89, 90, 96, 97, 98, 118, 119, 121, 123, 124, 127, 128, 131])
def test_forced_backward_plans_match_oracle(rn, plan):
    M, N, dt = 777, 8192, "bf16"
    d, t = dev_inputs(M, N, dt, 102)
    f = oracle.fwd(d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0)
    r = torch.from_numpy(f["rstd32"]).cuda()
    dx, dw, p = rn.rmsnorm_bwd_ex(t["dy"], t["x"], t["w"], r, force_plan=plan, force_ctas=100)
    assert p["plan_id"] == plan and p["ws_rows"] == 100 and p["ctas"] == 100 * p["cluster_size"]
    b = oracle.bwd(d["dy"], d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0, rstd=f["rstd32"])
    torch.cuda.synchronize()
    check_dx(to_host(dx, dt), b, dt)
    check_dw(to_host(dw, dt), b, dt)


def test_device_status_clean_after_cluster_rows(rn):
    """Backward kernels that share rows across a cluster wait, with a bound,
    for their peers' partial sums; none of the runs in this module may have
    given up."""
    for dt, N in (("bf16", 16384), ("f32", 16384), ("bf16", 65536)):
        _, t = dev_inputs(257, N, dt, 103)
        _, r = rn.rmsnorm_fwd(t["x"], t["w"])
        rn.rmsnorm_bwd(t["dy"], t["x"], t["w"], r)
    torch.cuda.synchronize()
    assert rn.lib().rmsnorm_device_status(0) == 0


@pytest.mark.parametrize("dt,N", [("bf16", 8192), ("f32", 16384), ("bf16", 4097), ("bf16", 128)])
def test_non_affine_equals_unit_weight_bitwise(rn, dt, N):
    """Without a weight the factor is exactly 1: y, rstd and dx equal those of
    a weight of ones with offset 0, bit for bit."""
    _, t = dev_inputs(500, N, dt, 104)
    ones = torch.ones_like(t["w"])
    y0, r0 = rn.rmsnorm_fwd(t["x"], ones, offset=0.0)
    y1, r1 = rn.rmsnorm_fwd(t["x"], None, offset=3.0)
    dx0, _ = rn.rmsnorm_bwd(t["dy"], t["x"], ones, r0, offset=0.0)
    dx1, dw1 = rn.rmsnorm_bwd(t["dy"], t["x"], None, r0, offset=3.0)
    torch.cuda.synchronize()
    assert dw1 is None
    assert cuda_bits_equal(y0, y1) and cuda_bits_equal(r0, r1) and cuda_bits_equal(dx0, dx1)


def test_non_affine_argument_rules(rn):
    _, t = dev_inputs(16, 256, "bf16", 105)
    _, r = rn.rmsnorm_fwd(t["x"], None)
    L = rn.lib()
    s = torch.cuda.current_stream().cuda_stream
    # a weight without dw, or dw without a weight, is refused
    assert L.rmsnorm_bwd(t["dy"].data_ptr(), t["x"].data_ptr(), t["w"].data_ptr(), r.data_ptr(),
                         t["dy"].data_ptr(), None, None, 0, 16, 256, 1, 1e-6, 0.0, s) == 1
    assert L.rmsnorm_bwd(t["dy"].data_ptr(), t["x"].data_ptr(), None, r.data_ptr(),
                         t["dy"].data_ptr(), t["w"].data_ptr(), None, 0, 16, 256, 1, 1e-6, 0.0, s) == 1


@pytest.mark.parametrize("dt,M,N,staged,vector,same_dw", [("bf16", 4096, 8192, 88, 27, True),
                                                          ("f32", 1031, 4096, 88, 27, True),
                                                          ("bf16", 2049, 4096, 95, 26, False),
                                                          ("f16", 777, 8192, 88, 27, True),
                                                          ("bf16", 301, 12288, 96, 42, True)])
@pytest.mark.parametrize("fused", [False, True])
def test_staged_backward_matches_register_backward_bitwise(rn, dt, M, N, staged, vector, same_dw, fused):
    """The staged backward (rows streamed into shared memory by bulk copies)
    does the register kernel's arithmetic on the same chunk mapping: dx is
    bit-identical, and so is dW where the register plan also keeps one
    partial row per CTA (with two row teams a CTA it adds them first)."""
    d = inputs.make_inputs(M, N, dt, 190 + N % 7, residual=fused, dres=fused)
    x, dy, w = (to_dev(d[k], dt) for k in ("x", "dy", "w"))
    dres = to_dev(d["dres"], dt) if fused else None
    _, rstd = rn.rmsnorm_fwd(x, w)
    a_dx, a_dw, ap = rn.rmsnorm_bwd_ex(dy, x, w, rstd, dresidual_out=dres, fused=fused, force_plan=staged,
                                       force_ctas=120)
    b_dx, b_dw, bp = rn.rmsnorm_bwd_ex(dy, x, w, rstd, dresidual_out=dres, fused=fused, force_plan=vector,
                                       force_ctas=120)
    torch.cuda.synchronize()
    assert ap["path_name"] == "staged" and bp["path_name"] == "vector"
    assert ap["ctas"] == bp["ctas"] == 120
    assert cuda_bits_equal(a_dx, b_dx)
    if same_dw:
        assert cuda_bits_equal(a_dw, b_dw)
    else:
        assert torch.allclose(a_dw.float(), b_dw.float(), rtol=1e-2, atol=1e-3)
    assert rn.lib().rmsnorm_device_status(1) == 0


@pytest.mark.parametrize("dt,M,N,reread,held", [("bf16", 1001, 16384, 118, 97), ("f16", 333, 12288, 119, 97),
                                                ("f32", 517, 8192, 118, 97), ("bf16", 61, 12288, 119, 97)])
@pytest.mark.parametrize("fused", [False, True])
def test_reread_staged_backward_matches_held_bitwise(rn, dt, M, N, reread, held, fused):
    """The re-read schedule of the staged backward (both passes read the
    row from its shared-memory stage; the last warp through a stage refills
    it) does the held schedule's arithmetic on the same geometry: dx and dW
    are bit-identical for the same number of partial rows, whatever the
    stage count."""
    d = inputs.make_inputs(M, N, dt, 230 + N % 5, residual=fused, dres=fused)
    x, dy, w = (to_dev(d[k], dt) for k in ("x", "dy", "w"))
    dres = to_dev(d["dres"], dt) if fused else None
    _, rstd = rn.rmsnorm_fwd(x, w)
    a_dx, a_dw, ap = rn.rmsnorm_bwd_ex(dy, x, w, rstd, dresidual_out=dres, fused=fused, force_plan=reread,
                                       force_ctas=120)
    b_dx, b_dw, bp = rn.rmsnorm_bwd_ex(dy, x, w, rstd, dresidual_out=dres, fused=fused, force_plan=held,
                                       force_ctas=120)
    torch.cuda.synchronize()
    assert ap["plan_id"] == reread and ap["path_name"] == "staged" and bp["plan_id"] == held
    assert ap["ctas"] == bp["ctas"] == min(120, M)
    assert cuda_bits_equal(a_dx, b_dx)
    assert cuda_bits_equal(a_dw, b_dw)
    assert rn.lib().rmsnorm_device_status(1) == 0



@pytest.mark.parametrize("dt,N,xoff", [("bf16", 4097, 0), ("bf16", 7168, 1), ("f32", 2050, 1), ("f16", 1003, 3)])
def test_generic_rows_independent_of_other_arrays_alignment(rn, dt, N, xoff):
    """A generic row splits by x's address alone: y, h, dy, dx and the
    residual buffers moved with 16-byte accesses (sharing x's address mod 16)
    or element by element (not sharing it) give the same bits, and so do
    the LayerNorm kernels."""
    M = 67
    d = inputs.make_inputs(M, N, dt, 330 + N % 9, residual=True, dres=True, beta=True)
    x = to_dev(d["x"], dt, offset=xoff)
    w = to_dev(d["w"], dt, offset=xoff)
    b = to_dev(d["beta"], dt, offset=xoff)
    outs = []
    for off in (xoff, xoff + 1, xoff + 2):
        res = to_dev(d["residual"], dt, offset=off)
        dy = to_dev(d["dy"], dt, offset=off)
        dres = to_dev(d["dres"], dt, offset=off)
        y = empty_dev((M, N), dt, offset=off)
        hout = empty_dev((M, N), dt, offset=off)
        dx = empty_dev((M, N), dt, offset=off)
        # (forced: arrays at one common offset would take the vectorised kernels)
        _, _, rstd, fp = rn.rmsnorm_fwd_ex(x, w, residual=res, residual_out=hout, y=y, force_plan=16)
        _, dw, bp = rn.rmsnorm_bwd_ex(dy, x, w, rstd, dresidual_out=dres, fused=True, dx=dx, force_plan=36)
        assert fp["path_name"] == "generic" and bp["path_name"] == "generic"
        lo = rn.layernorm_fwd(x, w, b, y=empty_dev((M, N), dt, offset=off), force_plan=16)
        lb = rn.layernorm_bwd(dy, x, w, lo["mean"], lo["rstd"], dx=empty_dev((M, N), dt, offset=off),
                              force_plan=72)
        torch.cuda.synchronize()
        outs.append([t.clone() for t in (y, hout, rstd, dx, dw, lo["y"], lo["mean"], lo["rstd"], lb["dx"],
                                         lb["dgamma"], lb["dbeta"])])
    for other in outs[1:]:
        for a, c in zip(outs[0], other):
            assert cuda_bits_equal(a, c)


@pytest.mark.parametrize("dt,M,N,cluster", [("bf16", 301, 16384, 123), ("f32", 77, 8192, 124), ("f16", 150, 12288, 123),
                                            ("bf16", 40, 16, 124), ("f32", 33, 4, 123), ("bf16", 64, 20480, 123)])
@pytest.mark.parametrize("fused", [False, True])
def test_cluster_staged_rows_match_oracle_any_partial_rows(rn, dt, M, N, cluster, fused):
    """A row shared by a cluster of staged CTAs (each streams an equal slice,
    the last ones shorter or empty; the row sums meet in distributed shared
    memory) against the oracle; dx is a function of the row alone, so it
    keeps its bits when the rows are spread over another number of units."""
    d, t = dev_inputs(M, N, dt, 340 + N % 7, residual=fused, dres=fused)
    f = oracle.fwd(d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0)
    r = torch.from_numpy(f["rstd32"]).cuda()
    kw = dict(dresidual_out=t.get("dres"), fused=fused, force_plan=cluster)
    a_dx, a_dw, ap = rn.rmsnorm_bwd_ex(t["dy"], t["x"], t["w"], r, force_ctas=30, **kw)
    b_dx, b_dw, bp = rn.rmsnorm_bwd_ex(t["dy"], t["x"], t["w"], r, force_ctas=7, **kw)
    b = oracle.bwd(d["dy"], d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0, rstd=f["rstd32"],
                   dres=d.get("dres") if fused else None)
    torch.cuda.synchronize()
    assert ap["path_name"] == "staged" and ap["cluster_size"] > 1 and ap["ws_rows"] == min(30, M)
    assert bp["ws_rows"] == 7 and bp["ctas"] == 7 * bp["cluster_size"]
    check_dx(to_host(a_dx, dt), b, dt)
    check_dw(to_host(a_dw, dt), b, dt)
    check_dw(to_host(b_dw, dt), b, dt)
    assert cuda_bits_equal(a_dx, b_dx)
    assert rn.lib().rmsnorm_device_status(1) == 0


@pytest.mark.parametrize("dt,M,N,plan", [("bf16", 203, 20488, 123), ("f32", 130, 16384, 123), ("bf16", 67, 40968, 124),
                                         ("f16", 45, 65536, 124), ("bf16", 3, 32768, 123)])
@pytest.mark.parametrize("fused", [False, True])
def test_cluster_staged_wide_rows_match_oracle(rn, dt, M, N, plan, fused):
    """Rows wider than one CTA's stages, each CTA of the cluster streaming a
    (ragged) slice, against the oracle."""
    d, t = dev_inputs(M, N, dt, 350 + N % 11, residual=fused, dres=fused)
    f = oracle.fwd(d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0)
    r = torch.from_numpy(f["rstd32"]).cuda()
    dx, dw, p = rn.rmsnorm_bwd_ex(t["dy"], t["x"], t["w"], r, dresidual_out=t.get("dres"), fused=fused,
                                  force_plan=plan)
    assert p["plan_id"] == plan and p["ctas"] == p["ws_rows"] * p["cluster_size"]
    b = oracle.bwd(d["dy"], d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0, rstd=f["rstd32"],
                   dres=d.get("dres") if fused else None)
    torch.cuda.synchronize()
    check_dx(to_host(dx, dt), b, dt)
    check_dw(to_host(dw, dt), b, dt)
    assert rn.lib().rmsnorm_device_status(1) == 0



@pytest.mark.parametrize("dt,M,N,staged,vector", [("bf16", 97, 32768, 139, 17), ("bf16", 130, 20480, 139, 17),
                                                  ("f32", 64, 16384, 139, 17), ("bf16", 33, 65536, 143, 18),
                                                  ("f16", 50, 40960, 143, 18), ("bf16", 200, 16384, 138, 8),
                                                  ("f32", 77, 6144, 138, 8), ("bf16", 70, 64, 139, 17)])
@pytest.mark.parametrize("fused", [False, True])
def test_staged_forward_matches_register_forward_bitwise(rn, dt, M, N, staged, vector, fused):
    """The staged forward (rows streamed through shared-memory stages by a
    persistent grid of CTAs or clusters) takes each thread's chunks in the
    register forward's order and reduces them in its tree: y, rstd and the
    fused residual_out are the same bits for the same geometry."""
    d, t = dev_inputs(M, N, dt, 380 + N % 7, residual=fused)
    res = t.get("residual")
    a_y, a_h, a_r, ap = rn.rmsnorm_fwd_ex(t["x"], t["w"], residual=res,
                                          residual_out=torch.empty_like(t["x"]) if fused else None, force_plan=staged)
    b_y, b_h, b_r, bp = rn.rmsnorm_fwd_ex(t["x"], t["w"], residual=res,
                                          residual_out=torch.empty_like(t["x"]) if fused else None, force_plan=vector)
    torch.cuda.synchronize()
    assert ap["plan_id"] == staged and ap["path_name"] == "staged" and bp["path_name"] == "vector"
    assert cuda_bits_equal(a_y, b_y) and cuda_bits_equal(a_r, b_r)
    if fused:
        assert cuda_bits_equal(a_h, b_h)
    assert rn.lib().rmsnorm_device_status(1) == 0


@pytest.mark.parametrize("dt,M,N,plan", [("bf16", 211, 20488, 141), ("f32", 67, 12280, 141), ("bf16", 45, 40968, 145),
                                         ("bf16", 19, 65536, 143), ("f16", 5, 24, 145), ("bf16", 301, 8192, 138)])
@pytest.mark.parametrize("fused", [False, True])
def test_staged_forward_matches_oracle(rn, dt, M, N, plan, fused):
    d, t = dev_inputs(M, N, dt, 390 + N % 5, residual=fused)
    y, h, r, p = rn.rmsnorm_fwd_ex(t["x"], t["w"], residual=t.get("residual"),
                                   residual_out=torch.empty_like(t["x"]) if fused else None, force_plan=plan)
    f = oracle.fwd(d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0, residual=d.get("residual") if fused else None)
    torch.cuda.synchronize()
    assert p["plan_id"] == plan and p["ctas"] == p["ws_rows"] * p["cluster_size"] and p["workspace_bytes"] == 0
    check_y(to_host(y, dt), f, dt)
    check_rstd(r.cpu().numpy(), f["rstd64"])
    if fused:
        assert np.array_equal(to_host(h, dt), f["h"])
    assert rn.lib().rmsnorm_device_status(1) == 0


def test_e4m3_forward_on_staged_plans_matches_register_plans_bitwise(rn):
    """Wide rows with an E4M3 output take the staged forward (the row max
    from one pass over the stage, the codes from another); its codes,
    1/scale and amax are the register cluster kernel's bits. A forced
    staged alternative (not compiled for E4M3) is refused."""
    _, t = dev_inputs(64, 32768, "bf16", 395, residual=True)
    with pytest.raises(rn.RMSNormError):
        rn.rmsnorm_fwd_fp8(t["x"], t["w"], scaling="row", force_plan=138)
    for scaling, scale in (("row", None), ("tensor", torch.tensor([3.0], device="cuda"))):
        for res in (None, t["residual"]):
            kw = dict(scaling=scaling, scale=scale, residual=res, amax=True)
            a = rn.rmsnorm_fwd_fp8(t["x"], t["w"], **kw)
            b = rn.rmsnorm_fwd_fp8(t["x"], t["w"], force_plan=17, **kw)
            torch.cuda.synchronize()
            assert a["plan"]["path_name"] == "staged" and a["plan"]["cluster_size"] == 2
            assert b["plan"]["path_name"] == "vector"
            for k in ("y", "rstd", "scale_inv", "amax") + (("residual_out",) if res is not None else ()):
                assert cuda_bits_equal(a[k], b[k]), (scaling, k)
    assert rn.lib().rmsnorm_device_status(1) == 0


@pytest.mark.parametrize("N", [20480, 65536])
def test_graph_replay_wide_rows_matches_direct(rn, N):
    """The staged cluster kernels (forward and backward, RMSNorm and
    LayerNorm, plain and fused) capture into a CUDA graph and replay to the
    direct calls' bits."""
    M = 64
    d, t = dev_inputs(M, N, "bf16", 420 + N % 7, residual=True, dres=True, beta=True)
    ws = torch.empty(rn.rmsnorm_bwd_workspace_bytes(M, N, torch.bfloat16), dtype=torch.uint8, device="cuda")
    lws = torch.empty(rn.layernorm_bwd_workspace_bytes(M, N, torch.bfloat16), dtype=torch.uint8, device="cuda")

    def run(out):
        y, h, r = rn.rmsnorm_add_fwd(t["x"], t["residual"], t["w"], y=out[0], residual_out=out[1], rstd=out[2])
        rn.rmsnorm_add_bwd(t["dy"], t["dres"], h, t["w"], r, dx=out[3], dw=out[4], workspace=ws)
        o = rn.layernorm_fwd(t["x"], t["w"], t["beta"], y=out[5], mean=out[6], rstd=out[7])
        rn.layernorm_bwd(t["dy"], t["x"], t["w"], o["mean"], o["rstd"], dx=out[8], dgamma=out[9], dbeta=out[10],
                         workspace=lws)

    def fresh():
        return [torch.empty_like(t["x"]), torch.empty_like(t["x"]), torch.empty(M, device="cuda"),
                torch.empty_like(t["x"]), torch.empty_like(t["w"]), torch.empty_like(t["x"]), torch.empty(M, device="cuda"),
                torch.empty(M, device="cuda"), torch.empty_like(t["x"]), torch.empty_like(t["w"]), torch.empty_like(t["w"])]
    ref = fresh()
    run(ref)
    out = fresh()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            run(out)
    for a in out:
        a.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(out, ref):
        assert cuda_bits_equal(a, b)
    assert rn.plan_query(rn.OP_FWD, M, N, rn.RMSNORM_BF16)["path_name"] == "staged"
    assert rn.lib().rmsnorm_device_status(1) == 0
