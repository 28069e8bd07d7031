"""Pins of the CPU oracle against facts that do not come from the oracle.

Every check here holds by mathematics: closed forms of special rows, exact
invariances, the finite-difference gradient of the forward, hand-derived
values, and the IEEE rounding rule for bf16 checked exhaustively and
against an independent implementation. A plausible slip in the oracle (a
sum instead of a mean, eps outside the square root, a dropped or sign-flipped
term of the gradient, a transposed w index, rounding through binary32)
fails at least one of these.

The RMSNorm definitions follow the Liger-Kernel page "perf(cutedsl): add
Blackwell fast path to RMSNorm" (llama mode, runtime offset) and the FlyDSL
page "[Perf] Optimize RMSNorm backward with staged reduction and vec8 I/O"
(fused-add backward: dx also serves as dresidual).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from row_wise_normalization_rmsnorm_gb300 import inputs


def f64(shape, seed, scale=1.0, loc=0.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale + loc


# ----------------------------------------------------------------- bf16 --

def test_bf16_decode_round_identity_exhaustive():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 7) & 0xFF
    frac = bits & 0x7F
    finite = ~((exp == 0xFF) & (frac != 0))          # drop NaNs
    b = bits[finite]
    assert np.array_equal(oracle.bf16_round(oracle.bf16_decode(b)), b)


def test_bf16_round_ties_to_even_and_neighbours():
    # every pair of adjacent positive finite bf16 values, normal and subnormal
    lo = np.arange(0, 0x7F7F, dtype=np.uint16)
    a = oracle.bf16_decode(lo)
    b = oracle.bf16_decode(lo + 1)
    mid = (a + b) / 2.0                               # exact in double
    got = oracle.bf16_round(mid)
    even = np.where((lo & 1) == 0, lo, lo + 1).astype(np.uint16)
    assert np.array_equal(got, even)
    below = np.nextafter(mid, -np.inf)
    above = np.nextafter(mid, np.inf)
    assert np.array_equal(oracle.bf16_round(below), lo)
    assert np.array_equal(oracle.bf16_round(above), (lo + 1).astype(np.uint16))
    # sign symmetry
    assert np.array_equal(oracle.bf16_round(-mid), even | np.uint16(0x8000))


def test_bf16_round_matches_torch_on_float32_values():
    # For values that are exact binary32 numbers, one-step rounding from
    # double equals torch's binary32 -> bf16 conversion (nearest, ties even).
    v = np.random.default_rng(7).standard_normal(200_000).astype(np.float32)
    v[:1000] *= np.float32(1e-30)
    v[1000:2000] *= np.float32(1e30)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_round(v.astype(np.float64)), ref)


def test_bf16_round_is_single_step():
    # 1 + 2^-8 is the midpoint between bf16 1.0 and 1.0078125; a hair above it
    # must round up. Going through binary32 first would land exactly on the
    # midpoint and then round down to the even neighbour 1.0.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert float(np.float32(v)) == 1.0 + 2.0 ** -8
    assert oracle.bf16_round(np.array([v]))[0] == 0x3F81
    assert oracle.bf16_round(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80


# ------------------------------------------------------------- forward --

def test_fwd_hand_example():
    # x = (3, 4): mean(x^2) = 12.5, rstd = 1/sqrt(12.5) = sqrt(2)/5.
    x = np.array([[3.0, 4.0]])
    w = np.array([1.0, 2.0])
    r = oracle.fwd(x, w, dtype="f64", eps=0.0, offset=0.0)
    s2 = math.sqrt(2.0)
    assert r["rstd64"][0] == pytest.approx(s2 / 5, rel=1e-15)
    assert r["y64"][0] == pytest.approx([3 * s2 / 5, 8 * s2 / 5], rel=1e-15)
    # with eps = 0.5 inside the root: mean + eps = 13
    r = oracle.fwd(x, w, dtype="f64", eps=0.5, offset=1.0)
    assert r["rstd64"][0] == pytest.approx(1 / math.sqrt(13.0), rel=1e-15)
    assert r["y64"][0] == pytest.approx([3 * 2 / math.sqrt(13), 4 * 3 / math.sqrt(13)], rel=1e-15)


@pytest.mark.parametrize("a", [0.75, -3.5, 1e-3])
@pytest.mark.parametrize("offset", [0.0, 1.0])
def test_fwd_constant_row_eps0(a, offset):
    N = 37
    w = f64(N, 1, 0.1, 1.0)
    x = np.full((2, N), a)
    r = oracle.fwd(x, w, dtype="f64", eps=0.0, offset=offset)
    np.testing.assert_allclose(r["y64"], np.sign(a) * (offset + w)[None, :].repeat(2, 0), rtol=1e-15)
    np.testing.assert_allclose(r["rstd64"], 1 / abs(a), rtol=1e-15)


def test_fwd_zero_row_eps_positive():
    eps = 0.01
    r = oracle.fwd(np.zeros((1, 16)), f64(16, 2), dtype="f64", eps=eps, offset=0.0)
    assert r["rstd64"][0] == pytest.approx(10.0, rel=1e-15)   # eps^-1/2
    assert np.all(r["y64"] == 0.0)


@pytest.mark.parametrize("k", [-3, 5])
def test_fwd_scale_invariance_eps0(k):
    x = f64((4, 50), 3)
    w = f64(50, 4, 0.1, 1.0)
    r1 = oracle.fwd(x, w, dtype="f64", eps=0.0, offset=0.0)
    r2 = oracle.fwd(x * 2.0 ** k, w, dtype="f64", eps=0.0, offset=0.0)
    assert np.array_equal(r1["y64"], r2["y64"])
    assert np.array_equal(r2["rstd64"], r1["rstd64"] * 2.0 ** -k)


@pytest.mark.parametrize("eps", [0.0, 0.3])
def test_fwd_norm_identity(eps):
    # sum_j (y_j / (o + w_j))^2 = N ms / (ms + eps): the mean, with eps under the root
    N = 64
    x = f64((5, N), 5)
    w = f64(N, 6, 0.1, 1.0)
    r = oracle.fwd(x, w, dtype="f64", eps=eps, offset=0.5)
    ms = np.mean(x * x, axis=1)
    lhs = np.sum((r["y64"] / (0.5 + w)) ** 2, axis=1)
    np.testing.assert_allclose(lhs, N * ms / (ms + eps), rtol=1e-13)


def test_fwd_n1_special_case():
    x = np.array([[0.5], [-2.0], [3.0]])
    w = np.array([1.25])
    eps = 0.2
    r = oracle.fwd(x, w, dtype="f64", eps=eps, offset=1.0)
    np.testing.assert_allclose(r["y64"][:, 0], x[:, 0] / np.sqrt(x[:, 0] ** 2 + eps) * 2.25, rtol=1e-15)


def test_fwd_rows_independent_and_threads():
    x = f64((33, 40), 8)
    w = f64(40, 9, 0.1, 1.0)
    full = oracle.fwd(x, w, dtype="f64", eps=1e-3, offset=0.0)
    part = oracle.fwd(x[10:20], w, dtype="f64", eps=1e-3, offset=0.0)
    thr = oracle.fwd(x, w, dtype="f64", eps=1e-3, offset=0.0, nthreads=4)
    assert np.array_equal(full["y64"][10:20], part["y64"])
    assert np.array_equal(full["y64"], thr["y64"])


def test_fwd_storage_rounding_bf16_and_f32():
    d = inputs.make_inputs(8, 96, "bf16", 11)
    r = oracle.fwd(d["x"], d["w"], dtype="bf16", eps=1e-6, offset=0.0)
    assert np.array_equal(r["y"], oracle.bf16_round(r["y64"]))
    assert np.array_equal(r["rstd32"], r["rstd64"].astype(np.float32))
    d = inputs.make_inputs(8, 96, "f32", 11)
    r = oracle.fwd(d["x"], d["w"], dtype="f32", eps=1e-6, offset=0.0)
    assert np.array_equal(r["y"], r["y64"].astype(np.float32))


def test_fused_add_fwd_is_fwd_of_rounded_sum():
    for dt in ("bf16", "f32"):
        d = inputs.make_inputs(6, 72, dt, 12, residual=True)
        r = oracle.fwd(d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0, residual=d["residual"])
        s = oracle.to_f64(d["x"], dt) + oracle.to_f64(d["residual"], dt)
        h = oracle.bf16_round(s) if dt == "bf16" else s.astype(np.float32)
        assert np.array_equal(r["h"], h)
        p = oracle.fwd(h, d["w"], dtype=dt, eps=1e-6, offset=0.0)
        assert np.array_equal(r["y"], p["y"]) and np.array_equal(r["rstd64"], p["rstd64"])


# ------------------------------------------------------------ backward --

def _bwd64(h, dy, w, eps, offset, dres=None):
    return oracle.bwd(dy, h, w, dtype="f64", eps=eps, offset=offset, dres=dres)


@pytest.mark.parametrize("offset", [0.0, 1.0])
def test_bwd_orthogonality_eps0(offset):
    # sum_j x_j dx_j = 0 when eps = 0, for any w and offset
    x = f64((6, 45), 20)
    dy = f64((6, 45), 21)
    w = f64(45, 22, 0.3, 0.2)
    r = _bwd64(x, dy, w, 0.0, offset)
    dot = np.sum(x * r["dx64"], axis=1)
    scale = np.sum(np.abs(x * r["dx64"]), axis=1)
    assert np.all(np.abs(dot) <= 1e-13 * scale)


def test_bwd_constant_row_eps0():
    N = 30
    x = np.full((3, N), -1.5)
    dy = f64((3, N), 23)
    w = f64(N, 24, 0.1, 1.0)
    r = _bwd64(x, dy, w, 0.0, 0.0)
    g = dy * w[None, :]
    rstd = 1 / 1.5
    np.testing.assert_allclose(r["dx64"], rstd * (g - g.mean(axis=1, keepdims=True)), rtol=1e-12, atol=1e-15)


def test_bwd_zero_row_eps_positive():
    dy = f64((1, 12), 25)
    w = f64(12, 26, 0.1, 1.0)
    r = _bwd64(np.zeros((1, 12)), dy, w, 0.04, 0.0)
    np.testing.assert_allclose(r["dx64"][0], 5.0 * dy[0] * w, rtol=1e-15)
    assert np.all(r["dw64"] == 0.0)


@pytest.mark.parametrize("k", [-2, 3])
def test_bwd_scaling_eps0(k):
    x = f64((5, 33), 27)
    dy = f64((5, 33), 28)
    w = f64(33, 29, 0.1, 1.0)
    r1 = _bwd64(x, dy, w, 0.0, 0.0)
    r2 = _bwd64(x * 2.0 ** k, dy, w, 0.0, 0.0)
    np.testing.assert_allclose(r2["dx64"], r1["dx64"] * 2.0 ** -k, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(r2["dw64"], r1["dw64"], rtol=1e-13, atol=1e-15)


def test_bwd_n1_textbook_derivative():
    # y = x (x^2+eps)^-1/2 (o+w): dy/dx = (o+w) eps / (x^2+eps)^(3/2)
    x = np.array([[0.7], [-1.3], [2.0]])
    dy = np.array([[1.0], [0.5], [-2.0]])
    w = np.array([0.9])
    eps = 0.3
    r = _bwd64(x, dy, w, eps, 1.0)
    want = dy[:, 0] * 1.9 * eps / (x[:, 0] ** 2 + eps) ** 1.5
    np.testing.assert_allclose(r["dx64"][:, 0], want, rtol=1e-14)
    np.testing.assert_allclose(r["dw64"][0], np.sum(dy[:, 0] * x[:, 0] / np.sqrt(x[:, 0] ** 2 + eps)), rtol=1e-14)


def _loss(x, w, dy, eps, offset, residual=None, dres=None):
    r = oracle.fwd(x, w, dtype="f64", eps=eps, offset=offset, residual=residual)
    L = float(np.sum(r["y64"] * dy))
    if dres is not None:
        L += float(np.sum((x + residual) * dres))
    return L


@pytest.mark.parametrize("N", [1, 5, 8])
@pytest.mark.parametrize("eps", [0.1, 1e-6])
@pytest.mark.parametrize("offset", [0.0, 1.0])
@pytest.mark.parametrize("fused", [False, True])
def test_bwd_matches_finite_differences(N, eps, offset, fused):
    """Central differences of L = sum y*dy (+ sum h*dres when fused) in x, w
    and the residual agree with the oracle's dx and dW."""
    M = 3
    rng = np.random.default_rng(100 + N)
    x = rng.standard_normal((M, N))
    w = rng.standard_normal(N) * 0.1 + (0.0 if offset else 1.0)
    dy = rng.standard_normal((M, N))
    res = rng.standard_normal((M, N)) if fused else None
    dres = rng.standard_normal((M, N)) if fused else None
    h = x + res if fused else x
    an = oracle.bwd(dy, h, w, dtype="f64", eps=eps, offset=offset, dres=dres)

    def fd(fun, v, idx):
        step = 1e-6 * max(1.0, abs(v[idx]))
        vp = v.copy(); vp[idx] += step
        vm = v.copy(); vm[idx] -= step
        return (fun(vp) - fun(vm)) / (2 * step)

    for idx in np.ndindex(M, N):
        gx = fd(lambda v: _loss(v, w, dy, eps, offset, res, dres), x, idx)
        tol = 1e-7 * max(abs(an["dx64"][idx]), an["dx_scale"][idx]) + 1e-9
        assert abs(gx - an["dx64"][idx]) <= tol, (idx, gx, an["dx64"][idx])
        if fused:
            gr = fd(lambda v: _loss(x, w, dy, eps, offset, v, dres), res, idx)
            assert abs(gr - an["dx64"][idx]) <= tol
    for j in range(N):
        gw = fd(lambda v: _loss(x, v, dy, eps, offset, res, dres), w, j)
        tol = 1e-7 * max(abs(an["dw64"][j]), an["dw_abs"][j]) + 1e-9
        assert abs(gw - an["dw64"][j]) <= tol, (j, gw, an["dw64"][j])


def test_bwd_dw_order_independence_and_brute_force():
    x = f64((40, 24), 30)
    dy = f64((40, 24), 31)
    w = f64(24, 32, 0.1, 1.0)
    a = oracle.bwd(dy, x, w, dtype="f64", eps=1e-6, offset=0.0, nthreads=1)
    b = oracle.bwd(dy, x, w, dtype="f64", eps=1e-6, offset=0.0, nthreads=5)
    np.testing.assert_allclose(a["dw64"], b["dw64"], rtol=1e-12, atol=1e-14)
    assert np.array_equal(a["dx64"], b["dx64"])
    rstd = 1 / np.sqrt(np.mean(x * x, axis=1) + 1e-6)
    brute = np.zeros(24)
    for i in range(40):
        for j in range(24):
            brute[j] += dy[i, j] * x[i, j] * rstd[i]
    np.testing.assert_allclose(a["dw64"], brute, rtol=1e-12, atol=1e-14)


def test_bwd_given_rstd_and_dw_only_pass():
    d = inputs.make_inputs(16, 64, "bf16", 33)
    f = oracle.fwd(d["x"], d["w"], dtype="bf16", eps=1e-6, offset=0.0)
    full = oracle.bwd(d["dy"], d["x"], d["w"], dtype="bf16", eps=1e-6, offset=0.0)
    given = oracle.bwd(d["dy"], d["x"], d["w"], dtype="bf16", eps=1e-6, offset=0.0, rstd=f["rstd32"])
    only = oracle.bwd(d["dy"], d["x"], d["w"], dtype="bf16", eps=1e-6, offset=0.0, want_dx=False)
    assert np.array_equal(full["dw64"], only["dw64"])
    # float32 rstd differs from the double one by <= 2^-24 relative; dx moves
    # by a few times that relative to the size of its terms
    assert np.all(np.abs(given["dx64"] - full["dx64"]) <= 1e-6 * full["dx_scale"])
    assert np.array_equal(full["dx"], oracle.bf16_round(full["dx64"]))
    assert np.array_equal(full["dw"], oracle.bf16_round(full["dw64"]))


def test_fused_bwd_zero_dres_equals_plain_plus_nothing():
    d = inputs.make_inputs(8, 48, "f32", 34, residual=True)
    h = oracle.fwd(d["x"], d["w"], dtype="f32", eps=1e-6, offset=0.0, residual=d["residual"])["h"]
    a = oracle.bwd(d["dy"], h, d["w"], dtype="f32", eps=1e-6, offset=0.0)
    b = oracle.bwd(d["dy"], h, d["w"], dtype="f32", eps=1e-6, offset=0.0,
                   dres=np.zeros_like(d["dy"]))
    assert np.array_equal(a["dx64"], b["dx64"])


# ------------------------------------------------------------ non-affine --

def test_non_affine_is_affine_with_unit_weight():
    # without a weight the factor is exactly 1 (offset unused)
    x = f64((5, 30), 40)
    dy = f64((5, 30), 41)
    a = oracle.fwd(x, None, dtype="f64", eps=1e-3, offset=7.0)
    b = oracle.fwd(x, np.ones(30), dtype="f64", eps=1e-3, offset=0.0)
    assert np.array_equal(a["y64"], b["y64"]) and np.array_equal(a["rstd64"], b["rstd64"])
    ga = oracle.bwd(dy, x, None, dtype="f64", eps=1e-3, offset=7.0)
    gb = oracle.bwd(dy, x, np.ones(30), dtype="f64", eps=1e-3, offset=0.0)
    assert np.array_equal(ga["dx64"], gb["dx64"])


def test_non_affine_hand_example_and_unit_rms():
    # x = (3, 4): y = x / sqrt(12.5); the output row has mean square 1 at eps 0
    r = oracle.fwd(np.array([[3.0, 4.0]]), None, dtype="f64", eps=0.0, offset=0.0)
    assert r["y64"][0] == pytest.approx([3 / math.sqrt(12.5), 4 / math.sqrt(12.5)], rel=1e-15)
    y = oracle.fwd(f64((4, 64), 42), None, dtype="f64", eps=0.0, offset=0.0)["y64"]
    np.testing.assert_allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-14)


@pytest.mark.parametrize("eps", [0.1, 1e-6])
def test_non_affine_bwd_matches_finite_differences(eps):
    M, N = 3, 6
    rng = np.random.default_rng(43)
    x = rng.standard_normal((M, N))
    dy = rng.standard_normal((M, N))
    an = oracle.bwd(dy, x, None, dtype="f64", eps=eps, offset=0.0)

    def loss(v):
        return float(np.sum(oracle.fwd(v, None, dtype="f64", eps=eps, offset=0.0)["y64"] * dy))

    for idx in np.ndindex(M, N):
        step = 1e-6 * max(1.0, abs(x[idx]))
        xp = x.copy(); xp[idx] += step
        xm = x.copy(); xm[idx] -= step
        fd = (loss(xp) - loss(xm)) / (2 * step)
        assert abs(fd - an["dx64"][idx]) <= 1e-7 * max(abs(an["dx64"][idx]), an["dx_scale"][idx]) + 1e-9


# ------------------------------------------------------------------ fp16 --

def test_f16_decode_round_identity_exhaustive():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 10) & 0x1F
    frac = bits & 0x3FF
    b = bits[~((exp == 0x1F) & (frac != 0))]           # drop NaNs
    v = b.view(np.float16).astype(np.float64)          # numpy's exact decode
    assert np.array_equal(oracle.f16_round(v).view(np.uint16), b)


def test_f16_round_ties_to_even_and_neighbours():
    lo = np.arange(0, 0x7BFF, dtype=np.uint16)          # adjacent finite pairs
    a = lo.view(np.float16).astype(np.float64)
    b = (lo + 1).astype(np.uint16).view(np.float16).astype(np.float64)
    mid = (a + b) / 2.0
    even = np.where((lo & 1) == 0, lo, lo + 1).astype(np.uint16)
    assert np.array_equal(oracle.f16_round(mid).view(np.uint16), even)
    assert np.array_equal(oracle.f16_round(np.nextafter(mid, -np.inf)).view(np.uint16), lo)
    assert np.array_equal(oracle.f16_round(np.nextafter(mid, np.inf)).view(np.uint16), (lo + 1).astype(np.uint16))


def test_f16_round_matches_numpy_double_to_half():
    # numpy converts float64 to float16 directly, nearest with ties to even
    v = np.random.default_rng(8).standard_normal(300_000)
    v[:20_000] *= 1e-5                                   # subnormal range
    v[20_000:30_000] *= 3e4                              # near the top of the range
    v = v[np.abs(v) < 65504.0]
    assert np.array_equal(oracle.f16_round(v), v.astype(np.float16))


def test_f16_storage_forward_rounds_once():
    d = inputs.make_inputs(8, 96, "f16", 13)
    r = oracle.fwd(d["x"], d["w"], dtype="f16", eps=1e-6, offset=0.0)
    assert np.array_equal(r["y"], oracle.f16_round(r["y64"]))
    r2 = oracle.fwd(oracle.to_f64(d["x"], "f16"), oracle.to_f64(d["w"], "f16"), dtype="f64", eps=1e-6,
                    offset=0.0)
    assert np.array_equal(r["y64"], r2["y64"])


# ------------------------------------------------- separate weight dtype --

def test_weight_dtype_only_changes_how_w_and_dw_are_stored():
    # bf16 activations with an fp32 weight: the arithmetic is the same as
    # with the weight's values given in double, and dW is stored as fp32
    d = inputs.make_inputs(12, 80, "bf16", 44, wdtype="f32")
    assert d["w"].dtype == np.float32
    a = oracle.fwd(d["x"], d["w"], dtype="bf16", wdtype="f32", eps=1e-6, offset=1.0)
    b = oracle.fwd(oracle.to_f64(d["x"], "bf16"), d["w"].astype(np.float64), dtype="f64", eps=1e-6, offset=1.0)
    assert np.array_equal(a["y64"], b["y64"]) and np.array_equal(a["y"], oracle.bf16_round(b["y64"]))
    ga = oracle.bwd(d["dy"], d["x"], d["w"], dtype="bf16", wdtype="f32", eps=1e-6, offset=1.0)
    gb = oracle.bwd(oracle.to_f64(d["dy"], "bf16"), oracle.to_f64(d["x"], "bf16"), d["w"].astype(np.float64),
                    dtype="f64", eps=1e-6, offset=1.0)
    assert np.array_equal(ga["dx64"], gb["dx64"]) and np.array_equal(ga["dw64"], gb["dw64"])
    assert ga["dw"].dtype == np.float32 and np.array_equal(ga["dw"], gb["dw64"].astype(np.float32))


# ------------------------------------------------------------------ E4M3 --
# The format (OCP "E4M3FN": bias 7, 3 fraction bits, no infinities, one NaN
# pattern per sign, largest finite 448) is pinned to torch's float8_e4m3fn,
# an independent implementation of the same format.

def _torch_e4m3_decode(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn) \
        .to(torch.float64).numpy()


def _torch_e4m3_round(v):
    # in-range float32-representable values only (torch maps overflow to NaN)
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_e4m3_decode_matches_torch_exhaustive():
    codes = np.arange(256, dtype=np.uint8)
    a, b = oracle.e4m3_decode(codes), _torch_e4m3_decode(codes)
    assert np.array_equal(np.isnan(a), np.isnan(b)) and np.isnan(a).sum() == 2
    assert np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)])
    assert np.nanmax(a) == 448.0 and a[1] == 2.0 ** -9 and a[8] == 2.0 ** -6


def test_e4m3_round_identity_exhaustive():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_round(oracle.e4m3_decode(codes)), codes)


def test_e4m3_round_ties_to_even_and_neighbours():
    lo = np.arange(0, 0x7E, dtype=np.uint8)               # adjacent finite pairs
    a, b = oracle.e4m3_decode(lo), oracle.e4m3_decode(lo + 1)
    mid = (a + b) / 2.0
    even = np.where((lo & 1) == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(oracle.e4m3_round(mid), even)
    assert np.array_equal(oracle.e4m3_round(np.nextafter(mid, -np.inf)), lo)
    assert np.array_equal(oracle.e4m3_round(np.nextafter(mid, np.inf)), (lo + 1).astype(np.uint8))
    assert np.array_equal(oracle.e4m3_round(-mid), even | 0x80)


def test_e4m3_round_saturates_and_keeps_nan():
    big = np.array([448.0, np.nextafter(448.0, np.inf), 463.9, 464.0, 480.0, 1e6, np.inf])
    assert np.all(oracle.e4m3_round(big) == 0x7E)
    assert np.all(oracle.e4m3_round(-big) == 0xFE)
    assert np.isnan(oracle.e4m3_decode(oracle.e4m3_round(np.array([np.nan])))[0])
    assert oracle.e4m3_round(np.array([2.0 ** -10]))[0] == 0            # half the smallest quantum, tie to 0
    assert oracle.e4m3_round(np.array([3 * 2.0 ** -10]))[0] == 2        # 1.5 quanta, tie to even (2)


def test_e4m3_round_matches_torch_on_float32_values():
    rng = np.random.default_rng(21)
    v = np.concatenate([rng.uniform(-447.0, 447.0, 200_000), rng.standard_normal(200_000) * 0.02,
                        rng.standard_normal(50_000) * 2.0 ** -8])
    v = v.astype(np.float32).astype(np.float64)
    assert np.array_equal(oracle.e4m3_round(v), _torch_e4m3_round(v))


# ------------------------------------------------------- fp8 forward --

def _quant_check(r, scale_of_row):
    """Codes of the fp8 forward against torch's E4M3 rounding of y * s.
    y * s can land exactly on a midpoint between two codes (bf16 inputs have
    few significant bits), and then the last bit of the double arithmetic
    decides; there either neighbour is accepted."""
    s = scale_of_row[:, None]
    v = r["y64"] * s
    inside = np.abs(v) < 447.0
    got, ref = r["yq"][inside], _torch_e4m3_round(v[inside])
    diff = got != ref
    if diff.any():
        g, f = got[diff].astype(np.int32), ref[diff].astype(np.int32)
        assert np.all((g >> 7) == (f >> 7)) and np.all(np.abs(g - f) == 1), "codes not adjacent"
        a, b = oracle.e4m3_decode(got[diff]), oracle.e4m3_decode(ref[diff])
        vv = v[inside][diff]
        assert np.all(np.abs(vv - (a + b) / 2.0) <= 1e-12 * np.abs(vv)), "not a tie"
        assert diff.sum() <= max(2, got.size // 500)
    assert np.all((r["yq"][~inside] & 0x7F) >= 0x7D)


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
def test_fp8_tensor_scaling_is_fwd_times_scale_rounded(dt):
    d = inputs.make_inputs(24, 160, dt, 61, outlier_frac=0.02)
    base = oracle.fwd(d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0)
    for scale in (1.0, 37.5, 0.125):
        r = oracle.fwd_fp8(d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0, scaling="tensor", scale=scale)
        assert np.array_equal(r["y64"], base["y64"]) and np.array_equal(r["rstd32"], base["rstd32"])
        _quant_check(r, np.full(24, scale))
        assert r["amax"] == np.abs(base["y64"]).max()
        assert np.all(r["scale_inv"] == 1.0 / scale)
        # dequantised values are within half an E4M3 step of y
        deq = oracle.e4m3_decode(r["yq"]) / scale
        y = base["y64"]
        ok = np.abs(deq - y) <= 2.0 ** -4 * np.abs(y) + 2.0 ** -10 / scale
        sat = np.abs(y * scale) >= 448.0
        assert np.all(ok | sat)


def test_fp8_tensor_scaling_saturates():
    d = inputs.make_inputs(8, 64, "bf16", 62)
    r = oracle.fwd_fp8(d["x"], d["w"], dtype="bf16", eps=1e-6, offset=0.0, scaling="tensor", scale=1000.0)
    big = np.abs(r["y64"] * 1000.0) >= 448.0
    assert big.any() and np.all((r["yq"][big] & 0x7F) == 0x7E)
    assert np.array_equal(r["yq"][big] >> 7, (r["y64"][big] < 0).astype(np.uint8))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_fp8_row_scaling_uses_each_rows_maximum(dt):
    d = inputs.make_inputs(32, 256, dt, 63, outlier_frac=0.02)
    base = oracle.fwd(d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0)
    r = oracle.fwd_fp8(d["x"], d["w"], dtype=dt, eps=1e-6, offset=0.0, scaling="row")
    amax = np.abs(base["y64"]).max(axis=1)
    assert np.array_equal(r["amax_row"], amax)
    assert np.allclose(r["scale_inv"] * 448.0, amax, rtol=1e-15, atol=0)
    _quant_check(r, 448.0 / amax)
    # the largest element of every row maps to the largest finite code
    assert np.all((r["yq"] & 0x7F).max(axis=1) == 0x7E)


def test_fp8_row_scaling_zero_row():
    x = np.zeros((2, 16), dtype=np.float32)
    x[1] = np.arange(16) - 7.5
    w = np.ones(16, dtype=np.float32)
    r = oracle.fwd_fp8(x, w, dtype="f32", eps=1e-6, offset=0.0, scaling="row")
    assert np.all(r["yq"][0] == 0) and r["scale_inv"][0] == 1.0 and r["amax_row"][0] == 0.0
    assert r["scale_inv"][1] > 0 and (r["yq"][1] & 0x7F).max() == 0x7E


def test_fp8_fused_add_quantises_the_fused_forward():
    d = inputs.make_inputs(16, 128, "bf16", 64, residual=True, w_mode="gemma")
    base = oracle.fwd(d["x"], d["w"], dtype="bf16", eps=1e-6, offset=1.0, residual=d["residual"])
    r = oracle.fwd_fp8(d["x"], d["w"], dtype="bf16", eps=1e-6, offset=1.0, residual=d["residual"],
                       scaling="row")
    assert np.array_equal(r["h"], base["h"]) and np.array_equal(r["y64"], base["y64"])
    _quant_check(r, 448.0 / np.abs(base["y64"]).max(axis=1))


# ------------------------------------------------------------- LayerNorm --

def test_ln_fwd_hand_example():
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    g = np.array([1.0, 2.0, 0.5, -1.0])
    b = np.array([0.0, 1.0, -1.0, 0.25])
    r = oracle.ln_fwd(x, g, b, dtype="f64", eps=0.25, offset=0.0)
    # mean 2.5, biased variance 1.25, rstd = 1 / sqrt(1.25 + 0.25)
    rstd = 1.0 / math.sqrt(1.5)
    assert r["mean64"][0] == 2.5 and abs(r["rstd64"][0] - rstd) < 1e-15
    # the saved fp32 statistics are the same values rounded once to binary32
    assert r["mean32"][0] == np.float32(2.5) and r["rstd32"][0] == np.float32(rstd)
    want = (x[0] - 2.5) * rstd * g + b
    assert np.allclose(r["y64"][0], want, rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("N", [2, 7, 64, 1000])
def test_ln_fwd_output_is_standardised(N):
    # gamma = 1, beta = 0, eps = 0: every row has mean 0 and (biased) variance 1
    x = inputs.make_inputs(5, N, "f32", 81, x_shift=3.0)["x"]
    r = oracle.ln_fwd(x, None, None, dtype="f32", eps=0.0, offset=0.0)
    y = r["y64"]
    assert np.allclose(y.mean(axis=1), 0.0, atol=1e-12)
    assert np.allclose((y * y).mean(axis=1), 1.0, rtol=1e-12)


def test_ln_fwd_shift_invariance():
    x = inputs.make_inputs(6, 96, "f32", 82)["x"].astype(np.float64)
    g = inputs.make_inputs(1, 96, "f32", 83)["w"].astype(np.float64)
    a = oracle.ln_fwd(x, g, None, dtype="f64", eps=1e-3, offset=0.0)
    b = oracle.ln_fwd(x + 1024.0, g, None, dtype="f64", eps=1e-3, offset=0.0)
    assert np.allclose(a["y64"], b["y64"], rtol=0, atol=1e-9)
    assert np.allclose(b["mean64"] - a["mean64"], 1024.0, rtol=0, atol=1e-9)


def test_ln_on_zero_mean_rows_is_rmsnorm():
    # a row with zero mean: var = mean(x^2), so LayerNorm = RMSNorm (+ beta)
    x = inputs.make_inputs(4, 64, "f32", 84)["x"].astype(np.float64)
    x = np.concatenate([x, -x], axis=1)               # exact zero mean
    w = np.linspace(0.5, 1.5, 128)
    b = np.linspace(-0.2, 0.2, 128)
    ln = oracle.ln_fwd(x, w, b, dtype="f64", eps=1e-5, offset=1.0)
    rms = oracle.fwd(x, w, dtype="f64", eps=1e-5, offset=1.0)
    assert np.allclose(ln["y64"] - b, rms["y64"], rtol=1e-13, atol=1e-13)
    assert np.allclose(ln["rstd64"], rms["rstd64"], rtol=1e-14)


def test_ln_n1_and_constant_rows():
    # N = 1 or a constant row: xhat = 0, y = beta, rstd = 1/sqrt(eps) and
    # dx = rstd (g - mean(g)) (zero for N = 1), dgamma = 0, dbeta = dy
    eps = 1e-6
    for x in (np.array([[3.5]]), np.full((1, 8), -2.0)):
        N = x.shape[1]
        gam = np.linspace(0.5, 1.7, N)
        b = np.linspace(-1, 1, N)
        r = oracle.ln_fwd(x, gam, b, dtype="f64", eps=eps, offset=0.0)
        assert np.array_equal(r["y64"], b[None, :])
        assert abs(r["rstd64"][0] - 1000.0) < 1e-9
        dy = np.linspace(0.3, 2.0, N)[None, :]
        d = oracle.ln_bwd(dy, x, gam, dtype="f64", eps=eps, offset=0.0)
        g = dy[0] * gam
        assert np.allclose(d["dx64"][0], 1000.0 * (g - g.mean()), rtol=1e-12, atol=1e-12)
        if N == 1:
            assert d["dx64"][0, 0] == 0.0
        assert np.array_equal(d["db64"], dy[0]) and np.all(d["dg64"] == 0.0)


def test_ln_fwd_storage_rounding_and_fused():
    d = inputs.make_inputs(8, 128, "bf16", 85, residual=True, beta=True, x_shift=0.5)
    r = oracle.ln_fwd(d["x"], d["w"], d["beta"], dtype="bf16", eps=1e-5, offset=0.0)
    assert np.array_equal(r["y"], oracle.bf16_round(r["y64"]))
    f = oracle.ln_fwd(d["x"], d["w"], d["beta"], dtype="bf16", eps=1e-5, offset=0.0, residual=d["residual"])
    hsum = oracle.bf16_round(oracle.to_f64(d["x"], "bf16") + oracle.to_f64(d["residual"], "bf16"))
    assert np.array_equal(f["h"], hsum)
    p = oracle.ln_fwd(hsum, d["w"], d["beta"], dtype="bf16", eps=1e-5, offset=0.0)
    assert np.array_equal(f["y"], p["y"]) and np.array_equal(f["rstd64"], p["rstd64"])


@pytest.mark.parametrize("eps", [1e-5, 0.0])
def test_ln_bwd_sums_and_orthogonality(eps):
    # y is invariant to shifting h, so sum_j dx_j = 0; at eps = 0 it is also
    # invariant to scaling (h - mean), so sum_j dx_j xhat_j = 0
    d = inputs.make_inputs(6, 200, "f32", 86, x_shift=1.0, w_mode="gemma")
    h = d["x"].astype(np.float64)
    r = oracle.ln_bwd(d["dy"].astype(np.float64), h, d["w"].astype(np.float64), dtype="f64", eps=eps,
                      offset=1.0)
    scale = np.abs(r["dx64"]).sum(axis=1)
    assert np.all(np.abs(r["dx64"].sum(axis=1)) <= 1e-12 * scale)
    if eps == 0.0:
        f = oracle.ln_fwd(h, None, None, dtype="f64", eps=0.0, offset=0.0)
        xhat = f["y64"]
        assert np.all(np.abs((r["dx64"] * xhat).sum(axis=1)) <= 1e-12 * scale * np.abs(xhat).max())


@pytest.mark.parametrize("N,eps,offset,fused", [(1, 0.1, 0.0, False), (5, 0.1, 1.0, False), (8, 1e-6, 0.0, True),
                                                 (13, 0.5, 1.0, True)])
def test_ln_bwd_matches_finite_differences(N, eps, offset, fused):
    rng = np.random.default_rng(87 + N)
    M = 3
    x = rng.standard_normal((M, N)) + 0.7
    r = rng.standard_normal((M, N)) if fused else None
    g = rng.standard_normal(N) * 0.3 + (0.0 if offset else 1.0)
    b = rng.standard_normal(N) * 0.1
    dy = rng.standard_normal((M, N))
    dres = rng.standard_normal((M, N)) if fused else None

    def loss(xv, gv, bv, rv):
        f = oracle.ln_fwd(xv, gv, bv, dtype="f64", eps=eps, offset=offset, residual=rv)
        L = (f["y64"] * dy).sum()
        if fused:
            L += ((xv + rv) * dres).sum()
        return L

    h = x + r if fused else x
    d = oracle.ln_bwd(dy, h, g, dtype="f64", eps=eps, offset=offset, dres=dres)
    step = 1e-6
    for arr, grad in ((x, d["dx64"]), (g, d["dg64"]), (b, d["db64"])) + (((r, d["dx64"]),) if fused else ()):
        num = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + step
            lp = loss(x, g, b, r)
            arr[idx] = old - step
            lm = loss(x, g, b, r)
            arr[idx] = old
            num[idx] = (lp - lm) / (2 * step)
        assert np.allclose(num, grad, rtol=1e-6, atol=1e-7), (num, grad)


def test_ln_bwd_param_grads_brute_force_and_given_stats():
    d = inputs.make_inputs(9, 40, "bf16", 88, x_shift=0.3)
    f = oracle.ln_fwd(d["x"], d["w"], None, dtype="bf16", eps=1e-5, offset=0.0)
    r = oracle.ln_bwd(d["dy"], d["x"], d["w"], dtype="bf16", eps=1e-5, offset=0.0, mean=f["mean32"],
                      rstd=f["rstd32"], nthreads=3)
    x = oracle.to_f64(d["x"], "bf16")
    dy = oracle.to_f64(d["dy"], "bf16")
    xhat = (x - f["mean32"].astype(np.float64)[:, None]) * f["rstd32"].astype(np.float64)[:, None]
    dg = np.zeros(40)
    db = np.zeros(40)
    for i in range(9):
        for j in range(40):
            dg[j] += dy[i, j] * xhat[i, j]
            db[j] += dy[i, j]
    assert np.allclose(r["dg64"], dg, rtol=1e-13, atol=1e-13)
    assert np.allclose(r["db64"], db, rtol=1e-13, atol=1e-13)
    assert np.array_equal(r["dg"], oracle.bf16_round(r["dg64"]))


# ---------------------------------------------------- tolerance scales --
# The backward also returns the scales that widen the dx and dW checks in
# the GPU parity tests: dx_scale = rstd (|g| + |xhat c|) [+ |dres|] (the
# terms whose difference is dx), dx_cscale = rstd |xhat| (1/N) sum |g xhat|
# (how far dx moves per unit relative error of the sum behind c) and
# dw_abs = sum over rows of |dy xhat| (the scale of dW's summation error).
# A scale that is too wide would let a wrong kernel pass, so each is pinned
# to values worked out by hand below (not by re-running its formula).

def test_bwd_tolerance_scales_hand_example():
    # Both rows x = (3, 4), w = 1, offset 0, eps 0: rstd = sqrt(2)/5 and
    # xhat = (3 sqrt(2)/5, 4 sqrt(2)/5).
    #   row 0, dy = (1, -1): g xhat = (3, -4) sqrt(2)/5, so c = -sqrt(2)/10
    #          and (1/N) sum |g xhat| = 7 sqrt(2)/10; |xhat c| = (0.12, 0.16)
    #   row 1, dy = (-1, 2): g xhat = (-3, 8) sqrt(2)/5, so c = sqrt(2)/2
    #          and (1/N) sum |g xhat| = 11 sqrt(2)/10; |xhat c| = (0.6, 0.8)
    s2 = math.sqrt(2.0)
    rs = s2 / 5
    x = np.array([[3.0, 4.0], [3.0, 4.0]])
    dy = np.array([[1.0, -1.0], [-1.0, 2.0]])
    r = _bwd64(x, dy, np.ones(2), 0.0, 0.0)
    np.testing.assert_allclose(r["dx64"], [[1.12 * rs, -0.84 * rs], [-1.6 * rs, 1.2 * rs]], rtol=1e-14)
    np.testing.assert_allclose(r["dx_scale"], [[1.12 * rs, 1.16 * rs], [1.6 * rs, 2.8 * rs]], rtol=1e-14)
    # rstd |xhat| cabs: row 0 (3, 4) 7/25 * rs ... = (0.84, 1.12) rs; row 1 (1.32, 1.76) rs
    np.testing.assert_allclose(r["dx_cscale"], [[0.84 * rs, 1.12 * rs], [1.32 * rs, 1.76 * rs]], rtol=1e-14)
    # column 0: |3| + |-3| (times sqrt(2)/5); column 1: |-4| + |8|. The signed
    # sums are 0 and 4 sqrt(2)/5, so |dW| is not the scale.
    np.testing.assert_allclose(r["dw_abs"], [6 * rs, 12 * rs], rtol=1e-14)
    np.testing.assert_allclose(r["dw64"], [0.0, 4 * rs], rtol=1e-14, atol=1e-15)


def test_bwd_tolerance_scales_with_dres_weight_and_offset():
    # Row x = (3, 4), dy = (1, -1), w = (0.5, 1.5) with offset 1 (factor
    # (1.5, 2.5)), dres = (0.5, -0.25): g = (1.5, -2.5),
    # g xhat = (4.5, -10) sqrt(2)/5, c = -5.5 sqrt(2)/10 = -0.55 sqrt(2),
    # (1/N) sum |g xhat| = 14.5 sqrt(2)/10; |xhat c| = (0.66, 0.88).
    s2 = math.sqrt(2.0)
    rs = s2 / 5
    x = np.array([[3.0, 4.0]])
    dy = np.array([[1.0, -1.0]])
    w = np.array([0.5, 1.5])
    dres = np.array([[0.5, -0.25]])
    r = _bwd64(x, dy, w, 0.0, 1.0, dres=dres)
    np.testing.assert_allclose(r["dx64"][0], [rs * (1.5 + 0.66) + 0.5, rs * (-2.5 + 0.88) - 0.25], rtol=1e-14)
    np.testing.assert_allclose(r["dx_scale"][0], [rs * (1.5 + 0.66) + 0.5, rs * (2.5 + 0.88) + 0.25], rtol=1e-14)
    # rstd |xhat| (1/N) sum |g xhat| = rs (3, 4) sqrt(2)/5 * 1.45 sqrt(2) = rs (1.74, 2.32)
    np.testing.assert_allclose(r["dx_cscale"][0], [1.74 * rs, 2.32 * rs], rtol=1e-14)
    # dW and its scale do not see the weight or the offset: sum |dy xhat|
    np.testing.assert_allclose(r["dw_abs"], [3 * rs, 4 * rs], rtol=1e-14)


def test_bwd_tolerance_scales_vanish_with_dy():
    # dy = 0: dx = dres exactly, and the only scale left is |dres|
    x = f64((3, 9), 40)
    dres = f64((3, 9), 41)
    r = _bwd64(x, np.zeros((3, 9)), f64(9, 42, 0.1, 1.0), 1e-3, 0.0, dres=dres)
    np.testing.assert_array_equal(r["dx64"], dres)
    np.testing.assert_array_equal(r["dx_scale"], np.abs(dres))
    np.testing.assert_array_equal(r["dx_cscale"], np.zeros((3, 9)))
    np.testing.assert_array_equal(r["dw_abs"], np.zeros(9))


def test_bwd_tolerance_scales_bound_each_term():
    # Random rows: each scale is at least the magnitude it bounds (the
    # triangle inequality), and dw_abs is the brute-force sum of |dy xhat|.
    x = f64((7, 33), 43)
    dy = f64((7, 33), 44)
    w = f64(33, 45, 0.1, 1.0)
    dres = f64((7, 33), 46)
    r = _bwd64(x, dy, w, 1e-6, 0.0, dres=dres)
    assert np.all(np.abs(r["dx64"]) <= r["dx_scale"] * (1 + 1e-14))
    rstd = 1 / np.sqrt(np.mean(x * x, axis=1) + 1e-6)
    xhat = x * rstd[:, None]
    g = dy * w[None, :]
    c = np.mean(g * xhat, axis=1)
    assert np.all(rstd[:, None] * np.abs(xhat * c[:, None]) <= r["dx_cscale"] * (1 + 1e-14))
    brute = np.zeros(33)
    for i in range(7):
        for j in range(33):
            brute[j] += abs(dy[i, j] * xhat[i, j])
    np.testing.assert_allclose(r["dw_abs"], brute, rtol=1e-13)


def test_ln_bwd_tolerance_scales_hand_example():
    # gamma = 1, offset 0, eps 0.
    #   row 0: x = (1, 1, 3, 3): mean 2, var 1, rstd 1, xhat = (-1, -1, 1, 1);
    #          dy = (1, -2, 0, 3): mean(g) = 0.5, mean|g| = 1.5,
    #          g xhat = (-1, 2, 0, 3): c = 1, mean|g xhat| = 1.5;
    #          dx = g - 0.5 - xhat = (1.5, -1.5, -1.5, 1.5)
    #   row 1: x = (0, 0, 0, 4): mean 1, var 3, rstd = 1/sqrt(3),
    #          xhat = (-1, -1, -1, 3)/sqrt(3); dy = (1, 0, 0, 1):
    #          mean(g) = mean|g| = 0.5, c = 1/(2 sqrt(3)), mean|g xhat| = 1/sqrt(3)
    r3 = 1 / math.sqrt(3.0)
    x = np.array([[1.0, 1.0, 3.0, 3.0], [0.0, 0.0, 0.0, 4.0]])
    dy = np.array([[1.0, -2.0, 0.0, 3.0], [1.0, 0.0, 0.0, 1.0]])
    r = oracle.ln_bwd(dy, x, np.ones(4), dtype="f64", eps=0.0, offset=0.0)
    np.testing.assert_allclose(r["dx64"][0], [1.5, -1.5, -1.5, 1.5], rtol=1e-14)
    # rstd (|g| + |mean g| + |xhat c|)
    np.testing.assert_allclose(r["dx_scale"][0], [2.5, 3.5, 1.5, 4.5], rtol=1e-14)
    np.testing.assert_allclose(r["dx_scale"][1], [r3 * (1 + 0.5 + 1 / 6), r3 * (0.5 + 1 / 6), r3 * (0.5 + 1 / 6),
                                                  r3 * (1 + 0.5 + 0.5)], rtol=1e-14)
    # rstd (mean|g| + |xhat| mean|g xhat|)
    np.testing.assert_allclose(r["dx_cscale"][0], [3.0, 3.0, 3.0, 3.0], rtol=1e-14)
    np.testing.assert_allclose(r["dx_cscale"][1], [r3 * (0.5 + 1 / 3)] * 3 + [r3 * 1.5], rtol=1e-14)
    # dgamma: sum dy xhat = (-1 - r3, 2, 0, 3 + sqrt(3)); its scale sum |dy xhat|
    np.testing.assert_allclose(r["dg64"], [-1 - r3, 2.0, 0.0, 3 + math.sqrt(3.0)], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(r["dg_abs"], [1 + r3, 2.0, 0.0, 3 + math.sqrt(3.0)], rtol=1e-14, atol=1e-15)
    # dbeta: sum dy = (2, -2, 0, 4); its scale sum |dy| = (2, 2, 0, 4)
    np.testing.assert_allclose(r["db64"], [2.0, -2.0, 0.0, 4.0], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(r["db_abs"], [2.0, 2.0, 0.0, 4.0], rtol=1e-14, atol=1e-15)


def test_ln_bwd_tolerance_scale_takes_dres():
    # the fused variant adds |dres| to the scale, as it adds dres to dx
    x = np.array([[1.0, 1.0, 3.0, 3.0]])
    dy = np.array([[1.0, -2.0, 0.0, 3.0]])
    dres = np.array([[0.25, -0.5, 1.0, -2.0]])
    r = oracle.ln_bwd(dy, x, np.ones(4), dtype="f64", eps=0.0, offset=0.0, dres=dres)
    np.testing.assert_allclose(r["dx64"][0], [1.75, -2.0, -0.5, -0.5], rtol=1e-14)
    np.testing.assert_allclose(r["dx_scale"][0], [2.75, 4.0, 2.5, 6.5], rtol=1e-14)
