"""GPU parity of the forward with E4M3 (fp8) output against the oracle.

y = E4M3(y' * s), y' the fp32 forward: per-tensor scaling with a given scale
(and the reported amax and 1/scale), per-row scaling with s_i = 448 / the
row's max |y'| (and the reported 1/s_i). Codes are compared with the
oracle's rounding of the exact scaled value; near a rounding midpoint either
neighbour is accepted (helpers.check_fp8). Shapes cover every plan family
the E4M3 kernels are built for: sub-warp and multi-warp teams, single-CTA
rows, cluster rows (bf16 N > 16384), and the generic kernel.
"""
import numpy as np
import pytest
import torch

import oracle
from helpers import check_fp8, check_rel, check_rstd, to_dev, to_host
from row_wise_normalization_rmsnorm_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rn():
    from row_wise_normalization_rmsnorm_gb300 import build
    build.build()
    import row_wise_normalization_rmsnorm_gb300 as pkg
    return pkg


def _run(rn, d, dt, scaling, scale=None, eps=1e-6, offset=0.0, fused=False, offset_elems=0, expect_path=None,
         amax=True, wdt=None):
    """wdt: the weight's storage type (default the activations')."""
    M, N = d["x"].shape
    x = to_dev(d["x"], dt, offset=offset_elems)
    w = to_dev(d["w"], wdt or dt, offset=offset_elems) if d["w"] is not None else None
    res = to_dev(d["residual"], dt, offset=offset_elems) if fused else None
    sc = torch.tensor([scale], dtype=torch.float32, device="cuda") if scale is not None else None
    buf = torch.full((M * N + offset_elems + 16,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN codes
    y = buf[offset_elems:offset_elems + M * N].view(M, N)
    out = rn.rmsnorm_fwd_fp8(x, w, scaling=scaling, scale=sc, residual=res, eps=eps, offset=offset, y=y,
                             amax=amax)
    f = oracle.fwd_fp8(d["x"], d["w"], dtype=dt, eps=eps, offset=offset, scaling=scaling, scale=scale,
                       residual=d.get("residual") if fused else None, wdtype=wdt)
    torch.cuda.synchronize()
    assert torch.all(buf[offset_elems + M * N:] == 0xFF), "store past the end of y"
    ties = check_fp8(y.cpu().numpy(), f)
    # exact midpoints are common: bf16 products scaled by 448 / amax often
    # land on one, and then the last fp32 bit decides
    assert ties <= max(2, M * N // 1000), ties
    check_rstd(out["rstd"].cpu().numpy(), f["rstd64"])
    if scaling == "row":
        check_rel(out["scale_inv"].cpu().numpy(), f["scale_inv"], 2.0 ** -19, "scale_inv")
    else:
        assert out["scale_inv"].item() == np.float32(1.0) / np.float32(scale)
    if amax:
        check_rel(out["amax"].cpu().numpy(), [f["amax"]], 2.0 ** -19, "amax")
    if fused:
        assert np.array_equal(to_host(out["residual_out"], dt), f["h"])
    if expect_path is not None:
        # "vector": a fast path (rows wider than 2048 chunks stream through shared memory)
        fast = ("vector", "staged") if expect_path == "vector" else (expect_path,)
        assert out["plan"]["path_name"] in fast, out["plan"]
    return out, f


SHAPES = [(333, 64), (257, 1024), (300, 4096), (129, 8192), (65, 16384), (101, 8193), (40, 3), (33, 32768),
          (17, 40968)]


@pytest.mark.parametrize("dt", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("M,N", SHAPES)
@pytest.mark.parametrize("scaling", ["row", "tensor"])
def test_fp8_shapes(rn, dt, M, N, scaling):
    d = inputs.make_inputs(M, N, dt, 150 + N % 17, outlier_frac=0.01)
    es = 4 if dt == "f32" else 2
    path = "vector" if (N * es) % 16 == 0 else "generic"
    _run(rn, d, dt, scaling, scale=37.5 if scaling == "tensor" else None, expect_path=path)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("M,N", [(333, 64), (257, 1024), (129, 8192), (65, 16384), (33, 32768), (40, 3),
                                 (101, 8193)])
@pytest.mark.parametrize("scaling", ["row", "tensor"])
@pytest.mark.parametrize("fused", [False, True])
def test_fp8_fp32_weight(rn, dt, M, N, scaling, fused):
    """An fp32 weight beside 16-bit activations (the key's wtype apart from
    its itype), on register, staged cluster and generic rows."""
    d = inputs.make_inputs(M, N, dt, 170 + N % 13, outlier_frac=0.01, wdtype="f32", residual=fused)
    path = "vector" if (N * 2) % 16 == 0 else "generic"
    out, _ = _run(rn, d, dt, scaling, scale=21.0 if scaling == "tensor" else None, fused=fused, expect_path=path,
                  wdt="f32")


@pytest.mark.parametrize("dt,N", [("bf16", 32768), ("bf16", 65536), ("f32", 16384), ("f32", 32768)])
def test_fp8_cluster_rows(rn, dt, N):
    d = inputs.make_inputs(9, N, dt, 151)
    out, _ = _run(rn, d, dt, "row", expect_path="vector")
    assert out["plan"]["cluster_size"] > 1


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_fp8_fused_add_gemma(rn, dt):
    d = inputs.make_inputs(513, 4096, dt, 152, w_mode="gemma", residual=True)
    _run(rn, d, dt, "row", offset=1.0, fused=True, expect_path="vector")
    _run(rn, d, dt, "tensor", scale=3.0, offset=1.0, fused=True, expect_path="vector")


def test_fp8_tensor_scale_saturates(rn):
    d = inputs.make_inputs(64, 2048, "bf16", 153)
    out, f = _run(rn, d, "bf16", "tensor", scale=2000.0)
    codes = out["y"].cpu().numpy()
    big = np.abs(f["scaled64"]) >= 448.0
    assert big.any() and np.all((codes[big] & 0x7F) == 0x7E)


def test_fp8_non_affine(rn):
    d = inputs.make_inputs(257, 2048, "bf16", 154)
    d["w"] = None
    _run(rn, d, "bf16", "row", expect_path="vector")


def test_fp8_misaligned_takes_generic(rn):
    d = inputs.make_inputs(300, 2048, "bf16", 155)
    _run(rn, d, "bf16", "row", offset_elems=1, expect_path="generic")


def test_fp8_zero_rows(rn):
    d = inputs.make_inputs(8, 1024, "bf16", 156)
    d["x"][3] = 0
    out, _ = _run(rn, d, "bf16", "row", expect_path="vector")
    assert out["scale_inv"][3].item() == 1.0
    assert torch.all((out["y"][3] & 0x7F) == 0)


def test_fp8_empty_batch_sets_amax_to_zero(rn):
    x = torch.empty((0, 1024), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(1024, dtype=torch.bfloat16, device="cuda")
    amax = torch.full((1,), 5.0, device="cuda")
    out = rn.rmsnorm_fwd_fp8(x, w, scaling="row", amax=amax)
    torch.cuda.synchronize()
    assert out["amax"].item() == 0.0


def test_fp8_full_size_sampled(rn):
    """The bench's shape: every row's scale and amax, codes of sampled rows."""
    M, N = 16384, 8192
    d = inputs.make_inputs(M, N, "bf16", inputs.SWEEP_SEED, outlier_frac=0.01)
    x, w = to_dev(d["x"], "bf16"), to_dev(d["w"], "bf16")
    out = rn.rmsnorm_fwd_fp8(x, w, scaling="row", amax=True)
    torch.cuda.synchronize()
    rows = np.random.default_rng(9).choice(M, 256, replace=False)
    f = oracle.fwd_fp8(d["x"][rows], d["w"], dtype="bf16", eps=1e-6, offset=0.0, scaling="row")
    check_fp8(out["y"].cpu().numpy()[rows], f)
    check_rel(out["scale_inv"].cpu().numpy()[rows], f["scale_inv"], 2.0 ** -19, "scale_inv")
    # the tensor amax is the largest row amax: 448 * max_i scale_inv_i
    si = out["scale_inv"].cpu().numpy().astype(np.float64)
    check_rel(out["amax"].cpu().numpy(), [448.0 * si.max()], 2.0 ** -19, "amax")
    assert out["plan"]["path_name"] in ("vector", "staged")


def test_fp8_codes_match_plain_forward_dequantised(rn):
    """Across the two output types of one kernel family: decode(E4M3) / s
    stays within half an E4M3 step of the bf16 forward's y."""
    d = inputs.make_inputs(512, 4096, "bf16", 157)
    x, w = to_dev(d["x"], "bf16"), to_dev(d["w"], "bf16")
    y16, _ = rn.rmsnorm_fwd(x, w)
    out = rn.rmsnorm_fwd_fp8(x, w, scaling="row")
    torch.cuda.synchronize()
    deq = oracle.e4m3_decode(out["y"].cpu().numpy()) * out["scale_inv"].cpu().numpy()[:, None].astype(np.float64)
    y = y16.float().cpu().numpy().astype(np.float64)
    amax = np.abs(y).max(axis=1, keepdims=True)
    assert np.all(np.abs(deq - y) <= 2.0 ** -4 * np.abs(y) + 2.0 ** -9 * amax / 448.0 + 2.0 ** -8 * np.abs(y))


@pytest.mark.parametrize("N,offs,path", [(4096, 0, "vector"), (32768, 0, "staged"), (4100, 1, "generic")])
@pytest.mark.parametrize("offset", [0.0, 1.0])
def test_fp8_row_scale_is_the_max_of_y_to_the_bit(rn, N, offs, path, offset):
    """Every E4M3 kernel forms y' = (h (offset + w)) rstd in fp32 and takes
    the row's max |y'| as rstd max_j |h_j (offset + w_j)|, which is the same
    number because rounding a product with rstd > 0 is monotone. So the
    reported 1/s is max_j |y'_j| / 448 with y' recomputed here in fp32 from
    the kernel's own rstd (numpy's float32 products round as the GPU's do),
    bit for bit: on the register path, the staged cluster path (whose max
    rides on the first pass's reduction) and the generic path."""
    M = 48
    d = inputs.make_inputs(M, N, "bf16", 177 + N % 13)
    x = to_dev(d["x"], "bf16", offset=offs)
    w = to_dev(d["w"], "bf16", offset=offs)
    out = rn.rmsnorm_fwd_fp8(x, w, scaling="row", offset=offset)
    torch.cuda.synchronize()
    assert out["plan"]["path_name"] == path, out["plan"]
    h = x.float().cpu().numpy()
    g = np.float32(offset) + w.float().cpu().numpy()
    rstd = out["rstd"].cpu().numpy()
    y = (h * g[None, :]).astype(np.float32) * rstd[:, None]
    amax = np.abs(y).max(axis=1)
    want = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    assert y.dtype == np.float32 and np.array_equal(out["scale_inv"].cpu().numpy(), want)
