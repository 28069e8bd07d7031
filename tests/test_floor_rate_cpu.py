"""How often a correct fp32 evaluation of dx needs the cancellation floor.

The GPU parity tests accept a dx element that is not within 1 bf16 ulp of
the oracle if it lies within the cancellation floor (the fp32 rounding bound
of g - xhat c plus the summation error of c), and cap how many elements may
use it (helpers.FLOOR_RATE_CAP). This file grounds that cap on the CPU: an
fp32 evaluation in numpy, each step rounded to binary32 (the products, the
row sum of g x, c, xhat, the difference and the final scaling, in the
kernel's order of operations), checked against the oracle exactly as the GPU
output is. Its rate of floor uses must sit well under the cap; an
evaluation with a deliberately coarse c (a relative error of 2^-12, far
beyond fp32 summation error) must exceed it, so the cap separates rounding
noise from a wrong step.

The oracle follows the backward of the Liger-Kernel page "perf(cutedsl):
add Blackwell fast path to RMSNorm" (llama mode) restated in the oracle's
header.
"""
import numpy as np

import oracle
from helpers import FLOOR_RATE_CAP, FLOOR_ULPS, reduction_ulps, ulp16_distance
from row_wise_normalization_rmsnorm_gb300 import inputs


def _fp32_dx(d, rstd32, c_rel_err=0.0):
    """dx in binary32 arithmetic, each operation rounded once."""
    x = oracle.to_f64(d["x"], "bf16").astype(np.float32)
    dy = oracle.to_f64(d["dy"], "bf16").astype(np.float32)
    w = oracle.to_f64(d["w"], "bf16").astype(np.float32)
    N = x.shape[1]
    r = rstd32.astype(np.float32)[:, None]
    g = dy * w[None, :]                                    # rounded products
    s = np.sum(g * x, axis=1, dtype=np.float32)            # fp32 pairwise row sum
    c = (s * r[:, 0]) / np.float32(N)
    c = (c.astype(np.float64) * (1.0 + c_rel_err)).astype(np.float32)
    xh = x * r
    # g - xhat c as one fused multiply-add (the product is exact in double)
    t = (g.astype(np.float64) - xh.astype(np.float64) * c[:, None].astype(np.float64)).astype(np.float32)
    return t * r


def _floor_uses(d, c_rel_err=0.0):
    f = oracle.fwd(d["x"], d["w"], dtype="bf16", eps=1e-6, offset=0.0, nthreads=4)
    b = oracle.bwd(d["dy"], d["x"], d["w"], dtype="bf16", eps=1e-6, offset=0.0, rstd=f["rstd32"], nthreads=4)
    v = _fp32_dx(d, f["rstd32"], c_rel_err)
    got = oracle.bf16_round(v.astype(np.float64))
    vd = oracle.to_f64(got, "bf16")
    N = v.shape[1]
    ok = ulp16_distance(got, b["dx"]) <= 1
    floor = FLOOR_ULPS * b["dx_scale"] + reduction_ulps(N) * b["dx_cscale"]
    near = np.abs(vd - b["dx64"]) <= floor
    return int((~ok).sum()), int((~ok & ~near).sum()), v.size


def test_correct_fp32_evaluation_stays_under_the_floor_cap():
    used = total = 0
    for M, N, seed, dys in ((1024, 8192, 901, 1.0), (2048, 2048, 902, 0.01)):
        d = inputs.make_inputs(M, N, "bf16", seed, dy_scale=dys)
        n, outside, size = _floor_uses(d)
        assert outside == 0          # the floor bounds every correct evaluation
        used += n
        total += size
    # some elements do need it (the floor is not vacuous) ...
    assert used > 0
    # ... but at under half the cap's rate
    assert used <= 0.5 * FLOOR_RATE_CAP * total, (used, total)


def test_a_coarse_row_sum_exceeds_the_cap():
    d = inputs.make_inputs(1024, 8192, "bf16", 903)
    n, _, size = _floor_uses(d, c_rel_err=2.0 ** -12)
    assert n > 2 + FLOOR_RATE_CAP * size, (n, size)
