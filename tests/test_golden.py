"""The oracle reproduces its stored regression fixture bit for bit."""
import json
import os

import numpy as np

import oracle
from row_wise_normalization_rmsnorm_gb300 import inputs

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_oracle_matches_stored_fixture():
    with open(os.path.join(HERE, "small_f32_64x256.json")) as fh:
        g = json.load(fh)
    arrays, p = inputs.workload_inputs(g["workload"])
    f = oracle.fwd(arrays["x"], arrays["w"], dtype="f32", eps=p["eps"], offset=p["offset"])
    b = oracle.bwd(arrays["dy"], arrays["x"], arrays["w"], dtype="f32", eps=p["eps"],
                   offset=p["offset"])
    unhex = lambda a: np.array([float.fromhex(v) for v in a])  # noqa: E731
    assert np.array_equal(f["rstd64"], unhex(g["rstd64"]))
    assert np.array_equal(b["dw64"], unhex(g["dw64"]))
    for r in g["rows"]:
        assert np.array_equal(f["y64"][r], unhex(g["y64"][str(r)]))
        assert np.array_equal(b["dx64"][r], unhex(g["dx64"][str(r)]))


def test_oracle_matches_stored_layernorm_and_e4m3_fixture():
    import sys
    sys.path.insert(0, HERE)
    import make_golden
    with open(os.path.join(HERE, "ln_fp8_bf16_32x128.json")) as fh:
        g = json.load(fh)
    d = make_golden.ln_fp8_inputs()
    f = oracle.ln_fwd(d["x"], d["w"], d["beta"], dtype="bf16", eps=g["eps"], offset=g["offset"],
                      residual=d["residual"])
    b = oracle.ln_bwd(d["dy"], f["h"], d["w"], dtype="bf16", eps=g["eps"], offset=g["offset"],
                      mean=f["mean32"], rstd=f["rstd32"], dres=d["dres"])
    q = oracle.fwd_fp8(d["x"], d["w"], dtype="bf16", eps=g["eps"], offset=g["offset"], scaling="row")
    unhex = lambda a: np.array([float.fromhex(v) for v in a])  # noqa: E731
    assert f["y"].reshape(-1).tolist() == g["ln_y"]
    assert np.array_equal(f["mean64"], unhex(g["ln_mean64"]))
    assert np.array_equal(f["rstd64"], unhex(g["ln_rstd64"]))
    assert b["dx"].reshape(-1).tolist() == g["ln_dx"]
    assert np.array_equal(b["dg64"], unhex(g["ln_dg64"]))
    assert np.array_equal(b["db64"], unhex(g["ln_db64"]))
    assert q["yq"].reshape(-1).tolist() == g["fp8_codes"]
    assert np.array_equal(q["scale_inv"], unhex(g["fp8_scale_inv"]))
