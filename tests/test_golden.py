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
