"""Write the oracle regression fixtures ``small_f32_64x256.json`` and
``ln_fp8_bf16_32x128.json``.

The RMSNorm pages print no worked numeric example, so no stored value here
comes from them. This fixture is the CPU oracle's own output on the seeded
64 x 256 fp32 workload (x, dy ~ N(0,1), w = 1 + 0.1 N(0,1), eps 1e-6,
offset 0), and its LayerNorm and E4M3 outputs on a seeded 32 x 128 bf16
workload (x ~ N(0.5, 1), beta ~ 0.1 N(0, 1), fused residual add, gemma
offset 1; per-row E4M3 codes). They guard the oracle against unintended
changes; the oracle's
correctness rests on tests/test_oracle_pins.py. Only ``oracle`` and the
seeded input generator are called.

Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from row_wise_normalization_rmsnorm_gb300 import inputs  # noqa: E402

ROWS = (0, 31, 63)


def main():
    arrays, p = inputs.workload_inputs("small_f32")
    f = oracle.fwd(arrays["x"], arrays["w"], dtype="f32", eps=p["eps"], offset=p["offset"])
    b = oracle.bwd(arrays["dy"], arrays["x"], arrays["w"], dtype="f32", eps=p["eps"],
                   offset=p["offset"])
    hx = lambda a: [float(v).hex() for v in a]  # noqa: E731
    out = {
        "workload": "small_f32", "M": p["M"], "N": p["N"], "eps": p["eps"], "offset": p["offset"],
        "seed": p["seed"], "rows": list(ROWS),
        "rstd64": hx(f["rstd64"]),
        "y64": {str(r): hx(f["y64"][r]) for r in ROWS},
        "dx64": {str(r): hx(b["dx64"][r]) for r in ROWS},
        "dw64": hx(b["dw64"]),
    }
    with open(os.path.join(HERE, "small_f32_64x256.json"), "w") as fh:
        json.dump(out, fh, indent=0)

    d = ln_fp8_inputs()
    f = oracle.ln_fwd(d["x"], d["w"], d["beta"], dtype="bf16", eps=1e-5, offset=1.0, residual=d["residual"])
    b = oracle.ln_bwd(d["dy"], f["h"], d["w"], dtype="bf16", eps=1e-5, offset=1.0, mean=f["mean32"],
                      rstd=f["rstd32"], dres=d["dres"])
    q = oracle.fwd_fp8(d["x"], d["w"], dtype="bf16", eps=1e-5, offset=1.0, scaling="row")
    out = {
        "M": 32, "N": 128, "seed": LN_SEED, "eps": 1e-5, "offset": 1.0,
        "ln_y": d_bits(f["y"]), "ln_mean64": hx(f["mean64"]), "ln_rstd64": hx(f["rstd64"]),
        "ln_dx": d_bits(b["dx"]), "ln_dg64": hx(b["dg64"]), "ln_db64": hx(b["db64"]),
        "fp8_codes": q["yq"].reshape(-1).tolist(), "fp8_scale_inv": hx(q["scale_inv"]),
    }
    with open(os.path.join(HERE, "ln_fp8_bf16_32x128.json"), "w") as fh:
        json.dump(out, fh, indent=0)


LN_SEED = 1900


def ln_fp8_inputs():
    return inputs.make_inputs(32, 128, "bf16", LN_SEED, w_mode="gemma", residual=True, dres=True, beta=True,
                              x_shift=0.5)


def d_bits(a):
    return [int(v) for v in a.reshape(-1)]


if __name__ == "__main__":
    main()
