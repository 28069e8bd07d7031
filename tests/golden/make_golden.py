"""Write the oracle regression fixture ``small_f32_64x256.json``.

The RMSNorm pages print no worked numeric example, so no stored value here
comes from them. This fixture is the CPU oracle's own output on the seeded
64 x 256 fp32 workload (x, dy ~ N(0,1), w = 1 + 0.1 N(0,1), eps 1e-6,
offset 0). It guards the oracle against unintended changes; the oracle's
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


if __name__ == "__main__":
    main()
