"""Writes qlinear_s8_yscale.json: the y_scale input of the int8 QLinearMatMul workload.

The workload asks for a per-tensor y_scale under which about 1% of the outputs
saturate (with y_zero_point = -9, an output saturates when x / y_scale rounds
above 136 or below -119).  This script draws the workload's seeded a, b, scales
and zero points (workloads.qlinear_s8), takes the first ROWS rows of a, computes
their exact int32 accumulators with the oracle (oracle.matmul on the
zero-point-shifted operands), forms the real values x = a_scale*b_scale*acc in
float64 and stores y_scale = the 99th percentile of max(x / 136.5, -x / 119.5),
rounded to float32.  It calls nothing but the oracle and the input generator.

    python tests/golden/make_qlinear_yscale.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads  # noqa: E402

ROWS = 64


def main():
    d = workloads.qlinear_s8(device="cpu", y_scale=1.0)
    a = d["a"][:ROWS].numpy().astype(np.int64) - d["a_zero_point"][:ROWS].numpy().astype(np.int64)
    b = d["b"].numpy().astype(np.int64) - d["b_zero_point"].numpy().astype(np.int64)
    acc = oracle.matmul(a, b)                       # exact (|acc| < 2^31 here)
    x = d["a_scale"][:ROWS].numpy().astype(np.float64) * d["b_scale"].numpy().astype(np.float64) * acc
    t = np.maximum(x / 136.5, -x / 119.5)
    y_scale = float(np.float32(np.quantile(t, 0.99)))
    out = {"y_scale": y_scale, "rows_sampled": ROWS, "quantile": 0.99,
           "written_by": "tests/golden/make_qlinear_yscale.py (oracle.matmul on seeded workload inputs)"}
    with open(os.path.join(HERE, "qlinear_s8_yscale.json"), "w") as f:
        json.dump(out, f, indent=1)
    print(out)


if __name__ == "__main__":
    main()
