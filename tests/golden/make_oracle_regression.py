"""Writes oracle_regression_small.json: a frozen fp64 oracle output on a tiny
seeded case.  Calls only the oracle and the seeded input module."""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from selective_state_space_109_b300 import inputs as I  # noqa: E402

spec = dict(batch=2, dim=6, dstate=8, seqlen=40, ngroups=2, io="f32", recipe="scaled",
            seed=3, with_z=True, with_h0=True)
x = I.make_scan_inputs(**spec).as_f64()
y, hf = oracle.scan(**x, return_final_state=True)
out = dict(inputs=spec, y_head=[float(v) for v in y.ravel()[:16]], y_sum=float(np.sum(y)),
           h_final_sumsq=float(np.sum(hf * hf)))
with open(os.path.join(HERE, "oracle_regression_small.json"), "w") as f:
    json.dump(out, f, indent=1)
print("wrote", os.path.join(HERE, "oracle_regression_small.json"))
