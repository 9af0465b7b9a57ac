"""Write tests/golden/oracle_small.json: a regression fixture of the CPU
oracle on a small literal input.

The pages print no worked numeric example for the operator, so no stored value
here comes from them.  This fixture is produced by the oracle alone (nothing
else is called) and guards the oracle against unintended changes; the oracle
itself is pinned by tests/pins.py.  Values are stored as float.hex strings.

Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

# Literal inputs: T = 5 rows, D = 4, two segments (rows 0-2 and 3-4), fp32.
X = [[1.0, 2.0, 3.0, 4.0], [-1.5, 0.5, 0.25, 8.0], [2.0, 2.0, 2.0, 2.0],
     [0.0, -3.0, 1.0, 0.125], [10.0, -10.0, 5.0, -5.0]]
DY = [[0.5, -1.0, 0.25, 2.0], [1.0, 1.0, -1.0, 0.0], [0.75, -0.5, 0.0, 1.5],
      [-2.0, 0.5, 0.5, 1.0], [0.125, 0.25, -0.375, 4.0]]
SHIFT = [[0.1, -0.2, 0.3, 0.0], [1.0, 0.5, -0.5, -1.0]]
SCALE = [[0.5, -0.25, 0.0, 1.0], [-0.5, 0.75, 0.2, 0.1]]
SEG = [0, 0, 0, 1, 1]
EPS = 1e-5


def inputs():
    f = lambda a: np.array(a, np.float32)  # noqa: E731
    return f(X), f(DY), f(SHIFT), f(SCALE), np.array(SEG, np.int32), EPS


def compute():
    x, dy, shift, scale, seg, eps = inputs()
    y, mean, rstd = oracle.adaln_fwd(x, shift, scale, seg, eps)
    dx, dshift, dscale = oracle.adaln_bwd(dy, x, scale, seg, eps)
    return dict(y=y, mean=mean, rstd=rstd, dx=dx, dshift=dshift, dscale=dscale)


def main():
    out = {"note": "oracle regression fixture; inputs are literal in make_golden.py",
           "eps": EPS}
    for k, v in compute().items():
        out[k] = [float(a).hex() for a in np.asarray(v).ravel()]
        out[k + "_shape"] = list(np.asarray(v).shape)
    with open(os.path.join(HERE, "oracle_small.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
