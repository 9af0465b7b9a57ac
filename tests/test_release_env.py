"""The release library reads no environment variable.

Launch-shape sweep variables (ADALN_RING_KB, ADALN_CTAS_PER_SM,
ADALN_FWD_SCHED) exist only in the tuning build (-DADALN_TUNING).  Were the
release library to honour them, the backward's grid, and with it the
summation order of dscale/dshift, would depend on the environment.
"""
import json
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "adaln_video_dit_gb300", "csrc")
KNOBS = {"ADALN_RING_KB": "32", "ADALN_CTAS_PER_SM": "1", "ADALN_FWD_SCHED": "device"}


def test_getenv_only_in_tuning_blocks():
    """Every getenv in the CUDA sources sits inside #ifdef ADALN_TUNING."""
    for name in sorted(os.listdir(CSRC)):
        if not name.endswith((".cu", ".cuh", ".h")):
            continue
        depth, tuning = 0, []
        with open(os.path.join(CSRC, name)) as f:
            for n, line in enumerate(f, 1):
                s = line.strip()
                if s.startswith("#if"):
                    tuning.append(s.startswith("#ifdef ADALN_TUNING"))
                elif s.startswith("#endif"):
                    tuning.pop()
                if re.search(r"\bgetenv\s*\(", s) and not s.startswith("//"):
                    assert any(tuning), f"{name}:{n} reads the environment outside ADALN_TUNING"
        assert not tuning, f"{name}: unbalanced #if"


CHILD = r"""
import hashlib, json, sys
sys.path.insert(0, %(root)r)
import numpy as np, torch
from adaln_video_dit_gb300 import _lib as L, inputs as I
out = {}
for which in (L.ADALN_KERNEL_FWD, L.ADALN_KERNEL_BWD_ROWS):
    for T, D, nseg in ((36864, 3072, 16), (32760, 5120, 1), (8192, 1536, 2)):
        out[f"{which}_{T}_{D}"] = L.adaln_launch_shape(which, T, D, nseg, torch.bfloat16)
c = I.random_case(5, 20000, 3072, 7, dtype="bf16")
bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
x, dy, sh, sc = (bf(c[k]) for k in ("x", "dy", "shift", "scale"))
seg = torch.from_numpy(c["seg_id"]).cuda()
y, m, r = L.adaln_fwd(x, sh, sc, seg, c["eps"])
dx, dsh, dsc = L.adaln_bwd(dy, x, m, r, sc, seg)
torch.cuda.synchronize()
for k, t in (("y", y), ("dx", dx), ("dshift", dsh), ("dscale", dsc)):
    out[k] = hashlib.sha256(t.cpu().contiguous().view(torch.uint8).numpy().tobytes()).hexdigest()
print(json.dumps(out))
"""


def _child(env_extra):
    env = {k: v for k, v in os.environ.items() if k not in KNOBS}
    env.update(env_extra)
    r = subprocess.run([sys.executable, "-c", CHILD % {"root": ROOT}], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.gpu
def test_release_library_ignores_tuning_variables(adaln):
    plain = _child({})
    knobs = _child(KNOBS)
    assert plain == knobs
