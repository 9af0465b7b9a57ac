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


MODES_CHILD = r"""
import ctypes, hashlib, json, sys
sys.path.insert(0, %(root)r)
import numpy as np, torch
from adaln_video_dit_gb300 import build as B, inputs as I
lib = ctypes.CDLL(B.build(tuning=True))
vp = ctypes.c_void_p
lib.adaln_fwd.argtypes = [vp, vp, vp, vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                          ctypes.c_int, ctypes.c_float, vp, vp, vp, vp]
c = I.random_case(9, 20000, 3072, 7, dtype="bf16")
bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
x, sh, sc = (bf(c[k]) for k in ("x", "shift", "scale"))
seg = torch.from_numpy(c["seg_id"]).cuda()
y = torch.empty_like(x); m = torch.empty(c["T"], device="cuda"); r = torch.empty_like(m)
P = lambda t: vp(t.data_ptr())
st = vp(torch.cuda.current_stream().cuda_stream)
assert lib.adaln_fwd(P(x), P(sh), P(sc), P(seg), c["T"], c["D"], c["nseg"], 1,
                     ctypes.c_float(c["eps"]), P(y), P(m), P(r), st) == 0
torch.cuda.synchronize()
print(json.dumps({k: hashlib.sha256(t.cpu().contiguous().view(torch.uint8).numpy().tobytes()).hexdigest()
                  for k, t in (("y", y), ("mean", m), ("rstd", r))}))
"""


@pytest.mark.gpu
def test_forward_claim_modes_give_the_same_bits(adaln):
    """The forward's rows may be streamed by any team (CTA ranges, device-wide
    units, or CTA ranges with a device-wide tail): every row's result is the
    same bit for bit.  The tuning build forces each mode."""
    outs = []
    for mode in ("cta", "device", "hybrid"):
        env = {k: v for k, v in os.environ.items() if k not in KNOBS}
        env["ADALN_FWD_SCHED"] = mode
        r = subprocess.run([sys.executable, "-c", MODES_CHILD % {"root": ROOT}], env=env,
                           capture_output=True, text=True, timeout=900)
        assert r.returncode == 0, r.stderr[-2000:]
        outs.append(json.loads(r.stdout.strip().splitlines()[-1]))
    assert outs[0] == outs[1] == outs[2]
