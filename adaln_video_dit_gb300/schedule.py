"""Dual-constraint bucketing and cost-model fitting (host side).

AdaptiveLoad, Technical summary section 2.A: a bucket of sequence length S
gets the batch size

    B_shape(S) = max(1, min(floor(M_mem / S), floor(M_comp / S**p)))

(a linear memory constraint B*S <= M_mem and a polynomial compute constraint
B*S**p <= M_comp), and the exponent p and bound M_comp come from "Shape
Benchmarking": timing steps over a grid of (B, S) and fitting

    step_time ~ a + b * B * S**p

by non-linear regression.  This module holds those two pieces and a shape
benchmark of the fused AdaLN operator itself (whose cost is linear in tokens,
so its fit gives p close to 1; a whole DiT block, dominated by attention,
gives p close to 2).
"""
import math

import numpy as np


def b_shape(S, m_mem, m_comp, p=2.0):
    """Batch size of a bucket of sequence length S."""
    if S <= 0:
        raise ValueError("S must be positive")
    return max(1, min(int(m_mem // S), int(math.floor(m_comp / float(S) ** p))))


def bucket_plan(lengths, m_mem, m_comp, p=2.0):
    """{S: B_shape(S)} for the distinct lengths of a corpus."""
    return {int(S): b_shape(int(S), m_mem, m_comp, p) for S in sorted(set(lengths))}


def cost_model(B, S, a, b, p):
    return a + b * np.asarray(B, float) * np.asarray(S, float) ** p


def fit_cost_model(B, S, t, p0=1.5, p_bounds=(0.5, 3.0)):
    """Least-squares fit of t ~ a + b*B*S**p.  Returns (a, b, p).

    For a fixed p the model is linear in (a, b), so the fit scans p with a
    golden-section search on the residual of the linear least-squares
    solution (variable projection); no starting values for a, b are needed.
    Relative residuals are minimised, so long and short steps weigh alike.
    """
    B = np.asarray(B, float)
    S = np.asarray(S, float)
    t = np.asarray(t, float)
    if not (B.shape == S.shape == t.shape) or B.size < 3:
        raise ValueError("need at least three (B, S, t) samples of equal shape")
    w = 1.0 / np.maximum(np.abs(t), 1e-30)

    def solve(p):
        A = np.stack([np.ones_like(B), B * S ** p], axis=1) * w[:, None]
        coef, *_ = np.linalg.lstsq(A, t * w, rcond=None)
        r = A @ coef - t * w
        return float(r @ r), coef

    lo, hi = p_bounds
    g = (math.sqrt(5.0) - 1.0) / 2.0
    x1, x2 = hi - g * (hi - lo), lo + g * (hi - lo)
    f1, f2 = solve(x1)[0], solve(x2)[0]
    for _ in range(100):
        if f1 <= f2:
            hi, x2, f2 = x2, x1, f1
            x1 = hi - g * (hi - lo)
            f1 = solve(x1)[0]
        else:
            lo, x1, f1 = x1, x2, f2
            x2 = lo + g * (hi - lo)
            f2 = solve(x2)[0]
        if hi - lo < 1e-10:
            break
    p = 0.5 * (lo + hi)
    _, (a, b) = solve(p)
    return float(a), float(b), float(p)


def m_comp_for_step_time(a, b, tau):
    """Compute bound M_comp that keeps a + b*B*S**p at or below tau."""
    if tau <= a:
        raise ValueError("target step time is below the fixed cost a")
    return (tau - a) / b


def shape_benchmark(shapes, D=5120, steps=20, warmup=3, seed=0):
    """Time the fused AdaLN forward + backward (bf16, on the current CUDA
    device) for each (B, S) in `shapes`; one segment per sample.  Returns a
    list of (B, S, ms): GPU time per step of back-to-back steps.  Outputs and
    workspace are allocated once, and the steps are queued behind a short
    device-side delay, so the host's per-call time is never on the measured
    path.  Needs a GPU and libadaln.so."""
    import torch

    from . import _lib as L
    from .autograd import sample_seg_ids

    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    out = []
    for B, S in shapes:
        T = B * S
        x = torch.randn(T, D, device="cuda", generator=g).to(torch.bfloat16)
        dy = torch.randn(T, D, device="cuda", generator=g).to(torch.bfloat16)
        mod = torch.randn(B, D, device="cuda", generator=g).to(torch.bfloat16)
        seg = sample_seg_ids(B, S, device="cuda")
        ws = torch.empty(L.adaln_bwd_workspace_size(T, D, B, torch.bfloat16), device="cuda",
                         dtype=torch.uint8)
        y, dx = torch.empty_like(x), torch.empty_like(x)
        m = torch.empty(T, device="cuda")
        r = torch.empty(T, device="cuda")
        dsh = torch.empty(B, D, device="cuda")
        dsc = torch.empty(B, D, device="cuda")

        def step():
            L.adaln_fwd(x, mod, mod, seg, 1e-6, y=y, mean=m, rstd=r)
            L.adaln_bwd(dy, x, m, r, mod, seg, dx=dx, dshift=dsh, dscale=dsc, workspace=ws)

        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(int(2e7))  # ~10 ms: the host queues every step meanwhile
        e0.record()
        for _ in range(steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        out.append((B, S, e0.elapsed_time(e1) / steps))
    return out
