"""Pins of the CPU oracle: checks against facts fixed by mathematics, not by
the oracle itself.  Each check takes the oracle's ctypes library (so that
tests/test_oracle_mutants.py can run the same checks against copies of the
oracle with planted mistakes) and raises AssertionError on a mismatch.

The operator is the fused AdaLN LayerNorm-Modulate of AdaptiveLoad
("Technical summary" section 2.B): y = xhat * (1 + scale_b) + shift_b with
xhat the biased LayerNorm of the row, and its backward (dx, and dscale_b /
dshift_b reduced over the sequence).
"""
import numpy as np

import oracle as O


def _f64_case(seed, T, D, nseg, lengths=None, x_scale=1.0):
    rng = np.random.default_rng(seed)
    if lengths is None:
        lengths = [T // nseg] * nseg
        lengths[-1] += T - sum(lengths)
    seg = np.repeat(np.arange(nseg, dtype=np.int32), lengths)
    x = rng.standard_normal((T, D)) * x_scale + rng.uniform(-2, 2, size=(T, 1))
    shift = rng.standard_normal((nseg, D)) * 0.5
    scale = rng.standard_normal((nseg, D)) * 0.5
    dy = rng.standard_normal((T, D))
    return x, shift, scale, seg, dy


def pin_closed_form_d2(lib):
    """D = 2: mean, rstd, y and dx in closed form.  With u = (a - b)/2 and
    r = 1/sqrt(u^2 + eps): xhat = (u r, -u r); dx_0 = -dx_1 = eps r^3 (g0 - g1)/2."""
    eps = 0.37
    x = np.array([[3.0, -1.0], [0.25, 2.0], [-5.0, -4.5]])
    shift = np.array([[0.1, -0.3]])
    scale = np.array([[0.7, -0.2]])
    dy = np.array([[1.5, -0.5], [2.0, 0.25], [-1.0, 3.0]])
    seg = np.zeros(3, np.int32)
    y, mean, rstd = O.adaln_fwd(x, shift, scale, seg, eps, lib=lib)
    dx, dshift, dscale = O.adaln_bwd(dy, x, scale, seg, eps, lib=lib)
    for t in range(3):
        a, b = x[t]
        u = (a - b) / 2
        r = 1.0 / np.sqrt(u * u + eps)
        assert abs(mean[t] - (a + b) / 2) < 1e-15
        assert abs(rstd[t] - r) < 1e-14 * r
        xh = np.array([u * r, -u * r])
        np.testing.assert_allclose(y[t], xh * (1 + scale[0]) + shift[0], rtol=1e-14, atol=1e-14)
        g = dy[t] * (1 + scale[0])
        d0 = eps * r ** 3 * (g[0] - g[1]) / 2
        np.testing.assert_allclose(dx[t], [d0, -d0], rtol=1e-13, atol=1e-15)
    xh_all = np.stack([np.array([(a - b) / 2, (b - a) / 2]) / np.sqrt(((a - b) / 2) ** 2 + eps)
                       for a, b in x])
    np.testing.assert_allclose(dshift[0], dy.sum(0), rtol=1e-15, atol=1e-15)
    np.testing.assert_allclose(dscale[0], (dy * xh_all).sum(0), rtol=1e-13, atol=1e-15)


def pin_constant_rows(lib):
    """A constant row has var = 0: xhat = 0, so y = shift exactly,
    rstd = 1/sqrt(eps), and dx = rstd (g - mean(g))."""
    eps = 1e-2
    T, D = 4, 8
    x = np.repeat(np.array([[2.5], [-1.0], [0.0], [7.0]]), D, axis=1)
    rng = np.random.default_rng(11)
    shift = rng.standard_normal((2, D))
    scale = rng.standard_normal((2, D))
    dy = rng.standard_normal((T, D))
    seg = np.array([0, 0, 1, 1], np.int32)
    y, mean, rstd = O.adaln_fwd(x, shift, scale, seg, eps, lib=lib)
    assert np.array_equal(y, shift[seg])
    np.testing.assert_allclose(mean, x[:, 0], rtol=0, atol=0)
    np.testing.assert_allclose(rstd, 1 / np.sqrt(eps), rtol=1e-15)
    dx, dshift, dscale = O.adaln_bwd(dy, x, scale, seg, eps, lib=lib)
    g = dy * (1 + scale[seg])
    np.testing.assert_allclose(dx, (g - g.mean(1, keepdims=True)) / np.sqrt(eps),
                               rtol=1e-13, atol=1e-13)
    assert np.all(dscale == 0.0)
    np.testing.assert_allclose(dshift, np.stack([dy[:2].sum(0), dy[2:].sum(0)]),
                               rtol=1e-15, atol=1e-15)


def pin_row_invariants(lib):
    """Per row: sum_d xhat = 0; mean_d xhat^2 = var/(var + eps) with var from
    numpy; sum_d dx = 0; sum_d dx xhat = rstd (sum_d g xhat) eps/(var + eps)."""
    eps = 0.05
    x, shift, scale, seg, dy = _f64_case(5, 16, 24, 2)
    zeros = np.zeros_like(shift)
    xhat, _, rstd = O.adaln_fwd(x, zeros, zeros, seg, eps, lib=lib)
    var = x.var(axis=1)
    np.testing.assert_allclose(xhat.sum(1), 0, atol=1e-12)
    np.testing.assert_allclose((xhat ** 2).mean(1), var / (var + eps), rtol=1e-12)
    np.testing.assert_allclose(rstd, 1 / np.sqrt(var + eps), rtol=1e-13)
    dx, _, _ = O.adaln_bwd(dy, x, scale, seg, eps, lib=lib)
    g = dy * (1 + scale[seg])
    np.testing.assert_allclose(dx.sum(1), 0, atol=1e-11)
    rhs = rstd * (g * xhat).sum(1) * eps / (var + eps)
    np.testing.assert_allclose((dx * xhat).sum(1), rhs, rtol=1e-9, atol=1e-12)


def _loss(x, shift, scale, seg, dy, eps, lib):
    y, _, _ = O.adaln_fwd(x, shift, scale, seg, eps, lib=lib)
    return float((y * dy).sum())


def pin_finite_differences(lib):
    """Central differences (fp64, h = 1e-6) of L = sum y * dy with respect to
    x, scale and shift match dx, dscale and dshift."""
    h = 1e-6
    for eps in (0.3, 1e-6):
        x, shift, scale, seg, dy = _f64_case(7, 5, 6, 2, lengths=[3, 2])
        dx, dshift, dscale = O.adaln_bwd(dy, x, scale, seg, eps, lib=lib)

        def fd(arr, which):
            out = np.empty_like(arr)
            for idx in np.ndindex(arr.shape):
                ap, am = arr.copy(), arr.copy()
                ap[idx] += h
                am[idx] -= h
                args_p = dict(x=x, shift=shift, scale=scale)
                args_m = dict(x=x, shift=shift, scale=scale)
                args_p[which], args_m[which] = ap, am
                lp = _loss(args_p["x"], args_p["shift"], args_p["scale"], seg, dy, eps, lib)
                lm = _loss(args_m["x"], args_m["shift"], args_m["scale"], seg, dy, eps, lib)
                out[idx] = (lp - lm) / (2 * h)
            return out

        for got, which in ((dx, "x"), (dscale, "scale"), (dshift, "shift")):
            want = fd({"x": x, "scale": scale, "shift": shift}[which], which)
            err = np.abs(got - want).max() / max(np.abs(want).max(), 1e-12)
            assert err < 1e-6, f"d{which}: relative error {err:.3g} at eps={eps}"


def pin_torch_layer_norm(lib):
    """Library special case: per segment, y = F.layer_norm(x_b, (D,),
    weight = 1 + scale_b, bias = shift_b, eps) in torch CPU fp64, and its
    autograd gives dx, dscale_b (= weight.grad) and dshift_b (= bias.grad).
    Includes an empty segment (its gradients are zero)."""
    import torch
    import torch.nn.functional as F
    eps = 1e-5
    T, D = 40, 32
    x, shift, scale, seg, dy = _f64_case(9, T, D, 4, lengths=[10, 0, 25, 5], x_scale=3.0)
    y, mean, rstd = O.adaln_fwd(x, shift, scale, seg, eps, lib=lib)
    dx, dshift, dscale = O.adaln_bwd(dy, x, scale, seg, eps, lib=lib)
    for b in range(4):
        rows = np.nonzero(seg == b)[0]
        if rows.size == 0:
            assert np.all(dshift[b] == 0) and np.all(dscale[b] == 0)
            continue
        xt = torch.tensor(x[rows], dtype=torch.float64, requires_grad=True)
        w = torch.tensor(1 + scale[b], dtype=torch.float64, requires_grad=True)
        bb = torch.tensor(shift[b], dtype=torch.float64, requires_grad=True)
        yt = F.layer_norm(xt, (D,), w, bb, eps)
        yt.backward(torch.tensor(dy[rows], dtype=torch.float64))
        np.testing.assert_allclose(y[rows], yt.detach().numpy(), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dx[rows], xt.grad.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dscale[b], w.grad.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dshift[b], bb.grad.numpy(), rtol=1e-12, atol=1e-12)


def pin_unfused_numpy(lib):
    """Brute-force unfused chain in numpy: LayerNorm from np.mean / np.var,
    then the multiply, then the add, as three separate array steps."""
    eps = 1e-6
    x, shift, scale, seg, dy = _f64_case(13, 33, 40, 3, lengths=[1, 30, 2])
    ln = (x - x.mean(1, keepdims=True)) / np.sqrt(x.var(1, keepdims=True) + eps)
    mul = ln * (1 + scale[seg])
    want = mul + shift[seg]
    y, _, _ = O.adaln_fwd(x, shift, scale, seg, eps, lib=lib)
    np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-12)


def pin_integer_dshift(lib):
    """dshift is the per-segment column sum of dy: with small integer dy in
    fp32 the sum is exact, so the comparison is bit-exact.  Segments are not
    required to be sorted by the definition."""
    rng = np.random.default_rng(17)
    T, D, nseg = 300, 16, 5
    seg = rng.integers(0, nseg, size=T).astype(np.int32)
    dy = rng.integers(-8, 9, size=(T, D)).astype(np.float32)
    x = rng.standard_normal((T, D)).astype(np.float32)
    scale = rng.standard_normal((nseg, D)).astype(np.float32)
    _, dshift, _ = O.adaln_bwd(dy, x, scale, seg, 1e-6, want_dx=False, lib=lib)
    want = np.zeros((nseg, D))
    for b in range(nseg):
        want[b] = dy[seg == b].astype(np.int64).sum(0)
    assert np.array_equal(dshift, want)


def pin_bf16_widening(lib):
    """bf16 inputs are widened exactly: the same values given as float64 give
    bit-identical results."""
    from adaln_video_dit_gb300 import inputs as I
    c = I.random_case(3, 20, 16, 2, dtype="bf16", lengths=[12, 8])
    xf = I.bf16_bits_to_f32(c["x"]).astype(np.float64)
    shf = I.bf16_bits_to_f32(c["shift"]).astype(np.float64)
    scf = I.bf16_bits_to_f32(c["scale"]).astype(np.float64)
    dyf = I.bf16_bits_to_f32(c["dy"]).astype(np.float64)
    a = O.adaln_fwd(c["x"], c["shift"], c["scale"], c["seg_id"], c["eps"], lib=lib)
    b = O.adaln_fwd(xf, shf, scf, c["seg_id"], c["eps"], lib=lib)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    a = O.adaln_bwd(c["dy"], c["x"], c["scale"], c["seg_id"], c["eps"], lib=lib)
    b = O.adaln_bwd(dyf, xf, scf, c["seg_id"], c["eps"], lib=lib)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


ALL = [pin_closed_form_d2, pin_constant_rows, pin_row_invariants,
       pin_finite_differences, pin_torch_layer_norm, pin_unfused_numpy,
       pin_integer_dshift, pin_bf16_widening]
