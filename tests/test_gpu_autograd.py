"""The fused operator as an autograd node: gradients against the CPU oracle,
and the tensors it keeps for the backward against the unfused chain."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import gpu_helpers as H
import oracle
from adaln_video_dit_gb300 import autograd as A
from adaln_video_dit_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_autograd_matches_oracle(adaln, dtype):
    B, N, D = 3, 700, 768
    c = I.random_case(91, B * N, D, B, dtype=dtype, lengths=[N] * B, dy_std=1.0)
    x = H.to_dev(c["x"]).view(B, N, D).requires_grad_(True)
    shift = H.to_dev(c["shift"]).requires_grad_(True)
    scale = H.to_dev(c["scale"]).requires_grad_(True)
    seg = A.sample_seg_ids(B, N, device="cuda")
    assert torch.equal(seg.cpu(), torch.from_numpy(c["seg_id"]))
    y = A.AdaLNModulate(c["eps"])(x, shift, scale, seg)
    y.backward(H.to_dev(c["dy"]).view(B, N, D))
    torch.cuda.synchronize()
    y_ref, _, _ = oracle.adaln_fwd(c["x"], c["shift"], c["scale"], c["seg_id"], c["eps"])
    dx_ref, dsh_ref, dsc_ref = oracle.adaln_bwd(c["dy"], c["x"], c["scale"], c["seg_id"], c["eps"])
    H.check_rowwise("y", dtype, H.to_f64(y.reshape(-1, D)), y_ref)
    H.check_rowwise("dx", dtype, H.to_f64(x.grad.reshape(-1, D)), dx_ref)
    # Parameter gradients come back in the parameters' dtype: for bf16
    # parameters one more rounding (2^-9 relative) on top of the fp32 sums.
    lim = 1e-4 if dtype == "f32" else 1e-3 + 2.0 ** -8
    for got, ref in ((shift.grad, dsh_ref), (scale.grad, dsc_ref)):
        assert got.dtype == shift.dtype
        err = H.normwise(H.to_f64(got), ref)
        assert err <= lim, err
    H.status_ok()


def _saved_bytes(fn):
    """Bytes of the distinct storages autograd keeps for the backward."""
    seen = {}

    def pack(t):
        try:
            key = t.untyped_storage().data_ptr()
            seen[key] = max(seen.get(key, 0), t.untyped_storage().nbytes())
        except RuntimeError:
            pass
        return t

    with torch.autograd.graph.saved_tensors_hooks(pack, lambda t: t):
        out = fn()
    return out, sum(seen.values())


def test_one_node_keeps_only_x_and_statistics(adaln):
    """The fused node saves x, mean/rstd (8 B/token), scale and seg_id; the
    unfused chain (layer_norm, gather, multiply, add) keeps the normalised
    activations and the gathered modulation rows as well."""
    B, N, D = 2, 2048, 1024
    dev = "cuda"
    x = torch.randn(B * N, D, device=dev, dtype=torch.bfloat16, requires_grad=True)
    shift = torch.randn(B, D, device=dev, dtype=torch.bfloat16, requires_grad=True)
    scale = torch.randn(B, D, device=dev, dtype=torch.bfloat16, requires_grad=True)
    seg = A.sample_seg_ids(B, N, device=dev)
    _, fused = _saved_bytes(lambda: A.adaln_modulate(x, shift, scale, seg))
    want = x.numel() * 2 + 8 * B * N + scale.numel() * 2 + 4 * B * N
    assert fused == want, (fused, want)

    def unfused():
        idx = seg.long()
        return F.layer_norm(x, (D,), eps=1e-6) * (1 + scale[idx]) + shift[idx]

    _, chain = _saved_bytes(unfused)
    assert chain >= 2.5 * x.numel() * 2, chain  # x, LN output, gathered (1 + scale)
    assert fused < 0.45 * chain
