"""The fused AdaLN operator as one autograd node.

AdaptiveLoad (Technical summary, section 2.B, "graph simplification"): the
LayerNorm -> multiply -> add chain of an adaLN modulation site collapses into
a single node whose intermediate statistics never become framework tensors.
`AdaLNModulateFunction` is that node: its forward is `adaln_fwd`, it saves
only x, the per-row mean and rstd (8 bytes per token), the modulation scale
and the segment ids, and its backward is `adaln_bwd`.  The unfused chain
instead keeps the normalised activations and the gathered (1 + scale) rows.

Layout: x is [..., D] (flattened to tokens [T, D]); shift and scale are
[nseg, D]; seg_id is int32 [T], non-decreasing, mapping each token to its
modulation row.  For a batch x [B, N, D] with one modulation row per sample,
`sample_seg_ids(B, N)` gives seg_id.
"""
import torch

from . import _lib


def sample_seg_ids(B, N, device=None):
    """seg_id for B samples of N tokens each, packed back to back."""
    return torch.arange(B, device=device, dtype=torch.int32).repeat_interleave(N)


class AdaLNModulateFunction(torch.autograd.Function):
    """y = LayerNorm(x) * (1 + scale[seg_id]) + shift[seg_id], fused."""

    @staticmethod
    def forward(ctx, x, shift, scale, seg_id, eps):
        shape = x.shape
        D = shape[-1]
        x2 = x.reshape(-1, D)
        if not x2.is_contiguous():
            x2 = x2.contiguous()
        y, mean, rstd = _lib.adaln_fwd(x2, shift.contiguous(), scale.contiguous(),
                                       seg_id, eps)
        ctx.save_for_backward(x2, mean, rstd, scale.contiguous(), seg_id)
        ctx.shape = shape
        ctx.mod_dtypes = (shift.dtype, scale.dtype)
        return y.reshape(shape)

    @staticmethod
    def backward(ctx, dy):
        x2, mean, rstd, scale, seg_id = ctx.saved_tensors
        dy2 = dy.reshape(x2.shape)
        if dy2.dtype != x2.dtype:
            dy2 = dy2.to(x2.dtype)
        if not dy2.is_contiguous():
            dy2 = dy2.contiguous()
        dx, dshift, dscale = _lib.adaln_bwd(dy2, x2, mean, rstd, scale, seg_id)
        return (dx.reshape(ctx.shape), dshift.to(ctx.mod_dtypes[0]),
                dscale.to(ctx.mod_dtypes[1]), None, None)


def adaln_modulate(x, shift, scale, seg_id, eps=1e-6):
    """Functional form of the fused operator (differentiable in x, shift, scale)."""
    return AdaLNModulateFunction.apply(x, shift, scale, seg_id, float(eps))


class AdaLNModulate(torch.nn.Module):
    """Module form: forward(x, shift, scale, seg_id) -> y."""

    def __init__(self, eps=1e-6):
        super().__init__()
        self.eps = float(eps)

    def forward(self, x, shift, scale, seg_id):
        return adaln_modulate(x, shift, scale, seg_id, self.eps)

    def extra_repr(self):
        return f"eps={self.eps}"
