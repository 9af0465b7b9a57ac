"""GB300-native fused AdaLN LayerNorm-Modulate (forward and backward).

The compute path is libadaln.so (hand-written sm_103a CUDA behind a C ABI,
declared in include/adaln.h); `adaln_video_dit_gb300._lib` is its thin ctypes
binding.  `adaln_video_dit_gb300.inputs` draws seeded synthetic workloads.
The binding is imported lazily so that the input generators load without a GPU.
"""

__all__ = ["inputs", "lib"]


def lib():
    """The ctypes binding of libadaln.so (raises if the library is missing)."""
    from . import _lib
    return _lib
