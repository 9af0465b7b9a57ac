"""Seeded input generators: determinism and the stated recipes."""
import numpy as np

from adaln_video_dit_gb300 import inputs as I


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.00390625, 1.005859375, 1.0078125 + 2 ** -9,
                     -3.14159, 65504.0, 1e-30], np.float32)
    bits = I.to_bf16_bits(vals)
    back = I.bf16_bits_to_f32(bits)
    # every result is a bf16 value nearest to the input
    for v, b in zip(vals, back):
        u = np.float32(b).view(np.uint32)
        lo = (u - np.uint32(0x10000)).view(np.float32)
        hi = (u + np.uint32(0x10000)).view(np.float32)
        assert abs(b - v) <= abs(lo - v) and abs(b - v) <= abs(hi - v)
    # ties go to the even mantissa: 1 + 2^-8 is halfway between 1 and 1 + 2^-7
    assert I.bf16_bits_to_f32(I.to_bf16_bits(np.float32(1 + 2 ** -8)))[()] == 1.0
    assert I.bf16_bits_to_f32(I.to_bf16_bits(np.float32(1 + 3 * 2 ** -8)))[()] == 1 + 2 ** -6


def test_workloads_are_deterministic_and_shaped():
    for c, (T, D, nseg, dt) in {1: (256, 128, 1, "f32"), 2: (8192, 1536, 2, "bf16")}.items():
        a, b = I.make(c), I.make(c)
        assert (a["T"], a["D"], a["nseg"], a["dtype"]) == (T, D, nseg, dt)
        for k in ("x", "dy", "shift", "scale", "seg_id"):
            assert np.array_equal(a[k], b[k])
        assert a["x"].shape == (T, D) and a["shift"].shape == (nseg, D)
        assert np.all(np.diff(a["seg_id"]) >= 0)


def test_long_video_truncated_has_outlier_channels():
    c = I.make(3, T_override=64)
    x = I.bf16_bits_to_f32(c["x"])
    col_std = x.std(0)
    assert (col_std > 20).sum() == round(0.001 * 5120)
    assert c["nseg"] == 1 and c["D"] == 5120


def test_b_shape_memory_bound_sets_every_bucket():
    assert [I.b_shape(S) for S in (256, 1024, 4096, 16384, 32760)] == [256, 64, 16, 4, 2]
    L = I.mixed_varlen_lengths()
    assert 16 <= len(L) <= 2048
    assert sum(L) == 524272


def test_mmdit_segments():
    seg = I.seg_ids_from_lengths([512, 4096] * 8)
    assert seg.shape == (36864,) and seg[511] == 0 and seg[512] == 1 and seg[-1] == 15
