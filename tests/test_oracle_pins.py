"""The CPU oracle against its pins (no GPU needed)."""
import numpy as np
import pytest

import pins


@pytest.mark.parametrize("pin", pins.ALL, ids=lambda f: f.__name__)
def test_pin(oracle, pin):
    pin(oracle.load())


def test_rows_subset_matches_full(oracle):
    from adaln_video_dit_gb300 import inputs as I
    c = I.random_case(21, 50, 24, 3, dtype="f32")
    rows = np.array([49, 0, 17, 17, 3], np.int64)
    y, m, r = oracle.adaln_fwd(c["x"], c["shift"], c["scale"], c["seg_id"], c["eps"])
    ys, ms, rs = oracle.adaln_fwd(c["x"], c["shift"], c["scale"], c["seg_id"], c["eps"], rows=rows)
    assert np.array_equal(ys, y[rows]) and np.array_equal(ms, m[rows]) and np.array_equal(rs, r[rows])
    dx, dsh, dsc = oracle.adaln_bwd(c["dy"], c["x"], c["scale"], c["seg_id"], c["eps"])
    dxs, dsh2, dsc2 = oracle.adaln_bwd(c["dy"], c["x"], c["scale"], c["seg_id"], c["eps"], rows=rows)
    assert np.array_equal(dxs, dx[rows])
    assert np.array_equal(dsh, dsh2) and np.array_equal(dsc, dsc2)


def test_thread_count_does_not_change_bits(oracle):
    from adaln_video_dit_gb300 import inputs as I
    c = I.random_case(22, 97, 40, 4, dtype="bf16")
    a = oracle.adaln_bwd(c["dy"], c["x"], c["scale"], c["seg_id"], c["eps"], nthreads=1)
    b = oracle.adaln_bwd(c["dy"], c["x"], c["scale"], c["seg_id"], c["eps"], nthreads=7)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_saved_stats_mode(oracle):
    from adaln_video_dit_gb300 import inputs as I
    c = I.random_case(23, 30, 64, 2, dtype="f32")
    m, r = oracle.row_stats(c["x"], c["eps"])
    own = oracle.adaln_bwd(c["dy"], c["x"], c["scale"], c["seg_id"], c["eps"])
    saved = oracle.adaln_bwd(c["dy"], c["x"], c["scale"], c["seg_id"], c["eps"],
                             mean=m.astype(np.float32), rstd=r.astype(np.float32))
    for u, v in zip(own, saved):
        np.testing.assert_allclose(v, u, rtol=1e-5, atol=1e-7)
    # The saved statistics are really used: shifting the means changes dscale.
    off = oracle.adaln_bwd(c["dy"], c["x"], c["scale"], c["seg_id"], c["eps"],
                           mean=(m + 1).astype(np.float32), rstd=r.astype(np.float32))
    assert not np.allclose(off[2], own[2])
    assert np.array_equal(off[1], own[1])


def test_seg_out_of_range_is_rejected(oracle):
    x = np.zeros((3, 8), np.float32)
    mod = np.zeros((2, 8), np.float32)
    with pytest.raises(ValueError):
        oracle.adaln_fwd(x, mod, mod, np.array([0, 2, 1], np.int32), 1e-6)
    with pytest.raises(ValueError):
        oracle.adaln_bwd(x, x, mod, np.array([0, -1, 1], np.int32), 1e-6)


def test_empty_input(oracle):
    x = np.zeros((0, 8), np.float32)
    mod = np.ones((3, 8), np.float32)
    y, m, r = oracle.adaln_fwd(x, mod, mod, np.zeros(0, np.int32), 1e-6)
    assert y.shape == (0, 8) and m.shape == (0,)
    dx, dsh, dsc = oracle.adaln_bwd(x, x, mod, np.zeros(0, np.int32), 1e-6)
    assert dx.shape == (0, 8) and np.all(dsh == 0) and np.all(dsc == 0)
