"""Dual-constraint bucketing and the cost-model fit (host side, no GPU)."""
import numpy as np
import pytest

from adaln_video_dit_gb300 import schedule as Sch


def test_b_shape_both_constraints():
    # memory-bound, compute-bound and the max(1, .) floor
    assert Sch.b_shape(1024, 65536, 2 ** 31, 2) == 64            # 65536 // 1024
    assert Sch.b_shape(1024, 65536, 2 ** 24, 2) == 16            # 2^24 // 2^20
    assert Sch.b_shape(100000, 65536, 2 ** 31, 2) == 1           # floor of 1
    assert Sch.b_shape(4096, 10 ** 9, 10 ** 9, 1.5) == int(10 ** 9 // 4096 ** 1.5)
    plan = Sch.bucket_plan([256, 1024, 256, 32760], 65536, 2 ** 31)
    assert plan == {256: 256, 1024: 64, 32760: 2}
    for S, B in plan.items():
        assert B * S <= 65536 and B * S ** 2 <= 2 ** 31 or B == 1
    with pytest.raises(ValueError):
        Sch.b_shape(0, 1, 1)


@pytest.mark.parametrize("a,b,p", [(3.0, 2e-6, 2.0), (0.5, 4e-4, 1.0), (10.0, 1e-5, 1.7)])
def test_fit_recovers_known_model(a, b, p):
    rng = np.random.default_rng(1)
    S = np.repeat([256, 1024, 4096, 16384], 4)
    B = np.concatenate([[1, 2, 4, 8]] * 4)
    t = Sch.cost_model(B, S, a, b, p) * (1 + 0.002 * rng.standard_normal(S.size))
    fa, fb, fp = Sch.fit_cost_model(B, S, t)
    assert abs(fp - p) < 0.02
    assert abs(fa - a) / a < 0.05 and abs(fb - b) / b < 0.1


def test_m_comp_from_step_budget():
    a, b, p = 2.0, 1e-6, 2.0
    m = Sch.m_comp_for_step_time(a, b, 10.0)
    S = 2048
    B = Sch.b_shape(S, 10 ** 9, m, p)
    assert Sch.cost_model(B, S, a, b, p) <= 10.0 + 1e-9
    assert Sch.cost_model(B + 1, S, a, b, p) > 10.0
    with pytest.raises(ValueError):
        Sch.m_comp_for_step_time(a, b, 1.0)
