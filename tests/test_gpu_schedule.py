"""Shape benchmarking of the fused operator and the cost-model fit on it.

The operator's cost is linear in the tokens of a batch, so the fitted
exponent of t ~ a + b*B*S**p must come out close to 1."""
import pytest

from adaln_video_dit_gb300 import schedule as Sch

pytestmark = pytest.mark.gpu


def test_shape_benchmark_fit_is_linear_in_tokens(adaln):
    shapes = [(B, S) for S in (8192, 16384, 32768) for B in (1, 2, 4)]
    res = Sch.shape_benchmark(shapes, D=2048, steps=10, warmup=2)
    B = [r[0] for r in res]
    S = [r[1] for r in res]
    t = [r[2] for r in res]
    a, b, p = Sch.fit_cost_model(B, S, t)
    assert 0.8 < p < 1.2, (a, b, p, res)
    assert b > 0
