"""The analytic speedup models against the figures the pages print (tests/golden)."""
import os

import pytest

from oracle import analytic as AN

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "speedup_models.txt")


def _rows():
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            yield line.split()[:6]


@pytest.mark.parametrize("row", list(_rows()))
def test_printed_figures(row):
    kind, a, b, c, val, tol = row
    if kind == "layer_skip":
        assert abs(AN.layer_skip_speedup(float(a), int(c), float(b)) - float(val)) <= float(tol)
    elif kind == "best_k":
        assert AN.best_k(float(a), float(b)) == int(val)
    elif kind == "best_k_in":
        assert AN.best_k(float(a), float(b)) in [int(x) for x in c.split(",")]
    elif kind == "below_all_k":
        assert all(AN.layer_skip_speedup(float(a), k, float(b)) < float(val) for k in range(1, 17))
    elif kind == "dspark":
        assert abs(AN.dspark_speedup(float(a), int(b), float(c)) - float(val)) <= float(tol)
    else:
        raise AssertionError(kind)


def test_expected_tokens_limits():
    # alpha -> 0: one token per round; alpha = 1: k + 1 (page's best / worst case)
    assert AN.expected_tokens(0.0, 5) == 1.0
    assert AN.expected_tokens(1.0, 5) == 6.0
    assert AN.expected_tokens_positional([1.0] * 4) == 5.0
    assert AN.expected_tokens_positional([0.0] * 4) == 1.0
    # geometric series equals the positional form with equal betas
    assert AN.expected_tokens(0.63, 5) == pytest.approx(AN.expected_tokens_positional([0.63] * 5))
