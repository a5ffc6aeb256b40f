"""The GPU/oracle comparison rules themselves, on hand-made results (CPU)."""
import numpy as np
import pytest

from parity_util import FLAG, compare, valid_output


def result(out, nacc, status=0, am=None, sm=1.0, lse_t=None, K=2):
    B = 1
    return {
        "out_tokens": np.array([out], dtype=np.int32),
        "num_accepted": np.array([nacc], dtype=np.int32),
        "seq_status": np.array([status], dtype=np.int32),
        "accept_margin": np.array([am if am is not None else [0.5] * K]),
        "sample_margin": np.array([sm]),
        "lse_t": np.array([lse_t if lse_t is not None else [1.0] * (K + 1)]),
        "lse_d": np.ones((B, K)),
        "log_ratio": np.zeros((B, K)),
    }


X = np.array([[3, 4]])


def test_exact_match_passes():
    st = compare(result([3, 9, -1], 1), result([3, 9, -1], 1), X, 2, 10)
    assert st["flagged_decisions"] == 0 and st["decisions"] == 3


def test_unflagged_difference_fails():
    with pytest.raises(AssertionError):
        compare(result([3, 8, -1], 1), result([3, 9, -1], 1), X, 2, 10)
    with pytest.raises(AssertionError):
        compare(result([7, -1, -1], 0), result([3, 9, -1], 1), X, 2, 10)


def test_flagged_sampling_may_differ_in_the_token_only():
    st = compare(result([3, 8, -1], 1), result([3, 9, -1], 1, sm=FLAG / 2), X, 2, 10)
    assert st["flagged_differing"] == 1
    with pytest.raises(AssertionError):  # but not in the accepted count
        compare(result([3, 4, 1], 2), result([3, 9, -1], 1, sm=FLAG / 2), X, 2, 10)


def test_flagged_acceptance_allows_either_branch():
    orc = result([3, 9, -1], 1, am=[0.3, FLAG / 3])
    compare(result([3, 4, 5], 2), orc, X, 2, 10)
    with pytest.raises(AssertionError):  # diverging before the flagged position is not allowed
        compare(result([6, -1, -1], 0), orc, X, 2, 10)


def test_normalisers_within_tolerance():
    compare(result([3, 9, -1], 1, lse_t=[10.0, 10.0, 10.0 + 5e-5]),
            result([3, 9, -1], 1, lse_t=[10.0, 10.0, 10.0]), X, 2, 10)
    with pytest.raises(AssertionError):
        compare(result([3, 9, -1], 1, lse_t=[10.0, 10.0, 10.0 + 2e-4]),
                result([3, 9, -1], 1, lse_t=[10.0, 10.0, 10.0]), X, 2, 10)


def test_invalid_sequences_must_match_status():
    compare(result([-1, -1, -1], -1, status=2), result([-1, -1, -1], -1, status=2), X, 2, 10)
    with pytest.raises(AssertionError):
        compare(result([3, 9, -1], 1, status=0), result([-1, -1, -1], -1, status=2), X, 2, 10)


def test_valid_output_rules():
    x = np.array([3, 4, 5])
    assert valid_output(np.array([3, 9, -1, -1]), 1, x, 3, 10)
    assert not valid_output(np.array([3, 9, 2, -1]), 1, x, 3, 10)
    assert not valid_output(np.array([4, 9, -1, -1]), 1, x, 3, 10)
    assert not valid_output(np.array([3, 10, -1, -1]), 1, x, 3, 10)


def test_oracle_flag_counts_counts_every_taken_decision():
    from parity_util import oracle_flag_counts
    orc = {
        "seq_status": np.array([0, 0, 1]),
        "num_accepted": np.array([1, 3, -1]),
        # seq 0 takes positions 0, 1 (1 is the rejection); seq 1 takes 0, 1, 2
        "accept_margin": np.array([[0.5, FLAG / 2, FLAG / 3],
                                   [FLAG / 2, 0.5, FLAG / 4],
                                   [0.0, 0.0, 0.0]]),
        "sample_margin": np.array([FLAG / 2, 0.5, 0.0]),
    }
    n, f = oracle_flag_counts(orc, 3)
    assert n == (2 + 1) + (3 + 1)
    assert f == 1 + 1 + 2  # seq 0: position 1 and the draw; seq 1: positions 0 and 2


def test_flag_budget_bounds():
    from parity_util import flag_count_plausible, flag_rate_upper_bound
    assert flag_count_plausible(0, 10) and flag_count_plausible(1, 100)
    assert not flag_count_plausible(3, 100)          # 3 in 100 at rate 1e-4: p ~ 1.6e-7
    assert flag_count_plausible(30, 300_000)         # mean 30 at the budget
    assert not flag_count_plausible(80, 300_000)
    ub = flag_rate_upper_bound(5, 300_000)
    assert 5 / 300_000 < ub < 1e-4
    assert flag_rate_upper_bound(40, 300_000) > 1e-4
