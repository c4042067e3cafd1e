"""Shared test setup: the `gpu` marker and import paths."""
import os
import sys

import numpy as np

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libeagle")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


# near-tie decisions met by the parity tests (counted, reported, excluded from the
# bit-exact comparison): test -> (excluded requests, requests)
NEAR_TIES = {}


def record_near_ties(test: str, excluded: int, total: int) -> None:
    NEAR_TIES[test] = (NEAR_TIES.get(test, (0, 0))[0] + int(excluded), NEAR_TIES.get(test, (0, 0))[1] + int(total))


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    if not NEAR_TIES:
        return
    terminalreporter.section("near-ties (requests excluded from the bit-exact comparison / requests)")
    for test, (ex, n) in sorted(NEAR_TIES.items()):
        terminalreporter.write_line(f"{test}: {ex} / {n}")


def near_tie_cap(n: int, rate: float) -> int:
    """Largest near-tie count a test accepts among n requests whose expected near-tie
    rate per request is `rate`: the 99.9% quantile of a Poisson with mean n * rate (at
    least 1).  Rates, per request: about 2e-5 per accept decision (|u - p/q| < 1e-5);
    at most 2e-7 V per draw over V tokens (a draw is near a bin edge when it lands
    within 1e-7 of the mass from one, i.e. with probability sum_i min(p_i, 2e-7))."""
    from scipy.stats import poisson
    return max(1, int(poisson.ppf(0.999, n * rate)))


def draw_rate(V: int, draws: int = 1) -> float:
    """Upper bound of a request's draw near-tie rate: every token's p above 2e-7."""
    return min(1.0, 2e-7 * V * draws)


def draw_rate_of(rows: np.ndarray, T: float = 1.0, draws: int = 1) -> float:
    """A request's draw near-tie rate from its distributions: the mean over the given
    logit rows (float values, last axis the vocabulary) of sum_i min(p_i, 2e-7), times
    the draws a request makes."""
    x = np.asarray(rows, np.float64).reshape(-1, rows.shape[-1]) / (T if T > 0 else 1.0)
    x = x - x.max(axis=1, keepdims=True)
    p = np.exp(x)
    p /= p.sum(axis=1, keepdims=True)
    return min(1.0, draws * float(np.minimum(p, 2e-7).sum(axis=1).mean()))
