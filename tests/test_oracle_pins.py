"""The CPU oracle against hand-derived values, closed forms, invariants and a
library routine.  CPU only."""
import numpy as np
import pytest

import oracle
from tests.oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.default())


def test_rows_match_full():
    """Row sampling returns exactly the rows of the full computation."""
    rng = np.random.default_rng(11)
    q = rng.standard_normal((2, 4, 9, 8))
    k = rng.standard_normal((2, 2, 13, 8))
    v = rng.standard_normal((2, 2, 13, 8))
    o, lse = oracle.attention(q, k, v, 0.5, True, 2)
    rows = np.array([[0, 0, 0], [1, 3, 8], [0, 2, 4], [1, 1, 5]])
    o2, l2 = oracle.attention_rows(q, k, v, 0.5, True, 2, rows)
    for n, (b, h, i) in enumerate(rows):
        assert np.array_equal(o2[n], o[b, h, i])
        assert l2[n] == lse[b, h, i]


def test_rejects_bad_shapes():
    q = np.zeros((1, 3, 2, 4))
    k = np.zeros((1, 2, 2, 4))
    with pytest.raises(ValueError):
        oracle.attention(q, k, k, 1.0)          # Hq % Hkv != 0
    with pytest.raises(ValueError):
        oracle.attention(np.zeros((1, 2, 2, 4)), k, k, 1.0, True, -1)
    q2 = np.zeros((1, 2, 2, 4))
    with pytest.raises(ValueError):
        oracle.attention(q2, k, k, 1.0, False, 0, window=2)  # window: causal only
    with pytest.raises(ValueError):
        oracle.attention(q2, k, k, 1.0, True, 0, window=-1)
    with pytest.raises(ValueError):
        # keys 0..1; the last query (position 2) with window 1 sees only key 2
        oracle.attention(q2, k, k, 1.0, True, 1, window=1)
    oracle.attention(q2, k, k, 1.0, True, 0, window=1)  # positions 0, 1: fine



def test_threads_positive():
    assert oracle.threads() >= 1
