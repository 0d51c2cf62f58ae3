"""The f64 oracle against facts that do not come from the oracle itself.

Each pin is described in ``oracle_pins.py``; this file runs every one of them
on the real oracle (CPU only)."""
import pytest

from tests import oracle_pins  # noqa: E402


@pytest.mark.parametrize("check", oracle_pins.ALL, ids=lambda c: c.__name__)
def test_oracle_pin(oracle_mod, check):
    check(oracle_mod.default())


def test_oracle_threads_do_not_change_bits(oracle_mod):
    import numpy as np
    rng = np.random.default_rng(3)
    q, k, v, t, L = oracle_pins.rand_case(rng, 3, 8, 2, 32, 8, [50, 3, 77])
    a = oracle_mod.decode_attn(q, k, v, t, L, 0.2, 0, threads=1)
    b = oracle_mod.decode_attn(q, k, v, t, L, 0.2, 0, threads=5)
    assert np.array_equal(a, b)


def test_oracle_row_subset_matches_full(oracle_mod):
    import numpy as np
    rng = np.random.default_rng(4)
    q, k, v, t, L = oracle_pins.rand_case(rng, 2, 4, 1, 16, 4, [21, 12])
    full = oracle_mod.decode_attn(q, k, v, t, L, 0.3, 5)
    rows = np.array([7, 0, 5])
    sub = oracle_mod.decode_attn(q, k, v, t, L, 0.3, 5, rows=rows)
    assert np.array_equal(sub, full.reshape(8, 16)[rows])
