"""The Markov parity rule itself, on the CPU: the oracle's own pick always
passes it, and a pick that cannot be the first argmax fails it."""

import numpy as np
import pytest

from oracle import draft as OD
from oracle_pins import rand_bf16
from parity import check_markov_row, markov_bounds, markov_possible_picks


def test_oracle_pick_is_always_possible():
    rng = np.random.default_rng(61)
    V = 3000
    W1 = rand_bf16(rng, (V, 256))
    W2 = rand_bf16(rng, (V, 256), std=0.25)
    base = rand_bf16(rng, (12, V), std=3.0)
    for j in range(12):
        tok = int(rng.integers(V))
        _, want, flag = OD.markov_step(base[j], W1, W2, tok)
        assert flag == 0
        lo, hi = markov_bounds(base[j], W1, W2, tok)
        assert np.all(lo <= hi)
        assert want in set(markov_possible_picks(lo, hi).tolist())
        assert check_markov_row(want, 0, base[j], W1, W2, tok, "self")


def test_wrong_pick_fails():
    rng = np.random.default_rng(62)
    V = 2000
    W1 = rand_bf16(rng, (V, 256))
    W2 = rand_bf16(rng, (V, 256), std=0.25)
    base = rand_bf16(rng, (1, V), std=3.0)
    tok = 5
    sc, want, _ = OD.markov_step(base[0], W1, W2, tok)
    vals = OD.bf16_to_f64(sc)
    worst = int(np.argmin(vals))
    with pytest.raises(AssertionError):
        check_markov_row(worst, 0, base[0], W1, W2, tok, "worst token")
    with pytest.raises(AssertionError):
        check_markov_row(want, 1, base[0], W1, W2, tok, "flag set on a finite row")


def test_possible_picks_rule():
    # scores fixed (lo == hi): only the first maximum is possible
    lo = np.array([1.0, 3.0, 2.0, 3.0])
    assert markov_possible_picks(lo, lo).tolist() == [1]
    # token 3 may reach 3.5 and beat token 1 -> both possible; token 0 may tie 3.0 and come first
    hi = np.array([3.0, 3.0, 2.0, 3.5])
    assert markov_possible_picks(lo, hi).tolist() == [0, 1, 3]
