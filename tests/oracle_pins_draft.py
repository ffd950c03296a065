"""Pins of the draft-side oracle (``oracle/draft.py``) to facts other than itself.

Each ``pin_*`` takes an implementation module (``oracle.draft``, or a copy of it
with a planted mistake) and raises AssertionError when it disagrees with what
the pages and the mathematics fix: hand-worked fixtures under ``tests/golden/``,
a closed form, a library routine, and brute force in exact rational arithmetic
on tiny inputs. None of them retypes the oracle's formula.
"""

import bisect
import math
import os
from fractions import Fraction

import numpy as np
import torch

from oracle_pins import GOLDEN, _lines, bits_value, exact_bits, rand_bf16

# --------------------------------------------------- exact bf16 arithmetic

_POS = None


def _positive_finite():
    """Every finite bf16 value >= 0 in increasing order, as (Fraction, pattern)."""
    global _POS
    if _POS is None:
        _POS = [(Fraction(bits_value(p)), p) for p in range(0x0000, 0x7F80)]
    return _POS


_HALF_PAST_MAX = Fraction(bits_value(0x7F7F)) + (Fraction(2) ** 128 - Fraction(bits_value(0x7F7F))) / 2


def brute_round(x):
    """Nearest bf16 to the rational x by search over every finite bf16 value;
    a tie goes to the even pattern; from the halfway point past the largest
    finite value on, infinity."""
    x = Fraction(x)
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    if a >= _HALF_PAST_MAX:
        return sign | 0x7F80
    vals = _positive_finite()
    keys = [v for v, _ in vals]
    k = bisect.bisect_left(keys, a)
    if k < len(vals) and vals[k][0] == a:
        return sign | vals[k][1]
    lo, hi = vals[k - 1], vals[k]
    dl, dh = a - lo[0], hi[0] - a
    if dl < dh or (dl == dh and lo[1] % 2 == 0):
        return sign | lo[1]
    return sign | hi[1]


def frac_of(p):
    return Fraction(bits_value(p))


# ------------------------------------------------------- rounding of float64

def pin_bf16_any_golden(impl):
    for line in _lines("bf16_rounding_any.txt"):
        parts = line.split()
        x, want = float.fromhex(parts[0]), int(parts[1], 16)
        got = int(impl.f64_to_bf16_rne_any(np.array([x]))[0])
        assert got == want, f"round({parts[0]}) = {got:04x}, want {want:04x}"


def pin_bf16_any_matches_torch_on_binary32(impl):
    """On values binary32 holds exactly, one-step rounding is torch's
    float -> bf16 cast (a library routine)."""
    rng = np.random.default_rng(51)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = impl.f64_to_bf16_rne_any(x.astype(np.float64))
    assert np.array_equal(got, want)


def pin_bf16_any_brute(impl):
    """Random float64 values, many of them a hair off a bf16 tie (where a
    double rounding through binary32 goes wrong), against ``brute_round``."""
    rng = np.random.default_rng(52)
    xs = list(rng.standard_normal(300) * 7.0)
    for _ in range(300):   # ties +- 2^-30 relative, and exact ties
        p = int(rng.integers(0x0080, 0x7F00))
        mid = (bits_value(p) + bits_value(p + 1)) / 2.0
        xs.append(mid * (1.0 + float(rng.choice([-1, 0, 1])) * 2.0 ** -30) * float(rng.choice([-1, 1])))
    got = impl.f64_to_bf16_rne_any(np.array(xs))
    for x, g in zip(xs, got):
        assert int(g) == brute_round(x), (x.hex(), hex(int(g)))


# -------------------------------------------------------------- Markov pick

def _markov_cases():
    cur = None
    for line in _lines("markov_worked.txt"):
        a = line.split()
        if a[0] == "case":
            cur = dict(name=a[1], V=int(a[2]), K=int(a[3]), prev=int(a[4]), W1=[], W2=[], base=[])
        elif a[0] in ("W1", "W2", "base"):
            cur[a[0]].append([int(x, 16) for x in a[1:]])
        elif a[0] == "expect":
            i = a.index("/")
            cur["picks"] = [int(x) for x in a[1:i]]
            cur["flags"] = [int(x) for x in a[i + 1:]]
            yield cur


def pin_markov_worked(impl):
    n = 0
    for c in _markov_cases():
        W1 = np.array(c["W1"], dtype=np.uint16)
        W2 = np.array(c["W2"], dtype=np.uint16)
        base = np.array(c["base"], dtype=np.uint16)
        assert W1.shape == (c["V"], c["K"]) and W2.shape == (c["V"], c["K"])
        picks, flags, _ = impl.markov_chain(base, W1, W2, c["prev"])
        assert [int(p) for p in picks] == c["picks"], (c["name"], list(picks))
        assert [int(f) for f in flags] == c["flags"], (c["name"], list(flags))
        n += 1
    assert n >= 9


def _permutation_head(rng, V):
    """W1 = identity and W2[v] = 16 * e_{pi^-1(v)}: the Markov term of token p
    is 16 at pi(p) and 0 elsewhere, so with |base| small the chain follows pi."""
    pi = rng.permutation(V)
    inv = np.argsort(pi)
    W1 = np.zeros((V, V), dtype=np.uint16)
    W1[np.arange(V), np.arange(V)] = exact_bits(1.0)
    W2 = np.zeros((V, V), dtype=np.uint16)
    W2[np.arange(V), inv] = exact_bits(16.0)
    return pi, W1, W2


def pin_markov_permutation_chain(impl):
    """Closed form: the chain's picks are pi(prev0), pi^2(prev0), ..."""
    rng = np.random.default_rng(53)
    V, n = 40, 6
    pi, W1, W2 = _permutation_head(rng, V)
    base = rand_bf16(rng, (n, V), std=1.0)
    assert np.abs(np.array([[bits_value(b) for b in row] for row in base])).max() < 6.0
    prev = 17
    picks, flags, _ = impl.markov_chain(base, W1, W2, prev)
    want, p = [], prev
    for _ in range(n):
        p = int(pi[p])
        want.append(p)
    assert [int(x) for x in picks] == want and not np.any(flags)


def pin_markov_streams(impl):
    """A verify table's draft rows: stream s's block holds r_s - 1 rows packed
    at draft row o_s - s, and each stream's chain starts from its own pending
    token (closed form of the permutation head per stream)."""
    rng = np.random.default_rng(54)
    V = 32
    pi, W1, W2 = _permutation_head(rng, V)
    rows = [3, 1, 5, 2]
    streams, off = [], 0
    for r in rows:
        streams.append((r, off, r + 10))
        off += r
    prev = np.array([4, 9, 30, 0], dtype=np.int32)
    n = sum(r - 1 for r in rows)
    base = rand_bf16(rng, (n, V), std=1.0)
    picks, flags, _ = impl.markov_all(streams, base, W1, W2, prev)
    assert len(picks) == n and not np.any(flags)
    k = 0
    for s, r in enumerate(rows):
        p = int(prev[s])
        for _ in range(r - 1):
            p = int(pi[p])
            assert int(picks[k]) == p, (s, k)
            k += 1


def pin_markov_brute(impl):
    """Tiny random head in exact rational arithmetic: exact dot, ``brute_round``
    of the dot, of the sum, and a scan keeping the first strictly larger."""
    rng = np.random.default_rng(55)
    V, K, n = 29, 6, 4
    W1 = rand_bf16(rng, (V, K), std=1.0)
    W2 = rand_bf16(rng, (V, K), std=0.5)
    base = rand_bf16(rng, (n, V), std=0.7)
    prev0 = 11
    picks, flags, scores = impl.markov_chain(base, W1, W2, prev0)
    prev = prev0
    for j in range(n):
        best, idx, row = None, -1, []
        for v in range(V):
            dot = sum(frac_of(W2[v, k]) * frac_of(W1[prev, k]) for k in range(K))
            sc = brute_round(frac_of(brute_round(dot)) + frac_of(base[j, v]))
            row.append(sc)
            val = frac_of(sc)
            if best is None or val > best:
                best, idx = val, v
        assert [int(b) for b in scores[j]] == row, j
        assert int(picks[j]) == idx and int(flags[j]) == 0, j
        prev = idx


# -------------------------------------------------------------- draft ids

def _draft_cases():
    c = None
    for line in _lines("draft_ids_cases.txt"):
        a = line.split()
        if a[0] == "case":
            c = dict(name=a[1], vocab=int(a[2]))
        elif a[0] == "expect":
            i = a.index("/")
            c["ids"] = [int(x) for x in a[1:i]]
            c["sflag"] = [int(x) for x in a[i + 1:]]
            yield c
        else:
            c[a[0]] = [int(x) for x in a[1:]]


def pin_draft_ids_golden(impl):
    n = 0
    for c in _draft_cases():
        streams, off = [], 0
        for r in c["rows"]:
            streams.append((r, off, r))
            off += r
        ids, dflag = impl.draft_ids_all(streams, c["prev"], c["drafts"],
                                        np.array(c["dflag"], dtype=np.uint8), c["vocab"])
        assert [int(x) for x in ids] == c["ids"], (c["name"], list(ids))
        assert [int(x) for x in dflag] == c["sflag"], (c["name"], list(dflag))
        n += 1
    assert n >= 4


DRAFT_PINS = [
    pin_bf16_any_golden, pin_bf16_any_matches_torch_on_binary32, pin_bf16_any_brute,
    pin_markov_worked, pin_markov_permutation_chain, pin_markov_streams, pin_markov_brute,
    pin_draft_ids_golden,
]
