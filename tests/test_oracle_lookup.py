"""Pins for the oracle's lookup (suffix match + copy), CPU only.

The rule (HyperQwen context-lookup article, "三步走", Step 1): the most recent
earlier occurrence of the longest 4..12-token suffix of the request's own
history, overlap allowed, and the tokens that follow it.  The oracle's early
exit scan is checked against exhaustive enumeration on every binary history
up to length 13, random histories over 3 symbols, hand-worked examples and
the closed form of primitive periodic histories.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden("lookup_examples.json")["cases"], ids=lambda c: c["name"])
def test_worked_examples(case):
    c, k, j = oracle.propose(case["h"])
    assert (k, j) == (case["k"], case["j"])
    assert c.tolist() == case["c"]


def test_all_binary_histories_match_enumeration():
    checked = 0
    for n in range(0, 14):
        for h in itertools.product((0, 1), repeat=n):
            got = oracle.lookup(h)
            want = brute.lookup_brute(h)
            assert got == want, (h, got, want)
            if got[0]:
                assert oracle.copy(h, *got).tolist() == brute.copy_brute(h, *got)
            checked += 1
    assert checked == 2 ** 14 - 1


def test_random_three_symbol_histories_match_enumeration():
    rng = np.random.default_rng(11)
    for _ in range(1500):
        n = int(rng.integers(0, 65))
        h = rng.integers(0, 3, size=n).tolist()
        got = oracle.lookup(h)
        assert got == brute.lookup_brute(h), h
        assert oracle.copy(h, *got).tolist() == brute.copy_brute(h, *got)


def test_random_histories_other_ranges():
    """min_k / max_k are parameters: the same enumeration holds for other ranges."""
    rng = np.random.default_rng(12)
    for lo, hi in ((1, 3), (2, 16), (4, 4), (6, 9)):
        p = oracle.Params.default(min_k=lo, max_k=hi)
        for _ in range(300):
            n = int(rng.integers(0, 48))
            h = rng.integers(0, 2 + int(rng.integers(0, 3)), size=n).tolist()
            assert oracle.lookup(h, p) == brute.lookup_brute(h, lo, hi), (lo, hi, h)


@pytest.mark.parametrize("p", list(range(1, 21)))
def test_primitive_periodic_closed_form(p):
    pattern = list(range(100, 100 + p))
    for n in range(p + 4, p + 45):
        h = [pattern[q % p] for q in range(n)]
        k, j, c = brute.periodic_closed_form(pattern, n)
        cc, kk, jj = oracle.propose(h)
        assert (kk, jj) == (k, j), (p, n)
        assert cc.tolist() == c


def test_short_histories_have_no_match():
    rng = np.random.default_rng(13)
    for n in range(0, 5):
        for _ in range(20):
            h = rng.integers(0, 2, size=n).tolist()
            assert oracle.lookup(h) == (0, -1)


def test_copy_is_cyclic_past_the_end():
    # match of period 3 that runs out after 3 tokens: the copy repeats them.
    h = [9, 9, 9, 9, 1, 2, 3, 1, 2, 3, 1, 2, 3]
    c, k, j = oracle.propose(h)
    assert (k, j) == (6, 10)  # the run of 9s stops the match at 6 tokens
    assert c.tolist() == [1, 2, 3] * 5 + [1]


def test_large_random_history_spot_checks():
    """Longer Zipf-like histories with planted copies: the early-exit scan
    agrees with enumeration restricted to the candidates that matter."""
    rng = np.random.default_rng(14)
    for _ in range(40):
        n = int(rng.integers(200, 600))
        h = rng.integers(0, 50, size=n)
        src = int(rng.integers(0, n - 40))
        ln = int(rng.integers(1, 20))
        h[n - ln:] = h[src:src + ln]
        h = h.tolist()
        assert oracle.lookup(h) == brute.lookup_brute(h)
