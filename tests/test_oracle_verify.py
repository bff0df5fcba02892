"""Pins for the oracle's greedy verification (argmax + accepted prefix), CPU only.

Greedy verification (HyperQwen context-lookup article, "三步走", last
paragraph; the Polish protocol page: the first rejected proposal ends the
run) accepts the drafts up to the first one that differs from the target's
argmax.  The argmax is checked against numpy.argmax, whose documentation
fixes the first occurrence on ties, on seeded bf16 and fp32 rows, and on
hand-built rows for ties, signed zeros, infinities and last-bit differences.
"""
import numpy as np
import pytest

import oracle
import workload as wl
from oracle import brute

SENT = -1


def _bf16(vals):
    return wl.f32_to_bf16_bits(np.array(vals, dtype=np.float32))


def test_argmax_matches_numpy_on_seeded_rows():
    rng = np.random.default_rng(21)
    for V in (1, 2, 7, 1024, 32000, 248320):
        for _ in range(3):
            x = rng.standard_normal(V).astype(np.float32)
            assert oracle.argmax_row(x) == int(np.argmax(x))
            b = wl.f32_to_bf16_bits(x)
            assert oracle.argmax_row(b) == int(np.argmax(wl.bf16_bits_to_f32(b)))


def test_argmax_matches_numpy_on_generator_rows():
    """Rows of the synthetic target (bf16 noise values tie often; the +8 truth is unique)."""
    w = wl.make_small("mixed", seed=3, B=2, V=248320, steps=2)
    g = wl.HostGen(w)
    ties = 0
    for b in range(2):
        P0 = w.prompts[b].size
        assert g.truth(b, P0) >= 0
        rows = g.logits_rows(b, P0, 16)
        f = wl.bf16_bits_to_f32(rows)
        for r in range(16):
            want = int(np.argmax(f[r]))
            assert oracle.argmax_row(rows[r]) == want
            ties += int((f[r] == f[r].max()).sum() > 1)
    assert ties == 0  # the boosted ground truth is the unique maximum here


@pytest.mark.parametrize("vals,want", [
    ([1.0, 1.0, 1.0, 1.0], 0),
    ([0.0, 1.0, 2.0, 3.0], 3),
    ([0.0, 3.0, 1.0, 3.0], 1),
    ([-0.0, 0.0, -1.0], 0),
    ([0.0, -0.0], 0),
    ([-1.0, -0.0, 0.0], 1),
    ([-np.inf, -np.inf], 0),
    ([-np.inf, -5.0, -np.inf], 1),
    ([np.inf, 1.0, np.inf], 0),
    ([-3.0, -2.0, -2.5], 1),
    ([1.0, np.nan, 5.0, np.nan], 1),
])
def test_argmax_hand_rows(vals, want):
    x = np.array(vals, dtype=np.float32)
    assert oracle.argmax_row(x) == want
    assert oracle.argmax_row(_bf16(vals)) == want


def test_argmax_bf16_last_mantissa_bit():
    row = np.array([0x3F80, 0x3F81, 0x3F80], dtype=np.uint16)  # 1.0, 1.0078125, 1.0
    assert oracle.argmax_row(row) == 1
    row = np.array([0xBF81, 0xBF80], dtype=np.uint16)  # -1.0078125, -1.0
    assert oracle.argmax_row(row) == 1


def test_argmax_plain_loop_agrees():
    rng = np.random.default_rng(22)
    for _ in range(50):
        x = rng.integers(-3, 4, size=int(rng.integers(1, 40))).astype(np.float32)
        assert oracle.argmax_row(x) == brute.first_argmax(x.tolist())


G = list(range(100, 116))


@pytest.mark.parametrize("L", [8, 16])
def test_accept_mismatch_at_each_slot(L):
    for m in range(0, L):  # drafts 1..m agree, draft m+1 (if any) differs
        blk = [7] + [G[r] for r in range(m)] + [999] * (16 - 1 - m)
        want = min(m, L - 1)
        assert oracle.accept(blk, G, L) == want
        assert brute.accept_brute(blk, G, L) == want


def test_accept_capped_by_block_length():
    blk = [7] + G[:15]  # every draft agrees, but an 8-block verifies only 7 of them
    assert oracle.accept(blk, G, 8) == 7
    assert oracle.accept(blk, G, 16) == 15
    assert oracle.accept(blk, G, 1) == 0


def test_accept_stops_at_sentinel():
    blk = [7] + G[:7] + [SENT] * 8
    assert oracle.accept(blk, G, 16) == 7
    blk = [7] + [SENT] * 15
    assert oracle.accept(blk, G, 16) == 0


def test_accept_random_against_brute():
    rng = np.random.default_rng(23)
    for _ in range(500):
        L = int(rng.choice([1, 2, 8, 16]))
        g = rng.integers(0, 3, size=16).tolist()
        blk = rng.integers(-1, 3, size=16).tolist()
        assert oracle.accept(blk, g, L) == brute.accept_brute(blk, g, L)
