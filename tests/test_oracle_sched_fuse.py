"""Pins for the oracle's scheduler and fusion rule, CPU only (hand-worked
traces and truth table in tests/golden, each citing the page section)."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
SENT = -1


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.mark.parametrize("tr", _golden("sched_traces.json")["traces"], ids=lambda t: t["name"])
def test_sched_traces(tr):
    s = oracle.Scheduler(oracle.Params.default(sticky=tr["sticky"]))
    prev_a = prev_L = 0
    got = []
    for k, a, want in zip(tr["k"], tr["a"], tr["L"]):
        L = s.step(k, prev_a, prev_L)
        got.append(L)
        assert a <= L - 1, "trace must be feasible"
        prev_a, prev_L = a, L
    assert got == tr["L"]


def test_sched_first_step_is_short_even_if_prev_given():
    s = oracle.Scheduler()
    assert s.step(12, 15, 16) == 8  # no previous step at t = 0


def test_sched_enter_streak_parameter():
    s = oracle.Scheduler(oracle.Params.default(enter_streak=1))
    assert [s.step(12, 7, 8) for _ in range(2)] == [8, 16]


LAST = 1000
C = [10 + i for i in range(16)]
M = {"both": [10, 11, 52, 53, 54, 55, 56], "first": [10, 51, 52, 53, 54, 55, 56], "second": [50, 11, 52, 53, 54, 55, 56],
     "none": [50, 51, 52, 53, 54, 55, 56]}


@pytest.mark.parametrize("row", _golden("fusion_table.json")["rows"],
                         ids=lambda r: f"k{r['k']}-{r['agree']}-L{r['L']}")
def test_fusion_truth_table(row):
    c = C if row["k"] > 0 else [SENT] * 16
    m = M[row["agree"]]
    blk = oracle.fuse(LAST, c, row["k"], m, row["L"]).tolist()
    head = c[:7] if row["head"] == "lookup" else m
    tail = c[7:15] if row["tail"] == "lookup" else [SENT] * 8
    assert blk == [LAST] + list(head) + list(tail)


def test_fusion_short_block_never_fills_tail():
    for k in range(0, 13):
        blk = oracle.fuse(5, C, k, M["both"], 8)
        assert (blk[8:] == SENT).all()
