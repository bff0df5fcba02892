"""Scheduler and fusion on the GPU against the hand-worked traces, the fusion
truth table and the oracle.  GPU."""
import json
import os

import numpy as np
import pytest
import torch

import context_lookup_speculative_gb300 as clk
import oracle

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _i32(x):
    return torch.tensor(np.asarray(x, dtype=np.int32), device="cuda")


@pytest.mark.parametrize("sticky", [0, 1, 3])
def test_sched_traces(sticky):
    traces = [t for t in _golden("sched_traces.json")["traces"] if t["sticky"] == sticky]
    if not traces:
        pytest.skip("no trace for this sticky value")
    B = len(traces)
    T = max(len(t["k"]) for t in traces)
    lk = clk.Lookup(max_slots=B, max_hist=64, params=clk.Params.default(sticky=sticky))
    s = _i32(range(B))
    clk.lookup_init(lk, s, _i32([1] * B), torch.tensor(np.arange(B + 1), dtype=torch.int64, device="cuda"))
    prev_a, length = _i32([0] * B), _i32([0] * B)
    got = [[] for _ in range(B)]
    for t in range(T):
        k = _i32([tr["k"][t] if t < len(tr["k"]) else 0 for tr in traces])
        clk.sched_step(lk, s, k, prev_a, length, length)
        L = length.cpu().numpy()
        for b, tr in enumerate(traces):
            if t < len(tr["k"]):
                got[b].append(int(L[b]))
        prev_a = _i32([tr["a"][t] if t < len(tr["a"]) else 0 for tr in traces])
    for b, tr in enumerate(traces):
        assert got[b] == tr["L"], tr["name"]


def test_sched_random_against_oracle():
    rng = np.random.default_rng(61)
    B, T = 64, 200
    params = [dict(sticky=int(rng.integers(0, 5)), enter_streak=int(rng.integers(1, 4)),
                  near_full_slack=int(rng.integers(0, 3))) for _ in range(4)]
    for kw in params:
        lk = clk.Lookup(max_slots=B, max_hist=64, params=clk.Params.default(**kw))
        s = _i32(range(B))
        clk.lookup_init(lk, s, _i32([1] * B), torch.tensor(np.arange(B + 1), dtype=torch.int64, device="cuda"))
        refs = [oracle.Scheduler(oracle.Params.default(**kw)) for _ in range(B)]
        pa = np.zeros(B, np.int32)
        pl = np.zeros(B, np.int32)
        length = _i32(pl)
        for t in range(T):
            k = rng.choice([0, 4, 5, 8, 12], size=B, p=[0.3, 0.1, 0.1, 0.2, 0.3]).astype(np.int32)
            clk.sched_step(lk, s, _i32(k), _i32(pa), length, length)
            L = length.cpu().numpy()
            want = np.array([refs[b].step(int(k[b]), int(pa[b]), int(pl[b])) for b in range(B)])
            assert np.array_equal(L, want), (kw, t)
            pa = np.array([rng.integers(0, L[b]) if rng.random() < 0.4 else L[b] - 1 for b in range(B)], np.int32)
            pl = L.astype(np.int32)
        for b in range(B):
            info = lk.slot_info(b)
            assert (info["mode"], info["streak"], info["miss"]) == (refs[b].s.mode, refs[b].s.streak, refs[b].s.miss)


C = [10 + i for i in range(16)]
M = {"both": [10, 11, 52, 53, 54, 55, 56], "first": [10, 51, 52, 53, 54, 55, 56],
     "second": [50, 11, 52, 53, 54, 55, 56], "none": [50, 51, 52, 53, 54, 55, 56]}


def test_fusion_truth_table():
    rows = _golden("fusion_table.json")["rows"]
    B = len(rows)
    p = clk.Params.default()
    draft = [C if r["k"] > 0 else [-1] * 16 for r in rows]
    head = [M[r["agree"]] for r in rows]
    blk = torch.zeros((B, 16), dtype=torch.int32, device="cuda")
    clk.fuse(p, _i32([1000] * B), _i32(draft), _i32([r["k"] for r in rows]), _i32(head),
             _i32([r["L"] for r in rows]), blk)
    got = blk.cpu().numpy()
    for b, r in enumerate(rows):
        hd = draft[b][:7] if r["head"] == "lookup" else head[b]
        tl = draft[b][7:15] if r["tail"] == "lookup" else [-1] * 8
        assert got[b].tolist() == [1000] + list(hd) + list(tl), r


@pytest.mark.parametrize("kw", [{}, dict(head=3, tail=4, head_agree_n=3, head_replace_k=10),
                                dict(head=0, tail=15, head_agree_n=0), dict(head=7, tail=0, head_agree_n=0)])
def test_fusion_random_against_oracle(kw):
    rng = np.random.default_rng(62)
    B = 500
    p = clk.Params.default(**kw)
    po = oracle.Params.default(**kw)
    k = rng.choice([0, 3, 4, 5, 6, 7, 8, 9, 12], size=B).astype(np.int32)
    draft = rng.integers(0, 3, size=(B, 16)).astype(np.int32)
    draft[k == 0] = -1
    head = rng.integers(0, 3, size=(B, max(p.head, 1))).astype(np.int32)[:, :p.head]
    L = rng.choice([p.short_len, p.long_len], size=B).astype(np.int32)
    last = rng.integers(0, 100, size=B).astype(np.int32)
    blk = torch.zeros((B, 16), dtype=torch.int32, device="cuda")
    clk.fuse(p, _i32(last), _i32(draft), _i32(k), torch.from_numpy(np.ascontiguousarray(head)).cuda(), _i32(L), blk)
    got = blk.cpu().numpy()
    for b in range(B):
        m = np.zeros(16, np.int32)
        m[:p.head] = head[b]
        want = oracle.fuse(int(last[b]), draft[b], int(k[b]), m, int(L[b]), po)
        assert got[b].tolist() == want.tolist(), b
