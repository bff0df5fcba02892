"""The derived metrics (hit rate, mean accepted length, tail share, accepted
length histograms per workload kind) against the same figures computed
directly from the oracle's per-step records (k, L, a) of a mixed batch."""
import numpy as np
import pytest

import oracle
import workload as wl
from context_lookup_speculative_gb300 import metrics


@pytest.fixture(scope="module")
def mixed_run():
    w = wl.make_small("mixed", seed=91, B=8, V=2048, steps=80)
    return w, oracle.run(w, threads=4)


def _direct(ref, idx, head=7, min_k=4, tail_k=4, tail=8):
    k = np.asarray(ref.k)[:, idx]
    L = np.asarray(ref.L)[:, idx]
    a = np.asarray(ref.a)[:, idx]
    hist = {"short": [int(((L == 8) & (a == x)).sum()) for x in range(16)],
            "long": [int(((L == 16) & (a == x)).sum()) for x in range(16)]}
    drafted = int((head + np.where((L == 16) & (k >= tail_k), tail, 0)).sum())
    return {"steps": k.size, "hits": int((k >= min_k).sum()), "long_steps": int((L == 16).sum()),
            "accepted": int(a.sum()), "emitted": int((a + 1).sum()), "drafted": drafted,
            "tail_accepted": int(np.maximum(a - head, 0).sum()), "accept_hist": hist}


def test_per_kind_metrics_match_the_step_records(mixed_run):
    w, ref = mixed_run
    got = metrics.by_kind(ref.counters, w.kinds)
    assert set(got) == {"all", "copy", "chat"}
    for kind in ("all", "copy", "chat"):
        idx = [i for i, kk in enumerate(w.kinds) if kind == "all" or kk == kind]
        d = _direct(ref, idx)
        g = got[kind]
        for f in ("steps", "hits", "long_steps", "accepted", "emitted", "drafted", "tail_accepted"):
            assert g[f] == d[f], (kind, f)
        assert g["accept_hist"] == d["accept_hist"], kind
        assert g["hit_rate"] == pytest.approx(d["hits"] / d["steps"], abs=1e-6)
        assert g["mean_accepted"] == pytest.approx(d["accepted"] / d["steps"], abs=1e-6)
        assert g["tail_share"] == pytest.approx(d["tail_accepted"] / d["accepted"], abs=1e-6)
        assert g["requests"] == len(idx)
    # copy-heavy requests reach the long block and accept past the head
    assert got["copy"]["long_share"] > got["chat"]["long_share"]
    assert got["copy"]["tail_accepted"] > 0


def test_delta_and_empty_sets(mixed_run):
    w, ref = mixed_run
    zero = [{f: 0 for f in metrics.FIELDS} | {"accept_hist": [[0] * 16, [0] * 16]} for _ in ref.counters]
    assert metrics.delta(ref.counters, zero) == ref.counters
    assert metrics.delta(ref.counters, ref.counters) == zero
    s = metrics.summarize(zero)
    assert s["steps"] == 0 and s["hit_rate"] is None and s["tail_share"] is None
    with pytest.raises(ValueError):
        metrics.by_kind(ref.counters, w.kinds[:-1])


def test_tail_share_hand_counts():
    # one request: 3 long steps accepting 15, 9 and 2 drafts, 1 short step accepting 7
    c = {"steps": 4, "hits": 4, "long_steps": 3, "drafted": 3 * 15 + 7, "accepted": 33, "emitted": 37,
         "accept_hist": [[0] * 16, [0] * 16]}
    c["accept_hist"][1][15] = 1
    c["accept_hist"][1][9] = 1
    c["accept_hist"][1][2] = 1
    c["accept_hist"][0][7] = 1
    s = metrics.summarize([c])
    assert s["tail_accepted"] == 8 + 2  # slots 8..15 of the first step, 8..9 of the second
    assert s["tail_share"] == pytest.approx(10 / 33, abs=1e-6)
    assert s["tokens_per_step"] == pytest.approx(37 / 4, abs=1e-6)


def test_short_blocks_only_count_no_long_steps():
    # with no tail (7 drafts, the pages' short setting) every block has
    # 1 + head slots, so no step is a long block whatever the scheduler's mode
    w = wl.make_small("copy", seed=92, B=4, V=2048, steps=48)
    ref = oracle.run(w, params=oracle.Params.default(tail=0), threads=4)
    s = metrics.summarize(ref.counters)
    assert s["long_steps"] == 0 and s["long_share"] == 0
    assert sum(s["accept_hist"]["long"]) == 0 and sum(s["accept_hist"]["short"]) == s["steps"]
    assert s["tail_accepted"] == 0 and (np.asarray(ref.L) == 8).all()
    assert s["drafted"] == 7 * s["steps"]
