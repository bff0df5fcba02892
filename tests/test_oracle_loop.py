"""Whole-loop pins for the oracle, CPU only.

Lossless invariant (HyperQwen context-lookup article, "三步走", last
paragraph: greedy verification never reads the draft distribution, so the
output is unchanged): because the synthetic target's logits are a pure
function of (request, absolute position), the tokens the speculative loop
emits must equal plain one-token-per-step argmax decoding of the same
logits, token for token, whatever the drafts and the schedule.
"""
import numpy as np
import pytest

import oracle
import workload as wl


def _plain_decode(gen, b, n0, count):
    rows = gen.logits_rows(b, n0, count)
    if rows.dtype == np.uint16:
        rows = wl.bf16_bits_to_f32(rows)
    return np.argmax(rows, axis=1).astype(np.int32)  # numpy: first occurrence on ties


def _check_lossless(w, res):
    gen = wl.HostGen(w)
    for i, b in enumerate(res.req_ids):
        n0 = w.prompts[b].size
        h = res.histories[i]
        assert np.array_equal(h[:n0], w.prompts[b])
        assert np.array_equal(h[n0:], _plain_decode(gen, b, n0, h.size - n0)), b


@pytest.mark.parametrize("kind", ["mixed", "periodic", "copy", "chat"])
@pytest.mark.parametrize("sticky", [0, 3])
def test_lossless_small_workloads(kind, sticky):
    w = wl.make_small(kind, seed=5, B=4, V=2048, steps=40)
    res = oracle.run(w, params=oracle.Params.default(sticky=sticky))
    _check_lossless(w, res)


def test_lossless_tiny_config():
    w = wl.make("0")
    _check_lossless(w, oracle.run(w))


@pytest.mark.parametrize("law", ["all_right", "all_wrong"])
def test_lossless_under_forced_head_laws(law):
    w = wl.make_small("mixed", seed=6, B=2, V=512, steps=30)
    gen = wl.HostGen(w)

    def head(b, t, n):
        truth = [gen.truth(b, n + i) for i in range(7)]
        return truth if law == "all_right" else [(x + 1) % w.V for x in truth]

    res = oracle.run(w, head=head, threads=1)
    _check_lossless(w, res)
    kept = (res.blk[:, :, 1:8] == res.blk[:, :, 1:8]).all(axis=2)
    for t in range(res.steps):
        for i in range(2):
            n = w.prompts[i].size + int((res.a[:t, i] + 1).sum())
            m = head(i, t, n)
            kept[t, i] = list(res.blk[t, i, 1:8]) == m
    if law == "all_right":
        # a kept all-right head is accepted in full unless the synthetic
        # target's noise beats the +8 boost somewhere in its 7 rows.
        assert (res.a[kept] >= 7).mean() > 0.97
    else:
        # a kept all-wrong head is rejected at its first slot.
        assert (res.a[kept] == 0).all()


def test_records_and_counters_are_consistent():
    w = wl.make_small("mixed", seed=7, B=4, V=1024, steps=50)
    res = oracle.run(w)
    for i in range(w.B):
        c = res.counters[i]
        k, L, a = res.k[:, i], res.L[:, i], res.a[:, i]
        assert c["steps"] == w.steps
        assert c["emitted"] == int((a + 1).sum()) == res.histories[i].size - w.prompts[i].size
        assert c["accepted"] == int(a.sum())
        assert c["hits"] == int((k >= 4).sum())
        assert c["long_steps"] == int((L == 16).sum())
        assert c["drafted"] == int((7 + 8 * ((L == 16) & (k >= 4))).sum())
        assert sum(map(sum, c["accept_hist"])) == w.steps
        assert set(np.unique(L)) <= {8, 16}
        assert (a <= L - 1).all()
        # emitted tokens are the argmax prefix, and blk[0] is the last token
        for t in range(w.steps):
            g = res.g[t, i]
            assert (g[L[t]:] == -1).all() and (g[:L[t]] >= 0).all()
        # j is -1 exactly when nothing matched
        assert ((k == 0) == (res.j[:, i] == -1)).all()
        assert (res.blk[:, i, 0] >= 0).all()


def test_generator_statistics():
    """Generator sanity (not parity): with no lookup hits the head law gives
    E[a] = sum_i prod_{s<i} (0.9 - 0.03 s) ~= 3.825 accepted drafts per
    8-token step."""
    expect = sum(np.prod([0.9 - 0.03 * s for s in range(i)]) for i in range(1, 8))
    assert abs(expect - 3.825) < 1e-3
    w = wl.make_small("chat", seed=8, B=8, V=248320, steps=60, L=(300, 600))
    res = oracle.run(w)
    miss = (res.k == 0) & (res.L == 8)
    mean_a = res.a[miss].mean()
    assert abs(mean_a - expect) < 0.35, mean_a
    # the tiny config's prompt has about 30% copied positions
    w0 = wl.make("0")
    h = w0.prompts[0]
    assert h.size == 2048


def test_time_split_covers_the_method_time():
    """The oracle's per-component times (lookup, scheduler + fusion, verify)
    are non-negative, fit inside the method time, and leave only the small
    append and bookkeeping rest uncounted."""
    w = wl.make_small("mixed", seed=3, B=4, V=4096, L=(200, 400), steps=12)
    res = oracle.run(w, threads=1, timed_from=2)
    parts = (res.lookup_s, res.sched_fuse_s, res.verify_s)
    assert all(x >= 0 for x in parts)
    assert sum(parts) <= res.method_s + 1e-6
    assert sum(parts) >= 0.5 * res.method_s
