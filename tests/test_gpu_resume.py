"""Checkpoint / resume of requests: snapshot every request's history,
scheduler state and counters in the middle of a decode loop, restore them
into another workspace under other slot numbers, and the loop continues
exactly as it would have without the interruption.  GPU."""
import numpy as np
import pytest
import torch

import context_lookup_speculative_gb300 as clk
import workload as wl
from workload import drive

pytestmark = pytest.mark.gpu


def _steps(st, gen, t0, n, rec):
    head = torch.zeros((gen.w.B, wl.HEAD), dtype=torch.int32, device="cuda")
    lg = gen.alloc_logits()
    for t in range(t0, t0 + n):
        gen.head(t, head)
        st.pre(head)
        gen.logits(lg)
        st.post(lg)
        gen.advance(st.emitted)
        rec.append((st.length.clone(), st.emitted.clone(), st.out_tok.clone()))


def test_resumed_loop_continues_bit_for_bit():
    w = wl.make_small("mixed", seed=321, B=10, V=4096, L=(300, 900), steps=24)
    B = w.B
    # A: 24 steps without interruption
    lk_a, slots_a = drive.make_lookup(w)
    st_a, gen_a, rec_a = clk.Step(lk_a, slots_a), wl.DevGen(w, device="cuda"), []
    _steps(st_a, gen_a, 0, 24, rec_a)
    # B: 12 steps, a snapshot of every request, a resume elsewhere, 12 more
    lk_b, slots_b = drive.make_lookup(w)
    st_b, gen_b, rec_b = clk.Step(lk_b, slots_b), wl.DevGen(w, device="cuda"), []
    _steps(st_b, gen_b, 0, 12, rec_b)
    snaps = [lk_b.snapshot(int(s)) for s in slots_b.tolist()]
    accept, length = st_b.accept.clone(), st_b.length.clone()
    del st_b, lk_b
    lk_c = clk.Lookup(max_slots=2 * B + 3, max_hist=w.max_hist, vocab=w.V)
    slots_c = torch.tensor([2 * B + 2 - 2 * b for b in range(B)], dtype=torch.int32, device="cuda")
    for b, snap in enumerate(snaps):
        lk_c.restore(int(slots_c[b]), snap)
    st_c = clk.Step(lk_c, slots_c)
    st_c.resume(accept, length)
    _steps(st_c, gen_b, 12, 12, rec_b)
    for t, (x, y) in enumerate(zip(rec_a, rec_b)):
        for name, p, q in zip(("length", "emitted", "out_tok"), x, y):
            assert torch.equal(p, q), (t, name)
    for b in range(B):
        sa, sc = int(slots_a[b]), int(slots_c[b])
        assert np.array_equal(lk_a.history(sa), lk_c.history(sc)), b
        assert lk_a.counters(sa) == lk_c.counters(sc), b
        ia, ic = lk_a.slot_info(sa), lk_c.slot_info(sc)
        assert {k: ia[k] for k in ("n", "mode", "streak", "miss", "has_prev", "cur_len")} == \
               {k: ic[k] for k in ("n", "mode", "streak", "miss", "has_prev", "cur_len")}, b
    assert lk_c.status() == (0, 0)
    assert sum(int(r[1].sum()) for r in rec_a[12:]) > 12 * B  # drafts were accepted after the resume


def test_restore_refuses_a_history_of_another_length():
    w = wl.make_small("chat", seed=5, B=2, V=1024, L=(100, 120), steps=2)
    lk, slots = drive.make_lookup(w)
    snap = lk.snapshot(0)
    snap["info"] = dict(snap["info"], n=snap["info"]["n"] + 1)
    with pytest.raises(clk.ClkError):
        lk.restore(1, snap)
