"""The two-launch decode step captured in one CUDA graph, as the benchmark
replays it (the verify launch a programmatic dependent of the proposal
launch inside the graph), gives exactly the eager step's tokens, lengths,
histories and counters; greedy and sampled.  GPU."""
import numpy as np
import pytest
import torch

import context_lookup_speculative_gb300 as clk
import workload as wl
from workload import drive

pytestmark = pytest.mark.gpu


def _eager(w, n, temp):
    """n eager steps; the generator positions each step starts from, and what
    every step emitted."""
    lk, slots = drive.make_lookup(w)
    st = clk.Step(lk, slots)
    gen = wl.DevGen(w, device="cuda")
    head = torch.zeros((w.B, wl.HEAD), dtype=torch.int32, device="cuda")
    lg = gen.alloc_logits()
    u = torch.zeros((w.B, 16, 2), dtype=torch.float32, device="cuda")
    t_inv = torch.full((w.B,), 1.0 / temp if temp else 1.0, device="cuda")
    pos, out, em, ln = [], [], [], []
    for t in range(n):
        pos.append(gen.pos.clone())
        gen.head(t, head)
        st.pre(head)
        gen.logits(lg)
        if temp:
            gen.uniforms(t, u)
            st.post_sample(lg, t_inv, u)
        else:
            st.post(lg)
        gen.advance(st.emitted)
        out.append(st.out_tok.clone())
        em.append(st.emitted.clone())
        ln.append(st.length.clone())
    torch.cuda.synchronize()
    return lk, slots, pos, torch.stack(out), torch.stack(em), torch.stack(ln)


def _graphed(w, n, temp, pos):
    """The same n steps from pre-generated inputs, captured as one graph and
    replayed once."""
    lk, slots = drive.make_lookup(w)
    st = clk.Step(lk, slots)
    gen = wl.DevGen(w, device="cuda")
    heads = torch.zeros((n, w.B, wl.HEAD), dtype=torch.int32, device="cuda")
    bufs = torch.empty((n, w.B, 16, w.V), dtype=gen.torch_dtype(), device="cuda")
    unis = torch.zeros((n, w.B, 16, 2), dtype=torch.float32, device="cuda")
    t_inv = torch.full((w.B,), 1.0 / temp if temp else 1.0, device="cuda")
    for t in range(n):
        gen.head(t, heads[t], pos=pos[t])
        gen.logits(bufs[t], pos=pos[t])
        gen.uniforms(t, unis[t])
    out = torch.zeros((n, w.B, 16), dtype=torch.int32, device="cuda")
    em = torch.zeros((n, w.B), dtype=torch.int32, device="cuda")
    ln = torch.zeros((n, w.B), dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for t in range(n):
                st.pre(heads[t])
                if temp:
                    st.post_sample(bufs[t], t_inv, unis[t])
                else:
                    st.post(bufs[t])
                out[t].copy_(st.out_tok)
                em[t].copy_(st.emitted)
                ln[t].copy_(st.length)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    return lk, slots, out, em, ln


@pytest.mark.parametrize("temp", [None, 0.5])
def test_graph_replay_equals_eager_steps(temp):
    w = wl.make_small("mixed", seed=123, B=12, V=4096, L=(300, 900), steps=10)
    n = 10
    lk_e, slots, pos, out_e, em_e, ln_e = _eager(w, n, temp)
    lk_g, _, out_g, em_g, ln_g = _graphed(w, n, temp, pos)
    assert torch.equal(ln_e, ln_g)
    assert torch.equal(em_e, em_g)
    assert torch.equal(out_e, out_g)
    for s in slots.tolist():
        assert np.array_equal(lk_e.history(s), lk_g.history(s))
        assert lk_e.counters(s) == lk_g.counters(s)
    assert lk_g.status() == (0, 0)
    assert (em_e > 1).any()  # drafts were accepted: the steps did real work
