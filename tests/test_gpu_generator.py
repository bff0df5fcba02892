"""The device generator produces the same bits as the host generator that
feeds the oracle (logit rows and head proposals).  GPU."""
import numpy as np
import pytest
import torch

import workload as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind,dtype,V", [("mixed", wl.BF16, 248320), ("periodic", wl.BF16, 32000),
                                          ("copy", wl.F32, 1024), ("chat", wl.BF16, 1000)])
def test_logits_and_head_match_host(kind, dtype, V):
    w = wl.make_small(kind, seed=31, B=3, V=V, steps=4, dtype=dtype)
    host = wl.HostGen(w)
    dev = wl.DevGen(w)
    pos = torch.tensor([w.prompts[b].size + 7 * b for b in range(w.B)], dtype=torch.int64, device="cuda")
    out = dev.alloc_logits()
    dev.logits(out, pos)
    head = torch.zeros((w.B, wl.HEAD), dtype=torch.int32, device="cuda")
    dev.head(5, head, pos)
    torch.cuda.synchronize()
    got = out.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == wl.BF16 else out.cpu().numpy()
    for b in range(w.B):
        P0 = int(pos[b])
        want = host.logits_rows(b, P0, wl.ROWS)
        assert np.array_equal(got[b].view(want.dtype) if dtype == wl.BF16 else got[b], want)
        assert np.array_equal(head[b].cpu().numpy(), host.head(b, 5, P0))


def test_advance_tracks_emitted():
    w = wl.make_small("mixed", seed=32, B=4, V=512, steps=2)
    dev = wl.DevGen(w)
    e = torch.tensor([1, 5, 16, 0], dtype=torch.int32, device="cuda")
    dev.advance(e)
    dev.advance(e)
    assert dev.pos.cpu().tolist() == [int(n) + 2 * int(x) for n, x in zip(w.n0, [1, 5, 16, 0])]


def test_device_uniforms_equal_host_uniforms():
    w = wl.make_small("mixed", seed=17, B=5, V=512, steps=8)
    hg, dg = wl.HostGen(w), wl.DevGen(w, device="cuda")
    out = torch.zeros((w.B, 16, 2), dtype=torch.float32, device="cuda")
    for t in (0, 1, 7, 123456):
        dg.uniforms(t, out)
        d = out.cpu().numpy()
        for b in range(w.B):
            h = hg.uniforms(b, t)
            assert np.array_equal(d[b].view(np.uint32), h.view(np.uint32)), (t, b)
            assert (h >= 0).all() and (h < 1).all()
