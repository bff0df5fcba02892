"""Drive the CUDA path over a synthetic workload and record every step.

Testbench code: the device generator supplies each step's head proposals and
target logits (the stand-ins for the draft and target models), the product
library runs the step, and every per-step field is recorded on the device
for comparison with the oracle.  Nothing here computes any part of the
method.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

import context_lookup_speculative_gb300 as clk
import workload as wl


@dataclasses.dataclass
class DeviceRun:
    k: np.ndarray
    j: np.ndarray
    L: np.ndarray
    a: np.ndarray
    c: np.ndarray
    blk: np.ndarray
    g: np.ndarray
    emitted: np.ndarray
    histories: list
    counters: list
    status: tuple


def make_lookup(w: wl.Workload, params=None, slots=None, max_hist=None, device="cuda"):
    B = w.B
    slots = torch.arange(B, dtype=torch.int32, device=device) if slots is None else slots
    lk = clk.Lookup(max_slots=int(slots.max().item()) + 1, max_hist=max_hist or w.max_hist, vocab=w.V,
                    params=params, device=device)
    ptok, poff = w.prompt_csr()
    clk.lookup_init(lk, slots, torch.from_numpy(ptok).to(device), torch.from_numpy(poff).to(device))
    return lk, slots


def run_device(w: wl.Workload, steps: Optional[int] = None, params=None, mode: str = "fused",
               device="cuda", record: bool = True, inv_temp: float = 0.0) -> DeviceRun:
    """Run `steps` decode steps of workload `w` on the GPU.

    mode "fused":   propose_fuse_sched + verify_append (the Step driver)
    mode "semi":    lookup_propose, fuse_sched, verify_append
    mode "unfused": lookup_propose, sched_step, fuse, verify_greedy, lookup_append
    mode "sample":  lookup_propose, sched_step, fuse, verify_sample (at
                    `inv_temp`, with the generator's uniforms), lookup_append;
                    the records' g holds the emitted tokens
    mode "sample_fused": propose_fuse_sched + verify_sample_append (the Step
                    driver's sampled step); g as for "sample"
    mode "sample_exact": as "sample" with verify_sample_exact (the
                    fixed-point weights)
    mode "sample_exact_fused": as "sample_fused" on the fixed-point weights
                    (verify_sample_exact_append)
    """
    steps = w.steps if steps is None else steps
    params = params or clk.Params.default()
    lk, slots = make_lookup(w, params, device=device)
    gen = wl.DevGen(w, device=device)
    st = clk.Step(lk, slots)
    B = w.B
    if params.head > wl.HEAD:
        raise ValueError(f"the synthetic draft model proposes {wl.HEAD} tokens; head must be <= {wl.HEAD}")
    head7 = torch.zeros((B, wl.HEAD), dtype=torch.int32, device=device)
    logits = gen.alloc_logits()
    i32 = dict(dtype=torch.int32, device=device)
    rec = {n: torch.zeros((steps, B), **i32) for n in ("k", "j", "L", "a", "e")}
    rec.update({n: torch.zeros((steps, B, clk.BLOCK), **i32) for n in ("c", "blk", "g")})
    scratch = clk.verify_scratch(B, device=device) if mode == "unfused" else None
    if mode in ("sample", "sample_fused", "sample_exact", "sample_exact_fused"):
        if not inv_temp > 0:
            raise ValueError("mode 'sample' needs inv_temp > 0")
        if mode == "sample_exact":
            sscratch = clk.verify_sample_exact_scratch(logits.dtype, w.V, B, device=device)
        else:
            sscratch = clk.verify_sample_scratch(logits.dtype, w.V, B, device=device)
        uni = torch.zeros((B, clk.BLOCK, 2), dtype=torch.float32, device=device)
        temps = torch.full((B,), float(inv_temp), dtype=torch.float32, device=device)
    last_tok = torch.from_numpy(np.array([p[-1] for p in w.prompts], dtype=np.int32)).to(device)
    for t in range(steps):
        gen.head(t, head7)
        head = head7[:, :params.head].contiguous()
        if mode in ("fused", "sample_fused", "sample_exact_fused"):
            st.pre(head)
        elif mode == "semi":
            clk.lookup_propose(lk, slots, st.draft, st.k, st.j)
            clk.fuse_sched(lk, slots, st.draft, st.k, head, st.accept, st.length, st.length, st.block)
        elif mode in ("unfused", "sample", "sample_exact"):
            clk.lookup_propose(lk, slots, st.draft, st.k, st.j)
            clk.sched_step(lk, slots, st.k, st.accept, st.length, st.length)
            clk.fuse(params, last_tok, st.draft, st.k, head, st.length, st.block)
        else:
            raise ValueError(mode)
        gen.logits(logits)
        if mode == "unfused":
            clk.verify_greedy(logits, st.block, st.length, st.argmax, st.accept, st.emitted, st.out_tok, scratch)
            clk.lookup_append(lk, slots, st.out_tok, st.emitted)
            last_tok = st.out_tok.gather(1, st.accept.long().unsqueeze(1)).squeeze(1).contiguous()
        elif mode in ("sample", "sample_exact"):
            gen.uniforms(t, uni)
            verify = clk.verify_sample_exact if mode == "sample_exact" else clk.verify_sample
            verify(logits, st.block, st.length, temps, uni, st.accept, st.emitted, st.out_tok, sscratch)
            clk.lookup_append(lk, slots, st.out_tok, st.emitted)
            last_tok = st.out_tok.gather(1, st.accept.long().unsqueeze(1)).squeeze(1).contiguous()
            st.argmax.copy_(st.out_tok)  # recorded as g
        elif mode in ("sample_fused", "sample_exact_fused"):
            gen.uniforms(t, uni)
            st.post_sample(logits, temps, uni, exact=mode == "sample_exact_fused")
            st.argmax.copy_(st.out_tok)  # recorded as g
        else:
            st.post(logits)
        gen.advance(st.emitted)
        if record:
            rec["k"][t].copy_(st.k)
            rec["j"][t].copy_(st.j)
            rec["L"][t].copy_(st.length)
            rec["a"][t].copy_(st.accept)
            rec["e"][t].copy_(st.emitted)
            rec["c"][t].copy_(st.draft)
            rec["blk"][t].copy_(st.block)
            rec["g"][t].copy_(st.argmax)
    torch.cuda.synchronize()
    status = lk.status()
    hists = [lk.history(int(s)) for s in slots.tolist()]
    counters = [lk.counters(int(s)) for s in slots.tolist()]
    r = {n: v.cpu().numpy() for n, v in rec.items()}
    return DeviceRun(k=r["k"], j=r["j"], L=r["L"], a=r["a"], c=r["c"], blk=r["blk"], g=r["g"], emitted=r["e"],
                     histories=hists, counters=counters, status=status)


def compare(dev: DeviceRun, ref, req_ids=None, steps=None) -> list:
    """Field-by-field mismatches between a device run and an oracle run
    (bit-exact: every field is an integer).  Returns a list of messages."""
    req_ids = list(range(dev.k.shape[1])) if req_ids is None else list(req_ids)
    steps = ref.steps if steps is None else steps
    msgs = []
    for name in ("k", "j", "L", "a", "c", "blk", "g"):
        d = getattr(dev, name)[:steps][:, req_ids]
        o = getattr(ref, name)[:steps]
        if not np.array_equal(d, o):
            bad = np.argwhere(d != o)
            t, i = int(bad[0][0]), int(bad[0][1])
            msgs.append(f"{name}: {len(bad)} mismatches, first at step {t} request {req_ids[i]}: "
                        f"gpu={d[t, i].tolist()} oracle={o[t, i].tolist()}")
    full = dev.k.shape[0] == ref.steps
    for i, b in enumerate(req_ids):
        if not full:
            break
        if not np.array_equal(dev.histories[b], ref.histories[i]):
            msgs.append(f"history of request {b} differs")
        if dev.counters[b] != ref.counters[i]:
            msgs.append(f"counters of request {b} differ: gpu={dev.counters[b]} oracle={ref.counters[i]}")
    if dev.status[0] != 0:
        msgs.append(f"device status {dev.status}")
    return msgs
