#!/usr/bin/env python3
"""Benchmark of the context-lookup speculative decoding hot path on GB300.

One step = one pass of the whole hot path over the batch: proposal (suffix
match + LZ77 copy), scheduler, fusion, greedy verification over the target
logits, and the commit of the emitted tokens into histories and index.  It
runs as the two fused launches of ``Step`` (propose_fuse_sched, then
verify_append).

Workload (default): the mixed serving batch, B=64, prompts U{2,000..32,000}
Zipf(1.1) tokens over V=248,320, half copy-heavy and half chat-like, bf16
logits [64, 16, 248320] with the +8 ground-truth boost; 8 warm-up steps and
504 timed steps = the workload's 512 steps.  Every timed step reads logits
generated beforehand into their own HBM buffers (inputs resident, larger
than L2, so nothing is served from a previous step's L2 lines).

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "spec steps/s and accepted tok/s (1 GB300), % of HBM roofline, vs CPU oracle"
UNIT = "spec steps/s"
CONFIG_NAMES = {"0": "tiny B=1 V=1024 fp32", "1": "restatement B=1 L=25000 V=248320 bf16",
                "2": "mixed serving batch B=64 L=2k-32k V=248320 bf16",
                "3": "periodic B=16 L=8192 V=32000 bf16", "4a": "long context B=8 L=262144 V=248320 bf16",
                "4b": "index stress B=256 L=4096 V=248320 bf16"}
# Lookup-side bytes per request per step that the method must move (besides
# the logits): suffix 48, index probes 9x8, one match check 48, copy 64,
# head 28, previous a/L 8, block+draft writes 128, k/j/L 12 (proposal
# launch); block read 64, argmax/out_tok writes 128, a/emitted 8, history
# append 64, index inserts 16 x 9 x 16 (verify launch).
LOOKUP_BYTES_PER_REQ = 48 + 72 + 48 + 64 + 28 + 8 + 128 + 12 + 64 + 128 + 8 + 64 + 16 * 9 * 16


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# The exact sampler is bound by arithmetic, not HBM.  Its algorithmic work per
# entry, in thread instructions: the scaled difference d (one fused
# multiply-add), the rounding split (three adds) and six Horner steps, all
# packed two entries to an instruction (5 per entry), plus six integer
# operations (the mantissa scaled, the shift amount, the funnel shift, the
# two of the rounding and the sum).  Peak: one warp instruction per scheduler
# per clock, four schedulers per SM.
FX_INSTR_PER_ENTRY = 11


def _alu_roofline(kernel: str, entries: float, seconds: float, clocks: dict, hbm: dict) -> dict:
    import torch

    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    mhz = float(clocks.get("sm_max_mhz") or 2070.0)
    peak = 4 * 32 * sms * mhz * 1e6 / 1e12  # thread instructions, T/s
    achieved = entries * FX_INSTR_PER_ENTRY / seconds / 1e12
    return {"bound": "alu", "kernel": kernel, "achieved": round(achieved, 3), "peak": round(peak, 3),
            "unit": "T thread-instructions/s", "frac": round(achieved / peak, 4),
            "peak_source": f"4 schedulers x 32 lanes x {sms} SMs x {mhz:.0f} MHz (one instruction per scheduler "
                           f"per clock)",
            "algorithmic_instructions_per_entry": FX_INSTR_PER_ENTRY, "entries_per_launch": int(entries),
            "hbm": hbm}


def _verify_sources_hash() -> str:
    h = hashlib.sha256()
    for f in ("clk_verify.cu", "clk_device.cuh"):
        with open(os.path.join(ROOT, "context_lookup_speculative_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic_ratio():
    """DRAM bytes (read + write) over algorithmic bytes of the verify launch,
    from the committed ncu capture of three full-size launches of this
    workload, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "k_verify_step_cfg2_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("source_hash") != _verify_sources_hash():
            return None
        return float(d["traffic_over_algorithmic"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", f"-lms={period_ms}"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        rows = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), util=float(f[4]),
                                 hw=f[6], hwt=f[7], swt=f[8], pcap=f[9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        busy = [r for r in rows if r["util"] > 0] or rows
        sm = sorted(r["sm"] for r in busy)
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                          ("pcap", "sw_power_cap")):
            if any(r[key].lower() == "active" for r in busy):
                reasons.append(name)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r["smax"] for r in rows), "reasons": reasons,
                "samples": len(busy)}


def _dist():
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local, dist


def shard_seed(base_seed: int, rank: int) -> int:
    """Each rank serves its own batch of the same recipe (weak scaling)."""
    return base_seed + 1000 * rank


def max_over_ranks(value: float, dist, world: int, device) -> float:
    if world == 1:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_ours(args, world, rank, local, dist):
    import numpy as np
    import torch

    import context_lookup_speculative_gb300 as clk
    import workload as wl
    from workload import drive

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    clk.lib()
    w = wl.make(args.config, seed=shard_seed(int(wl.DEFAULT_SEED[args.config]), rank))
    W, K = args.warmup, args.steps
    if W + K > w.steps:  # the workload's streams cover w.steps steps
        K = w.steps - W
    B, V = w.B, w.V
    params = clk.Params.default(**getattr(args, "overrides", {}))
    if params.head > wl.HEAD:
        raise ValueError(f"head {params.head}: the synthetic draft model proposes {wl.HEAD} tokens")
    stream = torch.cuda.current_stream(device)

    # Lookup state; the prompt ingestion (index build) is timed on its own.
    lk, slots = drive.make_lookup(w, params, device=device)
    ptok, poff = w.prompt_csr()
    d_ptok, d_poff = torch.from_numpy(ptok).to(device), torch.from_numpy(poff).to(device)
    gen = wl.DevGen(w, device=device)
    st = clk.Step(lk, slots)
    head = torch.zeros((B, params.head), dtype=torch.int32, device=device)
    head7 = torch.zeros((B, wl.HEAD), dtype=torch.int32, device=device)

    def gen_head(t, out, pos=None):
        """The first params.head of the synthetic model's proposals for step t."""
        if params.head == wl.HEAD:
            gen.head(t, out, pos=pos)
        else:
            gen.head(t, head7, pos=pos)
            out.copy_(head7[:, :params.head])

    logits = gen.alloc_logits()
    temp = getattr(args, "sampling", None)  # sampled verification at this temperature, else greedy
    if temp is not None and not temp > 0:
        raise ValueError("--sampling needs a temperature > 0")
    temps = torch.full((B,), 1.0 / temp if temp else 1.0, dtype=torch.float32, device=device)
    uni = torch.zeros((B, 16, 2), dtype=torch.float32, device=device)
    exact = bool(getattr(args, "exact", False)) and temp is not None  # sampling on the fixed-point weights

    def post(t, lg, u=None):
        """The step's verify launch: greedy, or sampled with step t's uniforms."""
        if temp is None:
            st.post(lg)
            return
        if u is None:
            gen.uniforms(t, uni)
            u = uni
        st.post_sample(lg, temps, u, exact=exact)

    def reinit():
        clk.lookup_init(lk, slots, d_ptok, d_poff)
        gen.reset()
        st.reset()

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    clk.lookup_init(lk, slots, d_ptok, d_poff)
    e1.record(stream)
    torch.cuda.synchronize()
    index_build_ms = e0.elapsed_time(e1)

    # Dry run: the positions every step starts from (the path is deterministic).
    reinit()
    pos_hist = torch.zeros((W + K + 1, B), dtype=torch.int64, device=device)
    for t in range(W + K):
        pos_hist[t].copy_(gen.pos)
        gen_head(t, head)
        st.pre(head)
        gen.logits(logits)
        post(t, logits)
        gen.advance(st.emitted)
    pos_hist[W + K].copy_(gen.pos)
    torch.cuda.synchronize()

    per_step = B * 16 * V * (2 if w.dtype == wl.BF16 else 4)
    chunk = max(1, min(K, int(args.input_gb * 2 ** 30 // per_step)))
    heads = torch.zeros((chunk, B, params.head), dtype=torch.int32, device=device)
    unis = torch.zeros((chunk, B, 16, 2), dtype=torch.float32, device=device)
    bufs = torch.empty((chunk, B, 16, V), dtype=gen.torch_dtype(), device=device)
    flush = torch.empty(2 * 160 * 2 ** 20, dtype=torch.uint8, device=device)  # > 2x the 129 MB L2
    del logits

    def warmup():
        reinit()
        lg = bufs[0]
        for t in range(W):
            gen_head(t, head)
            st.pre(head)
            gen.logits(lg)
            post(t, lg)
            gen.advance(st.emitted)
        torch.cuda.synchronize()

    def generate(t0, n):
        for i in range(n):
            gen_head(t0 + i, heads[i], pos=pos_hist[t0 + i])
            gen.logits(bufs[i], pos=pos_hist[t0 + i])
            if temp is not None:
                gen.uniforms(t0 + i, unis[i])
        flush.zero_()  # no step may find its logits in L2
        torch.cuda.synchronize()

    def capture(n, events=None, lens=None):
        """The n steps of a chunk as one CUDA graph (launched with one call, so
        no host time falls inside the timed region); `events` get recorded
        around every launch, `lens` receives each step's block lengths."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                if events is not None:
                    events[3 * i].record()
                st.pre(heads[i])
                if events is not None:
                    events[3 * i + 1].record()
                post(None, bufs[i], unis[i])
                if events is not None:
                    events[3 * i + 2].record()
                if lens is not None:
                    lens[i].copy_(st.length)
        return g

    # Pass B: the first steps once more with an event around every launch, for
    # each kernel's own duration (launches serialised by the events, so the
    # verify launches are made as launched alone: every CTA an even share).
    warmup()
    nb = min(chunk, K)
    generate(W, nb)
    lens_b = torch.zeros((nb, B), dtype=torch.int32, device=device)
    lk.set_alone(True)
    try:
        # events recorded inside a graph must be "external" to be timed
        ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(3 * nb)]
        graph = capture(nb, ev, lens_b)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        del graph
    except TypeError:  # a torch without external events: launch pass B directly
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3 * nb)]
        for i in range(nb):
            ev[3 * i].record(stream)
            st.pre(heads[i])
            ev[3 * i + 1].record(stream)
            post(None, bufs[i], unis[i])
            ev[3 * i + 2].record(stream)
            lens_b[i].copy_(st.length)
        torch.cuda.synchronize()
    lk.set_alone(False)
    pre_ms = sum(ev[3 * i].elapsed_time(ev[3 * i + 1]) for i in range(nb))
    verify_ms = sum(ev[3 * i + 1].elapsed_time(ev[3 * i + 2]) for i in range(nb))
    cb = lk.counters(-1)
    # logits bytes each pass-B verify launch had to read (for the ncu traffic comparison)
    esz_b = 2 if w.dtype == wl.BF16 else 4
    passb_bytes = [int(x) * V * esz_b for x in lens_b.sum(dim=1).tolist()]
    # Pass A (the measurement): warm-up again from the reset state, then the
    # timed steps back to back in chunks whose inputs are generated beforehand
    # into HBM, each chunk replayed as one CUDA graph; the two launches of a
    # step overlap (programmatic dependent launch) and nothing is recorded
    # between them.
    warmup()
    c_w = lk.counters(-1)
    rows_b = params.short_len * (cb["steps"] - c_w["steps"]) + \
        (params.long_len - params.short_len) * (cb["long_steps"] - c_w["long_steps"])
    clocks = ClockSampler(local)
    time.sleep(0.3)
    total_ms = 0.0
    launches = 0
    c_before = lk.counters(-1)
    slot_list = [int(x) for x in slots.tolist()]
    per_before = [lk.counters(x) for x in slot_list]
    t = W
    while t < W + K:
        n = min(chunk, W + K - t)
        generate(t, n)
        if world > 1:
            dist.barrier()
        graph = capture(n)
        torch.cuda.synchronize()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        graph.replay()
        end.record(stream)
        torch.cuda.synchronize()
        launches += 2 * n
        del graph
        if world > 1:
            dist.barrier()
        total_ms += start.elapsed_time(end)
        t += n
    clocks.stop()
    c_after = lk.counters(-1)
    per_after = [lk.counters(x) for x in slot_list]
    status = lk.status()
    # Determinism check: the timed steps ended where the dry run did.
    if status[0] != 0:
        raise RuntimeError(f"device status after the timed steps: {status}")
    hist_lens = torch.tensor([lk.slot_info(int(s))["n"] for s in slots.tolist()], dtype=torch.int64, device=device)
    if not torch.equal(hist_lens, pos_hist[W + K]):
        raise RuntimeError("timed steps diverged from the dry run")
    del bufs

    total_s = max_over_ranks(total_ms * 1e-3, dist, world, device)
    dc = {k: c_after[k] - c_before[k] for k in ("steps", "hits", "long_steps", "drafted", "accepted", "emitted")}
    rows = params.short_len * dc["steps"] + (params.long_len - params.short_len) * dc["long_steps"]
    esz = 2 if w.dtype == wl.BF16 else 4
    # sampled verification also re-reads one segment (exact: one chunk) of each request's drawn row
    draw_bytes = B * min(V, 1024 if exact else 16384) * esz if temp is not None else 0
    verify_bytes = rows * V * esz + draw_bytes * K      # logits rows read, all timed steps
    path_bytes = verify_bytes + LOOKUP_BYTES_PER_REQ * B * K
    peak, peak_kind = _peaks()
    verify_bytes_b = rows_b * V * esz + draw_bytes * nb  # the pass-B steps
    verify_gbs = verify_bytes_b / (verify_ms * 1e-3) / 1e9
    path_gbs = path_bytes / (total_ms * 1e-3) / 1e9
    ratio = _traffic_ratio()

    ablation = run_lookup_ablation(lk, slots, w, device) if args.ablation else None
    e2e = (run_e2e(args, w, params, d_ptok, d_poff, pos_hist, device, temp, exact)
           if (rank == 0 and not args.no_e2e) else None)
    cpu = run_cpu_baseline(args, w) if (rank == 0 and world == 1 and not args.no_cpu_baseline) else None

    lookup_cmp = None
    if cpu is not None:
        # [F] point 1: the incremental index against the full history scan.
        # GPU: the prompt ingestion (index build) once, then per step the
        # proposal launch alone (lookup, scheduler, fusion and the index
        # inserts of the tokens the previous step committed).  Oracle: the
        # full-scan lookup and copy per request-step (thread time).
        ptoks = int(sum(len(p) for p in w.prompts))
        ocore = cpu["one_core"]["us_per_request_step"]["lookup"]
        oall = cpu["us_per_request_step"]["lookup"]
        lookup_cmp = {
            "prompt_tokens": ptoks, "batch": B,
            "mean_history_tokens": int(hist_lens.float().mean().item()),
            "gpu_index_build_ms": round(index_build_ms, 3),
            "gpu_index_build_ns_per_prompt_token": round(index_build_ms * 1e6 / max(1, ptoks), 3),
            "gpu_propose_append_us_per_step": round(pre_ms * 1e3 / nb, 3),
            "gpu_propose_append_us_per_request_step": round(pre_ms * 1e3 / nb / B, 4),
            "oracle_full_scan_lookup_us_per_request_step": {"all_cores": oall, "one_core": ocore,
                                                            "cores": cpu["cores"]},
            "oracle_full_scan_lookup_us_per_step": {
                "all_cores": round(oall * B / max(1, min(cpu["cores"], B)), 3),
                "one_core": round(ocore * B, 3)},
            "note": "GPU proposal launch timed alone (events around it), launch overhead included; the oracle "
                    "times its lookup calls on the same histories over the cpu_baseline sample"}

    steps_s = world * K / total_s
    out = {
        "metric": METRIC if temp is None else METRIC + f", sampled verification at temperature {temp}" +
        (" on the exact (fixed-point) weights" if exact else ""),
        "value": round(steps_s, 2), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(total_s * 1e3 / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == wl.BF16 else "f32", "data": "synthetic",
        "config": {"workload": f"{w.name}: {CONFIG_NAMES[args.config]}, {W} warm-up + {K} timed of "
                               f"{w.steps} steps", "batch": B, "vocab": V, "block": "8 or 16",
                   "l2": "inputs larger than L2: every step reads its own pre-generated logits; "
                         "L2 flushed after each batch of generated inputs",
                   "parallelism": f"replicas x{world} (independent request batches)"},
        "tokens": {"accepted_tok_s": round(world * dc["accepted"] / total_s, 1),
                   "drafted_tok_s": round(world * dc["drafted"] / total_s, 1),
                   "emitted_tok_s": round(world * dc["emitted"] / total_s, 1),
                   "emitted_per_request_step": round(dc["emitted"] / max(1, dc["steps"]), 4),
                   "accepted_per_request_step": round(dc["accepted"] / max(1, dc["steps"]), 4),
                   "long_block_share": round(dc["long_steps"] / max(1, dc["steps"]), 4),
                   "by_kind": _kind_metrics(per_after, per_before, w.kinds, params.head)},
        "path": {"bytes_per_step": int(path_bytes // K), "verify_bytes_per_step": int(verify_bytes // K),
                 "achieved_gbs": round(path_gbs, 1), "frac": round(path_gbs / peak, 4),
                 "alone_us": {"propose_fuse_sched": round(pre_ms * 1e3 / nb, 3),
                              "verify_append": round(verify_ms * 1e3 / nb, 3),
                              "steps": nb, "note": "each launch timed alone (events between launches)"},
                 "overlapped_us_per_step": round(total_ms * 1e3 / K, 3),
                 "index_build_ms": round(index_build_ms, 3)},
        "roofline": {"bound": "hbm", "kernel": "k_verify_step (verify_append)" if temp is None else
                     ("k_sample_step_fx (verify_sample_exact_append)" if exact else
                      "k_sample_step (verify_sample_append)"),
                     "achieved": round(verify_bytes / total_s / 1e9, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(verify_bytes / total_s / 1e9 / peak, 4),
                     "peak_source": f"{peak_kind} hbm_gbs",
                     "traffic": None if ratio is None or args.config != "2" or temp is not None
                     else int(ratio * verify_bytes / K),
                     "traffic_note": "ncu dram read+write per launch, as the measured traffic/algorithmic ratio "
                                     "of three captured full-size launches times this run's bytes per launch",
                     "algorithmic_bytes_per_launch": int(verify_bytes // K),
                     "duration_us": round(total_ms * 1e3 / K, 3),
                     "measured": "in the timed region (CUDA events on the launching stream around the replayed "
                                 "graphs): one launch per step, back to back; each launch starts streaming "
                                 "while the previous one finishes, and the step's proposal launch runs inside "
                                 "that interval; duration_us = timed region / launches",
                     "isolated": {"duration_us": round(verify_ms * 1e3 / nb, 3),
                                  "achieved": round(verify_gbs, 1), "frac": round(verify_gbs / peak, 4),
                                  "algorithmic_bytes_per_launch": int(verify_bytes_b // nb),
                                  "first_launches_algorithmic_bytes": passb_bytes[:4],
                                  "note": "the first steps again, each launch alone (events around every "
                                          "launch serialise the two launches of a step and the steps)"}},
        "clocks": clocks.summary(),
        "gpu_launches": launches,
        "lookup_ablation": ablation,
        "lookup_vs_oracle": lookup_cmp,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if exact:  # the exact sampler is bound by arithmetic: its roofline in instructions, HBM beside it
        out["roofline"] = _alu_roofline(out["roofline"]["kernel"], verify_bytes / esz / K, total_s / K,
                                        out["clocks"], out["roofline"])
    return out


# Draft-block variants: the pages' 15-draft long block against 7 drafts only,
# the sticky exit on and off, and other splits of the block between the
# draft model's head and the lookup tail.
SWEEP = [
    ("15 drafts (7 head + 8 tail), sticky 3", {}),
    ("15 drafts, sticky 0 (exit on the first flag drop)", {"sticky": 0}),
    ("15 drafts, sticky 6", {"sticky": 6}),
    ("7 drafts (short blocks only)", {"tail": 0}),
    ("15 drafts as 5 head + 10 tail", {"head": 5, "tail": 10}),
    ("15 drafts as 3 head + 12 tail", {"head": 3, "tail": 12}),
]


def run_sweep(args, world, rank, local, dist):
    """The measured step (same timing as the headline) once per variant."""
    import copy

    rows = []
    for name, over in SWEEP:
        a = copy.copy(args)
        a.overrides, a.no_e2e, a.no_cpu_baseline, a.ablation = over, True, True, False
        r = run_ours(a, world, rank, local, dist)
        tk = r["tokens"]
        rows.append({"variant": name, "params": over, "value": r["value"], "ms_per_step": r["ms_per_step"],
                     "emitted_per_request_step": tk["emitted_per_request_step"],
                     "emitted_tok_s": tk["emitted_tok_s"], "long_block_share": tk["long_block_share"],
                     "tail_share": {k: v["tail_share"] for k, v in tk["by_kind"].items()},
                     "path_frac": r["path"]["frac"]})
    return {"metric": METRIC, "unit": UNIT, "n_gpus": world, "steps": r["steps"], "warmup": r["warmup"],
            "config": r["config"], "sweep": rows, "clocks": r.get("clocks")}


def run_sample_verify(args, world, rank, local, dist):
    """Sampling verification (clk_verify_sample) on the workload's shapes:
    each launch reads its own pre-generated logits (larger than L2) at
    temperature 0.3, with drafts that follow the synthetic target's favoured
    token except for 20 % random ones; long blocks for the copy-heavy
    requests, short ones for the chat-like.  CUDA events around every launch.
    With --exact: the exact sampler (clk_verify_sample_exact, fixed-point
    weights) on the same inputs."""
    import numpy as np
    import torch

    import context_lookup_speculative_gb300 as clk
    import workload as wl

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    clk.lib()
    w = wl.make(args.config, seed=shard_seed(int(wl.DEFAULT_SEED[args.config]), rank))
    B, V = w.B, w.V
    gen = wl.DevGen(w, device=device)
    per = B * 16 * V * (2 if w.dtype == wl.BF16 else 4)
    K = max(1, min(args.steps, int(args.input_gb * 2 ** 30 // per)))
    W = args.warmup
    g = torch.Generator(device=device).manual_seed(1234 + rank)
    bufs = torch.empty((K, B, 16, V), dtype=gen.torch_dtype(), device=device)
    blks = torch.empty((K, B, 16), dtype=torch.int32, device=device)
    for i in range(K):
        gen.logits(bufs[i], pos=gen.pos + 16 * i)
        fav = bufs[i].float().argmax(dim=2).int()
        noise = torch.rand((B, 16), generator=g, device=device) < 0.2
        rnd = torch.randint(0, V, (B, 16), generator=g, device=device, dtype=torch.int32)
        blks[i, :, 0] = 0
        blks[i, :, 1:] = torch.where(noise[:, 1:], rnd[:, 1:], fav[:, :15])
    long = torch.tensor([k == "copy" for k in w.kinds], device=device)
    L = torch.where(long, 16, 8).int()
    t = torch.full((B,), 1.0 / 0.3, device=device)
    u = torch.rand((K, B, 16, 2), generator=g, device=device)
    acc = torch.zeros(B, dtype=torch.int32, device=device)
    em, out = torch.zeros_like(acc), torch.zeros((B, 16), dtype=torch.int32, device=device)
    exact = bool(getattr(args, "exact", False))
    if exact:
        verify = clk.verify_sample_exact
        scratch = clk.verify_sample_exact_scratch(bufs.dtype, V, B, device=device)
    else:
        verify = clk.verify_sample
        scratch = clk.verify_sample_scratch(bufs.dtype, V, B, device=device)
    flush = torch.empty(2 * 160 * 2 ** 20, dtype=torch.uint8, device=device)
    for i in range(W):
        verify(bufs[i % K], blks[i % K], L, t, u[i % K], acc, em, out, scratch)
    flush.zero_()
    torch.cuda.synchronize()
    # The K launches as one CUDA graph with an event around each (no host
    # time between launches); eager launches if this torch has no external
    # events.
    emitted = torch.zeros(B, dtype=torch.int64, device=device)

    def launches(ev):
        for i in range(K):
            ev[2 * i].record()
            verify(bufs[i], blks[i], L, t, u[i], acc, em, out, scratch)
            ev[2 * i + 1].record()
            emitted.add_(em)

    clocks = ClockSampler(local)
    time.sleep(0.3)
    try:
        ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2 * K)]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            launches(ev)
        emitted.zero_()
        flush.zero_()
        torch.cuda.synchronize()
        graph.replay()
    except TypeError:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * K)]
        launches(ev)
    torch.cuda.synchronize()
    clocks.stop()
    us = [ev[2 * i].elapsed_time(ev[2 * i + 1]) * 1e3 for i in range(K)]
    mean_us = float(np.mean(us))
    esz = 2 if w.dtype == wl.BF16 else 4
    rows = int(L.sum().item())
    # the verified rows, plus the drawn row's segment (exact: its 1024-entry chunk)
    alg = rows * V * esz + B * min(V, 1024 if exact else 16384) * esz
    peak, peak_kind = _peaks()
    name = "exact sampled verify launches/s (fixed-point weights)" if exact else \
        "sampled verify launches/s (point-mass drafts)"
    kern = "k_sample_fx (verify_sample_exact)" if exact else "k_sample (verify_sample)"
    hbm_roof = {"bound": "hbm", "kernel": kern, "achieved": round(alg / mean_us / 1e3, 1),
                "peak": peak, "unit": "GB/s", "frac": round(alg / mean_us / 1e3 / peak, 4),
                "peak_source": peak_kind, "algorithmic_bytes_per_launch": alg}
    csum = clocks.summary()
    return {"metric": name, "value": round(1e6 / mean_us, 2),
            "unit": "launches/s", "n_gpus": world, "steps": K, "warmup": W, "us_per_launch": round(mean_us, 3),
            "higher_is_better": True, "dtype": "bf16" if w.dtype == wl.BF16 else "f32", "data": "synthetic",
            "config": {"workload": f"{w.name}: {CONFIG_NAMES[args.config]}", "batch": B, "vocab": V,
                       "temperature": 0.3, "block": "16 for copy-heavy requests, 8 for chat-like",
                       "l2": "every launch reads its own pre-generated logits (larger than L2)"},
            "roofline": hbm_roof if not exact else
            _alu_roofline(kern, rows * V + B * min(V, 1024), mean_us * 1e-6, csum, hbm_roof),
            "exp_per_launch": rows * V, "tokens_per_request_launch": round(emitted.sum().item() / (B * K), 4),
            "clocks": csum, "gpu_launches": K}


def _kind_metrics(after, before, kinds, head):
    """Hit rate, mean accepted length, tail share of the accepted drafts and
    accepted-length histograms over the timed steps, per workload kind."""
    from context_lookup_speculative_gb300 import metrics
    out = metrics.by_kind(metrics.delta(after, before), kinds, head)
    keep = ("requests", "steps", "hit_rate", "long_share", "mean_accepted", "tokens_per_step",
            "draft_acceptance", "tail_share", "accept_hist")
    return {k: {f: v[f] for f in keep} for k, v in out.items()}


def run_lookup_ablation(lk, slots, w, device, reps: int = 20):
    """The proposal by the incremental index against the pages' full history
    scan, both on the GPU from the same state (the one the timed steps left),
    per batch step, and whether their answers are identical."""
    import numpy as np
    import torch

    import context_lookup_speculative_gb300 as clk

    B = w.B
    z = lambda *sh: torch.zeros(sh, dtype=torch.int32, device=device)  # noqa: E731
    outs = {m: (z(B, 16), z(B), z(B)) for m in ("index", "scan", "scan_one_cta")}
    clk.lookup_propose(lk, slots, *outs["index"])  # indexes the last step's tokens first
    torch.cuda.synchronize()
    res = {}
    # the grid-wide scan, and the pages' form: one CTA per request
    scan1 = lambda *a: clk.lookup_propose_scan(*a, ctas_per_request=1)  # noqa: E731
    for mode, fn in (("index", clk.lookup_propose), ("scan", clk.lookup_propose_scan), ("scan_one_cta", scan1)):
        fn(lk, slots, *outs[mode])
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn(lk, slots, *outs[mode])
        b.record()
        torch.cuda.synchronize()
        res[f"gpu_{mode}_us"] = round(a.elapsed_time(b) * 1e3 / reps, 3)
    lens = [lk.slot_info(int(s))["n"] for s in slots.tolist()]
    res.update({
        "answers_identical": all(torch.equal(x, y) and torch.equal(x, y1)
                                 for x, y, y1 in zip(outs["index"], outs["scan"], outs["scan_one_cta"])),
        "history_tokens_mean": int(np.mean(lens)),
        "batch": B,
    })
    return res


ABLATION_SWEEP_B = (1, 64)
ABLATION_SWEEP_L = (1024, 4096, 16384, 65536, 262144)


def run_ablation_sweep(args, world, rank, local):
    """Where the incremental index overtakes the full history scan: for each
    batch size and history length, a lookup holding that many synthetic
    prompt tokens per request (the mixed recipe; its index built at
    ingestion), the proposal by the index and by the GPU full scan timed
    from the same state, and whether their answers are identical."""
    import torch

    import workload as wl
    from workload import drive

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    rows = []
    for B in ABLATION_SWEEP_B:
        for L in ABLATION_SWEEP_L:
            w = wl.make_small("mixed", seed=700 + B, B=B, V=32000, L=(L, L), steps=1)
            lk, slots = drive.make_lookup(w, device=device)
            r = run_lookup_ablation(lk, slots, w, device)
            rows.append({"batch": B, "history": L, "index_us": r["gpu_index_us"], "scan_us": r["gpu_scan_us"],
                         "scan_one_cta_us": r["gpu_scan_one_cta_us"], "answers_identical": r["answers_identical"]})
            del lk
            torch.cuda.empty_cache()
    if not all(r["answers_identical"] for r in rows):
        raise RuntimeError("ablation sweep: the index and the full scan disagree")
    return {"metric": "proposal latency: incremental index vs full history scan", "unit": "us per batch step",
            "data": "synthetic", "rows": rows}


def run_e2e(args, w, params, d_ptok, d_poff, pos_hist, device, temp=None, exact=False):
    """Same metric through the public API with host buffers.  Each step copies
    its head proposals (and, sampled at temperature `temp`, its uniforms) from
    pinned host memory, runs the two launches on the step's logits in pinned
    host memory, which the verify kernel reads in place over the host link
    (only the rows it verifies), and reads back the emitted tokens and
    counts.  The same steps with the whole [B, 16, V] logits copied to the
    device first are reported as `staged`; the two runs must emit the same
    tokens.  The steps run in chunks whose host inputs are prepared before
    each chunk's timed region (the host memory they take stays bounded); the
    figures sum the chunks' timed regions."""
    import numpy as np
    import torch

    import context_lookup_speculative_gb300 as clk
    import workload as wl
    from workload import drive

    W = args.warmup
    n = min(args.steps, args.e2e_steps, pos_hist.shape[0] - 1 - W)  # within the workload's steps
    B, V = w.B, w.V
    per_step = B * 16 * V * (2 if w.dtype == wl.BF16 else 4)
    chunk = max(1, min(n, int(args.e2e_gb * 2 ** 30 // per_step)))
    gen = wl.DevGen(w, device=device)
    head = torch.zeros((B, wl.HEAD), dtype=torch.int32, device=device)
    dl = gen.alloc_logits()
    # pinned host copies of one chunk's inputs
    h_heads = torch.empty((chunk, B, wl.HEAD), dtype=torch.int32, pin_memory=True)
    h_logits = torch.empty((chunk, B, 16, V), dtype=gen.torch_dtype(), pin_memory=True)
    h_unis = torch.empty((chunk, B, 16, 2), dtype=torch.float32, pin_memory=True)
    uni = torch.zeros((B, 16, 2), dtype=torch.float32, device=device)
    esz = dl.element_size()
    base = min(16, 1 + params.head)
    temps = torch.full((B,), 1.0 / temp if temp else 1.0, dtype=torch.float32, device=device)

    def fill(t0, m):
        """Host inputs of steps t0 .. t0+m-1 (untimed)."""
        for i in range(m):
            gen.head(t0 + i, head, pos=pos_hist[t0 + i])
            gen.logits(dl, pos=pos_hist[t0 + i])
            h_heads[i].copy_(head)
            h_logits[i].copy_(dl)
            gen.uniforms(t0 + i, uni)
            h_unis[i].copy_(uni)
        torch.cuda.synchronize()

    def post(st, lg):
        """The step's verify launch: greedy, or sampled with the uniforms in `uni`."""
        if temp is None:
            st.post(lg)
        else:
            st.post_sample(lg, temps, uni, exact=exact)

    def run(staged: bool):
        lk, slots = drive.make_lookup(w, params, device=device)
        st = clk.Step(lk, slots)
        g = wl.DevGen(w, device=device)
        for t in range(W):
            g.head(t, head)
            st.pre(head)
            g.logits(dl)
            if temp is not None:
                g.uniforms(t, uni)
            post(st, dl)
            g.advance(st.emitted)
        h_out = torch.empty((n, B, 16), dtype=torch.int32, pin_memory=True)
        h_em = torch.empty((n, B), dtype=torch.int32, pin_memory=True)
        lens = torch.zeros((n, 2, B), dtype=torch.int32, device=device)
        stream = torch.cuda.current_stream(device)
        ms, wall = 0.0, 0.0
        for c0 in range(0, n, chunk):
            m = min(chunk, n - c0)
            fill(W + c0, m)
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0 = time.perf_counter()
            start.record(stream)
            for i in range(m):
                head.copy_(h_heads[i], non_blocking=True)
                if temp is not None:
                    uni.copy_(h_unis[i], non_blocking=True)
                lens[c0 + i, 0].copy_(st.length)  # the previous step's lengths: the verify's prediction
                st.pre(head)
                lens[c0 + i, 1].copy_(st.length)
                if staged:
                    dl.copy_(h_logits[i], non_blocking=True)
                    post(st, dl)
                else:
                    post(st, h_logits[i])
                h_out[c0 + i].copy_(st.out_tok, non_blocking=True)
                h_em[c0 + i].copy_(st.emitted, non_blocking=True)
            end.record(stream)
            torch.cuda.synchronize()
            wall += time.perf_counter() - t0
            ms += start.elapsed_time(end)
        L = lens.cpu().numpy()
        pred = np.where((L[:, 0] >= 1) & (L[:, 0] <= 16), np.maximum(L[:, 0], base), base)
        rows = float(np.maximum(pred, L[:, 1]).sum()) / n  # rows the verify kernel reads per step
        return ms, wall, rows, h_out.numpy().copy(), h_em.numpy().copy()

    ms, wall, rows, out, em = run(staged=False)
    ms_s, wall_s, _, out_s, em_s = run(staged=True)
    if not (np.array_equal(out, out_s) and np.array_equal(em, em_s)):
        raise RuntimeError("e2e: host-resident and staged logits gave different tokens")
    head_b = B * wl.HEAD * 4 + (B * 16 * 2 * 4 if temp is not None else 0)  # heads (and uniforms)
    bo = B * 16 * 4 + B * 4
    return {"value": round(n / (ms * 1e-3), 2), "unit": UNIT,
            "h2d_bytes_per_step": int(head_b + rows * V * esz), "d2h_bytes_per_step": bo,
            "steps": n, "chunk_steps": chunk, "wall_s": round(wall, 4),
            "note": "head proposals (sampled: and uniforms) copied from pinned host memory; the verify kernel "
                    "reads the step's logits in place from pinned host memory over the host link, only the rows "
                    "it verifies; timed in chunks of chunk_steps steps (host inputs prepared between chunks)",
            "staged": {"value": round(n / (ms_s * 1e-3), 2), "unit": UNIT,
                       "h2d_bytes_per_step": head_b + B * 16 * V * esz, "wall_s": round(wall_s, 4),
                       "note": "the whole [B,16,V] logits copied to the device every step; same tokens"}}


def run_cpu_baseline(args, w):
    """The oracle as it stands, on this host's cores, over a bounded sample:
    all requests of the workload for the first `cpu_steps` steps."""
    import oracle

    steps = min(args.cpu_steps, w.steps)
    threads = os.cpu_count() or 1
    temp = getattr(args, "sampling", None)
    inv_temp = 1.0 / temp if temp else 0.0
    exact = bool(getattr(args, "exact", False)) and temp is not None
    res = oracle.run(w, steps=steps, threads=threads, inv_temp=inv_temp, exact=exact)
    used = min(threads, w.B)
    per_thread = res.method_s / used
    # the same steps of every (B/8)-th request on one core, scaled to the whole batch
    sub = list(range(0, w.B, max(1, w.B // 8)))
    one = oracle.run(w, req_ids=sub, steps=steps, threads=1, inv_temp=inv_temp, exact=exact)
    return {"value": round(steps / per_thread, 3), "unit": UNIT, "cores": used, "kind": "oracle",
            "sample": f"{w.B} requests x first {steps} steps of the same workload; full-scan lookup, copy, "
                      f"scheduler, fusion, argmax over every verified row, accept, append; host generation of "
                      f"the logit rows excluded ({res.provider_s / used:.2f} s/thread), wall incl. generation "
                      f"{res.wall_s:.2f} s", "cpu": _cpu_model(),
            "us_per_request_step": _oracle_parts(res, w.B * steps),
            "one_core": {"value": round(steps / (one.method_s * w.B / len(sub)), 3), "unit": UNIT, "cores": 1,
                         "sample": f"requests {sub[0]}, {sub[1] if len(sub) > 1 else sub[0]}, ... ({len(sub)} of "
                                   f"{w.B}) x first {steps} steps on one thread, scaled to {w.B} requests",
                         "us_per_request_step": _oracle_parts(one, len(sub) * steps)}}


def _oracle_parts(res, request_steps: int) -> dict:
    """The oracle's time per request-step by component (thread time, us)."""
    out = {k: round(getattr(res, k + "_s") * 1e6 / request_steps, 3)
           for k in ("lookup", "sched_fuse", "verify")}
    out["total"] = round(res.method_s * 1e6 / request_steps, 3)
    return out


def _cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def run_reference(args, world, rank):
    """The oracle timed on the host cores as the reference arm."""
    import oracle
    import workload as wl

    if rank != 0:
        return None
    w = wl.make(args.config)
    W, K = args.warmup, args.steps
    K = min(K, w.steps - W)
    threads = os.cpu_count() or 1
    res = oracle.run(w, steps=W + K, threads=threads, timed_from=W)
    used = min(threads, w.B)
    per_thread = res.method_s / used
    v = round(K / per_thread, 3)
    return {"metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": round(per_thread * 1e3 / K, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.dtype == wl.BF16 else "f32", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": f"{w.name}: {CONFIG_NAMES[args.config]}", "batch": w.B, "vocab": w.V},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": used, "kind": "oracle",
                             "sample": f"{w.B} requests x {W} warm-up + {K} timed steps, host generation of the "
                                       f"logit rows excluded", "cpu": _cpu_model(),
                             "us_per_request_step": _oracle_parts(res, w.B * K)},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=504)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="2", choices=sorted(CONFIG_NAMES))
    ap.add_argument("--input-gb", type=float, default=40.0, help="HBM for pre-generated timed inputs")
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--e2e-gb", type=float, default=4.0, help="pinned host memory for one e2e chunk of logits")
    ap.add_argument("--cpu-steps", type=int, default=128)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sampling", type=float, default=None, metavar="T",
                    help="verify by sampling (point-mass drafts) at temperature T instead of greedily")
    ap.add_argument("--sample-verify", action="store_true",
                    help="time the sampling verification (point-mass drafts) on --config's shapes, one JSON line")
    ap.add_argument("--exact", action="store_true",
                    help="with --sample-verify or --sampling: the exact sampler (fixed-point weights) instead")
    ap.add_argument("--sweep", action="store_true",
                    help="block-size and sticky variants of the measured step on --config, one JSON line")
    ap.add_argument("--ablation-sweep", action="store_true",
                    help="the index lookup against the full history scan over batch sizes and history lengths")
    ap.add_argument("--ablation", action="store_true",
                    help="also time the proposal by index vs by full history scan (GPU and CPU oracle)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local, dist = _dist()
    if args.impl == "reference":
        out = run_reference(args, world, rank)
        if out is not None:
            print(json.dumps(out), flush=True)
        return 0
    if world > 1:
        dist.init_process_group(backend="nccl")
    try:
        if args.sample_verify:
            out = run_sample_verify(args, world, rank, local, dist)
        elif args.sweep:
            out = run_sweep(args, world, rank, local, dist)
        elif args.ablation_sweep:
            out = run_ablation_sweep(args, world, rank, local)
        else:
            out = run_ours(args, world, rank, local, dist)
        if rank == 0:
            print(json.dumps(out), flush=True)
    finally:
        if world > 1:
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
