"""Whole decode loop on the GPU against the oracle, bit-exact on every
per-step field (k, j, L, draft, block, argmax rows, accepted count), the
final histories and the counters.  The full-size workloads run in the launch
configuration the benchmark times (the fused two-kernel step).  GPU."""
import os

import numpy as np
import pytest

import context_lookup_speculative_gb300 as clk
import oracle
import workload as wl
from workload import drive

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1


def _parity(w, steps=None, params=None, oparams=None, mode="fused", req_ids=None):
    dev = drive.run_device(w, steps=steps, params=params, mode=mode)
    ref = oracle.run(w, req_ids=req_ids, steps=steps, params=oparams, threads=THREADS)
    msgs = drive.compare(dev, ref, req_ids=req_ids)
    assert not msgs, "\n".join(msgs[:8])
    return dev, ref


@pytest.mark.parametrize("mode", ["fused", "semi", "unfused"])
@pytest.mark.parametrize("kind", ["mixed", "periodic", "copy", "chat"])
def test_small_workloads_all_modes(kind, mode):
    w = wl.make_small(kind, seed=71, B=6, V=4096, steps=64)
    _parity(w, mode=mode)


@pytest.mark.parametrize("sticky", [0, 1, 3, 6])
def test_sticky_variants(sticky):
    w = wl.make_small("mixed", seed=72, B=8, V=2048, steps=96)
    _parity(w, params=clk.Params.default(sticky=sticky), oparams=oracle.Params.default(sticky=sticky))


def test_fp32_and_block_variants():
    w = wl.make_small("copy", seed=73, B=4, V=1024, steps=64, dtype=wl.F32)
    _parity(w)
    kw = dict(head=3, tail=12, head_agree_n=1, head_replace_k=5)  # head <= the 7 synthetic proposals
    _parity(w, params=clk.Params.default(**kw), oparams=oracle.Params.default(**kw))


@pytest.mark.parametrize("kw", [{"tail": 0}, {"head": 5, "tail": 10}, {"head": 3, "tail": 12},
                                {"sticky": 6}])
def test_draft_block_variants(kw):
    """The variants the benchmark's sweep times: short blocks only, other
    head/tail splits of the 15 drafts, a longer sticky exit."""
    w = wl.make_small("mixed", seed=74, B=8, V=2048, steps=96)
    _parity(w, params=clk.Params.default(**kw), oparams=oracle.Params.default(**kw))


@pytest.mark.parametrize("mode", ["sample", "sample_fused"])
@pytest.mark.parametrize("kind", ["mixed", "periodic", "copy"])
def test_sampled_loop_at_near_zero_temperature_matches_the_greedy_oracle(kind, mode):
    """Sampling verification at inverse temperature 1e4 is greedy on these
    rows (each has a unique maximum): the whole sampled loop on the GPU
    equals the greedy oracle, records, histories and counters."""
    w = wl.make_small(kind, seed=75, B=6, V=4096, steps=48)
    dev = drive.run_device(w, mode=mode, inv_temp=1e4)
    ref = oracle.run(w, threads=THREADS)
    # the greedy oracle records argmax rows; the sampled run records the emitted tokens
    ref.g = np.where(np.arange(16)[None, None, :] <= ref.a[:, :, None], ref.g, -1)
    msgs = drive.compare(dev, ref)
    assert not msgs, "\n".join(msgs[:8])


@pytest.mark.parametrize("mode", ["sample", "sample_fused"])
@pytest.mark.parametrize("inv_temp", [1.0, 2.5])
def test_sampled_loop_matches_the_sampled_oracle(inv_temp, mode):
    """The sampled decode loop (lookup, scheduler, fusion, sampling verify,
    commit) against the oracle's sampled loop with the same uniforms: every
    record, history and counter equal (no decision of these seeded runs
    lies within rounding of its boundary)."""
    w = wl.make_small("mixed", seed=76, B=6, V=2048, steps=48)
    dev = drive.run_device(w, mode=mode, inv_temp=inv_temp)
    ref = oracle.run(w, threads=THREADS, inv_temp=inv_temp)
    msgs = drive.compare(dev, ref)
    assert not msgs, "\n".join(msgs[:8])
    assert (ref.a > 0).any()


def test_sampled_loop_full_size_mixed_batch():
    """The sampled step as the Step driver runs it, on the mixed serving
    batch's shapes (B=64, V=248,320, bf16) for 12 steps, against the
    oracle's sampled loop.  Temperature 0.25: the draws land on tokens of
    sizable probability.  (In the flat tail of a 248,320-token row one
    token's probability is about 4e-6; the draw's prefix sums are exact, but
    the float32 segment totals of the streaming pass place the segment
    boundaries to about 3e-8 of the row, so about one tail draw in a hundred
    can differ from the double-precision oracle by a token, which a loop
    then carries into its history.)"""
    w = wl.make("2").with_steps(12)
    dev = drive.run_device(w, mode="sample_fused", inv_temp=4.0)
    ref = oracle.run(w, threads=THREADS, inv_temp=4.0)
    msgs = drive.compare(dev, ref)
    assert not msgs, "\n".join(msgs[:8])


def test_maximum_batch_loop():
    """The fused two-launch step at B = CLK_MAX_BATCH (8,192) requests with
    short prompts, 3 steps, against the oracle (the fused verify's shared
    memory then needs the large-allocation opt-in)."""
    w = wl.make_small("mixed", seed=77, B=8192, V=64, L=(20, 60), steps=3)
    _parity(w)


def test_config0_tiny():
    _parity(wl.make("0"))


def test_config1_restatement_25k():
    _parity(wl.make("1"))


def test_config2_mixed_b64():
    dev, ref = _parity(wl.make("2"))
    assert (ref.L == 16).any() and (ref.L == 8).any()


def test_config3_periodic():
    dev, ref = _parity(wl.make("3"))
    # the noise drives flag drops, sticky exits and re-entries
    import numpy as np
    L = ref.L
    assert ((L[1:] == 8) & (L[:-1] == 16)).any() and ((L[1:] == 16) & (L[:-1] == 8)).any()
    assert (np.asarray(ref.j) > np.asarray(ref.k)).any()


def test_config4a_long_262k():
    _parity(wl.make("4a"))


def test_config4b_b256():
    _parity(wl.make("4b"))
