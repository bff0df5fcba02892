"""A model of the deferred index insertions of the proposal launch, run over
random sequences of library calls.  CPU only.

The model restates, per slot, the decisions `k_lookup_step` takes
(clk_lookup.cu) and the host rules of `launch_lookup_step`, the fused
verifies and the calls that rebuild a slot, with one launch at a time and
each launch's insertions becoming visible only when it has completed.  It
checks the two facts the lookup relies on:
- every k-gram ending before nidx_eff - 1 (the start of the positions the
  lookup warps check directly) was inserted by a launch that has completed,
  or by this launch's catch-up before its lookups;
- at most 32 end positions are pending for the direct check (kMaxPending),
  or the launch catches up first; and a launch that takes the record of the
  previous one, with at most one commit in between, never needs to.
A lookup warp may read the slot's nidx before or after the same launch's
insert warps raise it; the model draws either.
The mutants below break one rule each and must be caught."""
import random

import pytest

K_MAX_PENDING = 32  # pending end positions the lookup warps check directly
K_DEFER_MAX = 16    # positions a launch may leave to the next one
K_DEFER_BATCH = 32  # batches above this never leave insertions


class Slot:
    def __init__(self, n):
        self.n = n           # history length
        self.nidx = n        # published: k-grams ending before nidx - 1 are in the tables
        self.done = set(range(max(n - 1, 0)))  # end positions inserted by completed launches


class Model:
    """One slot (batch position 0), the handle's host state and the record halves."""

    def __init__(self, n, mutant=None):
        self.s = Slot(n)
        self.mutant = mutant
        self.ptag = 0
        self.defer_tag = 0
        self.vsince = 0
        self.early = False          # the last verify alternates scratch halves
        self.records = {}           # parity -> (tag, slot, z, w)
        self.commits = 0            # tokens committed since the last proposal

    # -- calls that rebuild the slot --------------------------------------
    def init(self, n):
        self.s = Slot(n)
        self.commits = 0
        self.defer_tag = 0

    def append(self, count):
        s = self.s
        s.n += count
        self.commits += count
        s.done |= set(range(max(s.nidx - 1, 0), s.n - 1))  # k_append indexes every pending position
        s.nidx = s.n
        self.defer_tag = 0

    # -- fused verifies (commit only) -------------------------------------
    def verify(self, count, paired):
        self.s.n += count
        self.commits += count
        self.early = paired
        if paired:
            self.vsince = 1

    # -- the proposal launch ----------------------------------------------
    def propose(self, batch, rng):
        s = self.s
        self.ptag = 1 if self.ptag >= (1 << 30) or self.ptag < 1 else self.ptag + 1
        tag, take = self.ptag, self.defer_tag
        pre = take != 0 and self.early and self.vsince
        defer = batch <= K_DEFER_BATCH
        inserted_here = set()
        prev = self.records.get(take & 1) if take else None
        prev_ok = prev is not None and prev[0] == take and prev[2] <= prev[3]
        mine = prev_ok and prev[1] == 0
        # before the wait: the insertions the previous launch left
        if pre and prev_ok and prev[2] < prev[3]:
            inserted_here |= set(range(max(prev[2] - 1, 0), prev[3] - 1))
        n = s.n
        # what this launch publishes (nidx) while it runs: its insert warps
        # may do that before a lookup warp reads the record, so the read may
        # see it (the race the design must tolerate)
        pub = prev[2] if prev_ok else 0
        if self.mutant == "publish_own":
            pub = max(pub, n)
        nidx_read = s.nidx if rng.random() < 0.5 else max(s.nidx, pub)
        nidx = min(nidx_read, n)
        if mine and self.mutant != "ignore_prev_z":
            nidx = max(nidx, min(prev[2], n))
        if self.mutant == "trust_own_pre" and pre and mine:
            nidx = max(nidx, min(prev[3], n))   # counts this launch's in-flight insertions as complete
        if mine and self.commits <= 16:
            # one commit since the recording launch: no catch-up needed
            assert n - nidx <= K_MAX_PENDING, "steady state needs a catch-up"
        if n - nidx > K_MAX_PENDING:
            # catch-up before the lookups: complete within this launch
            s.done |= set(range(max(nidx - 1, 0), n - 1))
            nidx = n
            s.nidx = max(s.nidx, n)
        # the lookup: positions below nidx - 1 must be complete, the rest few
        missing = [q for q in range(max(nidx - 1, 0)) if q not in s.done]
        assert not missing, ("lookup trusts positions not yet indexed", missing[:5])
        assert n - 1 - max(nidx - 1, 0) <= K_MAX_PENDING, "direct check window exceeded"
        covered = min(n, max(nidx, prev[3]) if (pre and mine and prev[2] < prev[3]) else nidx)
        limit = K_DEFER_MAX + (16 if self.mutant == "defer_too_much" else 0)
        deferred = defer and n - covered <= limit
        self.records[tag & 1] = (tag, 0, covered if deferred else n, n)
        if not deferred:
            inserted_here |= set(range(max(covered - 1, 0), n - 1))
        s.nidx = max(s.nidx, pub)
        # the launch completes: its insertions become visible
        s.done |= inserted_here
        self.defer_tag = tag
        self.vsince = 0
        self.commits = 0


def _run(seed, mutant=None, steps=400):
    rng = random.Random(seed)
    m = Model(rng.randint(1, 200), mutant)
    batch = rng.choice([1, 16, 32, 64])
    for _ in range(steps):
        r = rng.random()
        if r < 0.55:
            m.propose(batch, rng)
            if rng.random() < 0.9:
                m.verify(rng.randint(1, 16), paired=rng.random() < 0.8)
        elif r < 0.7:
            m.verify(rng.randint(1, 16), paired=rng.random() < 0.5)
        elif r < 0.8:
            m.propose(batch, rng)       # two proposals in a row
        elif r < 0.9:
            m.append(rng.randint(0, 16))
        elif r < 0.95:
            m.init(rng.randint(1, 300))
        else:
            batch = rng.choice([1, 16, 32, 64])


@pytest.mark.parametrize("seed", range(40))
def test_protocol_keeps_the_lookup_exact(seed):
    _run(seed)


@pytest.mark.parametrize("mutant", ["ignore_prev_z", "trust_own_pre", "defer_too_much", "publish_own"])
def test_protocol_mutants_are_caught(mutant):
    with pytest.raises(AssertionError):
        for seed in range(40):
            _run(seed, mutant)
