"""Decode metrics derived on the host from the per-request device counters.

HyperQwen 上下文复述加速 (section 代价与适用场景) measures, on chat traffic, what
share of the accepted tokens the tail positions of the draft block
contributed; the discussion under the same post asks for the hit rate and
the mean accepted length, reported per kind of workload together with the
distribution of accepted lengths.  These functions turn the counters that
`Lookup.counters(slot)` returns (steps, hits, long_steps, drafted, accepted,
emitted and the per-block-length histogram of accepted counts) into those
figures.  They only add and divide counter values; every step of the decode
itself runs on the device.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

FIELDS = ("steps", "hits", "long_steps", "drafted", "accepted", "emitted")
CLASSES = ("short", "long")  # accept_hist[0] counts short blocks, [1] long blocks


def delta(after: Sequence[dict], before: Sequence[dict]) -> List[dict]:
    """Per-request counters accumulated between two reads."""
    out = []
    for a, b in zip(after, before):
        d = {f: a[f] - b[f] for f in FIELDS}
        d["accept_hist"] = [[x - y for x, y in zip(ra, rb)] for ra, rb in zip(a["accept_hist"], b["accept_hist"])]
        out.append(d)
    return out


def summarize(counters: Sequence[dict], head: int = 7) -> Dict[str, object]:
    """Totals and derived rates over a set of requests.

    hit_rate: share of request-steps whose suffix matched (k >= min_k).
    long_share: share of request-steps verified as a long block.
    mean_accepted: accepted drafts per request-step (the accepted prefix a).
    tokens_per_step: emitted tokens per request-step (a + 1).
    draft_acceptance: accepted over drafted (non-sentinel) slots.
    tail_share: share of the accepted drafts that sat past the first `head`
    draft slots (block slots head+1 ..), i.e. that only a long block could
    have offered; a step that accepted a drafts contributed max(0, a - head).
    accept_hist: steps by accepted count a (0..15), per block length."""
    tot = {f: int(sum(c[f] for c in counters)) for f in FIELDS}
    hist = [[int(sum(c["accept_hist"][i][a] for c in counters)) for a in range(16)] for i in range(2)]
    tail = sum(max(0, a - head) * (hist[0][a] + hist[1][a]) for a in range(16))
    steps = tot["steps"]

    def ratio(x: float, y: float) -> Optional[float]:
        return round(x / y, 6) if y else None

    return {
        **tot,
        "requests": len(counters),
        "hit_rate": ratio(tot["hits"], steps),
        "long_share": ratio(tot["long_steps"], steps),
        "mean_accepted": ratio(tot["accepted"], steps),
        "tokens_per_step": ratio(tot["emitted"], steps),
        "draft_acceptance": ratio(tot["accepted"], tot["drafted"]),
        "tail_accepted": int(tail),
        "tail_share": ratio(tail, tot["accepted"]),
        "accept_hist": {CLASSES[i]: hist[i] for i in range(2)},
    }


def by_kind(counters: Sequence[dict], kinds: Sequence[str], head: int = 7) -> Dict[str, Dict[str, object]]:
    """summarize() over all requests and over each workload kind separately
    (e.g. "copy" and "chat" in a mixed serving batch)."""
    if len(counters) != len(kinds):
        raise ValueError("one kind per request")
    out = {"all": summarize(counters, head)}
    for k in sorted(set(kinds)):
        out[k] = summarize([c for c, kk in zip(counters, kinds) if kk == k], head)
    return out
