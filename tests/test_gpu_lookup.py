"""Lookup on the GPU (index build, incremental append, proposal) against the
oracle's full scan, element by element; error latching.  GPU."""
import numpy as np
import pytest
import torch

import context_lookup_speculative_gb300 as clk
import oracle

pytestmark = pytest.mark.gpu


def _csr(arrays):
    off = np.zeros(len(arrays) + 1, np.int64)
    off[1:] = np.cumsum([a.size for a in arrays])
    tok = np.concatenate(arrays).astype(np.int32) if arrays else np.zeros(0, np.int32)
    return torch.from_numpy(tok).cuda(), torch.from_numpy(off).cuda()


def _setup(hists, max_hist, slots=None, vocab=0, params=None):
    B = len(hists)
    slots = list(range(B)) if slots is None else slots
    lk = clk.Lookup(max_slots=max(slots) + 1, max_hist=max_hist, vocab=vocab, params=params)
    s = torch.tensor(slots, dtype=torch.int32, device="cuda")
    tok, off = _csr(hists)
    clk.lookup_init(lk, s, tok, off)
    return lk, s


def _propose(lk, s):
    B = s.numel()
    d = torch.zeros((B, 16), dtype=torch.int32, device="cuda")
    k = torch.zeros(B, dtype=torch.int32, device="cuda")
    j = torch.zeros(B, dtype=torch.int32, device="cuda")
    clk.lookup_propose(lk, s, d, k, j)
    torch.cuda.synchronize()
    return d.cpu().numpy(), k.cpu().numpy(), j.cpu().numpy()


def _expect(hists, params=None):
    return [oracle.propose(h, params) for h in hists]


def _assert_same(got, hists, params=None):
    d, k, j = got
    for b, (c, kk, jj) in enumerate(_expect(hists, params)):
        assert (k[b], j[b]) == (kk, jj), (b, hists[b][-16:], (k[b], j[b]), (kk, jj))
        assert d[b].tolist() == c.tolist(), b


def test_random_small_vocab_histories():
    rng = np.random.default_rng(51)
    hists = [rng.integers(0, int(rng.integers(2, 6)), size=int(rng.integers(1, 400))).astype(np.int32)
             for _ in range(200)]
    lk, s = _setup(hists, 512)
    _assert_same(_propose(lk, s), hists)
    assert lk.status() == (0, 0)


def test_periodic_and_planted_histories():
    rng = np.random.default_rng(52)
    hists = []
    for p in range(1, 41):
        pat = rng.integers(0, 32000, size=p).astype(np.int32)
        n = int(rng.integers(p + 1, 3000))
        h = pat[np.arange(n) % p].copy()
        noise = rng.random(n) < 0.05
        h[noise] = rng.integers(0, 32000, size=int(noise.sum()))
        hists.append(h)
    for _ in range(40):
        n = int(rng.integers(1000, 20000))
        h = rng.zipf(1.3, size=n).astype(np.int64) % 248320
        src = int(rng.integers(0, n // 2))
        ln = int(rng.integers(1, 30))
        h[n - ln:] = h[src:src + ln]
        hists.append(h.astype(np.int32))
    lk, s = _setup(hists, 20000)
    _assert_same(_propose(lk, s), hists)


def test_incremental_append_matches_full_scan():
    """Grow histories by random counts of tokens; after every append the
    proposal equals the oracle's full scan of the accumulated history."""
    rng = np.random.default_rng(53)
    B = 24
    hists = [rng.integers(0, 4, size=int(rng.integers(1, 30))).astype(np.int32) for _ in range(B)]
    lk, s = _setup(hists, 30 + 16 * 60, slots=[3 * b + 1 for b in range(B)])
    for step in range(60):
        cnt = rng.integers(0, 17, size=B).astype(np.int32)
        tok = rng.integers(0, 4 if step % 3 else 2, size=(B, 16)).astype(np.int32)
        # periodic bursts so long matches and overlaps occur
        for b in range(0, B, 4):
            tok[b] = np.resize(hists[b][-3:], 16)
        clk.lookup_append(lk, s, torch.from_numpy(tok).cuda(), torch.from_numpy(cnt).cuda())
        hists = [np.concatenate([h, tok[b, :cnt[b]]]) for b, h in enumerate(hists)]
        _assert_same(_propose(lk, s), hists)
    for b in range(B):
        assert np.array_equal(lk.history(3 * b + 1), hists[b])
    assert lk.status() == (0, 0)


def test_other_match_ranges():
    rng = np.random.default_rng(54)
    for lo, hi in ((1, 3), (2, 16), (6, 9)):
        p = clk.Params.default(min_k=lo, max_k=hi)
        po = oracle.Params.default(min_k=lo, max_k=hi)
        hists = [rng.integers(0, 3, size=int(rng.integers(1, 200))).astype(np.int32) for _ in range(50)]
        lk, s = _setup(hists, 256, params=p)
        _assert_same(_propose(lk, s), hists, po)


def test_capacity_overflow_is_latched_and_skipped():
    hists = [np.array([1, 2, 3, 4, 5], np.int32), np.array([7, 7, 7], np.int32)]
    lk, s = _setup(hists, 20)
    tok = torch.arange(32, dtype=torch.int32, device="cuda").reshape(2, 16)
    cnt = torch.tensor([16, 16], dtype=torch.int32, device="cuda")
    clk.lookup_append(lk, s, tok, cnt)   # slot 0 -> 21 > 20: refused; slot 1 -> 19: fine
    st, det = lk.status()
    assert st == clk.ECAPACITY and det == 0
    assert lk.history(0).tolist() == [1, 2, 3, 4, 5]
    assert lk.history(1).size == 19
    lk.status_clear()
    assert lk.status() == (0, 0)


def test_bad_inputs_are_latched():
    lk, s = _setup([np.array([1, 2, 3], np.int32)], 64, vocab=10)
    tok = torch.full((1, 16), 12, dtype=torch.int32, device="cuda")   # outside [0, vocab)
    clk.lookup_append(lk, s, tok, torch.tensor([2], dtype=torch.int32, device="cuda"))
    assert lk.status()[0] == clk.EINVAL
    assert lk.history(0).tolist() == [1, 2, 3]
    lk.status_clear()
    clk.lookup_append(lk, s, tok, torch.tensor([17], dtype=torch.int32, device="cuda"))  # count > 16
    assert lk.status()[0] == clk.EINVAL
    lk.status_clear()
    # an empty prompt leaves the slot empty; proposing from it is a state error
    lk2, s2 = _setup([np.array([], np.int32), np.array([4, 4, 4, 4, 4, 4], np.int32)], 64)
    assert lk2.status()[0] == clk.EINVAL
    lk2.status_clear()
    d, k, j = _propose(lk2, s2)
    assert lk2.status()[0] == clk.ESTATE
    assert k.tolist() == [0, 5] and j.tolist() == [-1, 5]
    # a prompt longer than max_hist
    lk3, _ = _setup([np.arange(70, dtype=np.int32)], 64)
    assert lk3.status()[0] == clk.ECAPACITY


def test_long_history_index_build():
    """A 262,144-token copy-heavy prompt: the index build and the proposal at
    several points of it (truncated prompts share the prefix)."""
    rng = np.random.default_rng(55)
    n = 262144
    base = (rng.zipf(1.1, size=n).astype(np.int64) % 248320).astype(np.int32)
    for _ in range(200):
        ln = int(rng.integers(1000, 8000))
        src = int(rng.integers(0, n - ln))
        dst = int(rng.integers(src + ln, n - ln + 1)) if src + ln < n - ln else src
        base[dst:dst + ln] = base[src:src + ln]
    cuts = [n, n - 1, n - 5000, 200000, 150001, 77777]
    hists = [base[:c].copy() for c in cuts]
    lk, s = _setup(hists, n + 64)
    _assert_same(_propose(lk, s), hists)


def _commit_by_verify(lk, s, rows_tokens):
    """Commit tokens through clk_verify_append: fp32 logits whose row r peaks at
    rows_tokens[b][r] and blocks that accept all 15 drafts (16 tokens)."""
    B = s.numel()
    V = 8
    x = torch.zeros((B, 16, V), dtype=torch.float32)
    blk = torch.full((B, 16), -1, dtype=torch.int32)
    for b in range(B):
        for r in range(16):
            x[b, r, rows_tokens[b][r]] = 1.0
            if r + 1 < 16:
                blk[b, r + 1] = int(rows_tokens[b][r])
    z = lambda *sh: torch.zeros(sh, dtype=torch.int32, device="cuda")  # noqa: E731
    g, a, e, out = z(B, 16), z(B), z(B), z(B, 16)
    L = torch.full((B,), 16, dtype=torch.int32, device="cuda")
    clk.verify_append(lk, s, x.cuda(), blk.cuda(), L, g, a, e, out)
    torch.cuda.synchronize()
    assert e.cpu().tolist() == [16] * B


@pytest.mark.parametrize("commits", [1, 2, 3, 5])
def test_commits_without_lookup_in_between(commits):
    """Several fused commits before the next proposal leave 16 x commits
    positions unindexed (more than the 32 the proposal checks directly for 3
    and more); the proposal must still equal the full scan, and so must a
    later unfused append."""
    rng = np.random.default_rng(56 + commits)
    B = 12
    hists = [rng.integers(0, 8, size=int(rng.integers(20, 120))).astype(np.int32) for _ in range(B)]
    lk, s = _setup(hists, 120 + 16 * 12, vocab=8)
    for _ in range(commits):
        toks = rng.integers(0, 8, size=(B, 16))
        toks[::3] = np.resize([1, 2, 3], 16)  # periodic runs: long, overlapping matches
        _commit_by_verify(lk, s, toks)
        hists = [np.concatenate([h, toks[b].astype(np.int32)]) for b, h in enumerate(hists)]
    n, nidx = lk.slot_info(0)["n"], lk.slot_info(0)["n_indexed"]
    assert nidx < n
    _assert_same(_propose(lk, s), hists)
    # n_indexed rises only when a later launch vouches for the insertions
    # (the next proposal), except after the catch-up of more than 32 pending
    # positions, which completes before the lookups run
    assert lk.slot_info(0)["n_indexed"] == (n if n - nidx > 32 else nidx)
    # commit again, then an unfused append on top of the pending positions
    toks = rng.integers(0, 8, size=(B, 16))
    _commit_by_verify(lk, s, toks)
    hists = [np.concatenate([h, toks[b].astype(np.int32)]) for b, h in enumerate(hists)]
    more = rng.integers(0, 8, size=(B, 16)).astype(np.int32)
    cnt = rng.integers(0, 17, size=B).astype(np.int32)
    clk.lookup_append(lk, s, torch.from_numpy(more).cuda(), torch.from_numpy(cnt).cuda())
    hists = [np.concatenate([h, more[b, :cnt[b]]]) for b, h in enumerate(hists)]
    _assert_same(_propose(lk, s), hists)
    for b in range(B):
        assert np.array_equal(lk.history(b), hists[b])
    assert lk.status() == (0, 0)


def _propose_scan(lk, s, ctas_per_request=0):
    B = s.numel()
    d = torch.zeros((B, 16), dtype=torch.int32, device="cuda")
    k = torch.zeros(B, dtype=torch.int32, device="cuda")
    j = torch.zeros(B, dtype=torch.int32, device="cuda")
    clk.lookup_propose_scan(lk, s, d, k, j, ctas_per_request=ctas_per_request)
    torch.cuda.synchronize()
    return d.cpu().numpy(), k.cpu().numpy(), j.cpu().numpy()


@pytest.mark.parametrize("kind", ["small_vocab", "periodic", "zipf_long"])
def test_full_scan_lookup_matches_oracle_and_index(kind):
    """The pages' full-scan lookup (clk_lookup_propose_scan) returns exactly the
    oracle's (k, j, draft), and the same as the index path."""
    rng = np.random.default_rng({"small_vocab": 61, "periodic": 62, "zipf_long": 63}[kind])
    if kind == "small_vocab":
        hists = [rng.integers(0, int(rng.integers(2, 6)), size=int(rng.integers(1, 9000))).astype(np.int32)
                 for _ in range(60)]
    elif kind == "periodic":
        hists = []
        for p in range(1, 41):
            pat = rng.integers(0, 32000, size=p).astype(np.int32)
            n = int(rng.integers(p + 1, 9000))
            h = pat[np.arange(n) % p].copy()
            noise = rng.random(n) < 0.05
            h[noise] = rng.integers(0, 32000, size=int(noise.sum()))
            hists.append(h)
    else:
        hists = []
        for _ in range(16):
            n = int(rng.integers(20000, 70000))
            h = (rng.zipf(1.1, size=n).astype(np.int64) % 248320).astype(np.int32)
            src = int(rng.integers(0, n // 2))
            ln = int(rng.integers(1, 40))
            h[n - ln:] = h[src:src + ln]
            hists.append(h)
    lk, s = _setup(hists, max(h.size for h in hists) + 32)
    got = _propose_scan(lk, s)
    _assert_same(got, hists)
    idx = _propose(lk, s)
    for a, b in zip(got, idx):
        assert np.array_equal(a, b)
    # the scan leaves no state behind: a second call gives the same answer
    again = _propose_scan(lk, s)
    for a, b in zip(got, again):
        assert np.array_equal(a, b)
    # one CTA per request (the pages' form), and other splits: the same answers
    for per in (1, 3, 7):
        for a, b in zip(got, _propose_scan(lk, s, ctas_per_request=per)):
            assert np.array_equal(a, b), per
    assert lk.status() == (0, 0)
    with pytest.raises(clk.ClkError):
        _propose_scan(lk, s, ctas_per_request=-1)


def test_insertions_left_to_the_next_proposal():
    """A proposal that still finds at most 16 end positions pending leaves
    their index insertions to the next proposal launch (an ins record); that
    launch runs them before its wait when a fused greedy verify came in
    between (the recording launch has then completed), else after it.  A
    launch never raises n_indexed over its own insertions: the next launch
    does, from the record.  Records of an older launch, or made stale by a
    re-initialisation, are never applied; every proposal equals the full
    scan."""
    rng = np.random.default_rng(58)
    B, V = 6, 5
    hists = [rng.integers(0, V, size=int(rng.integers(30, 90))).astype(np.int32) for _ in range(B)]
    lk, s = _setup(hists, 500, vocab=V)

    def commit():
        nonlocal hists
        toks = rng.integers(0, V, size=(B, 16))
        _commit_by_verify(lk, s, toks)
        hists = [np.concatenate([h, toks[b].astype(np.int32)]) for b, h in enumerate(hists)]

    def info():
        return [(lk.slot_info(b)["n"], lk.slot_info(b)["n_indexed"]) for b in range(B)]

    commit()  # 16 pending positions a slot
    before = info()
    _assert_same(_propose(lk, s), hists)
    assert info() == before  # left to the next proposal
    commit()
    _assert_same(_propose(lk, s), hists)  # runs them before its wait
    assert [ni for _, ni in info()] == [ni for _, ni in before]
    _assert_same(_propose(lk, s), hists)  # a second proposal vouches for them
    assert [ni for _, ni in info()] == [n for n, _ in before]
    commit()
    _assert_same(_propose(lk, s), hists)
    # a sampled verify in between: the next proposal takes nothing before its
    # wait and indexes the 32 pending positions itself
    x = torch.zeros((B, 16, V), dtype=torch.float32)
    x[:, :, 2] = 50.0
    blk = torch.full((B, 16), 2, dtype=torch.int32)
    L = torch.full((B,), 16, dtype=torch.int32, device="cuda")
    t = torch.ones(B, dtype=torch.float32, device="cuda")
    u = torch.full((B, 16, 2), 0.5, dtype=torch.float32, device="cuda")
    acc, em = torch.zeros(B, dtype=torch.int32, device="cuda"), torch.zeros(B, dtype=torch.int32, device="cuda")
    out = torch.zeros((B, 16), dtype=torch.int32, device="cuda")
    clk.verify_sample_append(lk, s, x.cuda(), blk.cuda(), L, t, u, acc, em, out,
                             clk.verify_sample_scratch(torch.float32, V, B))
    torch.cuda.synchronize()
    hists = [lk.history(b) for b in range(B)]
    assert all(n - ni > 32 for n, ni in info())
    _assert_same(_propose(lk, s), hists)
    _assert_same(_propose(lk, s), hists)
    assert all(n == ni for n, ni in info())
    # a re-initialisation between a recording proposal and the verify: the
    # records are dropped, the fresh index stays complete
    commit()
    _assert_same(_propose(lk, s), hists)
    fresh = [rng.integers(0, V, size=int(rng.integers(10, 40))).astype(np.int32) for _ in range(B)]
    tok, off = _csr(fresh)
    clk.lookup_init(lk, s, tok, off)
    hists = fresh
    assert all(ni == n for n, ni in info())
    commit()
    _assert_same(_propose(lk, s), hists)
    assert all(n - ni == 16 for n, ni in info())
    for _ in range(4):
        commit()
        _assert_same(_propose(lk, s), hists)
        assert all(n - ni == 32 for n, ni in info())
    assert lk.status() == (0, 0)
