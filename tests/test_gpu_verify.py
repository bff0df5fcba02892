"""Greedy verification on the GPU against the oracle, element by element.

Covers ragged block lengths, several tiles per row and a ragged tail, the
bf16 vector path, the fp32 path, the unaligned (scalar) path, hand-built
tie / signed-zero / infinity / NaN / last-bit rows placed so that equal
maxima fall in different CTAs, invalid lengths, and scratch reuse.  GPU."""
import numpy as np
import pytest
import torch

import context_lookup_speculative_gb300 as clk
import oracle
import workload as wl

pytestmark = pytest.mark.gpu
SENT = -1


def _oracle_rows(x_np, block, L):
    B = block.shape[0]
    g = np.full((B, 16), SENT, np.int32)
    a = np.zeros(B, np.int32)
    out = np.full((B, 16), SENT, np.int32)
    e = np.zeros(B, np.int32)
    for b in range(B):
        if not 1 <= L[b] <= 16:
            continue
        for r in range(L[b]):
            g[b, r] = oracle.argmax_row(x_np[b, r])
        a[b] = oracle.accept(block[b], g[b], int(L[b]))
        out[b, :a[b] + 1] = g[b, :a[b] + 1]
        e[b] = a[b] + 1
    return g, a, e, out


def _gpu(logits, block, L, scratch=None):
    B = block.shape[0]
    dev = logits.device
    blk = torch.from_numpy(block).to(dev)
    ln = torch.from_numpy(L.astype(np.int32)).to(dev)
    z = lambda *s: torch.full(s, 99, dtype=torch.int32, device=dev)  # noqa: E731
    g, a, e, out = z(B, 16), z(B), z(B), z(B, 16)
    scratch = clk.verify_scratch(B) if scratch is None else scratch
    clk.verify_greedy(logits, blk, ln, g, a, e, out, scratch)
    torch.cuda.synchronize()
    return g.cpu().numpy(), a.cpu().numpy(), e.cpu().numpy(), out.cpu().numpy()


def _np_view(logits):
    if logits.dtype == torch.bfloat16:
        return logits.view(torch.int16).cpu().numpy().view(np.uint16)
    return logits.cpu().numpy()


def _blocks_from(x_np, L, rng, p_agree=0.8):
    """Blocks whose drafts agree with the true argmax with probability p_agree."""
    B = L.size
    block = rng.integers(0, x_np.shape[2], size=(B, 16)).astype(np.int32)
    for b in range(B):
        for r in range(min(15, x_np.shape[1] - 1)):
            if rng.random() < p_agree:
                block[b, r + 1] = oracle.argmax_row(x_np[b, r])
    return block


def _check(logits, L, rng, **kw):
    x_np = _np_view(logits)
    block = _blocks_from(x_np, L, rng, **kw)
    got = _gpu(logits, block, L)
    want = _oracle_rows(x_np, block, L)
    for name, gg, ww in zip(("argmax", "accept", "emitted", "out_tok"), got, want):
        assert np.array_equal(gg, ww), (name, gg, ww)


@pytest.mark.parametrize("V", [8, 1000, 4096, 32000, 248320, 248321])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_seeded_rows(V, dtype):
    rng = np.random.default_rng(V)
    B = 5
    x = torch.from_numpy(rng.standard_normal((B, 16, V)).astype(np.float32)).to("cuda").to(dtype)
    L = rng.integers(1, 17, size=B)
    _check(x, L, rng)


def test_ragged_batch_of_300():
    rng = np.random.default_rng(3)
    B, V = 300, 4096
    # coarse values: many exact ties inside each row
    x = torch.from_numpy(rng.integers(-20, 20, size=(B, 16, V)).astype(np.float32)).to("cuda").to(torch.bfloat16)
    L = rng.choice([8, 16, 1, 2, 15], size=B)
    _check(x, L, rng, p_agree=0.95)


def test_generator_rows_full_width():
    """The synthetic target's bf16 rows at V = 248,320, all 16 rows."""
    w = wl.make_small("mixed", seed=41, B=4, V=248320, steps=4)
    gen = wl.DevGen(w)
    x = gen.alloc_logits()
    gen.logits(x)
    rng = np.random.default_rng(41)
    _check(x, np.array([16, 8, 16, 3]), rng, p_agree=0.97)


def _hand_rows(V, dtype):
    ninf = float("-inf")
    rows = np.zeros((10, V), np.float32)
    rows[0, :] = 1.0                                   # all equal -> 0
    rows[1, :] = (np.arange(V) % 97).astype(np.float32) / 128.0
    rows[1, V - 1] = 2.0                               # max at the last index
    rows[2, :] = -1.0
    rows[2, [5, V // 2, V - 3]] = 3.0                  # equal maxima far apart -> 5
    rows[3, :] = -1.0
    rows[3, 7] = -0.0
    rows[3, V - 9] = 0.0                               # -0 == +0 -> 7
    rows[4, :] = ninf                                  # all -inf -> 0
    rows[5, :] = ninf
    rows[5, V - 1] = -5.0                              # -> V-1
    rows[6, :] = 0.5
    rows[6, V // 3] = np.inf
    rows[6, V - 2] = np.nan                            # NaN beats +inf -> V-2
    rows[7, :] = 0.0
    rows[7, [3, V - 5]] = np.nan                       # first NaN -> 3
    rows[8, :] = -2.0
    rows[8, [11, V - 11]] = np.inf                     # -> 11
    rows[9, :] = 0.25
    expect = [0, V - 1, 5, 7, 0, V - 1, V - 2, 3, 11, None]
    x = torch.from_numpy(rows)
    if dtype == torch.bfloat16:
        xb = x.to(torch.bfloat16)
        bits = xb.view(torch.int16)
        bits[9, 100] = 0x3E81   # 0.251953125: one mantissa bit above 0.25 (0x3E80)
        bits[9, V - 7] = 0x3E81
        expect[9] = 100
        return xb, expect
    x[9, 100] = float(np.nextafter(np.float32(0.25), np.float32(1.0)))
    expect[9] = 100
    return x, expect


@pytest.mark.parametrize("V", [4096, 248320, 4099])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_hand_rows(V, dtype):
    rows, expect = _hand_rows(V, dtype)
    B = 10
    x = torch.zeros((B, 16, V), dtype=dtype)
    x[:, 0, :] = rows
    x = x.to("cuda")
    L = np.ones(B, np.int64)
    block = np.full((B, 16), -1, np.int32)
    g, a, e, out = _gpu(x, block, L)
    assert g[:, 0].tolist() == expect
    # and the oracle agrees on every one of them
    want = _oracle_rows(_np_view(x), block, L)
    assert np.array_equal(g, want[0])


def test_invalid_lengths_give_empty_outputs():
    rng = np.random.default_rng(5)
    x = torch.randn((4, 16, 512), device="cuda").to(torch.bfloat16)
    L = np.array([0, 17, 8, -3])
    block = np.zeros((4, 16), np.int32)
    g, a, e, out = _gpu(x, block, L)
    for b in (0, 1, 3):
        assert (g[b] == SENT).all() and (out[b] == SENT).all() and a[b] == 0 and e[b] == 0
    assert e[2] >= 1


def test_strided_and_unaligned_views():
    """Rows that are slices of a wider buffer (the scalar path) give the same answers."""
    rng = np.random.default_rng(6)
    base = torch.randn((3, 16, 4100), device="cuda").to(torch.bfloat16)
    x = base[:, :, 3:3 + 4093]           # row start not 16-byte aligned, V odd
    assert x.stride(2) == 1
    L = np.array([16, 5, 9])
    x_np = _np_view(x.contiguous())
    block = _blocks_from(x_np, L, rng)
    got = _gpu(x, block, L)
    want = _oracle_rows(x_np, block, L)
    for gg, ww in zip(got, want):
        assert np.array_equal(gg, ww)


def test_scratch_is_left_clean_for_reuse():
    rng = np.random.default_rng(7)
    x = torch.randn((6, 16, 32000), device="cuda").to(torch.bfloat16)
    L = rng.integers(1, 17, size=6)
    block = _blocks_from(_np_view(x), L, rng)
    scratch = clk.verify_scratch(6)
    first = _gpu(x, block, L, scratch)
    second = _gpu(x, block, L, scratch)
    for f, s in zip(first, second):
        assert np.array_equal(f, s)
    assert int(scratch.count_nonzero()) == 0


@pytest.mark.parametrize("hint", ["none", "short", "long", "mixed", "garbage"])
def test_fused_verify_results_do_not_depend_on_the_length_hint(hint):
    """clk_verify_append reads the rows of a predicted length before the
    proposal launch has finished; the prediction changes only what is read
    early, never the outputs or the committed tokens."""
    rng = np.random.default_rng(8)
    B, V = 40, 4096
    x = torch.from_numpy(rng.integers(-20, 20, size=(B, 16, V)).astype(np.float32)).to("cuda").to(torch.bfloat16)
    L = rng.choice([8, 16], size=B).astype(np.int32)
    L[::7] = 0  # invalid lengths take the empty result
    block = _blocks_from(_np_view(x), np.where(L > 0, L, 1), rng, p_agree=0.9)
    want = _oracle_rows(_np_view(x), block, L)
    hints = {"none": None, "short": np.full(B, 8), "long": np.full(B, 16),
             "mixed": rng.choice([8, 16], size=B), "garbage": rng.integers(-5, 40, size=B)}
    h = hints[hint]
    lk = clk.Lookup(max_slots=B, max_hist=64, vocab=V)
    s = torch.arange(B, dtype=torch.int32, device="cuda")
    clk.lookup_init(lk, s, torch.ones(B, dtype=torch.int32, device="cuda"),
                    torch.arange(B + 1, dtype=torch.int64, device="cuda"))
    z = lambda *sh: torch.full(sh, 77, dtype=torch.int32, device="cuda")  # noqa: E731
    g, a, e, out = z(B, 16), z(B), z(B), z(B, 16)
    hint_t = None if h is None else torch.from_numpy(h.astype(np.int32)).cuda()
    clk.verify_append(lk, s, x, torch.from_numpy(block).cuda(), torch.from_numpy(L).cuda(), g, a, e, out,
                      length_hint=hint_t)
    torch.cuda.synchronize()
    for name, gg, ww in zip(("argmax", "accept", "emitted", "out_tok"), (g, a, e, out), want):
        assert np.array_equal(gg.cpu().numpy(), ww), name
    for b in range(B):
        committed = want[3][b][:want[2][b]].tolist()
        assert lk.history(b).tolist() == [1] + committed
    assert lk.status()[0] == (clk.EINVAL if (L == 0).any() else 0)


@pytest.mark.parametrize("alone", [False, True])
def test_fused_verify_split_setting_changes_no_result(alone):
    """A launch large enough (67 MB of rows) that, expecting to overlap the
    proposal launch, it gives its trailing CTAs a smaller share; launched
    alone (clk_lookup_set_alone) it splits evenly.  Outputs and commits are
    the oracle's either way."""
    rng = np.random.default_rng(9)
    B, V = 64, 32768
    x = torch.from_numpy(rng.integers(-20, 20, size=(B, 16, V)).astype(np.float32)).to("cuda").to(torch.bfloat16)
    L = rng.choice([8, 16], size=B).astype(np.int32)
    block = _blocks_from(_np_view(x), L, rng, p_agree=0.9)
    want = _oracle_rows(_np_view(x), block, L)
    lk = clk.Lookup(max_slots=B, max_hist=64, vocab=V)
    lk.set_alone(alone)
    s = torch.arange(B, dtype=torch.int32, device="cuda")
    clk.lookup_init(lk, s, torch.ones(B, dtype=torch.int32, device="cuda"),
                    torch.arange(B + 1, dtype=torch.int64, device="cuda"))
    z = lambda *sh: torch.full(sh, 77, dtype=torch.int32, device="cuda")  # noqa: E731
    g, a, e, out = z(B, 16), z(B), z(B), z(B, 16)
    hint = torch.from_numpy(rng.choice([8, 16], size=B).astype(np.int32)).cuda()
    clk.verify_append(lk, s, x, torch.from_numpy(block).cuda(), torch.from_numpy(L).cuda(), g, a, e, out,
                      length_hint=hint)
    torch.cuda.synchronize()
    for name, gg, ww in zip(("argmax", "accept", "emitted", "out_tok"), (g, a, e, out), want):
        assert np.array_equal(gg.cpu().numpy(), ww), name
    for b in range(B):
        assert lk.history(b).tolist() == [1] + want[3][b][:want[2][b]].tolist()
    assert lk.status() == (0, 0)


def test_maximum_batch():
    """B = CLK_MAX_BATCH (8,192) requests: the stateless verify against the
    oracle, and the static-scratch entry's limit (1,024 requests)."""
    B, V = 8192, 64
    rng = np.random.default_rng(88)
    L = rng.integers(1, 17, size=B)
    x = torch.randn((B, 16, V), generator=torch.Generator(device="cuda").manual_seed(88), device="cuda")
    _check(x.to(torch.bfloat16).contiguous(), L, rng)
    # the static entry takes up to 1,024 requests and refuses more, launching nothing
    xb = x[:1025].to(torch.bfloat16).contiguous()
    blk = torch.zeros((1025, 16), dtype=torch.int32, device="cuda")
    ln = torch.full((1025,), 4, dtype=torch.int32, device="cuda")
    z = lambda *s: torch.zeros(s, dtype=torch.int32, device="cuda")  # noqa: E731
    g, a, e, out = z(1025, 16), z(1025), z(1025), z(1025, 16)
    with pytest.raises(clk.ClkError) as err:
        clk.verify_greedy_static(xb, blk, ln, g, a, e, out)
    assert err.value.code == clk.ECAPACITY
    clk.verify_greedy_static(xb[:1024], blk[:1024], ln[:1024], g[:1024], a[:1024], e[:1024], out[:1024])
    torch.cuda.synchronize()
    assert (e[:1024] >= 1).all()


@pytest.mark.parametrize("V", [5000, 5003])  # the 16-byte vector path and the scalar path
def test_pinned_host_logits_are_read_in_place(V):
    """Logits in pinned host memory: the stateless and fused greedy verifies
    and the sampler load them in place (unified addressing) and give exactly
    the results of the same logits in device memory, the oracle's for the
    greedy ones."""
    rng = np.random.default_rng(12)
    B = 24
    x = torch.from_numpy(rng.integers(-30, 30, size=(B, 16, V)).astype(np.float32)).to(torch.bfloat16)
    xd, xh = x.cuda(), x.pin_memory()
    L = rng.integers(1, 17, size=B).astype(np.int32)
    block = _blocks_from(_np_view(x), L, rng, p_agree=0.85)
    want = _oracle_rows(_np_view(x), block, L)
    bd, Ld = torch.from_numpy(block).cuda(), torch.from_numpy(L).cuda()
    z = lambda *sh: torch.full(sh, 77, dtype=torch.int32, device="cuda")  # noqa: E731
    for src in (xd, xh):
        g, a, e, out = z(B, 16), z(B), z(B), z(B, 16)
        clk.verify_greedy(src, bd, Ld, g, a, e, out, clk.verify_scratch(B))
        torch.cuda.synchronize()
        for name, gg, ww in zip(("argmax", "accept", "emitted", "out_tok"), (g, a, e, out), want):
            assert np.array_equal(gg.cpu().numpy(), ww), (name, src.is_cuda)
    s = torch.arange(B, dtype=torch.int32, device="cuda")
    hist = []
    for src in (xd, xh):
        lk = clk.Lookup(max_slots=B, max_hist=64, vocab=V)
        clk.lookup_init(lk, s, torch.ones(B, dtype=torch.int32, device="cuda"),
                        torch.arange(B + 1, dtype=torch.int64, device="cuda"))
        g, a, e, out = z(B, 16), z(B), z(B), z(B, 16)
        clk.verify_append(lk, s, src, bd, Ld, g, a, e, out, length_hint=torch.full_like(Ld, 8))
        torch.cuda.synchronize()
        for name, gg, ww in zip(("argmax", "accept", "emitted", "out_tok"), (g, a, e, out), want):
            assert np.array_equal(gg.cpu().numpy(), ww), (name, "fused", src.is_cuda)
        hist.append([lk.history(b).tolist() for b in range(B)])
    assert hist[0] == hist[1]
    t = torch.full((B,), 1.5, device="cuda")
    u = torch.rand((B, 16, 2), generator=torch.Generator(device="cuda").manual_seed(12), device="cuda")
    res = []
    for src in (xd, xh):
        a, e, out = z(B), z(B), z(B, 16)
        clk.verify_sample(src, bd, Ld, t, u, a, e, out, clk.verify_sample_scratch(x.dtype, V, B))
        torch.cuda.synchronize()
        res.append((a.cpu().numpy(), e.cpu().numpy(), out.cpu().numpy()))
    for p, q in zip(*res):
        assert np.array_equal(p, q)
