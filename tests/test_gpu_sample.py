"""Sampling verification (point-mass drafts) on the GPU against the oracle.

The kernel computes in float32 and the oracle in double, so a decision can
differ where the two sit within rounding of each other: an acceptance
uniform within a relative 1e-4 of the draft's probability, or a draw whose
target lies within 1e-4 of the total weight from a token boundary.  Every
request must either match the oracle exactly or be such a boundary case
(checked in double here), and boundary cases must be rare.  The tolerance
covers float32 sums of up to 2^18 terms combined in trees, the float32
product x * inv_temp, and the error bound of the hardware exponential
(about 2 ulp): together below 1e-5 relative.  GPU.
"""
import numpy as np
import pytest
import torch

import context_lookup_speculative_gb300 as clk
import oracle
import workload as wl

pytestmark = pytest.mark.gpu
SENT = -1
TOL = 1e-4


def _run(rows, blk, L, t, u):
    B = rows.shape[0]
    dev = rows.device
    acc = torch.full((B,), -7, dtype=torch.int32, device=dev)
    em = torch.full((B,), -7, dtype=torch.int32, device=dev)
    out = torch.full((B, 16), -7, dtype=torch.int32, device=dev)
    scratch = clk.verify_sample_scratch(rows.dtype, rows.shape[2], B, device=dev)
    clk.verify_sample(rows, blk, L, t, u, acc, em, out, scratch)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), em.cpu().numpy(), out.cpu().numpy(), scratch


def _host_rows(rows):
    if rows.dtype == torch.bfloat16:
        return rows.view(torch.int16).cpu().numpy().view(np.uint16)
    return rows.float().cpu().numpy()


def _weights(row, t):
    y = np.asarray(row, np.float64) * float(np.float32(t))
    return np.exp(y - y.max())


def _valid(rows_b, blk, L, t, u, a, out):
    """Whether (a, out) is a correct result when every decision within TOL
    of its boundary may go either way (double precision)."""
    if rows_b.dtype == np.uint16:
        rows_b = wl.bf16_bits_to_f32(rows_b)
    V = rows_b.shape[1]
    if not (0 <= a <= L - 1) or out[:a].tolist() != list(blk[1:a + 1]):
        return False
    for r in range(a + 1):
        if r == L - 1:
            break
        e = _weights(rows_b[r], t)
        c = blk[r + 1]
        p = e[c] / e.sum() if 0 <= c < V else 0.0
        ua = float(u[r, 0])
        if r < a and not ua < p * (1 + TOL) + 1e-30:
            return False
        if r == a and not ua >= p * (1 - TOL):
            return False
    e = _weights(rows_b[a], t)
    c = blk[a + 1] if a < L - 1 else SENT
    if 0 <= c < V:
        e[c] = 0.0
    tok = out[a]
    if not (0 <= tok < V) or e[tok] == 0.0:
        return False
    C = np.cumsum(e)
    Z = C[-1]
    target = float(u[a, 1]) * Z
    before = C[tok - 1] if tok > 0 else 0.0
    return before <= target + TOL * Z and C[tok] >= target - TOL * Z and (out[a + 1:] == SENT).all()


def _check(rows, blk, L, t, u, max_boundary_frac=0.01):
    acc, em, out, _ = _run(rows, blk, L, t, u)
    hr = _host_rows(rows)
    bl, Ln, tn, un = blk.cpu().numpy(), L.cpu().numpy(), t.cpu().numpy(), u.cpu().numpy()
    boundary = 0
    for b in range(rows.shape[0]):
        a_o, out_o = oracle.sample_verify(hr[b], bl[b], int(Ln[b]), float(tn[b]), un[b])
        ok_len = 1 <= Ln[b] <= 16 and tn[b] > 0 and np.isfinite(tn[b])
        if not ok_len:
            assert acc[b] == 0 and em[b] == 0 and (out[b] == SENT).all(), b
            continue
        assert em[b] == acc[b] + 1
        if acc[b] == a_o and out[b].tolist() == out_o.tolist():
            continue
        boundary += 1
        assert _valid(hr[b], bl[b], int(Ln[b]), float(tn[b]), un[b], int(acc[b]), out[b]), \
            (b, acc[b], out[b][:acc[b] + 1], a_o, out_o[:a_o + 1])
    assert boundary <= max(2, max_boundary_frac * rows.shape[0]), boundary
    return acc, out


def _case(B, V, dtype, seed, rows=16):
    # the raised logit grows with ln V so that the drafts it marks keep a
    # sizable probability at every vocabulary size and temperature
    spike = 3.0 + float(np.log(V))
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn((B, rows, V), generator=g, device="cuda") * 1.5
    # a raised token per row that the drafts often name, so drafts get accepted
    hot = torch.randint(0, V, (B, rows), generator=g, device="cuda")
    x.scatter_add_(2, hot.unsqueeze(2), torch.full((B, rows, 1), spike, device="cuda"))
    blk = torch.randint(0, V, (B, 16), generator=g, device="cuda", dtype=torch.int32)
    pick = torch.rand((B, 16), generator=g, device="cuda")
    blk[:, 1:] = torch.where(pick[:, 1:] < 0.7, hot[:, :15].int(), blk[:, 1:])
    blk[:, 1:] = torch.where(pick[:, 1:] > 0.95, torch.full_like(blk[:, 1:], SENT), blk[:, 1:])
    L = torch.randint(1, 17, (B,), generator=g, device="cuda", dtype=torch.int32)
    t = torch.tensor([0.5, 1.0, 2.0, 1.7], device="cuda")[torch.randint(0, 4, (B,), generator=g, device="cuda")]
    u = torch.rand((B, 16, 2), generator=g, device="cuda")
    return x.to(dtype).contiguous(), blk, L, t.float().contiguous(), u.contiguous()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V", [1000, 1003, 40000])
def test_parity_random_batches(dtype, V):
    x, blk, L, t, u = _case(64, V, dtype, seed=V + (1 if dtype == torch.float32 else 0))
    L[0], L[1], t[2], t[3] = 0, 17, 0.0, float("inf")  # invalid requests: empty results
    acc, _ = _check(x, blk, L, t, u)
    assert (acc[4:] > 0).any() and (acc[4:] == 0).any()


def test_parity_unaligned_rows_take_the_scalar_path():
    x, blk, L, t, u = _case(24, 4096, torch.bfloat16, seed=5, rows=17)
    _check(x[:, 1:, :], blk, L, t, u)  # a strided view, still 16-byte aligned: the vector path
    y = torch.zeros((24, 16, 4099), dtype=torch.bfloat16, device="cuda")
    y[:, :, 3:] = x[:, :16, :]
    _check(y[:, :, 3:], blk, L, t, u)


def test_draft_with_the_mass_is_accepted_and_the_bonus_follows_the_last_row():
    B, V = 32, 3000
    x = torch.zeros((B, 16, V), device="cuda")
    g = torch.Generator(device="cuda").manual_seed(11)
    hot = torch.randint(0, V, (B, 16), generator=g, device="cuda")
    x.scatter_(2, hot.unsqueeze(2), 60.0)  # every row has all its mass on one token
    blk = torch.cat([torch.zeros((B, 1), dtype=torch.int32, device="cuda"), hot[:, :15].int()], dim=1)
    L = torch.full((B,), 16, dtype=torch.int32, device="cuda")
    t = torch.ones(B, device="cuda")
    u = torch.rand((B, 16, 2), generator=g, device="cuda") * 0.999
    acc, out = _check(x.to(torch.bfloat16), blk, L, t, u)
    assert (acc == 15).all()
    assert (out[:, 15] == hot[:, 15].cpu().numpy()).all()


def test_results_repeat_exactly_and_the_scratch_is_reusable():
    x, blk, L, t, u = _case(48, 70000, torch.bfloat16, seed=21)
    r1 = _run(x, blk, L, t, u)
    acc = torch.zeros(48, dtype=torch.int32, device="cuda")
    em = torch.zeros_like(acc)
    out = torch.zeros((48, 16), dtype=torch.int32, device="cuda")
    for _ in range(3):  # the same scratch again: the counters were rewound
        clk.verify_sample(x, blk, L, t, u, acc, em, out, r1[3])
        torch.cuda.synchronize()
        assert (acc.cpu().numpy() == r1[0]).all() and (out.cpu().numpy() == r1[2]).all()


# chi-square 1e-4 upper-tail critical value for 15 degrees of freedom
CHI2_15DOF_1E4 = 44.3


@pytest.mark.parametrize("draft", [3, SENT])
def test_first_token_follows_the_target_on_the_gpu(draft):
    B, V = 8192, 16
    row = torch.randn((16, V), generator=torch.Generator(device="cuda").manual_seed(31), device="cuda")
    x = row.unsqueeze(0).expand(B, 16, V).contiguous()
    blk = torch.full((B, 16), draft, dtype=torch.int32, device="cuda")
    L = torch.full((B,), 4, dtype=torch.int32, device="cuda")
    t = torch.full((B,), 0.9, device="cuda")
    u = torch.rand((B, 16, 2), generator=torch.Generator(device="cuda").manual_seed(32), device="cuda")
    acc, em, out, _ = _run(x, blk, L, t, u)
    p0 = _weights(row[0].cpu().numpy(), 0.9)
    p0 /= p0.sum()
    counts = np.bincount(out[:, 0], minlength=V)
    chi2 = float(((counts - B * p0) ** 2 / (B * p0)).sum())
    assert chi2 < CHI2_15DOF_1E4
    pc = p0[draft] if draft >= 0 else 0.0
    assert abs(np.mean(acc >= 1) - pc) < 5 * np.sqrt(pc * (1 - pc) / B) + 1e-12


def test_full_vocabulary_rows_of_the_mixed_batch():
    w = wl.make("2")
    gen = wl.DevGen(w, device="cuda")
    lg = gen.alloc_logits()
    gen.logits(lg)
    B = w.B
    g = torch.Generator(device="cuda").manual_seed(41)
    # drafts: the ground-truth continuation the target favours, with noise
    hot = lg.float().argmax(dim=2).int()
    blk = torch.cat([torch.zeros((B, 1), dtype=torch.int32, device="cuda"), hot[:, :15]], dim=1)
    noise = torch.rand((B, 16), generator=g, device="cuda") < 0.2
    blk[:, 1:] = torch.where(noise[:, 1:], torch.randint(0, w.V, (B, 15), generator=g, device="cuda").int(), blk[:, 1:])
    L = torch.where(torch.rand(B, generator=g, device="cuda") < 0.5, 16, 8).int()
    t = torch.full((B,), 1.0 / 0.3, device="cuda")  # temperature 0.3
    u = torch.rand((B, 16, 2), generator=g, device="cuda")
    acc, _ = _check(lg, blk, L, t, u, max_boundary_frac=0.05)
    assert (acc > 0).any()


def test_bad_arguments_are_rejected():
    x, blk, L, t, u = _case(4, 1000, torch.bfloat16, seed=1)
    acc = torch.zeros(4, dtype=torch.int32, device="cuda")
    em, out = torch.zeros_like(acc), torch.zeros((4, 16), dtype=torch.int32, device="cuda")
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(clk.ClkError):
        clk.verify_sample(x, blk, L, t, u, acc, em, out, small)
    with pytest.raises(ValueError):
        clk.verify_sample(x, blk, L, t.double(), u, acc, em, out, small)


@pytest.mark.parametrize("hint", ["none", "short", "long", "exact", "garbage"])
def test_fused_sampler_results_do_not_depend_on_the_length_hint(hint):
    """clk_verify_sample_append streams the rows of a predicted length before
    the preceding launch has finished; the prediction changes only what is
    read early.  Every segment's pairs and the finisher's fixed-order
    combination are the same whichever CTA reads a row, so the outputs equal
    the stateless sampler's bit for bit (which is checked against the oracle
    here too), and each valid request commits exactly its emitted tokens."""
    B, V = 40, 4096
    x, blk, L, t, u = _case(B, V, torch.bfloat16, seed=90)
    L[::7] = 0  # invalid lengths and temperatures take the empty result
    t[3] = 0.0
    want_acc, want_out = _check(x, blk, L, t, u)
    rng = np.random.default_rng(90)
    hints = {"none": None, "short": np.full(B, 8), "long": np.full(B, 16), "exact": L.cpu().numpy(),
             "garbage": rng.integers(-5, 40, size=B)}
    h = hints[hint]
    lk = clk.Lookup(max_slots=B, max_hist=64, vocab=V)
    s = torch.arange(B, dtype=torch.int32, device="cuda")
    clk.lookup_init(lk, s, torch.ones(B, dtype=torch.int32, device="cuda"),
                    torch.arange(B + 1, dtype=torch.int64, device="cuda"))
    acc = torch.full((B,), 77, dtype=torch.int32, device="cuda")
    em, out = torch.full_like(acc, 77), torch.full((B, 16), 77, dtype=torch.int32, device="cuda")
    scratch = clk.verify_sample_scratch(x.dtype, V, B)
    hint_t = None if h is None else torch.from_numpy(np.asarray(h, np.int32)).cuda()
    clk.verify_sample_append(lk, s, x, blk, L, t, u, acc, em, out, scratch, length_hint=hint_t)
    torch.cuda.synchronize()
    assert np.array_equal(acc.cpu().numpy(), want_acc)
    assert np.array_equal(out.cpu().numpy(), want_out)
    emn, outn = em.cpu().numpy(), out.cpu().numpy()
    for b in range(B):
        assert lk.history(b).tolist() == [1] + outn[b][:emn[b]].tolist(), b
    assert lk.status()[0] == clk.EINVAL
    # the counters were rewound: the same call again gives the same answer
    lk2 = clk.Lookup(max_slots=B, max_hist=64, vocab=V)
    clk.lookup_init(lk2, s, torch.ones(B, dtype=torch.int32, device="cuda"),
                    torch.arange(B + 1, dtype=torch.int64, device="cuda"))
    clk.verify_sample_append(lk2, s, x, blk, L, t, u, acc, em, out, scratch, length_hint=hint_t)
    torch.cuda.synchronize()
    assert np.array_equal(acc.cpu().numpy(), want_acc) and np.array_equal(out.cpu().numpy(), want_out)


def test_fused_sampled_step_commits_and_rejects_invalid_requests():
    """verify_sample_append commits each valid request's emitted tokens to
    its history, and a request with an invalid length or temperature gets
    the empty result, commits nothing and latches CLK_EINVAL."""
    from workload import drive

    w = wl.make_small("mixed", seed=81, B=6, V=2048, steps=4)
    lk, slots = drive.make_lookup(w)
    st = clk.Step(lk, slots)
    head = torch.zeros((w.B, 7), dtype=torch.int32, device="cuda")
    gen = wl.DevGen(w, device="cuda")
    gen.head(0, head)
    st.pre(head)
    lg = gen.alloc_logits()
    gen.logits(lg)
    u = torch.zeros((w.B, 16, 2), dtype=torch.float32, device="cuda")
    gen.uniforms(0, u)
    length = st.length.clone()
    length[1] = 0
    t = torch.full((w.B,), 1.0, device="cuda")
    t[4] = -1.0
    before = [lk.history(int(s)).size for s in slots.tolist()]
    scratch = clk.verify_sample_scratch(lg.dtype, w.V, w.B)
    clk.verify_sample_append(lk, slots, lg, st.block, length, t, u, st.accept, st.emitted, st.out_tok, scratch)
    torch.cuda.synchronize()
    code, detail = lk.status()
    assert code == clk.EINVAL and detail in (1, 4)
    em = st.emitted.cpu().numpy()
    out = st.out_tok.cpu().numpy()
    after = [lk.history(int(s)) for s in slots.tolist()]
    for b in range(w.B):
        if b in (1, 4):
            assert em[b] == 0 and (out[b] == SENT).all() and after[b].size == before[b]
        else:
            assert em[b] >= 1 and after[b].size == before[b] + em[b]
            assert after[b][before[b]:].tolist() == out[b][:em[b]].tolist()
    lk.status_clear()
    assert lk.status()[0] == 0
