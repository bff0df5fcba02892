"""The exact sampler (clk_verify_sample_exact) on the GPU against the
oracle's or_sample_verify_exact, bit for bit: every acceptance and every
draw of the fixed-point weights is an integer comparison, so there is no
tolerance and no boundary case.  GPU."""
import ctypes
from fractions import Fraction

import numpy as np
import pytest
import torch

import context_lookup_speculative_gb300 as clk
import oracle
import workload as wl
from workload import drive

pytestmark = pytest.mark.gpu
SENT = -1
THREADS = 16
TAU_ONE = float(np.float32(0.6931471805599453))  # s = fl32(tau * fl32(log2 e)) = 1 exactly


def _run(rows, blk, L, t, u, scratch=None):
    B = rows.shape[0]
    dev = rows.device
    acc = torch.full((B,), -7, dtype=torch.int32, device=dev)
    em = torch.full((B,), -7, dtype=torch.int32, device=dev)
    out = torch.full((B, 16), -7, dtype=torch.int32, device=dev)
    if scratch is None:
        scratch = clk.verify_sample_exact_scratch(rows.dtype, rows.shape[2], B, device=dev)
    clk.verify_sample_exact(rows, blk, L, t, u, acc, em, out, scratch)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), em.cpu().numpy(), out.cpu().numpy(), scratch


def _host_rows(rows):
    if rows.dtype == torch.bfloat16:
        return rows.view(torch.int16).cpu().numpy().view(np.uint16)
    return rows.float().cpu().numpy()


def _check(rows, blk, L, t, u):
    acc, em, out, _ = _run(rows, blk, L, t, u)
    hr = _host_rows(rows)
    bl, Ln, tn, un = blk.cpu().numpy(), L.cpu().numpy(), t.cpu().numpy(), u.cpu().numpy()
    for b in range(rows.shape[0]):
        a_o, out_o = oracle.sample_verify_exact(hr[b], bl[b], int(Ln[b]), float(tn[b]), un[b])
        if a_o < 0:
            assert acc[b] == 0 and em[b] == 0 and (out[b] == SENT).all(), b
            continue
        assert acc[b] == a_o and em[b] == a_o + 1, (b, acc[b], a_o)
        assert out[b].tolist() == out_o.tolist(), (b, out[b][:a_o + 1], out_o[:a_o + 1])
    return acc, out


def _case(B, V, dtype, seed, rows=16, temps=(0.5, 1.0, 2.0, 1.7)):
    spike = 3.0 + float(np.log(V))
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn((B, rows, V), generator=g, device="cuda") * 1.5
    hot = torch.randint(0, V, (B, rows), generator=g, device="cuda")
    x.scatter_add_(2, hot.unsqueeze(2), torch.full((B, rows, 1), spike, device="cuda"))
    blk = torch.randint(0, V, (B, 16), generator=g, device="cuda", dtype=torch.int32)
    pick = torch.rand((B, 16), generator=g, device="cuda")
    blk[:, 1:] = torch.where(pick[:, 1:] < 0.7, hot[:, :15].int(), blk[:, 1:])
    blk[:, 1:] = torch.where(pick[:, 1:] > 0.95, torch.full_like(blk[:, 1:], SENT), blk[:, 1:])
    L = torch.randint(1, 17, (B,), generator=g, device="cuda", dtype=torch.int32)
    tt = torch.tensor(temps, device="cuda")
    t = tt[torch.randint(0, len(temps), (B,), generator=g, device="cuda")]
    # uniforms on the generator's 2^-24 grid, plus a few arbitrary floats
    u = torch.randint(0, 2 ** 24, (B, 16, 2), generator=g, device="cuda").float() / 2 ** 24
    u[:, ::5, 0] = torch.rand((B, 4), generator=g, device="cuda")
    return x.to(dtype).contiguous(), blk, L, t.float().contiguous(), u.contiguous()


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V", [1, 7, 1000, 1024, 1025, 3001, 40000])
def test_exact_parity_random_batches(dtype, V):
    x, blk, L, t, u = _case(48, V, dtype, seed=V + (1 if dtype == torch.float32 else 0))
    L[0], L[1], t[2], t[3] = 0, 17, 0.0, float("inf")  # invalid requests: empty results
    acc, _ = _check(x, blk, L, t, u)
    if V >= 1000:
        assert (acc[4:] > 0).any() and (acc[4:] == 0).any()


def test_exact_parity_unaligned_rows_take_the_scalar_path():
    x, blk, L, t, u = _case(24, 4096, torch.bfloat16, seed=5, rows=17)
    _check(x[:, 1:, :], blk, L, t, u)  # a strided view, 16-byte aligned: the vector path
    y = torch.zeros((24, 16, 4099), dtype=torch.bfloat16, device="cuda")
    y[:, :, 3:] = x[:, :16, :]
    _check(y[:, :, 3:], blk, L, t, u)
    z = torch.zeros((24, 16, 4097), dtype=torch.float32, device="cuda")
    z[:, :, 1:] = x[:, :16, :].float()
    _check(z[:, :, 1:], blk, L, t, u)


def test_exact_edge_values():
    """-inf entries and whole -inf chunks, an all -inf row, a chunk maximum
    past 2^22 (both: the empty result), a vanishing and a huge inverse
    temperature, uniforms 0, just below 1, 1 and NaN."""
    B, V = 12, 2500
    x, blk, L, t, u = _case(B, V, torch.float32, seed=21)
    L[:] = 16
    x[0, :, ::3] = float("-inf")
    x[1, 2, 1024:2048] = float("-inf")
    x[2, 5, :] = float("-inf")  # a row that cannot be weighed
    x[3, 7, 100] = 5.0e6  # |M s| > 2^22
    t[4] = 1e-30
    t[5] = 1e4
    u[6] = 0.0
    u[7] = float(np.float32(1.0 - 2 ** -24))
    u[8] = 1.0
    u[9, :, 1] = float("nan")
    _check(x, blk, L, t, u)
    # the block stops before the bad row: the request is valid
    L[2], L[3] = 5, 7
    _check(x, blk, L, t, u)


def test_exact_closed_form_thresholds():
    """Integer logits within 3 of their row's maximum at unit scale: weights
    in exact ratios 2^(x_i - x_j), so p(c) is a fraction and the GPU must
    accept exactly below it; uniforms at, just below and just above every
    draft's threshold."""
    rng = np.random.default_rng(9)
    B, V = 32, 3000
    x = np.zeros((B, 16, V), np.float32)
    for b in range(B):
        for r in range(16):
            top = int(rng.integers(-10, 10))
            x[b, r] = top - rng.integers(0, 4, V)
    blk = rng.integers(0, V, (B, 16)).astype(np.int32)
    u = (rng.integers(0, 2 ** 24, (B, 16, 2)) / 2 ** 24).astype(np.float32)
    expect_accept = np.zeros((B, 16), bool)
    for b in range(B):
        for r in range(15):
            lo = int(x[b, r].min())
            w = [1 << (int(v) - lo) for v in x[b, r]]
            p = Fraction(w[blk[b, r + 1]], sum(w))
            k = int(p * 2 ** 24) + int(rng.integers(-1, 2))
            u[b, r, 0] = np.float32(k / 2 ** 24)
            expect_accept[b, r] = Fraction(k, 2 ** 24) < p
    dev = dict(device="cuda")
    rows = torch.from_numpy(x).to(**dev)
    L = torch.full((B,), 16, dtype=torch.int32, **dev)
    t = torch.full((B,), TAU_ONE, dtype=torch.float32, **dev)
    acc, out = _check(rows, torch.from_numpy(blk).to(**dev), L, t, torch.from_numpy(u).to(**dev))
    for b in range(B):
        first_rej = int(np.argmin(expect_accept[b, :15])) if not expect_accept[b, :15].all() else 15
        assert acc[b] == first_rej, (b, acc[b], first_rej)


def test_exact_results_repeat_and_the_scratch_is_reusable():
    x, blk, L, t, u = _case(40, 5000, torch.bfloat16, seed=31)
    a1, e1, o1, scratch = _run(x, blk, L, t, u)
    a2, e2, o2, _ = _run(x, blk, L, t, u, scratch=scratch)
    assert (a1 == a2).all() and (e1 == e2).all() and (o1 == o2).all()
    # a smaller batch and another vocabulary on the same scratch
    y, blk2, L2, t2, u2 = _case(8, 3001, torch.bfloat16, seed=32)
    a3, _, o3, _ = _run(y, blk2, L2, t2, u2, scratch=scratch)
    hr = _host_rows(y)
    for b in range(8):
        a_o, out_o = oracle.sample_verify_exact(hr[b], blk2[b].cpu().numpy(), int(L2[b]), float(t2[b]),
                                                u2[b].cpu().numpy())
        assert a3[b] == max(a_o, 0) and (o3[b] == out_o).all()


def test_exact_full_vocabulary_rows_of_the_mixed_batch():
    """The mixed serving batch's shapes (B = 64, V = 248,320, bf16) at
    temperatures 0.25 and 0.7: flat-tail draws included, bit for bit."""
    for seed, temps in ((41, (4.0,)), (42, (float(np.float32(1 / 0.7)),))):
        x, blk, L, t, u = _case(64, 248320, torch.bfloat16, seed=seed, temps=temps)
        _check(x, blk, L, t, u)


def test_exact_bad_arguments_are_rejected():
    x, blk, L, t, u = _case(4, 64, torch.bfloat16, seed=51)
    acc = torch.zeros(4, dtype=torch.int32, device="cuda")
    em, out = torch.zeros_like(acc), torch.zeros((4, 16), dtype=torch.int32, device="cuda")
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(RuntimeError):
        clk.verify_sample_exact(x, blk, L, t, u, acc, em, out, small)
    size = ctypes.c_size_t()
    assert clk.lib().clk_verify_sample_exact_scratch_bytes(clk.BF16, 4194305, 4, ctypes.byref(size)) == -1
    assert clk.lib().clk_verify_sample_exact_scratch_bytes(clk.BF16, 4194304, 4, ctypes.byref(size)) == 0


@pytest.mark.parametrize("inv_temp", [1.0, 2.5])
def test_exact_sampled_loop_matches_the_oracle(inv_temp):
    """The decode loop with the exact sampler (lookup, scheduler, fusion,
    clk_verify_sample_exact, commit) against the oracle's loop on the same
    weights: every record, history and counter equal."""
    w = wl.make_small("mixed", seed=76, B=6, V=2048, steps=48)
    dev = drive.run_device(w, mode="sample_exact", inv_temp=inv_temp)
    ref = oracle.run(w, threads=THREADS, inv_temp=inv_temp, exact=True)
    msgs = drive.compare(dev, ref)
    assert not msgs, "\n".join(msgs[:8])


@pytest.mark.parametrize("inv_temp", [1.0, 2.5])
def test_exact_fused_sampled_loop_matches_the_oracle(inv_temp):
    """The decode loop as the Step driver runs it with the exact sampler
    fused with the commit (clk_verify_sample_exact_append): every record,
    history and counter equal to the oracle's loop on the same weights."""
    w = wl.make_small("mixed", seed=76, B=6, V=2048, steps=48)
    dev = drive.run_device(w, mode="sample_exact_fused", inv_temp=inv_temp)
    ref = oracle.run(w, threads=THREADS, inv_temp=inv_temp, exact=True)
    msgs = drive.compare(dev, ref)
    assert not msgs, "\n".join(msgs[:8])


@pytest.mark.parametrize("inv_temp", [4.0, float(np.float32(1 / 0.7))])
def test_exact_sampled_loop_full_size_mixed_batch_64_steps(inv_temp):
    """The mixed serving batch (B = 64, V = 248,320, bf16) for 64 steps of
    the exact sampled loop at temperatures 0.25 and 0.7, both as the Step
    driver runs it (the sampler fused with the commit, two launches a step)
    and unfused: every record, history and counter equal to the oracle's."""
    w = wl.make("2").with_steps(64)
    ref = oracle.run(w, threads=THREADS, inv_temp=inv_temp, exact=True)
    assert (ref.a > 0).any()
    for mode in ("sample_exact_fused", "sample_exact"):
        dev = drive.run_device(w, mode=mode, inv_temp=inv_temp)
        msgs = drive.compare(dev, ref)
        assert not msgs, mode + ": " + "\n".join(msgs[:8])


@pytest.mark.parametrize("hint", ["none", "short", "long", "exact", "garbage"])
def test_exact_fused_results_do_not_depend_on_the_length_hint(hint):
    """clk_verify_sample_exact_append reads the rows of a predicted length
    before the preceding launch has finished; every chunk's record is the same
    whichever CTA reads it, so the outputs equal the stateless exact sampler's
    bit for bit for any hint, and each valid request commits exactly its
    emitted tokens; invalid requests and a row that cannot be weighed commit
    nothing and latch CLK_EINVAL."""
    B, V = 40, 4096
    x, blk, L, t, u = _case(B, V, torch.bfloat16, seed=90)
    L[::7] = 0
    t[3] = 0.0
    x[5, 2, 17] = 5.0e6  # request 5: a row whose chunk maximum is past 2^22
    L[5] = 16
    want_acc, want_out = _check(x, blk, L, t, u)
    assert want_acc[5] == 0 and (want_out[5] == SENT).all()
    rng = np.random.default_rng(90)
    hints = {"none": None, "short": np.full(B, 8), "long": np.full(B, 16), "exact": L.cpu().numpy(),
             "garbage": rng.integers(-5, 40, size=B)}
    h = hints[hint]
    s = torch.arange(B, dtype=torch.int32, device="cuda")
    hint_t = None if h is None else torch.from_numpy(np.asarray(h, np.int32)).cuda()
    for halves in (1, 2):
        lk = clk.Lookup(max_slots=B, max_hist=64, vocab=V)
        clk.lookup_init(lk, s, torch.ones(B, dtype=torch.int32, device="cuda"),
                        torch.arange(B + 1, dtype=torch.int64, device="cuda"))
        acc = torch.full((B,), 77, dtype=torch.int32, device="cuda")
        em, out = torch.full_like(acc, 77), torch.full((B, 16), 77, dtype=torch.int32, device="cuda")
        scratch = clk.verify_sample_exact_scratch(x.dtype, V, B, halves=halves)
        clk.verify_sample_exact_append(lk, s, x, blk, L, t, u, acc, em, out, scratch, length_hint=hint_t)
        torch.cuda.synchronize()
        assert np.array_equal(acc.cpu().numpy(), want_acc)
        assert np.array_equal(out.cpu().numpy(), want_out)
        emn, outn = em.cpu().numpy(), out.cpu().numpy()
        for b in range(B):
            assert lk.history(b).tolist() == [1] + outn[b][:emn[b]].tolist(), b
        assert lk.status()[0] == clk.EINVAL
