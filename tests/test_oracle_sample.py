"""Pins of the oracle's sampling verification (point-mass drafts).

The rejection rule with a point-mass proposal has closed forms on simple
rows (all logits equal: every probability is 1/V; one raised logit: p(c) =
e^D / (e^D + V - 1)), and its defining property, the lossless one, is a
statement about distributions: the first emitted token is distributed as
the target's first row whatever the draft, a draft is accepted with the
target's probability of it, and after an accepted draft the next token
follows the next row.  These tests check the oracle against those facts,
and check that plausible mistakes planted in its source fail them.  CPU
only.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import workload as wl

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "clk_oracle.c")
SENT = -1


def _u(acc, smp):
    """[16, 2] uniforms: row r accepts with acc[r], samples with smp[r]."""
    u = np.zeros((16, 2), np.float32)
    u[:len(acc), 0] = acc
    u[:len(smp), 1] = smp
    return u


def _eligible(V, excl):
    return [v for v in range(V) if v != excl]


def _uniform_row_cases():
    """(V, draft, L, u_acc, u_smp, expected a, expected tokens) on rows whose
    logits are all equal, worked by hand: p = 1/V everywhere, a draft is
    accepted iff u < 1/V, the rejected row's token is eligible token number
    floor(u * (V - 1)) (the draft removed), the bonus is token floor(u * V)."""
    out = []
    # rejected at row 0: V = 8, draft 3, u_smp 0.5 -> target 3.5 of 7 -> 4th eligible (0,1,2,4) = 4
    out.append((8, 3, 4, [0.9], [0.5], 0, [4]))
    # boundary: u equal to p = 1/8 is not below it -> rejected
    out.append((8, 3, 4, [0.125], [0.1], 0, [_eligible(8, 3)[int(0.1 * 7)]]))
    # all three drafts accepted, bonus from row 3 with u 0.5 -> target 4 of 8 -> the running sum exceeds 4 at v = 4
    out.append((8, 3, 4, [0.05, 0.05, 0.05], [0.7, 0.7, 0.7, 0.5], 3, [3, 3, 3, 4]))
    # target an exact integer: V = 5, draft 0, u 0.5 -> 2 of 4 -> running sum exceeds 2 at the 3rd eligible = 3
    out.append((5, 0, 2, [0.9], [0.5], 0, [3]))
    # second draft rejected
    out.append((6, 2, 8, [0.1, 0.5], [0.3, 0.25], 1, [2, _eligible(6, 2)[int(0.25 * 5)]]))
    return out


@pytest.mark.parametrize("case", _uniform_row_cases())
def test_uniform_rows_closed_form(case):
    V, c, L, acc, smp, a_want, toks = case
    rows = np.zeros((16, V), np.float32)
    blk = [77] + [c] * 15
    a, out = oracle.sample_verify(rows, blk, L, 1.0, _u(acc, smp))
    assert a == a_want
    assert out[:a + 1].tolist() == toks
    assert (out[a + 1:] == SENT).all()


def test_raised_logit_acceptance_boundary():
    # one logit raised by D at the draft: p(c) = e^(D t) / (e^(D t) + V - 1) with inverse temperature t
    V, c, D = 10, 4, 2.0
    for t in (1.0, 0.5, 2.0):
        pc = np.exp(D * t) / (np.exp(D * t) + V - 1)
        rows = np.zeros((16, V), np.float32)
        rows[:, c] = D
        for u0, accepted in ((pc * (1 - 1e-5), True), (pc * (1 + 1e-5), False)):
            a, out = oracle.sample_verify(rows, [0] + [c] * 15, 2, t, _u([u0], [0.0, 0.0]))
            assert (a == 1) == accepted, (t, u0, pc)
            if not accepted:
                assert out[0] == 0  # u_smp = 0: the first eligible token


def test_temperature_scales_the_logits():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(16, 12)).astype(np.float32)
    for seed in range(40):
        u = np.random.default_rng(seed).random((16, 2)).astype(np.float32)
        blk = [0] + rng.integers(0, 12, 15).tolist()
        a1, o1 = oracle.sample_verify(x, blk, 16, 0.5, u)
        a2, o2 = oracle.sample_verify(x * 0.5, blk, 16, 1.0, u)
        assert a1 == a2 and o1.tolist() == o2.tolist()


def test_sentinel_draft_is_rejected_and_samples_the_whole_row():
    V = 8
    rows = np.zeros((16, V), np.float32)
    for u1 in (0.0, 0.3, 0.99):
        a, out = oracle.sample_verify(rows, [5] + [SENT] * 15, 8, 1.0, _u([0.0], [u1]))
        assert a == 0 and out[0] == int(u1 * V)
    # a draft outside the vocabulary behaves the same
    a, out = oracle.sample_verify(rows, [5, V + 3] + [0] * 14, 8, 1.0, _u([0.0], [0.3]))
    assert a == 0 and out[0] == int(0.3 * V)


def test_block_of_one_row_is_a_plain_sample():
    V = 8
    rows = np.zeros((16, V), np.float32)
    a, out = oracle.sample_verify(rows, [5] + [2] * 15, 1, 1.0, _u([0.0], [0.6]))
    assert a == 0 and out[0] == int(0.6 * V) and (out[1:] == SENT).all()


def test_each_row_is_its_own_distribution():
    # row 0 uniform over 8 tokens, row 1 with all its mass on token 5 (a
    # logit 40 above the rest): after row 0's draft is accepted the bonus is 5
    # whatever its uniform; a rejection at row 0 samples the uniform row.
    V = 8
    rows = np.zeros((16, V), np.float32)
    rows[1, 5] = 40.0
    for u1 in (0.001, 0.4, 0.97):  # not 0: every token has weight >= e^-40 > 0
        a, out = oracle.sample_verify(rows, [1, 2] + [0] * 14, 2, 1.0, _u([0.1], [0.0, u1]))
        assert a == 1 and out[:2].tolist() == [2, 5]
        a, out = oracle.sample_verify(rows, [1, 2] + [0] * 14, 2, 1.0, _u([0.9], [u1]))
        assert a == 0 and out[0] == _eligible(V, 2)[int(u1 * 7)]


def test_invalid_length():
    rows = np.zeros((16, 8), np.float32)
    for L in (0, 17, -2):
        a, out = oracle.sample_verify(rows, [0] * 16, L, 1.0, _u([], []))
        assert a == -1 and (out == SENT).all()


def test_bf16_rows_equal_their_widened_values():
    rng = np.random.default_rng(9)
    x = rng.normal(size=(16, 50)).astype(np.float32)
    bits = wl.f32_to_bf16_bits(x)
    xw = wl.bf16_bits_to_f32(bits)
    for seed in range(30):
        u = np.random.default_rng(100 + seed).random((16, 2)).astype(np.float32)
        blk = [0] + rng.integers(0, 50, 15).tolist()
        a1, o1 = oracle.sample_verify(bits, blk, 16, 1.3, u)
        a2, o2 = oracle.sample_verify(xw, blk, 16, 1.3, u)
        assert a1 == a2 and o1.tolist() == o2.tolist()


# chi-square critical value, 1e-4 upper tail: 5 degrees of freedom
CHI2_5DOF_1E4 = 25.74


def _softmax(x, t):
    y = np.asarray(x, np.float64) * t
    e = np.exp(y - y.max())
    return e / e.sum()


def _chi2(counts, p):
    n = counts.sum()
    return float(((counts - n * p) ** 2 / (n * p)).sum())


def _draws(rows, blk, L, t, n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        u = rng.random((16, 2)).astype(np.float32)
        out.append(oracle.sample_verify(rows, blk, L, t, u))
    return out


@pytest.mark.parametrize("draft", [0, 3, 5, SENT])
def test_first_token_follows_the_target_whatever_the_draft(draft):
    V, t, n = 6, 0.8, 12000
    rows = np.random.default_rng(21).normal(scale=1.5, size=(16, V)).astype(np.float32)
    p0 = _softmax(rows[0], t)
    res = _draws(rows, [9] + [draft] * 15, 2, t, n, seed=7 + draft)
    first = np.array([o[0] for _, o in res])
    assert _chi2(np.bincount(first, minlength=V), p0) < CHI2_5DOF_1E4
    acc = np.mean([a >= 1 for a, _ in res])
    pc = p0[draft] if draft >= 0 else 0.0
    assert abs(acc - pc) < 5 * np.sqrt(pc * (1 - pc) / n) + 1e-12


def test_token_after_an_accepted_draft_follows_the_next_row():
    V, t, n = 6, 1.0, 20000
    rows = np.random.default_rng(22).normal(scale=1.0, size=(16, V)).astype(np.float32)
    rows[0, 2] += 2.0  # draft 2 is likely at row 0
    p1 = _softmax(rows[1], t)
    res = _draws(rows, [9, 2, 4] + [0] * 13, 3, t, n, seed=8)
    second = np.array([o[1] for a, o in res if a >= 1 and o[0] == 2])
    assert second.size > 5000
    assert _chi2(np.bincount(second, minlength=V), p1) < CHI2_5DOF_1E4


def test_sample_weights_closed_forms():
    e = np.array([1.0, 2.0, 3.0, 4.0])
    # running sums 1, 3, 6, 10; the target is u * 10
    for u, want in ((0.0, 0), (0.05, 0), (0.1, 1), (0.29, 1), (0.3, 2), (0.6, 3), (0.999, 3)):
        assert oracle.sample_weights(e, -1, u) == want
    # token 1 removed: running sums 1, 4, 8 of 8
    for u, want in ((0.1, 0), (0.125, 2), (0.5, 3), (0.99, 3)):
        assert oracle.sample_weights(e, 1, u) == want
    # zero weights are never drawn
    assert oracle.sample_weights(np.array([0.0, 1.0, 0.0]), -1, 0.999) == 1


def _sample_pins_pass() -> bool:
    try:
        for case in _uniform_row_cases():
            test_uniform_rows_closed_form(case)
        test_raised_logit_acceptance_boundary()
        test_temperature_scales_the_logits()
        test_sentinel_draft_is_rejected_and_samples_the_whole_row()
        test_block_of_one_row_is_a_plain_sample()
        test_each_row_is_its_own_distribution()
        test_sample_weights_closed_forms()
        for d in (0, 3):
            test_first_token_follows_the_target_whatever_the_draft(d)
    except AssertionError:
        return False
    return True


MUTANTS = {
    "residual keeps the draft": ("tok = or_sample_weights(e, V, c, (double)u[2 * r + 1]);",
                                 "tok = or_sample_weights(e, V, -1, (double)u[2 * r + 1]);"),
    "accepts when u equals p": ("if ((double)u[2 * r] < pc) {", "if ((double)u[2 * r] <= pc) {"),
    "running sum reaching the target": ("if (run > target) return (int32_t)v;", "if (run >= target) return (int32_t)v;"),
    "temperature ignored": ("e[v] *= inv_temp;", "e[v] *= 1.0;"),
    "bonus drawn with the acceptance uniform": ("tok = or_sample_weights(e, V, -1, (double)u[2 * r + 1]);",
                                                "tok = or_sample_weights(e, V, -1, (double)u[2 * r]);"),
    "draft compared one slot early": ("const int32_t c = blk[r + 1];", "const int32_t c = blk[r];"),
    "rows one behind": ("(size_t)r * (size_t)row_stride * esz", "(size_t)(r > 0 ? r - 1 : 0) * (size_t)row_stride * esz"),
    "excluded weight kept in the total": ("if (v != excl) total += e[v];", "total += e[v];"),
}


def test_unmodified_sampler_passes():
    assert _sample_pins_pass()


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_sampler_mistake_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not unique: {name}"
    path = tmp_path / "clk_oracle_mut.c"
    path.write_text(src.replace(old, new, 1))
    so = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-D_POSIX_C_SOURCE=200809L", "-w", "-fPIC", "-shared", "-pthread",
                    "-o", str(so), str(path), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    real = oracle._lib()
    for fname in ("or_sample_weights", "or_sample_verify"):
        getattr(lib, fname).argtypes = getattr(real, fname).argtypes
        getattr(lib, fname).restype = getattr(real, fname).restype
    monkeypatch.setattr(oracle, "_lib", lambda: lib)
    assert not _sample_pins_pass(), f"pins did not catch: {name}"


def test_sampled_loop_at_near_zero_temperature_is_the_greedy_loop():
    # every synthetic row has a unique maximum (the ground truth's +8 lift):
    # at inverse temperature 1e4 the target is a point mass on it, so a draft
    # is accepted iff it is the argmax and the draw is the argmax
    for kind in ("mixed", "periodic"):
        w = wl.make_small(kind, seed=93, B=4, V=1024, steps=40)
        g = oracle.run(w, threads=4)
        s = oracle.run(w, threads=4, inv_temp=1e4)
        for f in ("k", "j", "L", "a", "blk"):
            assert np.array_equal(getattr(g, f), getattr(s, f)), (kind, f)
        assert all(np.array_equal(x, y) for x, y in zip(g.histories, s.histories))
        emitted = np.where(np.arange(16)[None, None, :] <= g.a[:, :, None], g.g, SENT)
        assert np.array_equal(emitted, s.g)


def test_sampled_loop_commits_its_draws():
    w = wl.make_small("copy", seed=94, B=3, V=512, steps=30)
    s = oracle.run(w, threads=3, inv_temp=0.8)
    gen = wl.HostGen(w)
    for i in range(w.B):
        n0 = w.prompts[i].size
        h = s.histories[i]
        toks = [int(x) for t in range(w.steps) for x in s.g[t, i][:s.a[t, i] + 1]]
        assert h[n0:].tolist() == toks
        # replaying step 0 by hand gives the same result
        rows = gen.logits_rows(i, n0, int(s.L[0, i]))
        a, out = oracle.sample_verify(rows, s.blk[0, i], int(s.L[0, i]), 0.8, gen.uniforms(i, 0))
        assert a == s.a[0, i] and out.tolist() == s.g[0, i].tolist()
