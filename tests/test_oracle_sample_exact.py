"""Pins of the oracle's exact sampler (or_sample_verify_exact): the sampling
rule on fixed-point weights, where every acceptance and draw is an integer
comparison.  CPU only.

What pins it to something other than itself:
- the weight Q(d) against 2^(d + 29.5) from numpy (the polynomial, the
  rounding split and the bit arithmetic), and its monotonicity;
- closed forms: at inverse temperature fl32(ln 2) the scale s is exactly 1,
  so integer logits within 3 of the row's maximum have weights in exact
  ratios 2^(x_i - x_j); then p(c) and the inverse CDF are exact fractions,
  and the sampler's decisions must equal the textbook rule computed with
  Python's Fraction, right at and beside every threshold, over several
  chunks with different references;
- agreement with the double-precision sampler (or_sample_verify) on random
  batches, every disagreement being a decision within 1e-5 of its boundary;
- planted mistakes in a copy of the C source, each caught by these pins.
"""
import ctypes
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "clk_oracle.c")
SENT = -1
TAU_ONE = float(np.float32(0.6931471805599453))  # fl32(ln 2): s = fl32(tau * fl32(log2 e)) = 1 exactly


def test_inverse_temperature_with_unit_scale():
    assert np.float32(np.float32(TAU_ONE) * np.float32(1.4426950408889634)) == np.float32(1.0)


# --------------------------------------------------------------------------
# The weight of one entry
# --------------------------------------------------------------------------

def _weight_fn(lib):
    return lambda x, s, R: int(lib.or_fx_weight(float(x), float(s), int(R)))


def _check_weights(fxw):
    """Q(d) ~ 2^(d + 29.5) within 2^-21 relative plus half a unit; 0 below
    -32; non-decreasing in d."""
    rng = np.random.default_rng(3)
    d = np.concatenate([rng.uniform(-31.0, 0.25, 4000), np.arange(-31, 1, dtype=np.float64),
                        np.arange(-31, 0, dtype=np.float64) + 0.5]).astype(np.float32)
    for x in d:
        q = fxw(x, 1.0, 0)
        ideal = 2.0 ** (float(x) + 29.5)
        if not abs(q - ideal) <= ideal * 2.0 ** -21 + 0.5:
            return False
    for x in (-32.5, -40.0, -1e6, -3e38, float("-inf")):
        if fxw(x, 1.0, 0) != 0:
            return False
    xs = np.sort(d)
    qs = [fxw(x, 1.0, 0) for x in xs]
    if not all(a <= b for a, b in zip(qs, qs[1:])):
        return False
    # d = fma(x, s, -R) is rounded once: x s - R exact in double, then float
    for _ in range(2000):
        x = np.float32(rng.uniform(-8, 8))
        sc = np.float32(rng.uniform(0.3, 6.0))
        R = int(np.ceil(np.float32(8 * sc)))
        d = np.float32(np.float64(x) * np.float64(sc) - R)
        if fxw(x, sc, R) != fxw(d, 1.0, 0):
            return False
    return True


def test_weight_follows_exp2():
    assert _check_weights(oracle.fx_weight)


def test_weight_uses_the_fused_multiply_add_against_the_reference():
    # d = fma(x, s, -R): one rounding.  x s - R with x s exactly an integer
    # plus a small remainder shows the difference from a rounded product.
    x, s = np.float32(1.0 + 2.0 ** -23), np.float32(3.0 - 2.0 ** -22)
    d = float(np.float64(x) * np.float64(s) - 3.0)  # exact in double, then one float rounding
    assert oracle.fx_weight(x, s, 3) == oracle.fx_weight(np.float32(d), 1.0, 0)


def test_chunk_references_and_totals():
    rng = np.random.default_rng(4)
    V = 3 * oracle.FX_CHUNK + 17
    row = (rng.standard_normal(V) * 3).astype(np.float32)
    row[oracle.FX_CHUNK:2 * oracle.FX_CHUNK] = -np.inf  # a chunk of -inf only
    t = 1.7
    S, R = oracle.fx_chunks(row, t)
    s = np.float32(np.float32(t) * np.float32(1.4426950408889634))
    for k in range(S.size):
        part = row[k * oracle.FX_CHUNK:(k + 1) * oracle.FX_CHUNK]
        if k == 1:
            assert S[k] == 0 and R[k] == -16777216
            continue
        assert R[k] == int(np.ceil(np.float32(part.max() * s)))
        z = part.astype(np.float64) * float(s) - R[k]
        ideal = float(np.sum(2.0 ** (z + 29.5)))
        assert abs(int(S[k]) - ideal) <= ideal * 2.0 ** -20 + part.size
    assert oracle.fx_chunks(np.full(10, -np.inf, np.float32), 1.0) is None  # nothing to weigh
    big = row.copy()
    big[5] = 3.0e6  # |M s| > 2^22
    assert oracle.fx_chunks(big, 1.0) is None


# --------------------------------------------------------------------------
# Closed forms: exact rational probabilities
# --------------------------------------------------------------------------

def _exact_rule(x, blk, L, u):
    """The textbook sampler on weights 2^x (integer x): accept iff
    u_acc < p(c), then the inverse CDF of the residual (or the last row)."""
    out = [SENT] * 16
    a = 0
    for r in range(L):
        lo = int(np.min(x[r]))
        w = [1 << (int(v) - lo) for v in x[r]]  # integer weights in the ratios 2^(x_i - x_j)
        c = blk[r + 1] if r < L - 1 else SENT
        if r < L - 1 and 0 <= c < len(w) and Fraction(float(u[r][0])) < Fraction(w[c], sum(w)):
            out[r] = c
            a += 1
            continue
        if 0 <= c < len(w):
            w[c] = 0
        tot, run, us = sum(w), 0, Fraction(float(u[r][1]))
        for i, wi in enumerate(w):
            run += wi
            if wi > 0 and Fraction(run, tot) > us:
                out[a] = i
                break
        return a, out
    raise AssertionError("not reached")


def _closed_form_cases(seed, n=40):
    """Rows of integer logits within 3 of the row maximum (chunks with
    different maxima), drafts and uniforms on the 2^-24 grid, some uniforms
    placed at and beside the thresholds."""
    rng = np.random.default_rng(seed)
    for _ in range(n):
        V = int(rng.choice([4, 7, 1024, 1500, 3000]))
        L = int(rng.integers(1, 17))
        top = int(rng.integers(-20, 20))
        x = np.full((16, V), top - 3, np.float32)
        # per chunk a maximum of top - 0..3, entries below it
        for r in range(16):
            for k in range(0, V, oracle.FX_CHUNK):
                m = top - int(rng.integers(0, 4)) if k else top
                e = min(V, k + oracle.FX_CHUNK)
                x[r, k:e] = m - rng.integers(0, 4 - (top - m), e - k)
                x[r, k] = m
        blk = rng.integers(-1, V, 16).astype(np.int32)
        u = (rng.integers(0, 2 ** 24, (16, 2)) / 2 ** 24).astype(np.float32)
        # uniforms at the acceptance thresholds (just below, at, just above)
        for r in range(15):
            c = blk[r + 1]
            if 0 <= c < V and rng.random() < 0.6:
                lo = int(np.min(x[r]))
                w = [1 << (int(v) - lo) for v in x[r]]
                p = Fraction(w[c], sum(w))
                k = int(p * 2 ** 24)
                u[r, 0] = np.float32((k + int(rng.integers(-1, 2))) / 2 ** 24)
        yield x, blk, L, u


def _closed_form_ok(verify, seed=11):
    for x, blk, L, u in _closed_form_cases(seed):
        a, out = verify(x, blk, L, TAU_ONE, u)
        ea, eout = _exact_rule(x, blk.tolist(), L, u.tolist())
        if a != ea or out.tolist() != eout:
            return False
    return True


def test_closed_form_decisions():
    assert _closed_form_ok(oracle.sample_verify_exact)


def test_closed_form_equal_weights_at_a_threshold():
    # four equal logits: p = 1/4 exactly; u = 1/4 is not below it (rejected),
    # the next grid point down is (accepted)
    x = np.zeros((16, 4), np.float32)
    blk = np.array([0, 2] + [SENT] * 14, np.int32)
    u = np.zeros((16, 2), np.float32)
    u[0, 0], u[0, 1] = 0.25, 0.5
    a, out = oracle.sample_verify_exact(x, blk, 2, TAU_ONE, u)
    assert a == 0 and out[0] == 1  # the residual {0, 1, 3}: running 1/3, 2/3 > 1/2 at token 1
    u[0, 0] = np.float32(0.25 - 2 ** -24)
    a, out = oracle.sample_verify_exact(x, blk, 2, TAU_ONE, u)
    assert a == 1 and out[0] == 2


# --------------------------------------------------------------------------
# Against the double-precision sampler
# --------------------------------------------------------------------------

def test_agrees_with_the_double_precision_sampler():
    rng = np.random.default_rng(5)
    n = differ = 0
    for _ in range(400):
        V = int(rng.integers(1, 9000))
        L = int(rng.integers(1, 17))
        rows = (rng.standard_normal((16, V)) * 1.5).astype(np.float32)
        blk = rng.integers(-1, V, 16).astype(np.int32)
        for r in range(15):
            if blk[r + 1] >= 0 and rng.random() < 0.7:
                rows[r, blk[r + 1]] += 3.0 + np.log(V)
        t = float(np.float32(rng.choice([0.25, 0.7, 1.0, 2.5, 4.0])))
        u = (rng.integers(0, 2 ** 24, (16, 2)) / 2 ** 24).astype(np.float32)
        a1, o1 = oracle.sample_verify(rows, blk, L, t, u)
        a2, o2 = oracle.sample_verify_exact(rows, blk, L, t, u)
        n += 1
        if a1 == a2 and (o1 == o2).all():
            continue
        differ += 1
        # the first differing decision must lie within 1e-5 of its boundary
        s = np.float32(np.float32(t) * np.float32(1.4426950408889634))
        r = min(a1, a2)
        z = rows[r].astype(np.float64) * float(s)
        e = 2.0 ** (z - z.max())
        c = blk[r + 1] if r < L - 1 else SENT
        if a1 != a2:
            p = e[c] / e.sum()
            assert abs(float(u[r, 0]) - p) <= 1e-5 * max(p, 1e-30) + 1e-12, (V, L, r)
        else:
            if 0 <= c < V:
                e[c] = 0.0
            C = np.cumsum(e) / e.sum()
            tok = min(o1[r], o2[r])
            assert abs(C[tok] - float(u[r, 1])) <= 1e-5, (V, L, r)
    assert differ <= 0.01 * n, differ


def test_exact_loop_equals_the_sampled_loop_on_a_small_workload():
    """The whole sampled decode loop on the fixed-point weights equals the
    double-precision loop on a seeded workload: no decision of these runs
    lies within the weights' rounding (about 1e-7) of its threshold."""
    import workload as wl
    w = wl.make_small("mixed", seed=76, B=6, V=2048, steps=48)
    for t in (1.0, 2.5):
        a = oracle.run(w, threads=2, inv_temp=t)
        b = oracle.run(w, threads=2, inv_temp=t, exact=True)
        assert np.array_equal(a.g, b.g) and np.array_equal(a.a, b.a)


def test_invalid_inputs_give_the_empty_result():
    x = np.zeros((16, 8), np.float32)
    blk = np.array([0] + [1] * 15, np.int32)
    u = np.full((16, 2), 0.5, np.float32)
    for L, t in ((0, 1.0), (17, 1.0), (4, 0.0), (4, float("inf")), (4, -1.0)):
        a, out = oracle.sample_verify_exact(x, blk, L, t, u)
        assert a == -1 and (out == SENT).all()
    y = x.copy()
    y[2, 3] = 5.0e6  # |M s| > 2^22 in a row the block covers
    assert oracle.sample_verify_exact(y, blk, 4, 1.0, u)[0] == -1
    assert oracle.sample_verify_exact(y, blk, 2, 1.0, u)[0] != -1  # row 2 not covered
    y = x.copy()
    y[1, :] = -np.inf
    assert oracle.sample_verify_exact(y, blk, 4, 1.0, u)[0] == -1


# --------------------------------------------------------------------------
# Planted mistakes
# --------------------------------------------------------------------------

MUTANTS = {
    "rounding split by floor": ("const float n = rintf(d);", "const float n = floorf(d);"),
    "polynomial one degree short": ("float f = c[6];\n    for (int k = 5; k >= 0; --k) f = fmaf(f, r, c[k]);",
                                    "float f = c[5];\n    for (int k = 4; k >= 0; --k) f = fmaf(f, r, c[k]);"),
    "product rounded before the reference": ("const float d = fmaf(x, s, -R);", "const float d = x * s - R;"),
    "row total ignores chunk references": ("for (int64_t k = 0; k < nc; ++k) T += or_fx_rowunits(Sr[k], Rr - Rrow[k]);",
                                           "for (int64_t k = 0; k < nc; ++k) T += Sr[k] << OR_FX_GUARD;"),
    "residual keeps the draft's weight": ("total += or_fx_rowunits(S[k] - (k == kx ? qx : 0), Rr - R[k]);",
                                          "total += or_fx_rowunits(S[k], Rr - R[k]);"),
    "chunk remainder not scaled back": ("const uint64_t tc = or_fx_chunkunits(t - before, Rr - R[k]);",
                                        "const uint64_t tc = t - before;"),
    "draw does not skip the draft": ("            if (v == excl) continue;\n", ""),
    "acceptance at equality": ("if (or_fx_mulshift(or_fx_unit(u[2 * r]), T) < w) {",
                               "if (or_fx_mulshift(or_fx_unit(u[2 * r]), T) <= w) {"),
    "product drops its low part": ("return (uint64_t)k * (v >> 24) + (((uint64_t)k * (v & 0xFFFFFFu)) >> 24);",
                                   "return (uint64_t)k * (v >> 24);"),
    "draft weight against the row reference": (
        "const uint64_t w = or_fx_rowunits(qc, Rr - Rrow[kc]);",
        "const uint64_t w = or_fx_q(or_row_value(row, dtype, cd), s, (float)Rr, c);"),
    "chunk reference from the first entry": ("if (x > M) M = x;", "if (v == v0) M = x;"),
    "weights rounded down": ("    return (((m << 7) >> sh) + 1) >> 1;", "    return (m << 6) >> sh;"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / "m.c"
    path.write_text(src.replace(old, new))
    out = tmp_path / "libm.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-D_POSIX_C_SOURCE=200809L", "-fPIC", "-shared",
                    "-pthread", "-o", str(out), str(path), "-lm"], check=True)
    lib = ctypes.CDLL(str(out))
    lib.or_fx_weight.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_int32]
    lib.or_fx_weight.restype = ctypes.c_uint64
    lib.or_sample_verify_exact.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p,
                                           ctypes.c_void_p]
    lib.or_sample_verify_exact.restype = ctypes.c_int32
    return lib


def _verify_with(lib):
    def verify(rows, blk, L, t, u):
        rows = np.ascontiguousarray(rows, np.float32)
        blk = np.ascontiguousarray(blk, np.int32)
        u = np.ascontiguousarray(u, np.float32)
        out = np.empty(16, np.int32)
        a = lib.or_sample_verify_exact(rows.ctypes.data, 1, rows.shape[1], rows.shape[1], blk.ctypes.data, int(L),
                                       float(t), u.ctypes.data, out.ctypes.data)
        return int(a), out
    return verify


def _pins_pass(lib) -> bool:
    if not _check_weights(_weight_fn(lib)):
        return False
    verify = _verify_with(lib)
    if not _closed_form_ok(verify):
        return False
    # the threshold case and random rows against the double sampler
    x = np.zeros((16, 4), np.float32)
    blk = np.array([0, 2] + [SENT] * 14, np.int32)
    u = np.zeros((16, 2), np.float32)
    u[0] = (0.25, 0.5)
    if verify(x, blk, 2, TAU_ONE, u)[0] != 0:
        return False
    rng = np.random.default_rng(6)
    for _ in range(60):
        V = int(rng.integers(1, 5000))
        rows = (rng.standard_normal((16, V)) * 2).astype(np.float32)
        b = rng.integers(-1, V, 16).astype(np.int32)
        uu = (rng.integers(0, 2 ** 24, (16, 2)) / 2 ** 24).astype(np.float32)
        L = int(rng.integers(1, 17))
        t = float(np.float32(rng.choice([0.5, 1.0, 2.0])))
        # (no decision of these seeded cases lies near its boundary)
        a1, o1 = verify(rows, b, L, t, uu)
        a2, o2 = oracle.sample_verify(rows, b, L, t, uu)
        if a1 != a2 or o1.tolist() != o2.tolist():
            return False
    return True


def test_unmutated_source_passes(tmp_path):
    assert _pins_pass(_build_mutant(tmp_path, "none", "#define OR_FX_CHUNK 1024", "#define OR_FX_CHUNK 1024"))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    assert not _pins_pass(_build_mutant(tmp_path, name, old, new)), name


def test_implied_distribution_is_close_to_the_softmax():
    """The exact sampler's distribution (each entry's weight in row units
    over the row's total) is within 1e-6 in total variation of the softmax
    computed in double, at several temperatures, including rows whose chunk
    maxima are far apart (a spike in one chunk)."""
    rng = np.random.default_rng(12)
    L2E = np.float32(1.4426950408889634)
    for t in (0.25, 1.0, 1.4285714, 4.0):
        for spike in (0.0, 8.0):
            V = 3000
            row = (rng.standard_normal(V) * 1.5).astype(np.float32)
            row[int(rng.integers(0, V))] += np.float32(spike)
            S, R = oracle.fx_chunks(row, t)
            s = np.float32(np.float32(t) * L2E)
            Rr = int(R.max())
            w = np.array([oracle.fx_weight(row[i], s, int(R[i // oracle.FX_CHUNK])) *
                          2.0 ** (int(R[i // oracle.FX_CHUNK]) - Rr) for i in range(V)])
            z = row.astype(np.float64) * float(s)
            p = 2.0 ** (z - z.max())
            tv = 0.5 * np.abs(w / w.sum() - p / p.sum()).sum()
            assert tv < 1e-6, (t, spike, tv)


def test_weight_rounding_is_unbiased():
    """Entries far below their chunk's reference have small integer weights;
    rounding them to the nearest integer (not down) leaves no systematic
    bias: over many such entries the mean error against 2^(d + 29.5) is a
    small fraction of a unit."""
    rng = np.random.default_rng(13)
    d = rng.uniform(-24.0, -14.0, 20000).astype(np.float32)
    ideal = 2.0 ** (d.astype(np.float64) + 29.5)
    err = np.array([oracle.fx_weight(x, 1.0, 0) for x in d]) - ideal
    assert abs(err.mean()) < 0.02, err.mean()
    assert (np.abs(err) <= 0.5 + ideal * 2.0 ** -21).all()
