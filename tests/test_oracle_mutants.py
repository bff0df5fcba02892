"""The oracle's pins are strong enough to catch plausible mistakes.

Each case plants one mistake (an off-by-one bound, a flipped comparison, a
dropped term, a wrong index) in a copy of the oracle's C source, builds it on
the CPU and checks that the pins reject it.  Nothing here touches a GPU.
"""
import ctypes
import json
import os
import subprocess

import numpy as np
import pytest

import oracle
import workload as wl
from oracle import brute

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "clk_oracle.c")

MUTANTS = {
    "lookup: j may not equal k": ("for (int64_t j = n - 1; j >= k; --j)", "for (int64_t j = n - 1; j > k; --j)"),
    "lookup: overlap at j = n-1 excluded": ("for (int64_t j = n - 1; j >= k; --j)", "for (int64_t j = n - 2; j >= k; --j)"),
    "lookup: shortest first": ("for (int32_t k = max_k; k >= min_k; --k)", "for (int32_t k = min_k; k <= max_k; ++k)"),
    "lookup: suffix off by one": ("if (h[j - k + i] != h[n - k + i])", "if (h[j - k + i] != h[n - k + i - 1])"),
    "lookup: oldest occurrence": ("for (int64_t j = n - 1; j >= k; --j)", "for (int64_t j = k; j <= n - 1; ++j)"),
    "copy: no cyclic continuation": ("c[i] = c[i - (n - j)];", "c[i] = h[n - 1];"),
    "copy: starts one late": ("else if (j + i < n)\n            c[i] = h[j + i];", "else if (j + i + 1 < n)\n            c[i] = h[j + i + 1];"),
    "sched: slack dropped": ("prev_a >= prev_L - 1 - p->near_full_slack", "prev_a >= prev_L - 1"),
    "sched: sticky off by one": ("if (s->miss > p->sticky)", "if (s->miss >= p->sticky)"),
    "sched: streak off by one": ("if (s->streak >= p->enter_streak)", "if (s->streak > p->enter_streak)"),
    "sched: first step counts as nearly full": ("s->has_prev && prev_a", "prev_a"),
    "sched: miss not reset by flag": ("            s->miss = 0;\n        else", "            s->miss = s->miss;\n        else"),
    "fuse: replace threshold": ("int take_head = k >= p->head_replace_k;", "int take_head = k > p->head_replace_k;"),
    "fuse: agreement on one token": ("for (int32_t i = 0; i < p->head_agree_n; ++i)", "for (int32_t i = 1; i < p->head_agree_n; ++i)"),
    "fuse: tail shifted": ("fill_tail ? c[p->head + i] : OR_SENT", "fill_tail ? c[p->head + i + 1] : OR_SENT"),
    "fuse: tail threshold": ("&& k >= p->tail_k;", "&& k > p->tail_k;"),
    "argmax f32: last occurrence": ("if (x[v] > x[best]) best = v;", "if (x[v] >= x[best]) best = v;"),
    "argmax bf16: last occurrence": ("if (f > bv) {", "if (f >= bv) {"),
    "argmax bf16: NaN ignored": ("if (isnan(or_bf16_value(x[v]))) return (int32_t)v;", "if (0) return (int32_t)v;"),
    "accept: block bound": ("while (a < L - 1 && blk[a + 1] == g[a]) a += 1;", "while (a < L && blk[a + 1] == g[a]) a += 1;"),
    "accept: compares the committed slot": ("while (a < L - 1 && blk[a + 1] == g[a]) a += 1;", "while (a < L - 1 && blk[a] == g[a]) a += 1;"),
    "loop: bonus token dropped": ("for (int32_t r = 0; r <= acc; ++r) h[n + r] = g[r];\n        n += acc + 1;",
                                  "for (int32_t r = 0; r < acc; ++r) h[n + r] = g[r];\n        n += acc;"),
    "loop: rows one position late": ("a->logits_fn(a->gen_ctx, b, n + r, row);", "a->logits_fn(a->gen_ctx, b, n + r + 1, row);"),
    "loop: last token from the draft": ("or_fuse(h[n - 1], c, k, m, L, p, blk);", "or_fuse(c[0], c, k, m, L, p, blk);"),
}


def _golden(name):
    with open(os.path.join(HERE, "golden", name)) as f:
        return json.load(f)


def _pins_pass() -> bool:
    """A compact run of the oracle pins; False at the first failed check."""
    for case in _golden("lookup_examples.json")["cases"]:
        c, k, j = oracle.propose(case["h"])
        if (k, j) != (case["k"], case["j"]) or c.tolist() != case["c"]:
            return False
    rng = np.random.default_rng(5)
    for _ in range(300):
        h = rng.integers(0, 3, size=int(rng.integers(0, 40))).tolist()
        kj = oracle.lookup(h)
        if kj != brute.lookup_brute(h) or oracle.copy(h, *kj).tolist() != brute.copy_brute(h, *kj):
            return False
    for tr in _golden("sched_traces.json")["traces"]:
        s = oracle.Scheduler(oracle.Params.default(sticky=tr["sticky"]))
        pa = pl = 0
        for k, a, want in zip(tr["k"], tr["a"], tr["L"]):
            L = s.step(k, pa, pl)
            if L != want:
                return False
            pa, pl = a, L
    C = [10 + i for i in range(16)]
    M = {"both": [10, 11, 52, 53, 54, 55, 56], "first": [10, 51, 52, 53, 54, 55, 56], "second": [50, 11, 52, 53, 54, 55, 56],
         "none": [50, 51, 52, 53, 54, 55, 56]}
    for row in _golden("fusion_table.json")["rows"]:
        c = C if row["k"] > 0 else [-1] * 16
        blk = oracle.fuse(1000, c, row["k"], M[row["agree"]], row["L"]).tolist()
        head = c[:7] if row["head"] == "lookup" else M[row["agree"]]
        tail = c[7:15] if row["tail"] == "lookup" else [-1] * 8
        if blk != [1000] + list(head) + list(tail):
            return False
    for vals, want in (([0.0, 3.0, 1.0, 3.0], 1), ([-0.0, 0.0, -1.0], 0), ([1.0, np.nan, 5.0, np.nan], 1)):
        x = np.array(vals, np.float32)
        if oracle.argmax_row(x) != want or oracle.argmax_row(wl.f32_to_bf16_bits(x)) != want:
            return False
    G = list(range(100, 116))
    for L in (8, 16):
        for m in range(L):
            blk = [7] + G[:m] + [999] * (15 - m)
            if oracle.accept(blk, G, L) != min(m, L - 1):
                return False
    if oracle.accept([7] + G[:15], G, 8) != 7:
        return False
    w = wl.make_small("mixed", seed=5, B=2, V=512, steps=20)
    res = oracle.run(w, threads=1)
    gen = wl.HostGen(w)
    for i in range(w.B):
        n0 = w.prompts[i].size
        h = res.histories[i]
        rows = wl.bf16_bits_to_f32(gen.logits_rows(i, n0, h.size - n0))
        if h.size == n0 or not np.array_equal(h[n0:], np.argmax(rows, axis=1)):
            return False
        if h.size != n0 + int((res.a[:, i] + 1).sum()) or res.counters[i]["emitted"] != h.size - n0:
            return False
        if not (res.blk[:, i, 0][1:] == h[n0 - 1 + np.cumsum(res.a[:-1, i] + 1)]).all():
            return False
    return True


def test_unmodified_oracle_passes():
    assert _pins_pass()


@pytest.mark.parametrize("name", list(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site not found: {name}"
    mutated = src.replace(old, new, 1)
    path = tmp_path / "clk_oracle_mut.c"
    path.write_text(mutated)
    so = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-D_POSIX_C_SOURCE=200809L", "-w", "-fPIC", "-shared", "-pthread",
                    "-o", str(so), str(path), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    real = oracle._lib()
    for fname in ("or_params_default", "or_lookup", "or_copy", "or_sched", "or_fuse", "or_argmax_f32",
                  "or_argmax_bf16", "or_accept", "or_run"):
        getattr(lib, fname).argtypes = getattr(real, fname).argtypes
        getattr(lib, fname).restype = getattr(real, fname).restype
    monkeypatch.setattr(oracle, "_lib", lambda: lib)
    assert not _pins_pass(), f"pins did not catch: {name}"
