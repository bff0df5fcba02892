"""CPU oracle of the context-lookup speculative decoding step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import, call, link or run
anything in this package.  The product package never imports it, and the two
share no code: this side is plain C (``clk_oracle.c``) plus a pure-Python
brute force (``brute.py``), written from the pages' definitions (HyperQwen
context-lookup article, "lookup 草稿的原理：三步走": steps 1-3 and the
greedy-verification paragraph).  Its only other input is the seeded workload
generator (``workload``), which serves both sides.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against brute force, closed forms, hand traces and numpy.argmax.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from functools import lru_cache
from typing import Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SENT = -1
BLOCK = 16
LIB_NAME = "liboracle.so"


def build(verbose: bool = False) -> str:
    """Compile clk_oracle.c into liboracle.so (plain -O2, no vector intrinsics)."""
    src = os.path.join(HERE, "clk_oracle.c")
    out = os.path.join(HERE, LIB_NAME)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-D_POSIX_C_SOURCE=200809L", "-Wall", "-fPIC", "-shared",
           "-pthread",
           "-o", out, src, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    return out


class Params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "min_k", "max_k", "head", "tail", "head_replace_k", "head_agree_k", "head_agree_n", "tail_k",
        "enter_streak", "sticky", "near_full_slack")]

    @classmethod
    def default(cls, **kw) -> "Params":
        p = cls()
        _lib().or_params_default(ctypes.byref(p))
        for k, v in kw.items():
            setattr(p, k, v)
        return p

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class SchedState(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("streak", ctypes.c_int32), ("miss", ctypes.c_int32),
                ("has_prev", ctypes.c_int32)]


class Counters(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("steps", "hits", "long_steps", "drafted", "accepted", "emitted")] + \
               [("accept_hist", (ctypes.c_int64 * 16) * 2)]

    def as_dict(self):
        d = {n: getattr(self, n) for n in ("steps", "hits", "long_steps", "drafted", "accepted", "emitted")}
        d["accept_hist"] = [[self.accept_hist[i][j] for j in range(16)] for i in range(2)]
        return d


_P = ctypes.c_void_p


class RunArgs(ctypes.Structure):
    _fields_ = [("params", _P), ("n_req", ctypes.c_int32), ("req_ids", _P), ("prompt", _P), ("prompt_off", _P),
                ("steps", ctypes.c_int32), ("V", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("threads", ctypes.c_int32), ("gen_ctx", _P), ("logits_fn", _P), ("head_fn", _P),
                ("uniform_fn", _P), ("inv_temp", ctypes.c_float), ("exact", ctypes.c_int32),
                ("rec_k", _P), ("rec_j", _P), ("rec_L", _P), ("rec_a", _P), ("rec_c", _P), ("rec_blk", _P),
                ("rec_g", _P), ("hist_out", _P), ("hist_off", _P), ("hist_len", _P), ("counters", _P),
                ("timed_from", ctypes.c_int32), ("pad", ctypes.c_int32),
                ("method_ns", ctypes.c_int64), ("provider_ns", ctypes.c_int64),
                ("lookup_ns", ctypes.c_int64), ("sched_fuse_ns", ctypes.c_int64), ("verify_ns", ctypes.c_int64)]


@lru_cache(maxsize=None)
def _lib() -> ctypes.CDLL:
    path = os.path.join(HERE, LIB_NAME)
    if not os.path.exists(path):
        build()
    lib = ctypes.CDLL(path)
    lib.or_params_default.argtypes = [ctypes.POINTER(Params)]
    lib.or_lookup.argtypes = [_P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_int64)]
    lib.or_lookup.restype = ctypes.c_int32
    lib.or_copy.argtypes = [_P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int64, _P]
    lib.or_sched.argtypes = [ctypes.POINTER(SchedState), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                             ctypes.POINTER(Params)]
    lib.or_sched.restype = ctypes.c_int32
    lib.or_fuse.argtypes = [ctypes.c_int32, _P, ctypes.c_int32, _P, ctypes.c_int32, ctypes.POINTER(Params), _P]
    lib.or_argmax_f32.argtypes = [_P, ctypes.c_int64]
    lib.or_argmax_f32.restype = ctypes.c_int32
    lib.or_argmax_bf16.argtypes = [_P, ctypes.c_int64]
    lib.or_argmax_bf16.restype = ctypes.c_int32
    lib.or_accept.argtypes = [_P, _P, ctypes.c_int32]
    lib.or_accept.restype = ctypes.c_int32
    lib.or_sample_weights.argtypes = [_P, ctypes.c_int64, ctypes.c_int32, ctypes.c_double]
    lib.or_sample_weights.restype = ctypes.c_int32
    lib.or_sample_verify.argtypes = [_P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64, _P, ctypes.c_int32,
                                     ctypes.c_float, _P, _P]
    lib.or_sample_verify.restype = ctypes.c_int32
    lib.or_sample_verify_exact.argtypes = lib.or_sample_verify.argtypes
    lib.or_sample_verify_exact.restype = ctypes.c_int32
    lib.or_fx_weight.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_int32]
    lib.or_fx_weight.restype = ctypes.c_uint64
    lib.or_fx_chunks.argtypes = [_P, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, _P, _P]
    lib.or_fx_chunks.restype = ctypes.c_int
    lib.or_fx_poly_coefs.argtypes = [_P]
    lib.or_run.argtypes = [ctypes.POINTER(RunArgs)]
    lib.or_run.restype = ctypes.c_int
    lib.or_counters_size.restype = ctypes.c_size_t
    lib.or_run_args_size.restype = ctypes.c_size_t
    assert lib.or_counters_size() == ctypes.sizeof(Counters)
    assert lib.or_run_args_size() == ctypes.sizeof(RunArgs)
    return lib


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


# --------------------------------------------------------------------------
# Single-operation wrappers (one request, one step)
# --------------------------------------------------------------------------
def lookup(h, params: Optional[Params] = None):
    """(k, j) of the longest-then-most-recent suffix match of history h."""
    p = params or Params.default()
    h = _i32(h)
    j = ctypes.c_int64()
    k = _lib().or_lookup(h.ctypes.data, h.size, p.min_k, p.max_k, ctypes.byref(j))
    return int(k), int(j.value)


def copy(h, k: int, j: int) -> np.ndarray:
    h = _i32(h)
    c = np.empty(BLOCK, np.int32)
    _lib().or_copy(h.ctypes.data, h.size, k, j, c.ctypes.data)
    return c


def propose(h, params: Optional[Params] = None):
    """(c[16], k, j): lookup followed by the copy."""
    k, j = lookup(h, params)
    return copy(h, k, j), k, j


class Scheduler:
    """One request's long-block scheduler."""

    def __init__(self, params: Optional[Params] = None):
        self.p = params or Params.default()
        self.s = SchedState(0, 0, 0, 0)

    def step(self, k: int, prev_a: int, prev_L: int) -> int:
        return int(_lib().or_sched(ctypes.byref(self.s), k, prev_a, prev_L, ctypes.byref(self.p)))

    @property
    def mode(self) -> int:
        return self.s.mode


def fuse(last: int, c, k: int, m, L: int, params: Optional[Params] = None) -> np.ndarray:
    p = params or Params.default()
    c = _i32(c)
    m = _i32(m)
    blk = np.empty(BLOCK, np.int32)
    _lib().or_fuse(last, c.ctypes.data, k, m.ctypes.data, L, ctypes.byref(p), blk.ctypes.data)
    return blk


def argmax_row(row: np.ndarray) -> int:
    """First index of the maximum; row is float32 or bf16 bits (uint16)."""
    if row.dtype == np.uint16:
        row = np.ascontiguousarray(row)
        return int(_lib().or_argmax_bf16(row.ctypes.data, row.size))
    row = np.ascontiguousarray(row, dtype=np.float32)
    return int(_lib().or_argmax_f32(row.ctypes.data, row.size))


def accept(blk, g, L: int) -> int:
    blk = _i32(blk)
    g = _i32(g)
    return int(_lib().or_accept(blk.ctypes.data, g.ctypes.data, L))


def sample_weights(e, excl: int, u: float) -> int:
    """Inverse-CDF sample of the weights e (float64) without token `excl`."""
    e = np.ascontiguousarray(e, dtype=np.float64)
    return int(_lib().or_sample_weights(e.ctypes.data, e.size, int(excl), float(u)))


def sample_verify(rows: np.ndarray, blk, L: int, inv_temp: float, u) -> tuple:
    """Sampling verification of one request with point-mass drafts.

    rows: [R >= L, V] float32 logits or bf16 bits (uint16); blk: 16 tokens;
    inv_temp: 1 / temperature (float32); u: [16, 2] float32 uniforms
    (acceptance, sample) per row.  Returns (accepted drafts a, out_tok[16]);
    a = -1 for an invalid L."""
    rows = np.ascontiguousarray(rows)
    if rows.dtype == np.uint16:
        dtype = 0
    else:
        rows = np.ascontiguousarray(rows, dtype=np.float32)
        dtype = 1
    blk = _i32(blk)
    u = np.ascontiguousarray(u, dtype=np.float32).reshape(BLOCK, 2)
    out = np.empty(BLOCK, np.int32)
    a = _lib().or_sample_verify(rows.ctypes.data, dtype, rows.shape[1], rows.shape[1], blk.ctypes.data, int(L),
                                float(inv_temp), u.ctypes.data, out.ctypes.data)
    return int(a), out


def _rows_dtype(rows):
    rows = np.ascontiguousarray(rows)
    if rows.dtype == np.uint16:
        return rows, 0
    return np.ascontiguousarray(rows, dtype=np.float32), 1


def sample_verify_exact(rows: np.ndarray, blk, L: int, inv_temp: float, u) -> tuple:
    """sample_verify on the fixed-point weights (or_sample_verify_exact):
    the same rule, every decision an integer comparison.  a = -1 (and no
    tokens) for an invalid L or temperature or a block that cannot be
    weighed."""
    rows, dtype = _rows_dtype(rows)
    blk = _i32(blk)
    u = np.ascontiguousarray(u, dtype=np.float32).reshape(BLOCK, 2)
    out = np.empty(BLOCK, np.int32)
    a = _lib().or_sample_verify_exact(rows.ctypes.data, dtype, rows.shape[1], rows.shape[1], blk.ctypes.data,
                                      int(L), float(inv_temp), u.ctypes.data, out.ctypes.data)
    return int(a), out


FX_CHUNK = 1024  # entries per chunk of the fixed-point weights


def fx_weight(x: float, s: float, R: int) -> int:
    """Fixed-point weight Q(fma(x, s, -R)) of one entry (x, s float32)."""
    return int(_lib().or_fx_weight(float(x), float(s), int(R)))


def fx_chunks(row: np.ndarray, inv_temp: float):
    """Chunk totals S and references R of one row, or None if the row cannot
    be weighed."""
    row, dtype = _rows_dtype(row)
    V = row.size
    nc = (V + FX_CHUNK - 1) // FX_CHUNK
    S = np.zeros(nc, np.uint64)
    R = np.zeros(nc, np.int32)
    rc = _lib().or_fx_chunks(row.ctypes.data, dtype, V, float(inv_temp), S.ctypes.data, R.ctypes.data)
    return None if rc != 0 else (S, R)


def fx_poly_coefs() -> np.ndarray:
    """The weight polynomial's 7 float32 Horner coefficients."""
    out = np.zeros(7, np.float32)
    _lib().or_fx_poly_coefs(out.ctypes.data)
    return out


# --------------------------------------------------------------------------
# The whole decode loop
# --------------------------------------------------------------------------
class RunResult:
    """Per-step records of an oracle run, arrays indexed [t, i(, slot)]."""

    def __init__(self, **kw):
        self.__dict__.update(kw)


def run(w, req_ids: Optional[Sequence[int]] = None, steps: Optional[int] = None,
        params: Optional[Params] = None, threads: Optional[int] = None, head=None,
        timed_from: int = 0, inv_temp: float = 0.0, exact: bool = False) -> RunResult:
    """Run the oracle decode loop of workload `w` for the given requests.

    The target logits and head proposals come from the host generator of the
    `workload` package (keyed by the original request ids).  `head`, if
    given, replaces the head proposals: a Python callable (b, t, n) -> 7
    tokens (small tests only: it runs under the GIL).  `timed_from`: the
    first step counted in method_s / provider_s (per-thread sums); method_s
    splits into lookup_s (suffix search + copy), sched_fuse_s (scheduler +
    fusion) and verify_s (argmax or draw + accepted prefix), the small rest
    being the history append and bookkeeping.
    `inv_temp` > 0 verifies by sampling (point-mass drafts) at that inverse
    temperature with the generator's uniforms; the records' `g` then holds
    each step's emitted tokens instead of the argmax rows.  `exact` samples
    on the fixed-point weights (sample_verify_exact)."""
    import workload as wl  # the seeded input generator shared by both sides

    p = params or Params.default()
    req_ids = list(range(w.B)) if req_ids is None else [int(r) for r in req_ids]
    steps = w.steps if steps is None else int(steps)
    threads = threads or min(len(req_ids), os.cpu_count() or 1)
    n = len(req_ids)
    gen = wl.HostGen(w)
    prompts = [w.prompts[r] for r in req_ids]
    ptok, poff = w.csr(prompts)
    caps = np.array([pp.size + BLOCK * steps for pp in prompts], dtype=np.int64)
    hoff = np.zeros(n + 1, np.int64)
    hoff[1:] = np.cumsum(caps)
    hist = np.zeros(int(hoff[-1]), np.int32)
    hlen = np.zeros(n, np.int64)
    ids = np.array(req_ids, np.int32)
    rec = {k: np.zeros((steps, n), np.int32) for k in ("k", "j", "L", "a")}
    rec.update({k: np.zeros((steps, n, BLOCK), np.int32) for k in ("c", "blk", "g")})
    counters = (Counters * n)()
    args = RunArgs()
    args.params = ctypes.cast(ctypes.pointer(p), _P)
    args.n_req = n
    args.req_ids = ids.ctypes.data
    args.prompt = ptok.ctypes.data
    args.prompt_off = poff.ctypes.data
    args.steps = steps
    args.V = w.V
    args.dtype = w.dtype
    args.threads = threads
    args.gen_ctx = gen.ctx_ptr
    args.logits_fn = gen.logits_fn
    args.head_fn = gen.head_fn
    args.uniform_fn = gen.uniform_fn
    args.inv_temp = float(inv_temp)
    args.exact = 1 if exact else 0
    if head is not None:
        proto = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                 ctypes.POINTER(ctypes.c_int32))

        def _cb(_ctx, b, t, n, out):
            vals = list(head(int(b), int(t), int(n)))
            for i in range(7):
                out[i] = int(vals[i])

        head_cb = proto(_cb)
        args.head_fn = ctypes.cast(head_cb, _P).value
    for k in ("k", "j", "L", "a", "c", "blk", "g"):
        setattr(args, "rec_" + k, rec[k].ctypes.data)
    args.hist_out = hist.ctypes.data
    args.hist_off = hoff.ctypes.data
    args.hist_len = hlen.ctypes.data
    args.counters = ctypes.cast(counters, _P)
    args.timed_from = int(timed_from)
    import time as _time
    t0 = _time.perf_counter()
    rc = _lib().or_run(ctypes.byref(args))
    wall = _time.perf_counter() - t0
    if rc != 0:
        raise RuntimeError(f"oracle run failed ({rc})")
    histories = [hist[hoff[i]:hoff[i] + hlen[i]].copy() for i in range(n)]
    return RunResult(req_ids=req_ids, steps=steps, threads=threads, histories=histories,
                     counters=[counters[i].as_dict() for i in range(n)],
                     method_s=args.method_ns * 1e-9, provider_s=args.provider_ns * 1e-9, wall_s=wall,
                     lookup_s=args.lookup_ns * 1e-9, sched_fuse_s=args.sched_fuse_ns * 1e-9,
                     verify_s=args.verify_ns * 1e-9, **rec)
