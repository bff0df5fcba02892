"""Seeded synthetic workloads for the context-lookup speculative decoding step.

This module builds the inputs that both the CUDA path and the CPU oracle
consume, and nothing else: it holds none of the method's arithmetic.

* Host arrays (numpy, seeded PCG64 per request): each request's prompt and its
  hidden ground-truth continuation, concatenated into one token *stream*.
* Per-step inputs, a pure function of (seed, request, absolute position) or
  (seed, request, step): the target logits of each verify row and the draft
  model's 7 head proposals.  Their rules live in ``gen_rules.h`` and are
  evaluated by a host library (``libclkgen_host.so``, handed to the oracle as
  callbacks) and a device library (``libclkgen_dev.so``, used by the GPU
  tests and the benchmark).  The two are cross-checked bit for bit.

The five workloads follow the pages' use cases (HyperQwen context-lookup
article, "先看效果" and "代价与适用场景": verbatim restatement of a long
document, mixed copy/chat serving batches, list-marker and indentation
repeats) at the sizes fixed for this hot path.  Every recipe choice that the
sizes leave open is documented on the builder that makes it.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import statistics
from functools import lru_cache
from typing import List, Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
HEAD = 7          # draft-model head proposals per step
ROWS = 16         # verify block width (1 committed token + 15 drafts)
BF16, F32 = 0, 1  # dtype codes shared with gen_host.c / gen_device.cu


# ---------------------------------------------------------------------------
# Value tables
# ---------------------------------------------------------------------------
@lru_cache(maxsize=None)
def normal_quantiles() -> np.ndarray:
    """Q[i] = inverse N(0,1) CDF at (i + 1/2) / 65536, in float64.

    Uses the standard library's NormalDist.inv_cdf (Wichura's AS241)."""
    nd = statistics.NormalDist()
    return np.array([nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)], dtype=np.float64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even), as uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


@lru_cache(maxsize=None)
def value_tables(dtype: int):
    """(T0, T8): the noise table and the boosted (+8) table in the stored type.

    bf16 entries are float32(Q) (resp. float32(Q + 8)) rounded to bf16."""
    q = normal_quantiles()
    if dtype == BF16:
        return (f32_to_bf16_bits(q.astype(np.float32)),
                f32_to_bf16_bits((q + 8.0).astype(np.float32)))
    return q.astype(np.float32), (q + 8.0).astype(np.float32)


# ---------------------------------------------------------------------------
# Token distributions
# ---------------------------------------------------------------------------
@lru_cache(maxsize=None)
def _zipf_cdf(V: int, s: float) -> np.ndarray:
    w = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    c = np.cumsum(w)
    return c / c[-1]


def zipf(rng: np.random.Generator, V: int, size: int, s: float = 1.1) -> np.ndarray:
    """Zipf(s) over a vocabulary of V: token id = rank - 1, by inverse CDF."""
    u = rng.random(size)
    t = np.searchsorted(_zipf_cdf(V, s), u, side="right")
    return np.minimum(t, V - 1).astype(np.int32)


def _substitute(rng, seg: np.ndarray, p: float, V: int) -> np.ndarray:
    if p <= 0.0:
        return seg
    seg = seg.copy()
    mask = rng.random(seg.size) < p
    seg[mask] = rng.integers(0, V, size=int(mask.sum()), dtype=np.int64).astype(np.int32)
    return seg


# ---------------------------------------------------------------------------
# Workload description
# ---------------------------------------------------------------------------
@dataclasses.dataclass
class Workload:
    """A batch of requests: prompt + hidden continuation per request."""

    name: str
    seed: int
    V: int
    dtype: int
    steps: int
    prompts: List[np.ndarray]
    streams: List[np.ndarray]  # prompt followed by the ground-truth continuation
    kinds: List[str]

    @property
    def B(self) -> int:
        return len(self.prompts)

    @property
    def n0(self) -> np.ndarray:
        return np.array([p.size for p in self.prompts], dtype=np.int64)

    @property
    def max_hist(self) -> int:
        """History capacity that holds the prompt plus every step's emitted tokens."""
        return int(self.n0.max()) + ROWS * self.steps

    def csr(self, arrays) -> tuple:
        off = np.zeros(len(arrays) + 1, dtype=np.int64)
        off[1:] = np.cumsum([a.size for a in arrays])
        tok = np.concatenate(arrays).astype(np.int32) if arrays else np.zeros(0, np.int32)
        return np.ascontiguousarray(tok), off

    def prompt_csr(self):
        return self.csr(self.prompts)

    def stream_csr(self):
        return self.csr(self.streams)

    def subset(self, idx) -> "Workload":
        """The same requests' data, reindexed 0..len(idx)-1 (the per-step draws
        are keyed by request index, so a subset is a different workload)."""
        idx = list(idx)
        return dataclasses.replace(self, name=f"{self.name}[sub]",
                                   prompts=[self.prompts[i] for i in idx],
                                   streams=[self.streams[i] for i in idx],
                                   kinds=[self.kinds[i] for i in idx])

    def with_steps(self, steps: int) -> "Workload":
        assert steps <= self.steps
        return dataclasses.replace(self, steps=steps)

    def verify_bytes_per_row(self) -> int:
        return self.V * (2 if self.dtype == BF16 else 4)


def _need(n0: int, steps: int) -> int:
    # rows read at most positions n + 15 with n <= n0 + 16*steps; head reads n + 6.
    return n0 + ROWS * steps + ROWS + 16


def _copy_heavy_stream(rng, prompt, V, steps, span_lo, span_hi, subst):
    """Continuation = back-to-back copies of random prompt spans of U{lo..hi}
    tokens, each token substituted by a uniform one with probability `subst`."""
    n0 = prompt.size
    need = _need(n0, steps)
    parts = [prompt]
    total = n0
    while total < need:
        span = int(rng.integers(span_lo, span_hi + 1))
        span = min(span, n0)
        src = int(rng.integers(0, n0 - span + 1))
        seg = _substitute(rng, prompt[src:src + span], subst, V)
        parts.append(seg)
        total += seg.size
    return np.concatenate(parts).astype(np.int32)


def _chat_stream(rng, prompt, V, steps, copy_p=0.03, lo=4, hi=10):
    """Continuation = fresh Zipf(1.1) tokens; at each position, with
    probability `copy_p`, a U{lo..hi}-token copy of an earlier span of the
    history (prompt and continuation so far, wholly before the position) starts."""
    n0 = prompt.size
    need = _need(n0, steps)
    out = np.empty(need, dtype=np.int32)
    out[:n0] = prompt
    fresh = zipf(rng, V, need - n0)
    starts = rng.random(need - n0)
    q = n0
    i = 0
    while q < need:
        if starts[i] < copy_p:
            ln = int(rng.integers(lo, hi + 1))
            ln = min(ln, need - q)
            src = int(rng.integers(0, q - ln + 1))
            out[q:q + ln] = out[src:src + ln]
            q += ln
            i += ln
        else:
            out[q] = fresh[i]
            q += 1
            i += 1
    return out


def _rng(seed: int, tag: int, b: int) -> np.random.Generator:
    return np.random.default_rng([seed, tag, b])


def _config0(seed: int) -> Workload:
    """B=1, V=1,024, fp32 logits, 2,048-token history, 64 steps.

    Prompt: Zipf(1.1) draws; at each position not inside a copy, with
    probability 0.3 / (0.7 * 40) a copy of a U{16..64}-token span lying wholly
    before the position starts (mean span 40, so about 30% of positions are
    copies).  Continuation: back-to-back 64-token prompt-span copies with 5%
    uniform substitution (the first is the specified hidden continuation,
    the rest keep the request stationary for the whole run)."""
    V, L, steps = 1024, 2048, 64
    rng = _rng(seed, 0, 0)
    p_start = 0.3 / (0.7 * 40.0)
    h = np.empty(L, dtype=np.int32)
    fresh = zipf(rng, V, L)
    q = 0
    while q < L:
        if rng.random() < p_start:
            ln = int(rng.integers(16, 65))
            if ln <= q:
                src = int(rng.integers(0, q - ln + 1))
                ln = min(ln, L - q)
                h[q:q + ln] = h[src:src + ln]
                q += ln
                continue
        h[q] = fresh[q]
        q += 1
    stream = _copy_heavy_stream(rng, h, V, steps, 64, 64, 0.05)
    return Workload("cfg0-tiny", seed, V, F32, steps, [h], [stream], ["copy"])


def _config1(seed: int) -> Workload:
    """B=1, V=248,320, 25,000-token Zipf(1.1) prompt, 2,000 steps; the
    continuation is back-to-back verbatim copies of 4,000-token prompt spans."""
    V, L, steps = 248320, 25000, 2000
    rng = _rng(seed, 1, 0)
    p = zipf(rng, V, L)
    stream = _copy_heavy_stream(rng, p, V, steps, 4000, 4000, 0.0)
    return Workload("cfg1-restate-25k", seed, V, BF16, steps, [p], [stream], ["copy"])


def _mixed(seed: int, tag: int, B: int, V: int, steps: int, lens, copy_span, subst, copy_frac=0.5,
           name="mixed") -> Workload:
    prompts, streams, kinds = [], [], []
    n_copy = int(round(B * copy_frac))
    for b in range(B):
        rng = _rng(seed, tag, b)
        L = int(lens(rng))
        p = zipf(rng, V, L)
        if b < n_copy:
            s = _copy_heavy_stream(rng, p, V, steps, copy_span[0], copy_span[1], subst)
            kinds.append("copy")
        else:
            s = _chat_stream(rng, p, V, steps)
            kinds.append("chat")
        prompts.append(p)
        streams.append(s)
    return Workload(name, seed, V, BF16, steps, prompts, streams, kinds)


def _config2(seed: int) -> Workload:
    """B=64 mixed serving batch, V=248,320, 512 steps.  Prompt lengths
    U{2,000..32,000} (read as decimal thousands), Zipf(1.1) prompts.  Requests
    0..31 are copy-heavy (U{50..2,000}-token prompt-span copies, 2% per-token
    substitution); 32..63 are chat-like (fresh Zipf with 3% short copies)."""
    return _mixed(seed, 2, 64, 248320, 512, lambda r: r.integers(2000, 32001), (50, 2000), 0.02,
                  name="cfg2-mixed-b64")


def _config3(seed: int) -> Workload:
    """B=16, V=32,000, L=8,192, 1,024 steps.  Per request a period p ~ U{3..40}
    and a pattern of p uniform tokens; every position of prompt and
    continuation is pattern[q mod p], replaced by a uniform token with
    probability 5%."""
    V, L, steps, B = 32000, 8192, 1024, 16
    prompts, streams = [], []
    for b in range(B):
        rng = _rng(seed, 3, b)
        p = int(rng.integers(3, 41))
        pat = rng.integers(0, V, size=p, dtype=np.int64).astype(np.int32)
        n = _need(L, steps)
        s = pat[np.arange(n) % p]
        s = _substitute(rng, s, 0.05, V)
        prompts.append(s[:L].copy())
        streams.append(s.astype(np.int32))
    return Workload("cfg3-periodic", seed, V, BF16, steps, prompts, streams, ["periodic"] * B)


def _config4a(seed: int) -> Workload:
    """B=8, L=262,144, V=248,320, 256 steps, copy-heavy with U{1,000..8,000}
    spans and 2% substitution."""
    return _mixed(seed, 40, 8, 248320, 256, lambda r: 262144, (1000, 8000), 0.02, copy_frac=1.0,
                  name="cfg4a-long-262k")


def _config4b(seed: int) -> Workload:
    """B=256, L=4,096, V=248,320, 256 steps, copy-heavy as the mixed batch
    (U{50..2,000} spans, 2% substitution)."""
    return _mixed(seed, 41, 256, 248320, 256, lambda r: 4096, (50, 2000), 0.02, copy_frac=1.0,
                  name="cfg4b-b256")


BUILDERS = {"0": _config0, "1": _config1, "2": _config2, "3": _config3, "4a": _config4a, "4b": _config4b}
DEFAULT_SEED = {"0": 0, "1": 1, "2": 2, "3": 3, "4a": 4, "4b": 4}


def make(cfg: str, seed: Optional[int] = None) -> Workload:
    """Build one of the named workloads ("0", "1", "2", "3", "4a", "4b")."""
    cfg = str(cfg)
    return BUILDERS[cfg](DEFAULT_SEED[cfg] if seed is None else seed)


def make_small(kind: str, seed: int, B: int = 4, V: int = 4096, L=(200, 2000), steps: int = 48,
               dtype: int = BF16) -> Workload:
    """Scaled-down variants of the recipes above, for fast tests.

    kind: "mixed" (half copy-heavy, half chat-like), "copy", "chat" or "periodic"."""
    if kind == "periodic":
        prompts, streams = [], []
        for b in range(B):
            rng = _rng(seed, 90, b)
            p = int(rng.integers(3, 41))
            Lb = int(rng.integers(L[0], L[1] + 1))
            pat = rng.integers(0, V, size=p, dtype=np.int64).astype(np.int32)
            n = _need(Lb, steps)
            s = _substitute(rng, pat[np.arange(n) % p], 0.05, V)
            prompts.append(s[:Lb].copy())
            streams.append(s.astype(np.int32))
        return Workload(f"small-periodic-{seed}", seed, V, dtype, steps, prompts, streams, ["periodic"] * B)
    frac = {"mixed": 0.5, "copy": 1.0, "chat": 0.0}[kind]
    w = _mixed(seed, 91, B, V, steps, lambda r: r.integers(L[0], L[1] + 1), (50, 400), 0.02,
               copy_frac=frac, name=f"small-{kind}-{seed}")
    w.dtype = dtype
    return w


# ---------------------------------------------------------------------------
# Native generator libraries
# ---------------------------------------------------------------------------
class HostCtx(ctypes.Structure):
    _fields_ = [("seed", ctypes.c_uint64), ("V", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("B", ctypes.c_int32), ("pad", ctypes.c_int32),
                ("stream", ctypes.c_void_p), ("stream_off", ctypes.c_void_p),
                ("t0_bf16", ctypes.c_void_p), ("t8_bf16", ctypes.c_void_p),
                ("t0_f32", ctypes.c_void_p), ("t8_f32", ctypes.c_void_p)]


DevCtx = HostCtx  # same field layout; the device context carries device pointers


def _load(name: str) -> ctypes.CDLL:
    path = os.path.join(HERE, name)
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run __graft_entry__.build() first")
    return ctypes.CDLL(path)


@lru_cache(maxsize=None)
def host_lib() -> ctypes.CDLL:
    lib = _load("libclkgen_host.so")
    lib.wl_logits_row.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p]
    lib.wl_logits_row.restype = None
    lib.wl_logits_block.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                    ctypes.c_void_p]
    lib.wl_logits_block.restype = None
    lib.wl_head.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p]
    lib.wl_head.restype = None
    lib.wl_truth.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64]
    lib.wl_truth.restype = ctypes.c_int32
    lib.wl_uniforms.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]
    lib.wl_uniforms.restype = None
    return lib


class HostGen:
    """Host-side per-step inputs of a workload (keeps its arrays alive)."""

    def __init__(self, w: Workload):
        self.w = w
        self.tok, self.off = w.stream_csr()
        t0b, t8b = value_tables(BF16)
        t0f, t8f = value_tables(F32)
        self._keep = [self.tok, self.off, t0b, t8b, t0f, t8f]
        self.ctx = HostCtx(w.seed, w.V, w.dtype, w.B, 0, self.tok.ctypes.data, self.off.ctypes.data,
                           t0b.ctypes.data, t8b.ctypes.data, t0f.ctypes.data, t8f.ctypes.data)
        self.lib = host_lib()

    @property
    def ctx_ptr(self) -> int:
        return ctypes.addressof(self.ctx)

    @property
    def logits_fn(self) -> int:
        return ctypes.cast(self.lib.wl_logits_row, ctypes.c_void_p).value

    @property
    def head_fn(self) -> int:
        return ctypes.cast(self.lib.wl_head, ctypes.c_void_p).value

    @property
    def uniform_fn(self) -> int:
        return ctypes.cast(self.lib.wl_uniforms, ctypes.c_void_p).value

    def uniforms(self, b: int, t: int) -> np.ndarray:
        """Step t's sampling uniforms of request b, float32 [16, 2]."""
        out = np.empty((ROWS, 2), dtype=np.float32)
        self.lib.wl_uniforms(self.ctx_ptr, b, t, out.ctypes.data)
        return out

    def np_dtype(self):
        return np.uint16 if self.w.dtype == BF16 else np.float32

    def logits_rows(self, b: int, P0: int, rows: int) -> np.ndarray:
        out = np.empty((rows, self.w.V), dtype=self.np_dtype())
        self.lib.wl_logits_block(self.ctx_ptr, b, P0, rows, out.ctypes.data)
        return out

    def head(self, b: int, t: int, n: int) -> np.ndarray:
        out = np.empty(HEAD, dtype=np.int32)
        self.lib.wl_head(self.ctx_ptr, b, t, n, out.ctypes.data)
        return out

    def truth(self, b: int, P: int) -> int:
        return int(self.lib.wl_truth(self.ctx_ptr, b, P))


@lru_cache(maxsize=None)
def dev_lib() -> ctypes.CDLL:
    lib = _load("libclkgen_dev.so")
    lib.wl_dev_logits.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                  ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p]
    lib.wl_dev_head.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                ctypes.c_void_p]
    lib.wl_dev_advance.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p]
    lib.wl_dev_uniforms.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    for f in (lib.wl_dev_logits, lib.wl_dev_head, lib.wl_dev_advance, lib.wl_dev_uniforms):
        f.restype = ctypes.c_int
    return lib


class DevGen:
    """Device-side per-step inputs of a workload (torch tensors on `device`).

    Keeps its own position array pos[B] (int64): the history length of every
    request, which starts at the prompt length and advances by the emitted
    count each step (``advance``)."""

    def __init__(self, w: Workload, device="cuda"):
        import torch
        self.torch = torch
        self.w = w
        tok, off = w.stream_csr()
        t0b, t8b = value_tables(BF16)
        t0f, t8f = value_tables(F32)
        self.d = {
            "tok": torch.from_numpy(tok).to(device),
            "off": torch.from_numpy(off).to(device),
            "t0b": torch.from_numpy(t0b.view(np.int16)).to(device),
            "t8b": torch.from_numpy(t8b.view(np.int16)).to(device),
            "t0f": torch.from_numpy(t0f).to(device),
            "t8f": torch.from_numpy(t8f).to(device),
        }
        d = self.d
        self.ctx = DevCtx(w.seed, w.V, w.dtype, w.B, 0, d["tok"].data_ptr(), d["off"].data_ptr(),
                          d["t0b"].data_ptr(), d["t8b"].data_ptr(), d["t0f"].data_ptr(), d["t8f"].data_ptr())
        self.pos = torch.from_numpy(w.n0.copy()).to(device)
        self.lib = dev_lib()
        self.device = device

    def torch_dtype(self):
        return self.torch.bfloat16 if self.w.dtype == BF16 else self.torch.float32

    def alloc_logits(self, rows: int = ROWS):
        return self.torch.empty((self.w.B, rows, self.w.V), dtype=self.torch_dtype(), device=self.device)

    def _stream(self):
        return self.torch.cuda.current_stream().cuda_stream

    def logits(self, out, pos=None):
        """Fill out[B, rows, V] for positions pos[b] + r (default: own pos)."""
        pos = self.pos if pos is None else pos
        if out.dim() != 3 or out.shape[0] != self.w.B or out.shape[2] != self.w.V or out.shape[1] > ROWS \
                or out.stride(2) != 1 or out.dtype != self.torch_dtype() or not out.is_cuda:
            raise ValueError(f"logits buffer must be [{self.w.B}, <=16, {self.w.V}] {self.torch_dtype()} on the GPU")
        if pos.shape != (self.w.B,) or pos.dtype != self.torch.int64:
            raise ValueError("pos must be int64 [B]")
        rc = self.lib.wl_dev_logits(ctypes.addressof(self.ctx), pos.data_ptr(), out.data_ptr(),
                                    out.stride(1), out.stride(0), out.shape[1], self._stream())
        if rc != 0:
            raise RuntimeError(f"wl_dev_logits failed ({rc})")
        return out

    def head(self, t: int, out, pos=None):
        """Fill out[B, 7] (contiguous int32) with step t's head proposals."""
        pos = self.pos if pos is None else pos
        if tuple(out.shape) != (self.w.B, HEAD) or out.dtype != self.torch.int32 or not out.is_contiguous() \
                or not out.is_cuda:
            raise ValueError(f"head buffer must be contiguous int32 [{self.w.B}, {HEAD}] on the GPU")
        if pos.shape != (self.w.B,) or pos.dtype != self.torch.int64:
            raise ValueError("pos must be int64 [B]")
        rc = self.lib.wl_dev_head(ctypes.addressof(self.ctx), pos.data_ptr(), t, out.data_ptr(), self._stream())
        if rc != 0:
            raise RuntimeError(f"wl_dev_head failed ({rc})")
        return out

    def uniforms(self, t: int, out):
        """Fill out[B, 16, 2] (contiguous float32) with step t's sampling uniforms."""
        if tuple(out.shape) != (self.w.B, ROWS, 2) or out.dtype != self.torch.float32 or not out.is_contiguous() \
                or not out.is_cuda:
            raise ValueError(f"uniform buffer must be contiguous float32 [{self.w.B}, {ROWS}, 2] on the GPU")
        rc = self.lib.wl_dev_uniforms(ctypes.addressof(self.ctx), t, out.data_ptr(), self._stream())
        if rc != 0:
            raise RuntimeError(f"wl_dev_uniforms failed ({rc})")
        return out

    def advance(self, emitted):
        if emitted.shape != (self.w.B,) or emitted.dtype != self.torch.int32 or not emitted.is_contiguous():
            raise ValueError("emitted must be contiguous int32 [B]")
        rc = self.lib.wl_dev_advance(self.pos.data_ptr(), emitted.data_ptr(), self.w.B, self._stream())
        if rc != 0:
            raise RuntimeError(f"wl_dev_advance failed ({rc})")

    def reset(self):
        self.pos.copy_(self.torch.from_numpy(self.w.n0.copy()))
