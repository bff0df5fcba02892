"""GB300 (sm_103a) hot path of context-lookup speculative decoding.

A thin ctypes binding over ``libclk.so`` (C ABI in ``include/clk.h``).  Every
step of the path runs in the library's CUDA kernels; this module only checks
tensors and passes their device pointers and the current CUDA stream.  There
is no fallback: if the library is missing, importing the binding's functions
raises.

Per decode step (HyperQwen context-lookup article, "lookup 草稿的原理：三步走"):

    lookup_propose    Step 1: longest 4..12 suffix match, most recent, LZ77 copy
    sched_step        Step 3: long-block scheduler (enter after 2, sticky 3)
    fuse              Step 2: head / tail fusion rule
    verify_greedy     greedy verification: argmax rows + accepted prefix
    lookup_append     commit the emitted tokens (incremental index update)

plus the fused launches ``propose_fuse_sched`` and ``verify_append`` that the
``Step`` driver uses (two kernels per step).
"""
from __future__ import annotations

import ctypes
import os
from functools import lru_cache
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libclk.so")

OK, EINVAL, ECAPACITY, ECUDA, ENOTIMPL, ESTATE = 0, -1, -2, -3, -4, -5
BF16, F32 = 0, 1
SENT = -1
BLOCK = 16
MAX_BATCH = 8192

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64


class ClkError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {code} ({status_string(code)})")
        self.code = code


class Params(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "min_k", "max_k", "head", "tail", "head_replace_k", "head_agree_k", "head_agree_n", "tail_k",
        "enter_streak", "sticky", "near_full_slack")]

    @classmethod
    def default(cls, **kw) -> "Params":
        p = cls()
        lib().clk_params_default(ctypes.byref(p))
        for k, v in kw.items():
            setattr(p, k, v)
        return p

    @property
    def long_len(self) -> int:
        return 1 + self.head + self.tail

    @property
    def short_len(self) -> int:
        return 1 + self.head


class Counters(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("steps", "hits", "long_steps", "drafted", "accepted", "emitted")] + \
               [("accept_hist", (ctypes.c_int64 * 16) * 2)]

    def as_dict(self):
        d = {n: getattr(self, n) for n in ("steps", "hits", "long_steps", "drafted", "accepted", "emitted")}
        d["accept_hist"] = [[self.accept_hist[i][j] for j in range(16)] for i in range(2)]
        return d


class SlotInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("n", "mode", "streak", "miss", "has_prev", "cur_len", "n_indexed")]


# (name, restype, argtypes) of every exported entry point
_SIGS = [
    ("clk_params_default", None, [_P]),
    ("clk_params_check", ctypes.c_int, [_P]),
    ("clk_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("clk_lookup_workspace_bytes", ctypes.c_int, [_P, _I32, _I64, ctypes.POINTER(ctypes.c_size_t)]),
    ("clk_lookup_create", ctypes.c_int, [ctypes.POINTER(_P), _P, _I32, _I64, _I32, _P, ctypes.c_size_t]),
    ("clk_lookup_reset", ctypes.c_int, [_P, _P]),
    ("clk_lookup_set_alone", ctypes.c_int, [_P, _I32]),
    ("clk_lookup_init", ctypes.c_int, [_P, _P, _I32, _P, _P, _P]),
    ("clk_lookup_append", ctypes.c_int, [_P, _P, _I32, _P, _P, _P]),
    ("clk_lookup_propose", ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P]),
    ("clk_lookup_propose_scan", ctypes.c_int, [_P, _P, _I32, _I32, _P, _P, _P, _P]),
    ("clk_sched_step", ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _P]),
    ("clk_fuse", ctypes.c_int, [_P, _I32, _P, _P, _P, _P, _P, _P, _P]),
    ("clk_fuse_sched", ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P]),
    ("clk_propose_fuse_sched", ctypes.c_int, [_P, _P, _I32, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    ("clk_verify_scratch_bytes", ctypes.c_int, [_I32, ctypes.POINTER(ctypes.c_size_t)]),
    ("clk_verify_scratch_init", ctypes.c_int, [_P, ctypes.c_size_t, _P]),
    ("clk_verify_greedy", ctypes.c_int, [_P, _I32, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P, _P,
                                         ctypes.c_size_t, _P]),
    ("clk_verify_greedy_static", ctypes.c_int, [_P, _I32, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P, _P]),
    ("clk_verify_append", ctypes.c_int, [_P, _P, _P, _I32, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P, _P,
                                         _P]),
    ("clk_verify_sample_scratch_bytes", ctypes.c_int, [_I32, _I32, _I32, ctypes.POINTER(ctypes.c_size_t)]),
    ("clk_verify_sample", ctypes.c_int, [_P, _I32, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                                         ctypes.c_size_t, _P]),
    ("clk_verify_sample_exact_scratch_bytes", ctypes.c_int, [_I32, _I32, _I32, ctypes.POINTER(ctypes.c_size_t)]),
    ("clk_verify_sample_exact", ctypes.c_int, [_P, _I32, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                                               ctypes.c_size_t, _P]),
    ("clk_verify_sample_append", ctypes.c_int, [_P, _P, _P, _I32, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P,
                                                _P, _P, _P, ctypes.c_size_t, _P]),
    ("clk_verify_sample_exact_append", ctypes.c_int, [_P, _P, _P, _I32, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P,
                                                      _P, _P, _P, _P, ctypes.c_size_t, _P]),
    ("clk_status", ctypes.c_int, [_P, ctypes.POINTER(_I32), ctypes.POINTER(_I32), _P]),
    ("clk_status_clear", ctypes.c_int, [_P, _P]),
    ("clk_read_counters", ctypes.c_int, [_P, _I32, _P, _P]),
    ("clk_read_slot_info", ctypes.c_int, [_P, _I32, _P, _P]),
    ("clk_lookup_read_history", ctypes.c_int, [_P, _I32, _P, _I64, ctypes.POINTER(_I64), _P]),
    ("clk_lookup_restore_state", ctypes.c_int, [_P, _I32, _P, _P, _P]),
    ("clk_lookup_destroy", None, [_P]),
]


@lru_cache(maxsize=None)
def lib() -> ctypes.CDLL:
    """The loaded libclk.so; raises if it has not been built."""
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    for name, res, args in _SIGS:
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


def status_string(code: int) -> str:
    return lib().clk_status_string(code).decode()


def _check(fn: str, rc: int):
    if rc != OK:
        raise ClkError(fn, rc)


def _stream(stream=None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor], dtype=torch.int32, shape=None, name="tensor") -> int:
    if t is None:
        return 0
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _logits_args(logits: torch.Tensor):
    # a CUDA tensor, or a pinned host tensor that the kernels read in place
    if not (logits.is_cuda or logits.is_pinned()) or logits.dim() != 3:
        raise ValueError("logits must be a CUDA tensor or a pinned host tensor [B, rows, V]")
    if logits.dtype == torch.bfloat16:
        dt = BF16
    elif logits.dtype == torch.float32:
        dt = F32
    else:
        raise ValueError("logits must be bfloat16 or float32")
    if logits.stride(2) != 1:
        raise ValueError("logits rows must be contiguous")
    return dt, logits.stride(1), logits.stride(0), logits.shape[2]


class Lookup:
    """Histories, k-gram index and scheduler state of up to `max_slots` requests.

    Owns its device workspace (a torch uint8 tensor) and the C handle."""

    def __init__(self, max_slots: int, max_hist: int, vocab: int = 0, params: Optional[Params] = None,
                 device="cuda", stream=None):
        self.params = params or Params.default()
        L = lib()
        nbytes = ctypes.c_size_t()
        _check("clk_lookup_workspace_bytes",
               L.clk_lookup_workspace_bytes(ctypes.byref(self.params), max_slots, max_hist, ctypes.byref(nbytes)))
        self.workspace_bytes = nbytes.value
        # 256-byte alignment: torch's caching allocator returns 512-byte aligned blocks.
        self.workspace = torch.empty(self.workspace_bytes, dtype=torch.uint8, device=device)
        h = _P()
        _check("clk_lookup_create", L.clk_lookup_create(ctypes.byref(h), ctypes.byref(self.params), max_slots,
                                                        max_hist, vocab, self.workspace.data_ptr(),
                                                        self.workspace_bytes))
        self.handle = h
        self.max_slots, self.max_hist, self.vocab = max_slots, max_hist, vocab
        _check("clk_lookup_reset", L.clk_lookup_reset(self.handle, _stream(stream)))

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            try:
                lib().clk_lookup_destroy(h)
            except Exception:
                pass
            self.handle = None

    def set_alone(self, alone: bool):
        """clk_lookup_set_alone: True when the fused verify calls are launched
        with nothing to overlap (timing only; results are the same)."""
        _check("clk_lookup_set_alone", lib().clk_lookup_set_alone(self.handle, 1 if alone else 0))

    # -- inspection (synchronising) -------------------------------------
    def status(self, stream=None):
        st, det = _I32(), _I32()
        _check("clk_status", lib().clk_status(self.handle, ctypes.byref(st), ctypes.byref(det), _stream(stream)))
        return st.value, det.value

    def status_clear(self, stream=None):
        _check("clk_status_clear", lib().clk_status_clear(self.handle, _stream(stream)))

    def counters(self, slot: int = -1, stream=None) -> dict:
        c = Counters()
        _check("clk_read_counters", lib().clk_read_counters(self.handle, slot, ctypes.byref(c), _stream(stream)))
        return c.as_dict()

    def slot_info(self, slot: int, stream=None) -> dict:
        s = SlotInfo()
        _check("clk_read_slot_info", lib().clk_read_slot_info(self.handle, slot, ctypes.byref(s), _stream(stream)))
        return {n: getattr(s, n) for n, _ in SlotInfo._fields_}

    def history(self, slot: int, stream=None):
        import numpy as np
        n = _I64()
        _check("clk_lookup_read_history",
               lib().clk_lookup_read_history(self.handle, slot, None, 0, ctypes.byref(n), _stream(stream)))
        out = np.empty(n.value, dtype=np.int32)
        _check("clk_lookup_read_history",
               lib().clk_lookup_read_history(self.handle, slot, out.ctypes.data, n.value, ctypes.byref(n),
                                             _stream(stream)))
        return out

    # -- checkpoint / resume ----------------------------------------------
    def snapshot(self, slot: int, stream=None) -> dict:
        """Everything needed to resume request `slot` elsewhere: its history,
        scheduler state and counters (host copies; synchronising)."""
        return {"history": self.history(slot, stream), "info": self.slot_info(slot, stream),
                "counters": self.counters(slot, stream)}

    def restore(self, slot: int, snap: dict, stream=None):
        """Resume a snapshot in `slot` of this lookup (same parameters): the
        history is ingested again (which rebuilds its index), then the
        scheduler state and counters are written back (synchronising)."""
        import numpy as np
        dev = self.workspace.device
        hist = np.ascontiguousarray(snap["history"], dtype=np.int32)
        s = torch.tensor([slot], dtype=torch.int32, device=dev)
        off = torch.tensor([0, hist.size], dtype=torch.int64, device=dev)
        lookup_init(self, s, torch.from_numpy(hist).to(dev), off, stream=stream)
        info = SlotInfo(**{n: int(snap["info"][n]) for n, _ in SlotInfo._fields_})
        c = Counters(**{n: int(snap["counters"][n]) for n in
                        ("steps", "hits", "long_steps", "drafted", "accepted", "emitted")})
        for i in range(2):
            for j in range(16):
                c.accept_hist[i][j] = int(snap["counters"]["accept_hist"][i][j])
        _check("clk_lookup_restore_state",
               lib().clk_lookup_restore_state(self.handle, slot, ctypes.byref(info), ctypes.byref(c),
                                              _stream(stream)))


# ---------------------------------------------------------------------------
# Entry points (same names as the C ABI without the clk_ prefix)
# ---------------------------------------------------------------------------
def lookup_init(h: Lookup, slots, prompt, prompt_off, stream=None):
    B = slots.numel()
    _check("clk_lookup_init", lib().clk_lookup_init(h.handle, _ptr(slots, name="slots"), B,
                                                    _ptr(prompt, name="prompt"),
                                                    _ptr(prompt_off, torch.int64, (B + 1,), "prompt_off"),
                                                    _stream(stream)))


def lookup_append(h: Lookup, slots, tok, count, stream=None):
    B = slots.numel()
    _check("clk_lookup_append", lib().clk_lookup_append(h.handle, _ptr(slots, name="slots"), B,
                                                        _ptr(tok, shape=(B, BLOCK), name="tok"),
                                                        _ptr(count, shape=(B,), name="count"), _stream(stream)))


def lookup_propose(h: Lookup, slots, draft, k, j, stream=None):
    B = slots.numel()
    _check("clk_lookup_propose", lib().clk_lookup_propose(h.handle, _ptr(slots, name="slots"), B,
                                                          _ptr(draft, shape=(B, BLOCK), name="draft"),
                                                          _ptr(k, shape=(B,), name="k"), _ptr(j, shape=(B,), name="j"),
                                                          _stream(stream)))


def lookup_propose_scan(h: Lookup, slots, draft, k, j, stream=None, ctas_per_request: int = 0):
    """The proposal by a full history scan (clk_lookup_propose_scan);
    ctas_per_request=1 is the pages' one-program-per-request form."""
    B = slots.numel()
    _check("clk_lookup_propose_scan",
           lib().clk_lookup_propose_scan(h.handle, _ptr(slots, name="slots"), B, int(ctas_per_request),
                                         _ptr(draft, shape=(B, BLOCK)), _ptr(k, shape=(B,)), _ptr(j, shape=(B,)),
                                         _stream(stream)))


def sched_step(h: Lookup, slots, k, prev_accept, prev_len, length, stream=None):
    B = slots.numel()
    _check("clk_sched_step", lib().clk_sched_step(h.handle, _ptr(slots, name="slots"), B, _ptr(k, shape=(B,)),
                                                  _ptr(prev_accept, shape=(B,)), _ptr(prev_len, shape=(B,)),
                                                  _ptr(length, shape=(B,)), _stream(stream)))


def fuse(params: Params, last_tok, draft, k, head, length, block, stream=None):
    B = last_tok.numel()
    _check("clk_fuse", lib().clk_fuse(ctypes.byref(params), B, _ptr(last_tok, shape=(B,)),
                                      _ptr(draft, shape=(B, BLOCK)), _ptr(k, shape=(B,)),
                                      _ptr(head, shape=(B, params.head)), _ptr(length, shape=(B,)),
                                      _ptr(block, shape=(B, BLOCK)), _stream(stream)))


def fuse_sched(h: Lookup, slots, draft, k, head, prev_accept, prev_len, length, block, stream=None):
    B = slots.numel()
    _check("clk_fuse_sched", lib().clk_fuse_sched(h.handle, _ptr(slots), B, _ptr(draft, shape=(B, BLOCK)),
                                                  _ptr(k, shape=(B,)), _ptr(head, shape=(B, h.params.head)),
                                                  _ptr(prev_accept, shape=(B,)), _ptr(prev_len, shape=(B,)),
                                                  _ptr(length, shape=(B,)), _ptr(block, shape=(B, BLOCK)),
                                                  _stream(stream)))


def propose_fuse_sched(h: Lookup, slots, head, prev_accept, prev_len, draft, k, j, length, block, stream=None):
    B = slots.numel()
    _check("clk_propose_fuse_sched",
           lib().clk_propose_fuse_sched(h.handle, _ptr(slots), B, _ptr(head, shape=(B, h.params.head)),
                                        _ptr(prev_accept, shape=(B,)), _ptr(prev_len, shape=(B,)),
                                        _ptr(draft, shape=(B, BLOCK)), _ptr(k, shape=(B,)), _ptr(j, shape=(B,)),
                                        _ptr(length, shape=(B,)), _ptr(block, shape=(B, BLOCK)), _stream(stream)))


def verify_scratch_bytes(B: int) -> int:
    n = ctypes.c_size_t()
    _check("clk_verify_scratch_bytes", lib().clk_verify_scratch_bytes(B, ctypes.byref(n)))
    return n.value


def verify_scratch(B: int, device="cuda", stream=None) -> torch.Tensor:
    """A zeroed scratch buffer for verify_greedy with up to B requests."""
    t = torch.empty(verify_scratch_bytes(B), dtype=torch.uint8, device=device)
    _check("clk_verify_scratch_init", lib().clk_verify_scratch_init(t.data_ptr(), t.numel(), _stream(stream)))
    return t


def verify_greedy(logits, block, length, argmax, accept, emitted, out_tok, scratch, stream=None):
    dt, rs, qs, V = _logits_args(logits)
    B = block.shape[0]
    _check("clk_verify_greedy",
           lib().clk_verify_greedy(logits.data_ptr(), dt, rs, qs, V, B, _ptr(block, shape=(B, BLOCK)),
                                   _ptr(length, shape=(B,)), _ptr(argmax, shape=(B, BLOCK)),
                                   _ptr(accept, shape=(B,)), _ptr(emitted, shape=(B,)),
                                   _ptr(out_tok, shape=(B, BLOCK)), _ptr(scratch, torch.uint8, name="scratch"),
                                   scratch.numel(), _stream(stream)))


def verify_greedy_static(logits, block, length, argmax, accept, emitted, out_tok, stream=None):
    """verify_greedy with the library's own fixed scratch (no buffer from the
    caller, nothing allocated); B <= 1024; calls must not overlap on the GPU."""
    dt, rs, qs, V = _logits_args(logits)
    B = block.shape[0]
    _check("clk_verify_greedy_static",
           lib().clk_verify_greedy_static(logits.data_ptr(), dt, rs, qs, V, B, _ptr(block, shape=(B, BLOCK)),
                                          _ptr(length, shape=(B,)), _ptr(argmax, shape=(B, BLOCK)),
                                          _ptr(accept, shape=(B,)), _ptr(emitted, shape=(B,)),
                                          _ptr(out_tok, shape=(B, BLOCK)), _stream(stream)))


def verify_sample_scratch(logits_dtype, V: int, B: int, device="cuda", stream=None, halves: int = 1) -> torch.Tensor:
    """A zeroed scratch buffer for verify_sample with vocabulary V and up to
    B requests (logits_dtype: torch.bfloat16 or torch.float32).  halves=2:
    two halves (each the needed size rounded up to 256 bytes), which
    verify_sample_append alternates so that a call may start while the
    previous one finishes."""
    dt = BF16 if logits_dtype == torch.bfloat16 else F32
    n = ctypes.c_size_t()
    _check("clk_verify_sample_scratch_bytes", lib().clk_verify_sample_scratch_bytes(dt, V, B, ctypes.byref(n)))
    size = n.value if halves == 1 else 2 * ((n.value + 255) // 256 * 256)
    t = torch.empty(size, dtype=torch.uint8, device=device)
    _check("clk_verify_scratch_init", lib().clk_verify_scratch_init(t.data_ptr(), t.numel(), _stream(stream)))
    return t


def verify_sample(logits, block, length, inv_temp, uniform, accept, emitted, out_tok, scratch, stream=None):
    """Sampling verification with point-mass drafts (clk_verify_sample).
    inv_temp: float32 [B]; uniform: float32 [B, 16, 2]."""
    dt, rs, qs, V = _logits_args(logits)
    B = block.shape[0]
    _check("clk_verify_sample",
           lib().clk_verify_sample(logits.data_ptr(), dt, rs, qs, V, B, _ptr(block, shape=(B, BLOCK)),
                                   _ptr(length, shape=(B,)), _ptr(inv_temp, torch.float32, (B,), "inv_temp"),
                                   _ptr(uniform, torch.float32, (B, BLOCK, 2), "uniform"),
                                   _ptr(accept, shape=(B,)), _ptr(emitted, shape=(B,)),
                                   _ptr(out_tok, shape=(B, BLOCK)), _ptr(scratch, torch.uint8, name="scratch"),
                                   scratch.numel(), _stream(stream)))


def verify_sample_exact_scratch(logits_dtype, V: int, B: int, device="cuda", stream=None,
                                halves: int = 1) -> torch.Tensor:
    """A zeroed scratch buffer for verify_sample_exact with vocabulary V and
    up to B requests; halves=2: two halves for the fused calls to alternate
    (as verify_sample_scratch)."""
    dt = BF16 if logits_dtype == torch.bfloat16 else F32
    n = ctypes.c_size_t()
    _check("clk_verify_sample_exact_scratch_bytes",
           lib().clk_verify_sample_exact_scratch_bytes(dt, V, B, ctypes.byref(n)))
    size = n.value if halves == 1 else 2 * ((n.value + 255) // 256 * 256)
    t = torch.empty(size, dtype=torch.uint8, device=device)
    _check("clk_verify_scratch_init", lib().clk_verify_scratch_init(t.data_ptr(), t.numel(), _stream(stream)))
    return t


def verify_sample_exact(logits, block, length, inv_temp, uniform, accept, emitted, out_tok, scratch, stream=None):
    """Sampling verification on the fixed-point weights
    (clk_verify_sample_exact): the rule of verify_sample with every decision
    an integer comparison."""
    dt, rs, qs, V = _logits_args(logits)
    B = block.shape[0]
    _check("clk_verify_sample_exact",
           lib().clk_verify_sample_exact(logits.data_ptr(), dt, rs, qs, V, B, _ptr(block, shape=(B, BLOCK)),
                                         _ptr(length, shape=(B,)), _ptr(inv_temp, torch.float32, (B,), "inv_temp"),
                                         _ptr(uniform, torch.float32, (B, BLOCK, 2), "uniform"),
                                         _ptr(accept, shape=(B,)), _ptr(emitted, shape=(B,)),
                                         _ptr(out_tok, shape=(B, BLOCK)), _ptr(scratch, torch.uint8, name="scratch"),
                                         scratch.numel(), _stream(stream)))


def verify_sample_append(h: Lookup, slots, logits, block, length, inv_temp, uniform, accept, emitted, out_tok,
                         scratch, stream=None, length_hint=None):
    """Sampling verification fused with the token commit (clk_verify_sample_append);
    ``length_hint`` (int32 [B] or None) predicts the block lengths."""
    dt, rs, qs, V = _logits_args(logits)
    B = slots.numel()
    _check("clk_verify_sample_append",
           lib().clk_verify_sample_append(h.handle, _ptr(slots), logits.data_ptr(), dt, rs, qs, V, B,
                                          _ptr(block, shape=(B, BLOCK)), _ptr(length, shape=(B,)),
                                          _ptr(length_hint, shape=(B,), name="length_hint"),
                                          _ptr(inv_temp, torch.float32, (B,), "inv_temp"),
                                          _ptr(uniform, torch.float32, (B, BLOCK, 2), "uniform"),
                                          _ptr(accept, shape=(B,)), _ptr(emitted, shape=(B,)),
                                          _ptr(out_tok, shape=(B, BLOCK)), _ptr(scratch, torch.uint8, name="scratch"),
                                          scratch.numel(), _stream(stream)))


def verify_sample_exact_append(h: Lookup, slots, logits, block, length, inv_temp, uniform, accept, emitted, out_tok,
                               scratch, stream=None, length_hint=None):
    """Exact sampling verification (fixed-point weights) fused with the
    token commit (clk_verify_sample_exact_append)."""
    dt, rs, qs, V = _logits_args(logits)
    B = slots.numel()
    _check("clk_verify_sample_exact_append",
           lib().clk_verify_sample_exact_append(h.handle, _ptr(slots), logits.data_ptr(), dt, rs, qs, V, B,
                                                _ptr(block, shape=(B, BLOCK)), _ptr(length, shape=(B,)),
                                                _ptr(length_hint, shape=(B,), name="length_hint"),
                                                _ptr(inv_temp, torch.float32, (B,), "inv_temp"),
                                                _ptr(uniform, torch.float32, (B, BLOCK, 2), "uniform"),
                                                _ptr(accept, shape=(B,)), _ptr(emitted, shape=(B,)),
                                                _ptr(out_tok, shape=(B, BLOCK)),
                                                _ptr(scratch, torch.uint8, name="scratch"), scratch.numel(),
                                                _stream(stream)))


def verify_append(h: Lookup, slots, logits, block, length, argmax, accept, emitted, out_tok, stream=None,
                  length_hint=None):
    dt, rs, qs, V = _logits_args(logits)
    B = slots.numel()
    _check("clk_verify_append",
           lib().clk_verify_append(h.handle, _ptr(slots), logits.data_ptr(), dt, rs, qs, V, B,
                                   _ptr(block, shape=(B, BLOCK)), _ptr(length, shape=(B,)),
                                   _ptr(length_hint, shape=(B,), name="length_hint"),
                                   _ptr(argmax, shape=(B, BLOCK)), _ptr(accept, shape=(B,)),
                                   _ptr(emitted, shape=(B,)), _ptr(out_tok, shape=(B, BLOCK)), _stream(stream)))


# ---------------------------------------------------------------------------
# Step driver: two launches per decode step
# ---------------------------------------------------------------------------
class Step:
    """Per-step buffers of one batch and the two launches of a step.

    ``pre(head)``    -> propose + scheduler + fusion: draft, k, j, length, block
    ``post(logits)`` -> verify + commit: argmax, accept, emitted, out_tok
    ``post_sample(logits, inv_temp, uniform)`` -> the same step verified by
    sampling (point-mass drafts): accept, emitted, out_tok; ``exact=True``
    samples on the fixed-point weights (clk_verify_sample_exact_append)
    The previous step's accept/length feed the scheduler.  The block lengths
    alternate between two buffers, so that ``post`` can pass the previous
    step's lengths as the verify launch's prediction while ``pre`` writes the
    new ones; ``length`` is the buffer of the latest ``pre``.  The buffers are
    owned here, so their pointers are resolved once; a call only checks the
    tensor it is given.  The logits must hold all 1 + head + tail rows of
    every request."""

    def __init__(self, lookup: Lookup, slots: torch.Tensor):
        self.h = lookup
        self.slots = slots
        B = slots.numel()
        dev = slots.device
        z = lambda *s: torch.zeros(s, dtype=torch.int32, device=dev)  # noqa: E731
        self.B = B
        self.draft, self.k, self.j = z(B, BLOCK), z(B), z(B)
        self._len = [z(B), z(B)]
        self._cur = 0
        self.block = z(B, BLOCK)
        self.argmax, self.accept, self.emitted, self.out_tok = z(B, BLOCK), z(B), z(B), z(B, BLOCK)
        _ptr(slots, shape=(B,), name="slots")
        self._p = {n: getattr(self, n).data_ptr() for n in
                   ("slots", "draft", "k", "j", "block", "argmax", "accept", "emitted", "out_tok")}
        self._lp = [t.data_ptr() for t in self._len]
        self._head_shape = (B, lookup.params.head)
        self._rows = lookup.params.long_len
        self._lib = lib()
        self._sscratch = None

    @property
    def length(self) -> torch.Tensor:
        return self._len[self._cur]

    def reset(self):
        """Forget the previous step (after the slots are set up again)."""
        for t in self._len:
            t.zero_()
        self.accept.zero_()

    def resume(self, accept, length):
        """Continue from a checkpoint: the previous step's accepted counts and
        block lengths (int32 [B], as ``accept`` and ``length`` held them when
        the lookup was snapshotted), the inputs of the next scheduler step."""
        for t, name in ((accept, "accept"), (length, "length")):
            if tuple(t.shape) != (self.B,):
                raise ValueError(f"{name} must have shape ({self.B},)")
        for t in self._len:
            t.copy_(length)
        self.accept.copy_(accept)

    def pre(self, head, stream=None):
        if tuple(head.shape) != self._head_shape or head.dtype != torch.int32 or not head.is_cuda \
                or not head.is_contiguous():
            raise ValueError(f"head must be contiguous int32 {self._head_shape} on the GPU")
        p, prev, new = self._p, self._cur, self._cur ^ 1
        _check("clk_propose_fuse_sched",
               self._lib.clk_propose_fuse_sched(self.h.handle, p["slots"], self.B, head.data_ptr(), p["accept"],
                                                self._lp[prev], p["draft"], p["k"], p["j"], self._lp[new],
                                                p["block"], _stream(stream)))
        self._cur = new

    def post(self, logits, stream=None):
        dt, rs, qs, V = _logits_args(logits)
        if logits.shape[0] != self.B or logits.shape[1] < self._rows:
            raise ValueError(f"logits must be [{self.B}, >= {self._rows}, V]")
        p = self._p
        _check("clk_verify_append",
               self._lib.clk_verify_append(self.h.handle, p["slots"], logits.data_ptr(), dt, rs, qs, V, self.B,
                                           p["block"], self._lp[self._cur], self._lp[self._cur ^ 1], p["argmax"],
                                           p["accept"], p["emitted"], p["out_tok"], _stream(stream)))

    def post_sample(self, logits, inv_temp, uniform, stream=None, exact: bool = False):
        """Verify the block by sampling at inverse temperatures inv_temp
        (float32 [B]) with the uniforms uniform (float32 [B, 16, 2]), and
        commit the emitted tokens.  Like ``post`` it passes the previous
        step's lengths as the prediction of the new ones.  exact=True: on the
        fixed-point weights (clk_verify_sample_exact_append)."""
        dt, rs, qs, V = _logits_args(logits)
        if logits.shape[0] != self.B or logits.shape[1] < self._rows:
            raise ValueError(f"logits must be [{self.B}, >= {self._rows}, V]")
        key = (logits.dtype, V, bool(exact))
        if self._sscratch is None or self._sscratch[0] != key:
            make = verify_sample_exact_scratch if exact else verify_sample_scratch
            self._sscratch = (key, make(logits.dtype, V, self.B, device=self.slots.device, stream=stream, halves=2))
        p = self._p
        sc = self._sscratch[1]
        name = "clk_verify_sample_exact_append" if exact else "clk_verify_sample_append"
        _check(name,
               getattr(self._lib, name)(self.h.handle, p["slots"], logits.data_ptr(), dt, rs, qs, V,
                                                  self.B, p["block"], self._lp[self._cur], self._lp[self._cur ^ 1],
                                                  _ptr(inv_temp, torch.float32, (self.B,), "inv_temp"),
                                                  _ptr(uniform, torch.float32, (self.B, BLOCK, 2), "uniform"),
                                                  p["accept"], p["emitted"], p["out_tok"], sc.data_ptr(), sc.numel(),
                                                  _stream(stream)))
