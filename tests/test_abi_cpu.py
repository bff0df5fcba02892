"""The C-ABI library loads, exports every symbol include/clk.h declares, and
its host-only entry points behave; the CUDA path and the oracle share no
code.  CPU only: no call here launches a kernel."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "clk.h")
PKG = os.path.join(ROOT, "context_lookup_speculative_gb300")


@pytest.fixture(scope="module")
def clk():
    import context_lookup_speculative_gb300 as clk_mod
    if not os.path.exists(clk_mod.LIB_PATH):
        from context_lookup_speculative_gb300 import build
        build.build()
    return clk_mod


def _declared():
    src = open(HEADER).read()
    return set(re.findall(r"^CLK_API\s+(?:int|void|const char\*)\s+(clk_\w+)\(", src, flags=re.M))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("clk_lookup_init", "clk_lookup_append", "clk_lookup_propose", "clk_fuse", "clk_sched_step",
              "clk_verify_greedy", "clk_fuse_sched", "clk_propose_fuse_sched", "clk_verify_append"):
        assert n in names
    assert len(names) >= 20


def test_library_exports_every_declared_symbol(clk):
    out = subprocess.run(["nm", "-D", "--defined-only", clk.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    declared = _declared()
    assert declared <= exported, declared - exported
    # nothing else leaks out of the library
    assert {s for s in exported if s.startswith("clk_")} == declared
    lib = ctypes.CDLL(clk.LIB_PATH)
    for n in declared:
        assert getattr(lib, n) is not None


def test_binding_covers_every_declared_symbol(clk):
    assert {n for n, _, _ in clk._SIGS} == _declared()
    clk.lib()


def test_params_defaults_and_checks(clk):
    p = clk.Params.default()
    assert (p.min_k, p.max_k, p.head, p.tail, p.head_replace_k, p.head_agree_k, p.head_agree_n, p.tail_k,
            p.enter_streak, p.sticky, p.near_full_slack) == (4, 12, 7, 8, 8, 6, 2, 4, 2, 3, 1)
    assert p.long_len == 16 and p.short_len == 8
    L = clk.lib()
    assert L.clk_params_check(ctypes.byref(p)) == 0
    for field, bad in (("min_k", 0), ("max_k", 17), ("max_k", 3), ("tail", 9), ("head_agree_n", 8),
                       ("enter_streak", 0), ("sticky", -1)):
        q = clk.Params.default(**{field: bad})
        assert L.clk_params_check(ctypes.byref(q)) == clk.EINVAL, field
    assert L.clk_params_check(None) == clk.EINVAL


def test_workspace_sizing(clk):
    L = clk.lib()
    p = clk.Params.default()
    n = ctypes.c_size_t()

    def ws(slots, hist):
        rc = L.clk_lookup_workspace_bytes(ctypes.byref(p), slots, hist, ctypes.byref(n))
        return rc, n.value

    rc, small = ws(1, 100)
    assert rc == 0 and small > 0
    rc, big = ws(64, 40192)
    assert rc == 0
    # 9 tables of 2^17 4-byte entries per slot dominate: about 302 MB for 64 slots
    assert 9 * 2 ** 17 * 4 * 64 < big < 1.1 * 9 * 2 ** 17 * 4 * 64 + 64 * 40192 * 4 * 1.1
    assert ws(0, 100)[0] == clk.EINVAL
    assert ws(1, 0)[0] == clk.EINVAL
    assert L.clk_lookup_workspace_bytes(None, 1, 100, ctypes.byref(n)) == clk.EINVAL
    assert L.clk_verify_scratch_bytes(64, ctypes.byref(n)) == 0 and n.value == 64 * 17 * 8
    assert L.clk_verify_scratch_bytes(-1, ctypes.byref(n)) == clk.EINVAL
    assert L.clk_verify_scratch_bytes(clk.MAX_BATCH + 1, ctypes.byref(n)) == clk.EINVAL


def test_host_side_rejections_launch_nothing(clk):
    L = clk.lib()
    p = clk.Params.default()
    h = ctypes.c_void_p()
    assert L.clk_lookup_create(ctypes.byref(h), ctypes.byref(p), 4, 100, 0, None, 0) == clk.EINVAL
    assert L.clk_lookup_create(ctypes.byref(h), ctypes.byref(p), 4, 100, 0, 0x1001, 1 << 30) == clk.EINVAL  # unaligned
    assert L.clk_lookup_create(None, ctypes.byref(p), 4, 100, 0, 0x1000, 1 << 30) == clk.EINVAL
    assert L.clk_lookup_init(None, None, 1, None, None, None) == clk.ESTATE
    assert L.clk_lookup_propose(None, None, 1, None, None, None, None) == clk.ESTATE
    assert L.clk_verify_greedy(None, 0, 8, 8, 8, 1, None, None, None, None, None, None, None, 0, None) == clk.EINVAL
    assert L.clk_verify_greedy(0x1000, 7, 8, 128, 8, 1, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000,
                               0x1000, 1 << 20, None) == clk.EINVAL  # bad dtype
    assert L.clk_fuse(None, 1, None, None, None, None, None, None, None) == clk.EINVAL
    bad = clk.Params.default(tail=12)
    assert L.clk_fuse(ctypes.byref(bad), 1, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, 0x1000, None) == clk.EINVAL
    assert clk.status_string(clk.ECAPACITY) == "capacity exceeded"


def test_handle_over_fake_workspace_validates_batches(clk):
    """A handle is host-only; a batch larger than max_slots is refused before any launch."""
    L = clk.lib()
    p = clk.Params.default()
    n = ctypes.c_size_t()
    L.clk_lookup_workspace_bytes(ctypes.byref(p), 4, 100, ctypes.byref(n))
    h = ctypes.c_void_p()
    assert L.clk_lookup_create(ctypes.byref(h), ctypes.byref(p), 4, 100, 0, 1 << 20, n.value) == 0
    try:
        assert L.clk_lookup_propose(h, 0x1000, 5, 0x1000, 0x1000, 0x1000, None) == clk.EINVAL
        assert L.clk_lookup_append(h, 0x1000, -1, 0x1000, 0x1000, None) == clk.EINVAL
        assert L.clk_lookup_propose(h, 0x1000, 0, 0x1000, 0x1000, 0x1000, None) == 0  # empty batch: no-op
        # the launch setting is host state only
        assert L.clk_lookup_set_alone(h, 1) == 0 and L.clk_lookup_set_alone(h, 0) == 0
        assert L.clk_lookup_set_alone(None, 1) == clk.ESTATE
        assert L.clk_read_counters(h, 9, ctypes.byref(clk.Counters()), None) == clk.EINVAL
        # a resume refuses a bad slot or scheduler state before touching the device
        ok = clk.SlotInfo(n=5, mode=1, streak=0, miss=2, has_prev=1, cur_len=16, n_indexed=5)
        c = clk.Counters()
        assert L.clk_lookup_restore_state(h, 9, ctypes.byref(ok), ctypes.byref(c), None) == clk.EINVAL
        assert L.clk_lookup_restore_state(h, 0, None, ctypes.byref(c), None) == clk.EINVAL
        assert L.clk_lookup_restore_state(h, 0, ctypes.byref(ok), None, None) == clk.EINVAL
        for field, bad in (("mode", 2), ("streak", -1), ("miss", -1), ("has_prev", 2), ("cur_len", 17)):
            info = clk.SlotInfo(n=5, mode=1, streak=0, miss=2, has_prev=1, cur_len=16, n_indexed=5)
            setattr(info, field, bad)
            assert L.clk_lookup_restore_state(h, 0, ctypes.byref(info), ctypes.byref(c), None) == clk.EINVAL, field
    finally:
        L.clk_lookup_destroy(h)


def _sources(d, exts):
    for root, _, files in os.walk(d):
        if "_build" in root or "__pycache__" in root:
            continue
        for f in files:
            if f.endswith(exts):
                yield os.path.join(root, f)


def test_cuda_path_and_oracle_share_nothing():
    for path in _sources(PKG, (".py", ".cu", ".cuh", ".h")):
        text = open(path).read()
        assert not re.search(r"\boracle\b|clk_oracle|or_lookup", text), path
        assert "gen_rules.h" not in text and "import workload" not in text, path
    for path in _sources(os.path.join(ROOT, "oracle"), (".py", ".c", ".h")):
        text = open(path).read()
        assert "context_lookup_speculative_gb300" not in text and "clk.h" not in text, path
        assert "clk_device" not in text, path
