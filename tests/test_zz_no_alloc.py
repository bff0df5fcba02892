"""clk_verify_greedy_static: verification for callers that cannot allocate.

Some callers cannot give the library a scratch buffer: a plugin that only
receives its input and output pointers, or an engine whose device memory is
already committed to its own pools.  For them the library keeps the verify
scratch in a fixed array of its own.  These tests call that entry point
through the C ABI:
- twice in a row, with different batches (the second call runs over
  whatever the first left in the shared array), checking every output
  against the ordinary entry point that takes a caller buffer;
- after filling the array with garbage (through a hook that only a test
  build of the library exports), checking that the call clears what it uses:
  the outputs still equal the caller-buffer entry point's and the oracle's
  argmax rows and accepted counts;
- with batches above the fixed maximum, which are refused.
This file is collected last on purpose.  GPU."""
import ctypes
import os

import numpy as np
import pytest
import torch

import context_lookup_speculative_gb300 as clk
import oracle

pytestmark = pytest.mark.gpu

STATIC_MAX_BATCH = 1024  # CLK_STATIC_VERIFY_MAX_BATCH in include/clk.h
_P, _I32, _I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
_STATIC_ARGS = [_P, _I32, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P, _P]


def _case(seed, B, V, dtype):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.integers(-30, 30, size=(B, 16, V)).astype(np.float32)).to(dtype).cuda()
    L = torch.from_numpy(rng.integers(1, 17, size=B).astype(np.int32)).cuda()
    # drafts mostly equal to the row argmax so that accepted prefixes vary
    g = x.float().argmax(dim=2).to(torch.int32).cpu().numpy()
    blk = rng.integers(0, V, size=(B, 16)).astype(np.int32)
    agree = rng.random((B, 15)) < 0.85
    blk[:, 1:][agree] = g[:, :15][agree]
    return x, torch.from_numpy(blk).cuda(), L


def _outputs(B):
    return [torch.full(s, 77, dtype=torch.int32, device="cuda") for s in ((B, 16), (B,), (B,), (B, 16))]


def _dtype_code(x):
    return clk.BF16 if x.dtype == torch.bfloat16 else clk.F32


def _call_static(x, blk, L, outs, lib=None):
    B, _, V = x.shape
    stream = torch.cuda.current_stream().cuda_stream
    return (lib or clk.lib()).clk_verify_greedy_static(
        x.data_ptr(), _dtype_code(x), x.stride(1), x.stride(0), V, B, blk.data_ptr(), L.data_ptr(),
        outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(), outs[3].data_ptr(), stream)


def _call_with_buffer(x, blk, L, outs):
    B, _, V = x.shape
    scratch = clk.verify_scratch(B)
    stream = torch.cuda.current_stream().cuda_stream
    return clk.lib().clk_verify_greedy(
        x.data_ptr(), _dtype_code(x), x.stride(1), x.stride(0), V, B, blk.data_ptr(), L.data_ptr(),
        outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(), outs[3].data_ptr(), scratch.data_ptr(),
        ctypes.c_size_t(scratch.numel()), stream)


def _assert_same(got, want):
    for g, w in zip(got, want):
        assert torch.equal(g, w)  # integer outputs: exact


def _assert_oracle(x, blk, L, got):
    """Argmax rows and accepted counts against the oracle (first index of the
    maximum of each row, then the accepted prefix)."""
    # bf16 rows go to the oracle as their bit patterns, float32 rows as floats
    xs = x.view(torch.int16).cpu().numpy().view(np.uint16) if x.dtype == torch.bfloat16 else x.cpu().numpy()
    bs, ls = blk.cpu().numpy(), L.cpu().numpy()
    am, acc = got[0].cpu().numpy(), got[1].cpu().numpy()
    for b in range(xs.shape[0]):
        g = np.array([oracle.argmax_row(xs[b, r]) for r in range(ls[b])], dtype=np.int64)
        assert am[b, :ls[b]].tolist() == g.tolist(), b
        assert acc[b] == oracle.accept(bs[b], g, int(ls[b])), b


@pytest.fixture(scope="module")
def hooks_lib():
    """A test build of the library that also exports clk_test_fill_static_scratch."""
    from context_lookup_speculative_gb300 import build

    out_dir = os.path.join(build.HERE, "_build", "hooks")
    path = build.build(out=os.path.join(out_dir, "libclk.so"), build_dir=out_dir, extra=["-DCLK_TEST_HOOKS"])
    lib = ctypes.CDLL(path)
    lib.clk_verify_greedy_static.restype = ctypes.c_int
    lib.clk_verify_greedy_static.argtypes = _STATIC_ARGS
    lib.clk_test_fill_static_scratch.restype = ctypes.c_int
    lib.clk_test_fill_static_scratch.argtypes = [ctypes.c_int, _P]
    return lib


def test_static_scratch_matches_caller_scratch_on_two_calls_in_a_row():
    cases = [_case(1, 300, 32000, torch.bfloat16), _case(2, 57, 4096, torch.float32)]
    for x, blk, L in cases:
        got, want = _outputs(x.shape[0]), _outputs(x.shape[0])
        assert _call_static(x, blk, L, got) == clk.OK
        assert _call_with_buffer(x, blk, L, want) == clk.OK
        torch.cuda.synchronize()
        _assert_same(got, want)


def test_static_scratch_is_cleared_before_use(hooks_lib):
    """Garbage in the fixed array (every byte 0xFF: row keys above any real
    key, counters past any total) would, if left, keep wrong row maxima and
    stop every request from finishing.  Each call must clear what it uses."""
    stream = torch.cuda.current_stream().cuda_stream
    cases = [_case(3, 200, 8192, torch.bfloat16), _case(4, 33, 1000, torch.float32)]
    for i, (x, blk, L) in enumerate(cases):
        assert hooks_lib.clk_test_fill_static_scratch(0xFF, stream) == clk.OK
        got, want = _outputs(x.shape[0]), _outputs(x.shape[0])
        assert _call_static(x, blk, L, got, lib=hooks_lib) == clk.OK
        assert _call_with_buffer(x, blk, L, want) == clk.OK
        torch.cuda.synchronize()
        _assert_same(got, want)
        _assert_oracle(x, blk, L, got)


@pytest.mark.parametrize("B", [STATIC_MAX_BATCH + 1, clk.MAX_BATCH + 1])
def test_static_scratch_refuses_batches_above_its_maximum(B):
    x = torch.zeros((B, 1, 8), dtype=torch.bfloat16, device="cuda")
    blk = torch.zeros((B, 16), dtype=torch.int32, device="cuda")
    L = torch.ones(B, dtype=torch.int32, device="cuda")
    outs = _outputs(B)
    assert _call_static(x, blk, L, outs) == clk.ECAPACITY
    torch.cuda.synchronize()
    assert int(outs[1][0]) == 77  # nothing was launched
