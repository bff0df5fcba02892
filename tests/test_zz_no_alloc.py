"""clk_verify_greedy_static: verification for callers that cannot allocate.

Some callers cannot give the library a scratch buffer: a plugin that only
receives its input and output pointers, or an engine whose device memory is
already committed to its own pools.  For them the library keeps the verify
scratch in a fixed array of its own.  This test calls that entry point
through the C ABI twice in a row, with different batches (the second call
runs over whatever the first left in the shared array), and checks every
output against the ordinary entry point that takes a caller buffer.  It
also checks that a batch above the fixed maximum is refused.  This file is
collected last on purpose.  GPU."""
import ctypes

import numpy as np
import pytest
import torch

import context_lookup_speculative_gb300 as clk

pytestmark = pytest.mark.gpu

STATIC_MAX_BATCH = 1024  # CLK_STATIC_VERIFY_MAX_BATCH in include/clk.h


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


def _call_static(x, blk, L, outs):
    B, _, V = x.shape
    stream = torch.cuda.current_stream().cuda_stream
    return clk.lib().clk_verify_greedy_static(
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


def test_static_scratch_matches_caller_scratch_on_two_calls_in_a_row():
    cases = [_case(1, 300, 32000, torch.bfloat16), _case(2, 57, 4096, torch.float32)]
    for x, blk, L in cases:
        got, want = _outputs(x.shape[0]), _outputs(x.shape[0])
        assert _call_static(x, blk, L, got) == clk.OK
        assert _call_with_buffer(x, blk, L, want) == clk.OK
        torch.cuda.synchronize()
        for g, w in zip(got, want):
            assert torch.equal(g, w)  # integer outputs: exact


def test_static_scratch_refuses_batches_above_its_maximum():
    B = STATIC_MAX_BATCH + 1
    x = torch.zeros((B, 1, 8), dtype=torch.bfloat16, device="cuda")
    blk = torch.zeros((B, 16), dtype=torch.int32, device="cuda")
    L = torch.ones(B, dtype=torch.int32, device="cuda")
    outs = _outputs(B)
    assert _call_static(x, blk, L, outs) == clk.ECAPACITY
    torch.cuda.synchronize()
    assert int(outs[1][0]) == 77  # nothing was launched
