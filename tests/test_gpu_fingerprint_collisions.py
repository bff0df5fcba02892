"""The index's fingerprint branches, exercised on the GPU.

An index entry keeps only a few bits of its k-gram's hash as a fingerprint,
so two different k-grams can carry equal fingerprints.  Exactness then rests
on two branches: an insert that meets an entry with its fingerprint but other
tokens keeps probing, and a lookup that meets one skips it.  With full-width
fingerprints (13 to 16 bits at these history sizes) these branches run about
once in thousands of probes, too rarely to test.  This test builds the
library with 2-bit fingerprints (CLK_TEST_FP_BITS=2): a quarter of the
occupied entries a probe meets then carry its fingerprint without being its
k-gram.  It runs the lookup tests (random small vocabularies, periodic
histories, incremental appends, other match ranges, many commits without a
lookup in between) and the decode-loop tests on small workloads and on the
periodic and restatement workloads at full size, against that build,
bit-exact against the oracle as always.  GPU."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = ["tests/test_gpu_lookup.py", "tests/test_gpu_loop.py"]
SELECT = ("not maximum_batch and not config2 and not config4 and not full_size and not sampled "
          "and not fp32_and_block")


def test_parity_with_two_bit_fingerprints():
    from context_lookup_speculative_gb300 import build

    out_dir = os.path.join(build.HERE, "_build", "fp2")
    lib = build.build(out=os.path.join(out_dir, "libclk.so"), build_dir=out_dir, extra=["-DCLK_TEST_FP_BITS=2"])
    env = dict(os.environ, CLK_TEST_LIBRARY=lib)
    cmd = [sys.executable, "-m", "pytest", "-x", "-p", "no:cacheprovider", *TESTS, "-k", SELECT]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert f"clk library under test: {lib}" in r.stdout
    assert " passed" in r.stdout and " failed" not in r.stdout
