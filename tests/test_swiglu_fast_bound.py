"""CPU check of the bound the SwiGLU kernels' fast path relies on: the
denominator 1 + exp_spec(t) evaluated with fused multiply-adds stays within
2 binary32 ulps (4 * 2^-24 relative) of the specification's separately
rounded evaluation for every binary32 t in [-17, 88] (the fast path's
range; the kernels send other arguments to the exact path).  The check runs
a plain C restatement of both evaluations (tests/dplus1_bound.c) over every
16th binary32 value by default and over all 2.2e9 of them with
W8_EXHAUSTIVE=1 (about three minutes)."""

import os
import re
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_fast_denominator_within_two_ulps(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "dplus1_bound")
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-fno-fast-math", "-o", exe,
                    os.path.join(HERE, "dplus1_bound.c"), "-lm"], check=True)
    stride = "1" if os.environ.get("W8_EXHAUSTIVE") == "1" else "16"
    out = subprocess.run([exe, stride], check=True, capture_output=True, text=True, timeout=1200).stdout
    m = re.search(r"n=(\d+) differ=(\d+) max_ulp=(\d+) max_rel_over_2\^-24=([0-9.]+)", out)
    assert m, out
    n, differ, max_ulp, max_rel = int(m[1]), int(m[2]), int(m[3]), float(m[4])
    assert n > 100_000_000 // int(stride)
    assert max_ulp <= 2 and max_rel <= 4.0, out
    assert differ / n < 0.01, out      # the two agree on more than 99% of arguments
