"""Worker of the exhaustive E4M3 encoding check (run in spawned processes):
the oracle's software encoder on one range of binary32 bit patterns, compared
with the codes the GPU produced for the same range."""

import numpy as np

import oracle as O


def check_range(start, got):
    """Compare the GPU's codes `got` for the bit patterns start .. start +
    len(got) - 1 with the oracle's.  Returns (mismatches among non-NaN
    inputs, the first such (pattern, gpu, oracle) or None, the set of codes
    the GPU gave for NaN inputs)."""
    bits = (np.arange(got.size, dtype=np.uint64) + np.uint64(start)).astype(np.uint32)
    f = bits.view(np.float32)
    with np.errstate(invalid="ignore", over="ignore"):
        want = O.e4m3_encode(f)
    nan = np.isnan(f)
    bad = (got != want) & ~nan
    n_bad = int(bad.sum())
    first = None
    if n_bad:
        i = int(np.argmax(bad))
        first = (int(bits[i]), int(got[i]), int(want[i]))
    return n_bad, first, sorted(set(np.unique(got[nan]).tolist()))
