"""The E4M3 encoding every code-producing kernel ends with (the hardware's
saturating round-to-nearest-even conversion, exported on its own as
fp8_e4m3_from_f32) against the oracle's software encoder: exhaustively, on
all 2^32 binary32 bit patterns, and on a ragged small case.

The oracle's encoder follows the E4M3 definition (the (4, 3)-bit format of
diffusers issue #15170, Logs; saturation at +-448 as the static quantization
of cosmos-framework PR #157, Verification, clamps before rounding).  NaN
inputs may give either NaN code: the hardware returns one canonical NaN; the
test records which."""

import multiprocessing as mp
import os

import numpy as np
import pytest
import torch

import oracle as O
from gpu_util import W  # noqa: F401

pytestmark = pytest.mark.gpu

CHUNK = 1 << 24


def test_ragged_and_special_values(W):
    rng = np.random.default_rng(3)
    f = np.concatenate([
        rng.normal(0.0, 100.0, 997).astype(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 448.0, 464.0, -464.0, 2.0 ** -10, 2.0 ** -9 * 1.5,
                  7.5 * 2.0 ** -9, 1e-45, -1e-45, 3.4e38], dtype=np.float32)])
    for n in (f.size, f.size - 1, f.size - 2, f.size - 3, 3, 1):
        x = torch.from_numpy(f[:n].copy()).cuda()
        got = W.fp8_e4m3_from_f32(x).cpu().numpy()
        with np.errstate(invalid="ignore"):
            want = O.e4m3_encode(f[:n])
        nan = np.isnan(f[:n])
        assert np.array_equal(got[~nan], want[~nan]), n
        assert np.all((got[nan] & 0x7F) == 0x7F)


def test_every_binary32_bit_pattern(W):
    """All 2^32 inputs, 2^24 at a time: the GPU converts each range, a pool
    of spawned processes runs the oracle on it and compares."""
    import codec_worker
    bits = torch.arange(CHUNK, dtype=torch.int32, device="cuda")
    q = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    procs = max(1, min(16, os.cpu_count() or 1))
    total_bad, firsts, nan_codes = 0, [], set()
    with mp.get_context("spawn").Pool(procs) as pool:
        pending = []
        for c in range(1 << 8):
            start = c * CHUNK
            start_i32 = start - (1 << 32) if start >= (1 << 31) else start
            x = (bits + start_i32).view(torch.float32)
            W.fp8_e4m3_from_f32(x, out=q)
            pending.append(pool.apply_async(codec_worker.check_range, (start, q.cpu().numpy())))
            if len(pending) >= 2 * procs:
                n_bad, first, nans = pending.pop(0).get()
                total_bad += n_bad
                firsts += [first] if first else []
                nan_codes |= set(nans)
        for p in pending:
            n_bad, first, nans = p.get()
            total_bad += n_bad
            firsts += [first] if first else []
            nan_codes |= set(nans)
    W.poll_device_error()
    assert total_bad == 0, (total_bad, [tuple(hex(v) for v in f) for f in firsts[:5]])
    assert nan_codes and nan_codes <= {0x7F, 0xFF}, nan_codes
