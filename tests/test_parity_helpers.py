"""CPU checks of the check the GPU tests apply to the fused gate/up +
SwiGLU kernels: it accepts every output a correct kernel can produce (the
SwiGLU of gate/up values rounded from any sum within the binary32
accumulation bound) and rejects plausible mistakes (gate and up swapped, a
sign flip, the wrong output scale, a dropped SiLU)."""

import numpy as np
import pytest

import oracle as O
from gpu_util import accumulation_window, assert_swiglu_consistent, swiglu_range

K = 4096


def _case(seed, n=20000):
    rng = np.random.default_rng(seed)
    g64 = rng.normal(0.0, 2.0, n)
    u64 = rng.normal(0.0, 1.0, n)
    # sums of |terms| between 1x and 100x the result, some results near zero
    g64[:200] *= 1e-4
    u64[200:400] *= 1e-4
    abs_g = np.abs(g64) * rng.uniform(1, 100, n) + 1e-3
    abs_u = np.abs(u64) * rng.uniform(1, 100, n) + 1e-3
    # a correct kernel: bf16 of some binary32 sum within the accumulation bound
    eg = 2.0 * K * 2.0 ** -24 * abs_g
    eu = 2.0 * K * 2.0 ** -24 * abs_u
    gk = O.bf16_round(g64 + rng.uniform(-1, 1, n) * eg)
    uk = O.bf16_round(u64 + rng.uniform(-1, 1, n) * eu)
    wg = accumulation_window(g64, abs_g, K)
    wu = accumulation_window(u64, abs_u, K)
    return g64, u64, O.bf16_round(g64), O.bf16_round(u64), gk, uk, wg, wu


@pytest.mark.parametrize("out", ["bf16", "e4m3"])
def test_accepts_what_a_correct_kernel_may_produce(out):
    g64, u64, gb, ub, gk, uk, wg, wu = _case(1)
    s = np.float32(0.01)
    spec = (lambda g, u: O.swiglu_2in_bf16(g, u)) if out == "bf16" else (lambda g, u: O.swiglu_2in_fp8(g, u, s))
    got, want = spec(gk, uk), spec(gb, ub)
    assert (got != want).any()              # the case exercises the window
    assert_swiglu_consistent(got, want, g64, u64, wg, wu, out, s, max_frac=1.0)


@pytest.mark.parametrize("out", ["bf16", "e4m3"])
def test_rejects_plausible_mistakes(out):
    g64, u64, gb, ub, gk, uk, wg, wu = _case(2)
    s = np.float32(0.01)
    spec = (lambda g, u: O.swiglu_2in_bf16(g, u)) if out == "bf16" else (lambda g, u: O.swiglu_2in_fp8(g, u, s))
    want = spec(gb, ub)
    mistakes = [spec(uk, gk),                                     # gate and up swapped
                spec(gk ^ np.uint16(0x8000), uk),                 # sign of the gate flipped
                O.bf16_round(O.bf16_decode(gk).astype(np.float64) * O.bf16_decode(uk))
                if out == "bf16" else O.e4m3_encode(O.bf16_decode(gk) * O.bf16_decode(uk) / s)]  # no SiLU
    if out == "e4m3":
        mistakes.append(O.swiglu_2in_fp8(gk, uk, np.float32(0.02)))   # wrong output scale
    for bad in mistakes:
        with pytest.raises(AssertionError):
            assert_swiglu_consistent(bad, want, g64, u64, wg, wu, out, s, max_frac=1.0)


def test_swiglu_range_contains_sampled_points():
    rng = np.random.default_rng(3)
    lo = rng.normal(0, 3, 2000)
    hi = lo + rng.uniform(0, 2, 2000)
    ulo = rng.normal(0, 1, 2000)
    uhi = ulo + rng.uniform(0, 1, 2000)
    hmin, hmax = swiglu_range(lo, hi, ulo, uhi)
    for t in np.linspace(0, 1, 41):
        for v in np.linspace(0, 1, 5):
            g = lo + t * (hi - lo)
            u = ulo + v * (uhi - ulo)
            h = g / (1 + np.exp(-g)) * u
            assert np.all((hmin - 1e-12 <= h) & (h <= hmax + 1e-12))
