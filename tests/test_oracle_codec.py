"""Pins of the oracle's E4M3 and bf16 codecs against the format definition,
a brute-force nearest search and torch's own float8/bfloat16 casts."""

import fractions

import numpy as np
import pytest
import torch

import oracle as O
from conftest import golden_lines


def test_golden_e4m3_values():
    for code, value in golden_lines("e4m3_codes.txt"):
        c = int(code, 16)
        got = O.e4m3_decode(np.array([c], np.uint8))[0]
        if value == "nan":
            assert np.isnan(got)
        else:
            assert got == float(value) and np.signbit(got) == value.startswith("-")
            assert O.e4m3_encode(np.array([got], np.float32))[0] == c


def test_all_256_codes_round_trip():
    codes, vals = O.e4m3_all_values()
    assert np.array_equal(O.e4m3_encode(vals), codes)


def test_decode_matches_torch_float8():
    codes, vals = O.e4m3_all_values()
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    assert np.array_equal(ref, vals, equal_nan=True)


def test_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    n = 400_000
    v = (rng.standard_normal(n) * np.exp(rng.uniform(-16, 7, n))).astype(np.float32)
    v = np.clip(v, -448, 448)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(O.e4m3_encode(v), ref)


def _brute_nearest(v):
    """Nearest finite E4M3 code by exhaustive search; ties to the even code."""
    codes, vals = O.e4m3_all_values()
    fin = ~np.isnan(vals)
    best = None
    for c, x in zip(codes[fin], vals[fin]):
        d = abs(fractions.Fraction(float(x)) - fractions.Fraction(float(v)))
        key = (d, int(c) & 1)
        if best is None or key < best[0]:
            best = (key, int(c), float(x))
    return best


def test_encode_brute_force_nearest():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(300) * np.exp(rng.uniform(-12, 6, 300))).astype(np.float32)
    v = np.clip(v, -448, 448)
    got = O.e4m3_encode(v)
    for x, c in zip(v, got):
        _, bc, bx = _brute_nearest(x)
        # +0 and -0 are both nearest for tiny values; the sign must follow x
        assert O.e4m3_decode(np.array([c], np.uint8))[0] == bx
        assert (int(c) >> 7) == int(np.signbit(x))


@pytest.mark.parametrize("v,code", [
    (2.0 ** -10, 0x00),            # half of the smallest subnormal: tie to even (0)
    (3 * 2.0 ** -10, 0x02),        # 1.5 subnormal quanta: tie to even (2)
    (7.5 * 2.0 ** -9, 0x08),       # between the largest subnormal and 2^-6: tie to even code
    (1.0625, 0x38),                # 1 + 1/16: tie between 1.0 and 1.125, even mantissa
    (1.1875, 0x3A),                # 1 + 3/16: tie, rounds up to the even mantissa 1.25
    (464.0, 0x7E),                 # midpoint 448/480: ties to even, 448
    (465.0, 0x7E),                 # above: saturates
    (1e30, 0x7E),
    (np.inf, 0x7E),
    (-np.inf, 0xFE),
    (-1e-12, 0x80),                # negative underflow keeps the sign
])
def test_encode_special_cases(v, code):
    assert O.e4m3_encode(np.array([v], np.float32))[0] == code


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(2)
    v32 = (rng.standard_normal(200_000) * np.exp(rng.uniform(-80, 80, 200_000))).astype(np.float32)
    v32 = np.concatenate([v32, np.array([0.0, -0.0, np.inf, -np.inf, 3.4e38, 1e-40, -1e-45], np.float32)])
    ref = torch.from_numpy(v32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.bf16_round(v32), ref)
    # float64 inputs: rounded once, directly from the double
    v64 = rng.standard_normal(10_000) * 3.0
    f = [fractions.Fraction(float(x)) for x in v64[:200]]
    got = O.bf16_decode(O.bf16_round(v64[:200])).astype(np.float64)
    for x, g in zip(f, got):
        # the rounding error is at most half a bf16 ulp (2^-8 relative to the binade)
        assert abs(fractions.Fraction(float(g)) - x) <= abs(x) * fractions.Fraction(1, 256)


def test_bf16_decode_exact():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(O.bf16_decode(bits), ref, equal_nan=True)


def test_fp16_decode_matches_numpy():
    """Every binary16 pattern decodes to numpy's own widening (a library
    routine independent of the oracle's field arithmetic)."""
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    assert np.array_equal(O.fp16_decode(bits), ref, equal_nan=True)


def test_fp16_round_matches_numpy_and_format_edges():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal(300_000) * 10.0 ** rng.integers(-9, 6, 300_000)).astype(np.float32)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(O.fp16_round(v), ref)
    # format edges written from the definition
    edges = {65504.0: 0x7BFF, 65519.0: 0x7BFF, 65520.0: 0x7C00, -1e9: 0xFC00,
             2.0 ** -24: 0x0001, 2.0 ** -25: 0x0000, 3 * 2.0 ** -26: 0x0001, 3 * 2.0 ** -25: 0x0002,
             2.0 ** -14: 0x0400, -0.0: 0x8000, 1.0 + 2.0 ** -11: 0x3C00, 1.0 + 3 * 2.0 ** -11: 0x3C02}
    for val, code in edges.items():
        assert int(O.fp16_round(np.float64(val))) == code, (val, code)
    assert int(O.fp16_round(np.float32(np.inf))) == 0x7C00
