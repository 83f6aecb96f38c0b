"""Helpers shared by the GPU parity tests: host <-> device marshalling of
bit patterns, seeded problem set-ups, and the GEMM error metric."""

import numpy as np
import pytest
import torch

import oracle as O
from w8a16_linear_gb300 import synth

# GEMM tolerance: max|y_gpu - y_exact| / max|y_exact| <= 2^-8 + margin.
# A correctly rounded bf16 output alone can reach 2^-8 (half a bf16 ulp of
# the largest element, relative to that element when it sits at the bottom of
# its binade); the F32 accumulation adds ~K * 2^-24 relative at most.
GEMM_TOL = 4.0e-3


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev_u8(codes):
    return torch.from_numpy(np.ascontiguousarray(codes)).cuda()


def dev_f32(v):
    return torch.tensor([float(v)], dtype=torch.float32, device="cuda")


def host_bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_u8(t):
    return t.contiguous().view(torch.uint8).cpu().numpy()


def amax_scale(vals):
    return np.float32(np.abs(np.asarray(vals, np.float64)).max() / 448.0)


def gemm_err(y_bits, y64):
    got = O.bf16_decode(y_bits).astype(np.float64)
    return float(np.abs(got - y64).max() / max(np.abs(y64).max(), 1e-300))


def frac_rounded_equal(y_bits, y64):
    return float(np.mean(y_bits == O.bf16_round(y64)))


def abs_product_sums(mode, x_bits, s_in, qw, s_w):
    """sum_k |a_mk b_nk| of the products a W8A8 ("A8") or W8A16 ("A16")
    linear adds up, times the A8 epilogue scale: what bounds the rounding
    error of any binary32 summation of them."""
    if mode == "A8":
        a = np.abs(O.e4m3_decode(O.quant_static(x_bits, s_in)).astype(np.float64))
        b = np.abs(O.e4m3_decode(qw).astype(np.float64))
        return float(np.float32(s_in)) * float(np.float32(s_w)) * (a @ b.T)
    a = np.abs(O.bf16_decode(x_bits).astype(np.float64))
    b = np.abs(O.bf16_decode(O.dequant_weight_bf16(qw, s_w)).astype(np.float64))
    return a @ b.T


def accumulation_window(y64, abs_sum, K):
    """Half-width of the interval that holds a kernel's bf16 output of a
    linear whose exact value is y64: any order of binary32 additions of the
    K exact products (rounded to nearest or toward zero) is within
    2 K 2^-24 sum|terms| of the exact sum; the epilogue scale adds one
    binary32 rounding and the bf16 rounding at most 2^-8 of the result."""
    e = 2.0 * K * 2.0 ** -24 * abs_sum + 2.0 ** -24 * np.abs(y64)
    return e + 2.0 ** -8 * (np.abs(y64) + e)


_SILU_ARGMIN = -1.2784645427610738


def _silu(g):
    return g / (1.0 + np.exp(-g))


def swiglu_range(g_lo, g_hi, u_lo, u_hi):
    """Smallest and largest SiLU(g) * u over the boxes [g_lo, g_hi] x
    [u_lo, u_hi] (float64, elementwise): u enters linearly, and SiLU has
    one interior extremum (its minimum)."""
    gm = np.where((g_lo < _SILU_ARGMIN) & (_SILU_ARGMIN < g_hi), _SILU_ARGMIN, g_lo)
    s = [_silu(g_lo), _silu(g_hi), _silu(gm)]
    s_lo, s_hi = np.minimum.reduce(s), np.maximum.reduce(s)
    c = [s_lo * u_lo, s_lo * u_hi, s_hi * u_lo, s_hi * u_hi]
    return np.minimum.reduce(c), np.maximum.reduce(c)


def assert_swiglu_consistent(got, want, g64, u64, wg, wu, out, s_out=None, max_frac=2e-3):
    """Outputs of a fused gate/up GEMM + SwiGLU against the oracle.

    ``want`` is the oracle's SwiGLU of the correctly rounded bf16 gate/up.
    The kernel rounds its own binary32 accumulations, so its bf16 gate and
    up can differ from the correctly rounded ones -- by one ulp usually,
    by more where the sum cancels.  Every differing output must be the
    SwiGLU of some gate in [g64 - wg, g64 + wg] and up in [u64 - wu, u64 + wu]
    (the accumulation windows, ``accumulation_window``): its value must lie
    in the range of SiLU(g) * u over that box, widened by the
    specification's own error (2^-20 relative, a bound on its 4-ulp
    agreement with SiLU(g) * u) and by the output rounding (bf16: 2^-8
    relative; E4M3 with ``s_out``: 2^-4 relative, 2^-10 absolute, and
    saturation at 448).  The share of differing outputs must stay below
    ``max_frac``."""
    diff = got != want
    assert diff.mean() <= max_frac, diff.mean()
    if not diff.any():
        return
    g, u, dg, du = g64[diff], u64[diff], wg[diff], wu[diff]
    lo, hi = swiglu_range(g - dg, g + dg, u - du, u + du)
    lo = lo - 2.0 ** -20 * np.abs(lo)
    hi = hi + 2.0 ** -20 * np.abs(hi)
    if out == "bf16":
        v = O.bf16_decode(got[diff]).astype(np.float64)
        ok = (lo - 2.0 ** -8 * np.abs(lo) <= v) & (v <= hi + 2.0 ** -8 * np.abs(hi))
    else:
        s = float(np.float32(s_out))
        t_lo, t_hi = lo / s, hi / s
        t_lo = np.clip(t_lo - 2.0 ** -4 * np.abs(t_lo) - 2.0 ** -10, -448.0, 448.0)
        t_hi = np.clip(t_hi + 2.0 ** -4 * np.abs(t_hi) + 2.0 ** -10, -448.0, 448.0)
        v = O.e4m3_decode(got[diff]).astype(np.float64)
        ok = (t_lo <= v) & (v <= t_hi)
    assert ok.all(), (int((~ok).sum()), got[diff][~ok][:8], want[diff][~ok][:8], lo[~ok][:4], hi[~ok][:4])


def linear_problem(M, K, N, x_std=0.25, outliers=0.001, w_std=0.02, seed_x=0, seed_w=1, seed_cal=2,
                   w_mult=1.0):
    """x bf16 [M,K], E4M3 weight [N,K], calibrated s_in and s_w."""
    x = synth.activations_bf16(seed_x, (M, K), x_std, outlier_frac=outliers)
    xc = synth.activations_bf16(seed_cal, (min(M, 4096), K), x_std, outlier_frac=outliers)
    s_in = amax_scale(O.bf16_decode(xc))
    w = synth.normal_f32(seed_w, (N, K), w_std) * np.float32(w_mult)
    s_w = amax_scale(w)
    qw = O.e4m3_encode(w / s_w)
    return x, qw, s_in, s_w


@pytest.fixture(scope="session")
def W():
    import __graft_entry__ as g
    g.build()
    import w8a16_linear_gb300 as W
    W.device_check()
    return W
