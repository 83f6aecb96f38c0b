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


def bf16_neighbour(bits, d):
    """The bf16 bit pattern ``d`` steps away from ``bits`` in the order of
    the values (finite inputs; +0 and -0 are the same point)."""
    b = np.asarray(bits, np.uint16).astype(np.int64)
    o = np.where(b & 0x8000, -(b & 0x7FFF), b) + int(d)
    return np.where(o >= 0, o, 0x8000 | (-o)).astype(np.uint16)


def assert_swiglu_within_one_ulp(got, want, g_rn, u_rn, spec, max_frac):
    """Outputs of a fused gate/up GEMM + SwiGLU against the oracle.

    ``want = spec(g_rn, u_rn)`` with ``g_rn``, ``u_rn`` the correctly rounded
    bf16 gate/up.  The kernel rounds its own F32 accumulations, whose order
    differs from the exact sum, so its bf16 gate or up may sit one bf16 ulp
    away from the correctly rounded value.  Every output that differs must
    therefore be ``spec(g', u')`` for g' and u' each within one ulp of
    ``g_rn`` and ``u_rn``; no other difference is accepted, and the share of
    differing outputs must stay below ``max_frac``."""
    diff = got != want
    assert diff.mean() <= max_frac, diff.mean()
    if not diff.any():
        return
    g, u, gd = g_rn[diff], u_rn[diff], got[diff]
    explained = np.zeros(gd.shape, bool)
    for dg in (-1, 0, 1):
        for du in (-1, 0, 1):
            if dg == 0 and du == 0:
                continue
            explained |= spec(bf16_neighbour(g, dg), bf16_neighbour(u, du)) == gd
    assert explained.all(), (int((~explained).sum()), gd[~explained][:8], want[diff][~explained][:8])


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
