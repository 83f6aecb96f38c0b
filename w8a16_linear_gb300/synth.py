"""Seeded synthetic inputs shaped like the workloads of a static-FP8
diffusion transformer (4096-wide projections, ~20k latent tokens).

This module only draws random numbers.  It holds none of the linear
layer's arithmetic (no quantization, no scales, no GEMM), so the tests can
feed the same inputs to the CUDA path and to the CPU oracle.

All draws use a torch CPU generator seeded per tensor, so a given
``(seed, shape)`` always gives the same values on every machine.  bf16
activations are returned as their uint16 bit patterns.
"""

import numpy as np
import torch


def _gen(seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal_f32(seed, shape, std):
    """float32 N(0, std^2) draw."""
    t = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32) * float(std)
    return t.numpy()


def activations_bf16(seed, shape, std, outlier_frac=0.0, outlier_mult=8.0, mean=0.0):
    """bf16 activations ~ N(mean, std^2), with a fraction of randomly placed
    elements multiplied by ``outlier_mult`` (heavy-tailed channels of a
    diffusion transformer's hidden state).  Returns uint16 bf16 bits."""
    g = _gen(seed)
    t = torch.randn(*shape, generator=g, dtype=torch.float32) * float(std)
    if outlier_frac > 0:
        n = t.numel()
        k = max(1, int(round(n * outlier_frac)))
        idx = torch.randint(0, n, (k,), generator=g)
        t.view(-1)[idx] *= float(outlier_mult)
    if mean:
        t += float(mean)
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def activations_f16(seed, shape, std):
    """float16 activations ~ N(0, std^2); returns uint16 binary16 bits."""
    t = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32) * float(std)
    return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)


def uniform_f32(seed, shape, lo, hi):
    """float32 U[lo, hi) draw."""
    t = torch.rand(*shape, generator=_gen(seed), dtype=torch.float32)
    return (t * float(hi - lo) + float(lo)).numpy()


def random_bf16_bits(seed, shape, lo_bits=0, hi_bits=1 << 16):
    """Uniformly random bf16 bit patterns in ``[lo_bits, hi_bits)``."""
    t = torch.randint(lo_bits, hi_bits, tuple(shape), generator=_gen(seed), dtype=torch.int32)
    return t.numpy().astype(np.uint16)


def random_rows(seed, m, k):
    """``k`` distinct sorted row indices out of ``m`` (sampled checks)."""
    p = torch.randperm(m, generator=_gen(seed))[:k]
    return np.sort(p.numpy())
