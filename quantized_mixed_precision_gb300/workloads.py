"""Seeded synthetic inputs for the five hot-path workloads.

This module only draws random numbers and holds shapes; it contains none of
the quantise / pack / GEMM arithmetic, so both the CUDA library's tests and
the CPU oracle can be fed from it without sharing any of the method.

Recipe (one ``numpy.random.default_rng(seed)`` stream per workload, arrays
drawn in the order activations, weights, scales):

* int8 operands: uniform integers in [-128, 127] (inclusive).
* int4 codes: uniform integers in [-8, 7].
* ternary codes: uniform over {-1, 0, 1} (P(0) = 1/3).
* normal fp16 tensors: float32 standard normals times the std, cast to fp16
  with round-to-nearest-even.
* uniform fp16 scales: float64 uniform in [lo, hi), cast to fp32, then fp16.

The shapes are those of the pages' workloads: the BitBLAS guide's 256^3 test
and 1024^3 / 4096^3 tuning squares, LLM-layer weights N x K with a dynamic
activation row count M in [1, 1024], and BitNet-b1.58 style ternary weights.
No dataset or trained weight is involved.
"""

from __future__ import annotations

import numpy as np


def rng_for(seed: int = 0) -> np.random.Generator:
    return np.random.default_rng(seed)


def int8_uniform(rng, shape):
    return rng.integers(-128, 128, size=shape, dtype=np.int8)


def int4_uniform(rng, shape):
    return rng.integers(-8, 8, size=shape, dtype=np.int8)


def int2_uniform(rng, shape):
    """All four 2-bit two's-complement codes, {-2, -1, 0, 1}."""
    return rng.integers(-2, 2, size=shape, dtype=np.int8)


def ternary(rng, shape):
    return rng.integers(-1, 2, size=shape, dtype=np.int8)


def normal_f16(rng, shape, std=1.0):
    return (rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float16)


def uniform_f16(rng, shape, lo, hi):
    return rng.uniform(lo, hi, size=shape).astype(np.float32).astype(np.float16)


# --------------------------------------------------------------------------
# The five workloads.  Each returns a dict of host numpy arrays.
# --------------------------------------------------------------------------
CFG0 = dict(M=256, N=256, K=256)                  # INT8 x INT4, int32 out
CFG1 = dict(M=1024, N=4096, K=4096)               # quantise + INT8 x INT8, fp16 out
CFG2 = dict(M=4096, N=4096, K=4096)               # INT8 x INT4 + per-column dequant
CFG3 = dict(N=11008, K=4096, Ms=(1, 4, 16, 64, 256, 1024))   # fp16 x INT4
CFG4 = dict(N=8192, K=8192, Ms=(1, 128, 1024))    # INT8 x ternary, fp16 out


def cfg0(seed=0, M=256, N=256, K=256):
    rng = rng_for(seed)
    return dict(A=int8_uniform(rng, (M, K)), B=int4_uniform(rng, (N, K)))


def cfg1(seed=0, M=1024, N=4096, K=4096):
    """fp16 activations X ~ N(0, 1) and fp16 weights W ~ N(0, 0.02)."""
    rng = rng_for(seed)
    x = normal_f16(rng, (M, K), 1.0)
    w = normal_f16(rng, (N, K), 0.02)
    return dict(X=x, W=w)


def cfg2(seed=0, M=4096, N=4096, K=4096):
    rng = rng_for(seed)
    a = int8_uniform(rng, (M, K))
    b = int4_uniform(rng, (N, K))
    s = uniform_f16(rng, (N,), 1e-3, 1e-2)
    return dict(A=a, B=b, scale=s)


def cfg3(seed=0, M=1, N=11008, K=4096, source=True):
    """fp16 X ~ N(0, 1); 4-bit codes uniform in [-8, 7]; and the Normal(0,
    0.02) source matrix whose per-row absmax / 7 gives the channel scale
    (the scale itself is computed by the quantiser under test or by the
    oracle, never here)."""
    rng = rng_for(seed)
    x = normal_f16(rng, (M, K), 1.0)
    w = int4_uniform(rng, (N, K))
    out = dict(X=x, W=w)
    if source:
        out["S"] = normal_f16(rng, (N, K), 0.02)
    return out


def cfg4(seed=0, M=1, N=8192, K=8192):
    rng = rng_for(seed)
    a = int8_uniform(rng, (M, K))
    b = ternary(rng, (N, K))
    s = uniform_f16(rng, (N,), 0.5, 2.0)
    return dict(A=a, B=b, scale=s)
