"""Seeded synthetic GEMM inputs, shared by the tests, bench.py and the oracle
checks.

This module holds no GEMM arithmetic: it only draws numbers and quantises
them to the input formats (fp16, bf16, FP8 E4M3 / E5M2).  Both the CUDA path and the oracle are fed
the same host bytes produced here.

Generator.  Each matrix has its own 64-bit seed.  Element e (row-major index)
of a matrix uses the SplitMix64 output for counter e (Steele, Lea and Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014; the finaliser
constants are Stafford's "Mix13" variant as published with SplitMix64):

    x   = seed + (c + 1) * 0x9E3779B97F4A7C15          (mod 2^64)
    x   = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9
    x   = (x ^ (x >> 27)) * 0x94D049BB133111EB
    out = x ^ (x >> 31)

u = (out >> 11) * 2^-53 is uniform on [0, 1) with 53 random bits.

Distributions:
    uniform[lo, hi]  : lo + (hi - lo) * u           (counter c = e)
    normal(0, s^2)   : s * sqrt(-2 ln(1 - u1)) * cos(2 pi u2), Box-Muller with
                       u1 from counter 2e and u2 from counter 2e + 1 (only the
                       cosine branch is used)
    integers [lo,hi] : lo + floor((hi - lo + 1) * u)

Quantisation to the input format: fp16 by numpy's float64 -> float16
conversion (round to nearest, ties to even); bf16 by float64 -> float32
(ties to even) and then float32 -> bf16 keeping the upper 16 bits with ties
to even; FP8 E4M3 / E5M2 by float64 -> float32 -> torch's float8
conversion (ties to even).  Integers in [-2, 2] and all the values the workloads use are
representable, so the second rounding only shapes random real inputs.
"""
import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def splitmix64(seed, start, count):
    """SplitMix64 outputs for counters start .. start + count - 1."""
    with np.errstate(over="ignore"):
        c = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        x = np.uint64(seed) + c * GOLDEN
        x = (x ^ (x >> np.uint64(30))) * _M1
        x = (x ^ (x >> np.uint64(27))) * _M2
        return x ^ (x >> np.uint64(31))


def uniform01(seed, start, count):
    """53-bit uniforms on [0, 1) for counters start .. start + count - 1."""
    return (splitmix64(seed, start, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def f16_bits(x):
    """float64 -> IEEE binary16 bits (round to nearest, ties to even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def bf16_bits(x):
    """float64 -> float32 -> bfloat16 bits (each step ties to even)."""
    u = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32)
    u = u.astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    return ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def fp8_bits(x, dtype):
    """float64 -> FP8 E4M3 / E5M2 bits via float32 (each step ties to even;
    values must be within the format's finite range)."""
    import torch
    t = torch.from_numpy(np.asarray(x, dtype=np.float64).astype(np.float32))
    tdt = torch.float8_e4m3fn if dtype == "e4m3" else torch.float8_e5m2
    return t.to(tdt).view(torch.uint8).numpy().copy()


def quantise(x, dtype):
    if dtype in ("f16", "fp16", "float16"):
        return f16_bits(x)
    if dtype in ("bf16", "bfloat16"):
        return bf16_bits(x)
    if dtype in ("e4m3", "e5m2"):
        return fp8_bits(x, dtype)
    raise ValueError("input dtype must be f16, bf16, e4m3 or e5m2, got %r" % (dtype,))


def elem_dtype(dtype):
    """numpy storage type of the input format's bit patterns."""
    return np.uint8 if dtype in ("e4m3", "e5m2") else np.uint16


def _draw(dist, seed, start, count):
    kind = dist[0]
    if kind == "uniform":
        lo, hi = dist[1], dist[2]
        return lo + (hi - lo) * uniform01(seed, start, count)
    if kind == "normal":
        sigma = dist[1]
        u = uniform01(seed, 2 * start, 2 * count)
        u1, u2 = u[0::2], u[1::2]
        return sigma * np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * np.pi * u2)
    if kind == "int":
        lo, hi = dist[1], dist[2]
        return lo + np.floor((hi - lo + 1) * uniform01(seed, start, count))
    raise ValueError("unknown distribution %r" % (dist,))


def matrix(rows, cols, dist, seed, dtype, out=None):
    """A rows x cols row-major matrix of input bits (numpy uint16 for
    fp16/bf16, uint8 for e4m3/e5m2).

    dist is ("uniform", lo, hi), ("normal", sigma) or ("int", lo, hi).
    `out` may be a preallocated (rows, cols) array of that storage type (for
    example a pinned host buffer viewed through numpy).
    """
    n = rows * cols
    if out is None:
        out = np.empty((rows, cols), dtype=elem_dtype(dtype))
    flat = out.reshape(-1)

    def fill(s):
        c = min(_CHUNK, n - s)
        flat[s:s + c] = quantise(_draw(dist, seed, s, c), dtype)

    # Every element depends only on its own counter, so chunks are filled
    # independently, on several threads for large matrices (numpy releases
    # the interpreter lock inside these array operations).
    starts = range(0, n, _CHUNK)
    if len(starts) <= 1:
        for s in starts:
            fill(s)
    else:
        import concurrent.futures as cf
        import os
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(starts), os.cpu_count() or 1, 16))) as ex:
            list(ex.map(fill, starts))
    return out


from .workloads import (WORKLOADS, EXTRA_WORKLOADS, ATTN_WORKLOADS, MLA_WORKLOADS, workload,  # noqa: E402,F401
                        attn_workload, mla_workload, mla_inputs, inputs, stored)
