"""The five seeded GEMM workloads: shapes, formats, distributions and seeds.

Seeds: A uses 0x7E5A0000 + index, B uses 0x7E5A0000 + index + 0x100, where
index is the workload's position in this table (0-based).  A is generated
before B; both are row-major.
"""
import numpy as np

_SEED_BASE = 0x7E5A0000

# name -> description; "exact" marks integer-valued inputs whose fp32 partial
# sums are exact, so the result is checked bit for bit.
WORKLOADS = {
    "gemm_256_f16_f32": dict(
        index=0, M=256, N=256, K=256, dtype_in="f16", dtype_out="f32",
        dist_a=("uniform", -1.0, 1.0), dist_b=("uniform", -1.0, 1.0),
        exact=False, cluster=None),
    "gemm_4096_bf16": dict(
        index=1, M=4096, N=4096, K=4096, dtype_in="bf16", dtype_out="bf16",
        dist_a=("normal", 1.0), dist_b=("normal", 1.0),
        exact=False, cluster=None),
    "skinny_128x28672x8192_bf16": dict(
        index=2, M=128, N=28672, K=8192, dtype_in="bf16", dtype_out="bf16",
        dist_a=("normal", 1.0), dist_b=("normal", 0.02),
        exact=False, cluster=None),
    "gemm_16384x16384x8192_bf16": dict(
        index=3, M=16384, N=16384, K=8192, dtype_in="bf16", dtype_out="bf16",
        dist_a=("uniform", -1.0, 1.0), dist_b=("uniform", -1.0, 1.0),
        exact=False, cluster=(2, 1)),
    "longk_1024x1024x65536_int_f32": dict(
        index=4, M=1024, N=1024, K=65536, dtype_in="bf16", dtype_out="f32",
        dist_a=("int", -2, 2), dist_b=("int", -2, 2),
        exact=True, cluster=None),
}


def workload(name):
    w = dict(WORKLOADS[name])
    w["name"] = name
    w["seed_a"] = _SEED_BASE + w["index"]
    w["seed_b"] = _SEED_BASE + w["index"] + 0x100
    w["flops"] = 2 * w["M"] * w["N"] * w["K"]
    return w


def inputs(name, out_a=None, out_b=None):
    """(A_bits, B_bits) numpy uint16 arrays for a named workload."""
    from . import matrix
    w = workload(name)
    A = matrix(w["M"], w["K"], w["dist_a"], w["seed_a"], w["dtype_in"], out=out_a)
    B = matrix(w["K"], w["N"], w["dist_b"], w["seed_b"], w["dtype_in"], out=out_b)
    return A, B


def out_nbytes(dtype_out):
    return 4 if dtype_out == "f32" else 2


def out_numpy_dtype(dtype_out):
    return np.float32 if dtype_out == "f32" else np.uint16
