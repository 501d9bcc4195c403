"""Parity of the DSMEM cluster split against the fp64 oracle: the cs CTAs
of a cs x 1 cluster (cs = 2, 4, 8) compute cs consecutive parts of every
tile's K range; CTA r receives the fp32 sum of parts 0..r-1 from CTA r - 1
through distributed shared memory, chunk by chunk, adds its own and passes
it on, and the last CTA stores C (the parts summed in K order).
"""
import time

import numpy as np
import pytest

import oracle
import synth
from gpu_util import TORCH_DT, run_gemm, to_dev

pytestmark = pytest.mark.gpu

SIZES = [2, 4, 8]


def CS(cs):
    return dict(block_m=128, cluster_split=cs)


def _ints(rows, cols, seed, din="bf16", lo=-4, hi=4):
    return synth.matrix(rows, cols, ("int", lo, hi), seed, din)


def _check(C, A, B, din, dout, exact):
    ref, sabs, _ = oracle.gemm(A, B, din)
    ok, info = oracle.accept(C, ref, sabs, dout, exact=exact)
    assert ok, info


@pytest.mark.parametrize("cs", SIZES)
@pytest.mark.parametrize("block_n", [64, 128, 192, 256])
@pytest.mark.parametrize("dout", ["f32", "bf16"])
def test_integer_exact(cs, block_n, dout):
    M, N, K = 640, 768, 1088  # K = 17 slices: parts of unequal length
    A = _ints(M, K, 61)
    B = _ints(K, N, 62)
    C, cfg = run_gemm(A, B, "bf16", dout, block_n=block_n, **CS(cs))
    assert cfg["cluster_split"] == cs and cfg["grid"] % cs == 0
    _check(C, A, B, "bf16", dout, exact=True)


@pytest.mark.parametrize("cs", SIZES)
@pytest.mark.parametrize("shape", [(129, 264, 136), (1000, 1288, 328), (128, 128, 128), (2048, 1024, 4096),
                                   (128, 256, 520)])
def test_ragged_and_multi_round(cs, shape):
    M, N, K = shape
    if -(-K // 64) < cs:
        pytest.skip("fewer K slices than CTAs per cluster (the planner refuses it)")
    A = _ints(M, K, 63)
    B = _ints(K, N, 64)
    C, _ = run_gemm(A, B, "bf16", "f32", **CS(cs))
    _check(C, A, B, "bf16", "f32", exact=True)


@pytest.mark.parametrize("cs", SIZES)
def test_one_slice_per_cta(cs):
    # K = cs slices: every CTA of the cluster contributes exactly one
    M, N, K = 256, 512, 64 * cs
    A = _ints(M, K, 69)
    B = _ints(K, N, 70)
    C, _ = run_gemm(A, B, "bf16", "f32", **CS(cs))
    _check(C, A, B, "bf16", "f32", exact=True)


@pytest.mark.parametrize("cs", SIZES)
@pytest.mark.parametrize("din,dout", [("f16", "f32"), ("f16", "f16"), ("bf16", "bf16")])
def test_random_inputs_and_repeatable_bits(cs, din, dout):
    M, N, K = 512, 1024, 2048
    A = synth.matrix(M, K, ("uniform", -1.0, 1.0), 65, din)
    B = synth.matrix(K, N, ("uniform", -1.0, 1.0), 66, din)
    outs, _ = run_gemm(A, B, din, dout, repeat=2, **CS(cs))
    assert np.array_equal(outs[0], outs[1])
    _check(outs[0], A, B, din, dout, exact=False)


def test_skinny_projection_shape():
    # the shape of the weight-streaming projection (M = 128, K = 8192), its
    # K range cut into 8 parts per tile; checked against the oracle on
    # integer inputs, bit for bit
    M, N, K = 128, 4096, 8192
    A = _ints(M, K, 71, lo=-2, hi=2)
    B = _ints(K, N, 72, lo=-2, hi=2)
    C, cfg = run_gemm(A, B, "bf16", "f32", **CS(8))
    assert cfg["cluster_split"] == 8
    _check(C, A, B, "bf16", "f32", exact=True)


@pytest.mark.parametrize("cs", [2, 8])
def test_expired_wait_reports_timeout_and_the_context_survives(cs):
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    M, N, K = 512, 512, 1024
    A_bits = _ints(M, K, 67, lo=-2, hi=2)
    B_bits = _ints(K, N, 68, lo=-2, hi=2)
    A, B = to_dev(A_bits, "bf16"), to_dev(B_bits, "bf16")
    C = torch.zeros((M, N), dtype=TORCH_DT["f32"], device="cuda")
    plan = tsgemm.Plan(M, N, K, "bf16", "f32", timeout_ms=50, debug_flags=tsgemm.DEBUG_SKIP_FIRST_LOAD, **CS(cs))
    t0 = time.time()
    plan.run(A, B, C)
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    assert plan.status() == tsgemm.ERR_TIMEOUT
    plan.close()
    out, _ = run_gemm(A_bits, B_bits, "bf16", "f32", **CS(cs))
    _check(out, A_bits, B_bits, "bf16", "f32", exact=True)
