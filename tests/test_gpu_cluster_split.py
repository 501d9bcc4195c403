"""Parity of the DSMEM cluster split against the fp64 oracle: the two CTAs
of a 2 x 1 cluster compute the two halves of every tile's K range, and
CTA 1 hands its fp32 accumulator to CTA 0 through distributed shared
memory, chunk by chunk; CTA 0 adds it after its own (K order) and stores C.
"""
import time

import numpy as np
import pytest

import oracle
import synth
from gpu_util import TORCH_DT, run_gemm, to_dev

pytestmark = pytest.mark.gpu

CS = dict(block_m=128, cluster_split=2)


def _ints(rows, cols, seed, din="bf16", lo=-4, hi=4):
    return synth.matrix(rows, cols, ("int", lo, hi), seed, din)


def _check(C, A, B, din, dout, exact):
    ref, sabs, _ = oracle.gemm(A, B, din)
    ok, info = oracle.accept(C, ref, sabs, dout, exact=exact)
    assert ok, info


@pytest.mark.parametrize("block_n", [64, 128, 192, 256])
@pytest.mark.parametrize("dout", ["f32", "bf16"])
def test_integer_exact(block_n, dout):
    M, N, K = 640, 768, 1088  # K = 17 slices: the halves are 8 and 9 slices
    A = _ints(M, K, 61)
    B = _ints(K, N, 62)
    C, cfg = run_gemm(A, B, "bf16", dout, block_n=block_n, **CS)
    assert cfg["cluster_split"] == 2 and cfg["grid"] % 2 == 0
    _check(C, A, B, "bf16", dout, exact=True)


@pytest.mark.parametrize("shape", [(129, 264, 136), (1000, 1288, 328), (128, 128, 128), (2048, 1024, 4096)])
def test_ragged_and_multi_round(shape):
    M, N, K = shape
    A = _ints(M, K, 63)
    B = _ints(K, N, 64)
    C, _ = run_gemm(A, B, "bf16", "f32", **CS)
    _check(C, A, B, "bf16", "f32", exact=True)


@pytest.mark.parametrize("din,dout", [("f16", "f32"), ("f16", "f16"), ("bf16", "bf16")])
def test_random_inputs_and_repeatable_bits(din, dout):
    M, N, K = 512, 1024, 2048
    A = synth.matrix(M, K, ("uniform", -1.0, 1.0), 65, din)
    B = synth.matrix(K, N, ("uniform", -1.0, 1.0), 66, din)
    outs, _ = run_gemm(A, B, din, dout, repeat=2, **CS)
    assert np.array_equal(outs[0], outs[1])
    _check(outs[0], A, B, din, dout, exact=False)


def test_expired_wait_reports_timeout_and_the_context_survives():
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    M, N, K = 512, 512, 1024
    A_bits = _ints(M, K, 67, lo=-2, hi=2)
    B_bits = _ints(K, N, 68, lo=-2, hi=2)
    A, B = to_dev(A_bits, "bf16"), to_dev(B_bits, "bf16")
    C = torch.zeros((M, N), dtype=TORCH_DT["f32"], device="cuda")
    plan = tsgemm.Plan(M, N, K, "bf16", "f32", timeout_ms=50, debug_flags=tsgemm.DEBUG_SKIP_FIRST_LOAD, **CS)
    t0 = time.time()
    plan.run(A, B, C)
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    assert plan.status() == tsgemm.ERR_TIMEOUT
    plan.close()
    out, _ = run_gemm(A_bits, B_bits, "bf16", "f32", **CS)
    _check(out, A_bits, B_bits, "bf16", "f32", exact=True)
