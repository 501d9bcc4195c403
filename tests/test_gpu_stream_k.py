"""Parity of stream-K scheduling against the fp64 oracle.

The K slices of the schedule's last tiles are spread evenly over all CTAs
(or CTA pairs); a tile cut between CTAs is finished by the CTA that holds
its first K slices, which adds the other parts' fp32 partials in K order.
The cases cover the owner reading one partial and several, from the idle
operand ring (bulk copies) and straight from global memory, one-SM tiles,
CTA pairs, the 8-bit inputs, ragged shapes and an
expired bounded wait.  Integer inputs make every order of fp32 addition
exact, so those results are compared bit for bit.
"""
import time

import numpy as np
import pytest

import oracle
import synth
from gpu_util import TORCH_DT, run_gemm, to_dev

pytestmark = pytest.mark.gpu


def _ints(rows, cols, seed, din="bf16", lo=-4, hi=4):
    return synth.matrix(rows, cols, ("int", lo, hi), seed, din)


def _check(C, A, B, din, dout, exact):
    ref, sabs, _ = oracle.gemm(A, B, din)
    ok, info = oracle.accept(C, ref, sabs, dout, exact=exact)
    assert ok, info


CASES = [
    # (M, N, K, force): pairs, tiles cut in ~5 parts (owner reads from global)
    (1024, 1024, 4096, dict(block_m=256, block_n=256, stream_k_tiles=16)),
    # pairs, two rounds of whole tiles then tiles cut in two (ring-staged)
    (4096, 4096, 1024, dict(block_m=256, block_n=256, stream_k_tiles=104)),
    # one-SM 128 x 128 tiles cut in up to 3 parts (ring-staged)
    (1024, 1024, 2048, dict(block_m=128, block_n=128, stream_k_tiles=64)),
    # one-SM, ragged M / N / K, a few tiles
    (1000, 1288, 328, dict(block_m=128, block_n=128, stream_k_tiles=30)),
    # pairs, ragged N
    (2048, 2304, 1024, dict(block_m=256, block_n=256, stream_k_tiles=20)),
    # pairs with 128-wide tiles
    (1536, 1536, 2560, dict(block_m=256, block_n=128, stream_k_tiles=30)),
]


@pytest.mark.parametrize("M,N,K,force", CASES)
@pytest.mark.parametrize("dout", ["f32", "bf16"])
def test_integer_exact(M, N, K, force, dout):
    A = _ints(M, K, 51)
    B = _ints(K, N, 52)
    C, cfg = run_gemm(A, B, "bf16", dout, **force)
    assert cfg["stream_k_tiles"] == force["stream_k_tiles"]
    _check(C, A, B, "bf16", dout, exact=True)


@pytest.mark.parametrize("layout", ["rcr", "crr", "ccr"])
def test_layouts(layout):
    M, N, K = 1024, 1024, 2048
    A = _ints(M, K, 53)
    B = _ints(K, N, 54)
    C, _ = run_gemm(A, B, "bf16", "f32", layout=layout, block_m=256, block_n=256, stream_k_tiles=16)
    _check(C, A, B, "bf16", "f32", exact=True)


@pytest.mark.parametrize("M,N,K,force", CASES[:3])
def test_random_inputs_and_repeatable_bits(M, N, K, force):
    A = synth.matrix(M, K, ("normal", 1.0), 55, "bf16")
    B = synth.matrix(K, N, ("normal", 1.0), 56, "bf16")
    outs, _ = run_gemm(A, B, "bf16", "f32", repeat=2, **force)
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    _check(outs[0], A, B, "bf16", "f32", exact=False)


def test_fp8():
    M, N, K = 2048, 2048, 2048
    A = _ints(M, K, 57, "e4m3")
    B = _ints(K, N, 58, "e4m3")
    C, _ = run_gemm(A, B, "e4m3", "f32", layout="rcr", block_m=256, block_n=256, stream_k_tiles=64)
    _check(C, A, B, "e4m3", "f32", exact=True)


def test_expired_wait_reports_timeout_and_the_context_survives():
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    M, N, K = 1024, 1024, 2048
    A_bits = _ints(M, K, 59, lo=-2, hi=2)
    B_bits = _ints(K, N, 60, lo=-2, hi=2)
    A, B = to_dev(A_bits, "bf16"), to_dev(B_bits, "bf16")
    C = torch.zeros((M, N), dtype=TORCH_DT["f32"], device="cuda")
    plan = tsgemm.Plan(M, N, K, "bf16", "f32", block_m=256, block_n=256, stream_k_tiles=16, timeout_ms=50,
                       debug_flags=tsgemm.DEBUG_SKIP_FIRST_LOAD)
    t0 = time.time()
    plan.run(A, B, C)
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    assert plan.status() == tsgemm.ERR_TIMEOUT
    plan.close()
    out, _ = run_gemm(A_bits, B_bits, "bf16", "f32", block_m=256, block_n=256, stream_k_tiles=16)
    _check(out, A_bits, B_bits, "bf16", "f32", exact=True)
