"""Parity of the two-pair cluster form (4 CTAs: two CTA pairs computing
adjacent 256 x 256 tiles of the same A rows, the A tiles shared by TMA
multicast) against the fp64 oracle.

Covers every operand layout, output format and the 8-bit inputs, ragged
shapes whose last tile column has no partner tile (the second pair then
runs on zero-filled B and its stores are clipped), split-K on all units and
on the tail wave, and a bounded wait that runs out.
"""
import time

import numpy as np
import pytest

import oracle
import synth
from gpu_util import TORCH_DT, run_gemm, to_dev

pytestmark = pytest.mark.gpu

MC = dict(block_m=256, block_n=256, cluster_n=2)


def _ints(rows, cols, seed, din="bf16", lo=-4, hi=4):
    return synth.matrix(rows, cols, ("int", lo, hi), seed, din)


def _check(C, A, B, din, dout, exact):
    ref, sabs, _ = oracle.gemm(A, B, din)
    ok, info = oracle.accept(C, ref, sabs, dout, exact=exact)
    assert ok, info


def test_plan_uses_two_pairs_per_cluster():
    from hierarchical_gemm_gb300 import tsgemm
    plan = tsgemm.Plan(1024, 1024, 512, "bf16", "bf16", **MC)
    cfg = plan.config
    plan.close()
    assert cfg["cluster_n"] == 2 and cfg["grid"] % 4 == 0
    assert cfg["units"] == 4 * 2  # 4 tile rows x 2 column pairs


@pytest.mark.parametrize("layout", ["rrr", "rcr", "crr", "ccr"])
def test_permutation_and_identity(layout):
    r = np.random.default_rng(31)
    n = 512
    perm = r.permutation(n)
    P = np.zeros((n, n))
    P[np.arange(n), perm] = 1.0
    Pb = synth.quantise(P, "bf16")
    B = _ints(n, 768, 32, lo=-16, hi=16)
    C, cfg = run_gemm(Pb, B, "bf16", "bf16", layout=layout, **MC)
    assert cfg["cluster_n"] == 2
    _check(C, Pb, B, "bf16", "bf16", exact=True)
    A = _ints(768, n, 33, lo=-16, hi=16)
    C, _ = run_gemm(A, Pb, "bf16", "bf16", layout=layout, **MC)
    _check(C, A, Pb, "bf16", "bf16", exact=True)


@pytest.mark.parametrize("shape", [(512, 512, 512), (300, 264, 200), (1000, 1288, 328), (256, 256, 64)])
@pytest.mark.parametrize("layout", ["rrr", "rcr"])
@pytest.mark.parametrize("dout", ["f32", "bf16"])
def test_integer_shapes(shape, layout, dout):
    M, N, K = shape
    A = _ints(M, K, 34)
    B = _ints(K, N, 35)
    C, _ = run_gemm(A, B, "bf16", dout, layout=layout, **MC)
    _check(C, A, B, "bf16", dout, exact=True)


@pytest.mark.parametrize("splits,split_tiles", [(2, 0), (3, 0), (2, 3), (4, 1)])
def test_split_k(splits, split_tiles):
    M, N, K = 1024, 1536, 2048
    A = _ints(M, K, 36)
    B = _ints(K, N, 37)
    force = dict(MC, splits=splits)
    if split_tiles:
        force["split_tiles"] = split_tiles
    C, cfg = run_gemm(A, B, "bf16", "f32", **force)
    assert cfg["splits"] == splits
    _check(C, A, B, "bf16", "f32", exact=True)


@pytest.mark.parametrize("din,dout", [("f16", "f32"), ("f16", "f16"), ("bf16", "bf16")])
def test_random_inputs(din, dout):
    M, N, K = 768, 1024, 1600
    A = synth.matrix(M, K, ("uniform", -1.0, 1.0), 38, din)
    B = synth.matrix(K, N, ("uniform", -1.0, 1.0), 39, din)
    C, _ = run_gemm(A, B, din, dout, **MC)
    _check(C, A, B, din, dout, exact=False)


@pytest.mark.parametrize("din", ["e4m3", "e5m2"])
def test_fp8(din):
    M, N, K = 768, 1280, 1040
    A = _ints(M, K, 40, din)
    B = _ints(K, N, 41, din)
    C, _ = run_gemm(A, B, din, "f32", layout="rcr", **MC)
    _check(C, A, B, din, "f32", exact=True)
    A = synth.matrix(M, K, ("normal", 1.0), 42, din)
    B = synth.matrix(K, N, ("normal", 1.0), 43, din)
    C, _ = run_gemm(A, B, din, "bf16", layout="rcr", **MC)
    _check(C, A, B, din, "bf16", exact=False)


def test_4096_bf16_sampled():
    M = N = K = 4096
    A = synth.matrix(M, K, ("normal", 1.0), 44, "bf16")
    B = synth.matrix(K, N, ("normal", 1.0), 45, "bf16")
    C, cfg = run_gemm(A, B, "bf16", "bf16", **MC)
    r = np.random.default_rng(46)
    rows = np.concatenate([r.integers(0, M, 4096), np.full(N, 777), np.arange(M)])
    cols = np.concatenate([r.integers(0, N, 4096), np.arange(N), np.full(M, 2049)])
    ref, sabs = oracle.gemm_sampled(A, B, "bf16", rows, cols)
    ok, info = oracle.accept(C[rows, cols], ref, sabs, "bf16", exact=False)
    assert ok, (cfg, info)


def test_expired_wait_reports_timeout_and_the_context_survives():
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    M, N, K = 512, 1024, 1024
    A_bits = _ints(M, K, 47, lo=-2, hi=2)
    B_bits = _ints(K, N, 48, lo=-2, hi=2)
    A, B = to_dev(A_bits, "bf16"), to_dev(B_bits, "bf16")
    C = torch.zeros((M, N), dtype=TORCH_DT["f32"], device="cuda")
    plan = tsgemm.Plan(M, N, K, "bf16", "f32", splits=1, timeout_ms=50,
                       debug_flags=tsgemm.DEBUG_SKIP_FIRST_LOAD, **MC)
    t0 = time.time()
    plan.run(A, B, C)
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    assert plan.status() == tsgemm.ERR_TIMEOUT
    plan.close()
    out, _ = run_gemm(A_bits, B_bits, "bf16", "f32", **MC)
    _check(out, A_bits, B_bits, "bf16", "f32", exact=True)
