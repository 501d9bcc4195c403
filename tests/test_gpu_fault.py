"""Failure detection without a GPU fault: a bounded device wait that runs out.

The plan's test-only flag makes the first CTA (or CTA pair) skip one operand
load, so a barrier that the MMA issuer waits on is never completed.  Every
device wait is bounded in time (here 50 ms): the kernel must record
TSGEMM_ERR_TIMEOUT in the plan's status word, let its in-flight copies land,
free tensor memory and return -- the stream synchronises in well under a
second and the context stays usable for the next GEMM.
"""
import time

import pytest

import oracle
import synth
from gpu_util import TORCH_DT, from_dev, run_gemm, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("block_m", [128, 256])
def test_expired_wait_reports_timeout_and_the_context_survives(block_m):
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    M, N, K = 512, 512, 1024
    A_bits = synth.matrix(M, K, ("int", -2, 2), 0xFA01, "bf16")
    B_bits = synth.matrix(K, N, ("int", -2, 2), 0xFA02, "bf16")
    A, B = to_dev(A_bits, "bf16"), to_dev(B_bits, "bf16")
    C = torch.zeros((M, N), dtype=TORCH_DT["f32"], device="cuda")
    plan = tsgemm.Plan(M, N, K, "bf16", "f32", block_m=block_m, block_n=128, splits=1, timeout_ms=50,
                       debug_flags=tsgemm.DEBUG_SKIP_FIRST_LOAD)
    assert plan.config["timeout_ms"] == 50
    t0 = time.time()
    plan.run(A, B, C)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert elapsed < 10.0, "the bounded waits took %.1f s" % elapsed
    assert plan.status() == tsgemm.ERR_TIMEOUT
    assert plan.status() == tsgemm.OK  # reading the timeout cleared it
    plan.close()
    # The device is still healthy: the same GEMM without the fault is exact.
    out, _ = run_gemm(A_bits, B_bits, "bf16", "f32", block_m=block_m)
    ref, sabs, _ = oracle.gemm(A_bits, B_bits, "bf16")
    ok, info = oracle.accept(out, ref, sabs, "f32", exact=True)
    assert ok, info


def test_timeout_does_not_disturb_other_ctas():
    # CTAs other than the first are not affected by the injected fault: the
    # tiles they own are still correct.
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    M, N, K = 1024, 512, 512
    A_bits = synth.matrix(M, K, ("int", -2, 2), 0xFA03, "bf16")
    B_bits = synth.matrix(K, N, ("int", -2, 2), 0xFA04, "bf16")
    A, B = to_dev(A_bits, "bf16"), to_dev(B_bits, "bf16")
    C = torch.full((M, N), float("nan"), dtype=TORCH_DT["f32"], device="cuda")
    plan = tsgemm.Plan(M, N, K, "bf16", "f32", block_m=128, block_n=128, splits=1, group_m=1,
                       timeout_ms=50, debug_flags=tsgemm.DEBUG_SKIP_FIRST_LOAD)
    cfg = plan.config
    plan.run(A, B, C)
    torch.cuda.synchronize()
    assert plan.status() == tsgemm.ERR_TIMEOUT
    got = from_dev(C, "f32")
    ref, sabs, _ = oracle.gemm(A_bits, B_bits, "bf16")
    # With group_m = 1 tile t is (t % tiles_m, t / tiles_m); CTA 0 owns the
    # units 0, grid, 2 * grid, ...; every other tile must be exact.
    tiles_m, tiles_n = M // 128, N // 128
    bad_tiles = {u for u in range(0, tiles_m * tiles_n, cfg["grid"])}
    for t in range(tiles_m * tiles_n):
        if t in bad_tiles:
            continue
        tm, tn = t % tiles_m, t // tiles_m
        blk = (slice(tm * 128, tm * 128 + 128), slice(tn * 128, tn * 128 + 128))
        ok, info = oracle.accept(got[blk], ref[blk], sabs[blk], "f32", exact=True)
        assert ok, (t, info)
    plan.close()
