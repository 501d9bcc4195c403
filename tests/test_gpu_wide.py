"""Parity of the 256 x 512 CTA-pair tiles against the fp64 oracle.

A wide tile's two 256-column halves are the two accumulators of tensor
memory; each K slice's A feeds two N = 256 MMAs, each CTA holding one
128-column piece of B per half.  The planner takes them for large
whole-tile schedules (see test_wide_pair_tiles_rule in the host tests);
here they are forced on shapes that exercise ragged edges, both B
layouts, 8-bit inputs and stream-K over wide tiles.
"""
import pytest

import oracle
import synth
from gpu_util import run_gemm

pytestmark = pytest.mark.gpu

W = dict(block_m=256, block_n=512)


def _ints(rows, cols, seed, din="bf16", lo=-3, hi=3):
    return synth.matrix(rows, cols, ("int", lo, hi), seed, din)


def _check(C, A, B, din, dout, exact):
    ref, sabs, _ = oracle.gemm(A, B, din)
    ok, info = oracle.accept(C, ref, sabs, dout, exact=exact)
    assert ok, info


@pytest.mark.parametrize("layout", ["rrr", "rcr"])
@pytest.mark.parametrize("M,N,K,dout", [(512, 1024, 640, "f32"), (256, 512, 64, "bf16"), (1000, 1504, 704, "f32"),
                                        (2048, 2560, 1088, "bf16"), (300, 600, 200, "f16")])
def test_integer_exact(layout, M, N, K, dout):
    din = "f16" if dout == "f16" else "bf16"
    A = _ints(M, K, 71 + M, din)
    B = _ints(K, N, 72 + N, din)
    C, cfg = run_gemm(A, B, din, dout, layout=layout, **W)
    assert cfg["block_n"] == 512 and cfg["stream_k_tiles"] == 0
    _check(C, A, B, din, dout, exact=True)


def test_random_inputs():
    A = synth.matrix(768, 1024, ("normal", 1.0), 73, "bf16")
    B = synth.matrix(1024, 1536, ("normal", 1.0), 74, "bf16")
    C, _ = run_gemm(A, B, "bf16", "bf16", **W)
    _check(C, A, B, "bf16", "bf16", exact=False)


def test_e4m3():
    A = synth.matrix(512, 1024, ("normal", 1.0), 75, "e4m3")
    B = synth.matrix(1024, 1024, ("normal", 1.0), 76, "e4m3")
    C, _ = run_gemm(A, B, "e4m3", "bf16", layout="rcr", **W)
    _check(C, A, B, "e4m3", "bf16", exact=False)


@pytest.mark.parametrize("M,N,K,sk", [(1024, 2048, 4096, 4), (2048, 2560, 1088, 10), (4096, 4096, 4096, 52),
                                      (4096, 4096, 4096, 128)])
def test_stream_k_over_wide_tiles(M, N, K, sk):
    A = _ints(M, K, 77 + M, lo=-2, hi=2)
    B = _ints(K, N, 78 + N, lo=-2, hi=2)
    C, cfg = run_gemm(A, B, "bf16", "f32", stream_k_tiles=sk, **W)
    assert cfg["stream_k_tiles"] == sk
    _check(C, A, B, "bf16", "f32", exact=True)


def test_stream_k_over_wide_tiles_e4m3():
    A = _ints(4096, 4096, 79, "e4m3", lo=-2, hi=2)
    B = _ints(4096, 4096, 80, "e4m3", lo=-2, hi=2)
    C, _ = run_gemm(A, B, "e4m3", "f32", layout="rcr", stream_k_tiles=52, **W)
    _check(C, A, B, "e4m3", "f32", exact=True)


def test_planner_choice_8192_cubed_sampled():
    # the planner's own choice for 8192^3 is the wide tile; every row of a
    # few tile rows against the oracle on integer inputs (exact)
    import numpy as np
    A = _ints(8192, 8192, 81, lo=-2, hi=2)
    B = _ints(8192, 8192, 82, lo=-2, hi=2)
    C, cfg = run_gemm(A, B, "bf16", "f32")
    assert cfg["block_n"] == 512
    rows = np.r_[0:3, 255:258, 4095:4098, 8189:8192]
    ref, sabs, _ = oracle.gemm(A[rows], B, "bf16")
    ok, info = oracle.accept(C[rows], ref, sabs, "f32", exact=True)
    assert ok, info
