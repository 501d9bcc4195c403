"""Parity of the 8-bit float GEMM (E4M3 / E5M2 inputs, tcgen05 kind::f8f6f4)
against the fp64 oracle, element by element.

The operands are stored K-major (the RCR layout: A M x K, B N x K).
Acceptance is the one of the 16-bit path: bit-exact on integer inputs whose
fp32 partial sums are exact, else |C - ref| <= 1e-3 * sum_k |a_ik b_kj| +
1e-5 (plus half an output ulp for 16-bit outputs).  Integers up to 16 are
exact in E4M3 and up to 8 in E5M2.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TORCH_DT, from_dev, run_gemm, to_dev

pytestmark = pytest.mark.gpu

FORMATS = ["e4m3", "e5m2"]


def _ints(rows, cols, seed, din, lo=-4, hi=4):
    return synth.matrix(rows, cols, ("int", lo, hi), seed, din)


def _bits_of(x, din):
    return synth.quantise(np.asarray(x, dtype=np.float64), din)


def _check(C, A, B, din, dout, exact):
    ref, sabs, _ = oracle.gemm(A, B, din)
    ok, info = oracle.accept(C, ref, sabs, dout, exact=exact)
    assert ok, info


@pytest.mark.parametrize("din", FORMATS)
@pytest.mark.parametrize("dout", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("n", [256, 208])  # K rows are bytes: multiples of 16
def test_identity_left(din, dout, n):
    eye = _bits_of(np.eye(n), din)
    B = _ints(n, 264, 11, din, -8, 8)
    C, _ = run_gemm(eye, B, din, dout, layout="rcr")
    _check(C, eye, B, din, dout, exact=True)


@pytest.mark.parametrize("din", FORMATS)
@pytest.mark.parametrize("n", [384, 144])
def test_identity_right(din, n):
    eye = _bits_of(np.eye(n), din)
    A = _ints(300, n, 12, din, -8, 8)
    C, _ = run_gemm(A, eye, din, "f32", layout="rcr")
    _check(C, A, eye, din, "f32", exact=True)


TILES = [(128, 64), (128, 128), (128, 192), (128, 256), (256, 128), (256, 256)]


@pytest.mark.parametrize("block_m,block_n", TILES)
def test_permutation_both_sides(block_m, block_n):
    din = "e4m3"
    r = np.random.default_rng(13)
    n = 512
    perm = r.permutation(n)
    P = np.zeros((n, n))
    P[np.arange(n), perm] = 1.0
    Pb = _bits_of(P, din)
    B = _ints(n, 320, 14, din, -16, 16)
    C, cfg = run_gemm(Pb, B, din, "bf16", layout="rcr", block_m=block_m, block_n=block_n)
    assert (cfg["block_m"], cfg["block_n"]) == (block_m, block_n)
    _check(C, Pb, B, din, "bf16", exact=True)
    A = _ints(256, n, 15, din, -16, 16)
    C, _ = run_gemm(A, Pb, din, "bf16", layout="rcr", block_m=block_m, block_n=block_n)
    _check(C, A, Pb, din, "bf16", exact=True)


@pytest.mark.parametrize("din", FORMATS)
@pytest.mark.parametrize("block_m,block_n", TILES)
@pytest.mark.parametrize("splits", [1, 3])
def test_integer_exact_ragged(din, block_m, block_n, splits):
    # M, N and K all ragged: K = 5 slices of 128 plus 48
    M, N, K = 333, 264, 5 * 128 + 48
    A = _ints(M, K, 16, din)
    B = _ints(K, N, 17, din)
    C, cfg = run_gemm(A, B, din, "f32", layout="rcr", block_m=block_m, block_n=block_n, splits=splits)
    assert cfg["splits"] == splits
    _check(C, A, B, din, "f32", exact=True)


@pytest.mark.parametrize("din", FORMATS)
def test_rank_one_closed_form(din):
    r = np.random.default_rng(18)
    M, N, K = 256, 384, 1024
    u, v = r.integers(-2, 3, M), r.integers(-2, 3, N)
    p, q = r.integers(-2, 3, K), r.integers(-2, 3, K)
    A = _bits_of(np.outer(u, p), din)
    B = _bits_of(np.outer(q, v), din)
    C, _ = run_gemm(A, B, din, "f32", layout="rcr")
    assert np.array_equal(C, (np.dot(p, q) * np.outer(u, v)).astype(np.float32))


@pytest.mark.parametrize("din", FORMATS)
@pytest.mark.parametrize("K", [128, 4096 + 16])
def test_all_ones_counts_every_slice(din, K):
    A = _bits_of(np.ones((256, K)), din)
    B = _bits_of(np.ones((K, 256)), din)
    C, _ = run_gemm(A, B, din, "f32", layout="rcr", splits=4 if K > 1024 else 1)
    assert np.all(C == K)


@pytest.mark.parametrize("din", FORMATS)
@pytest.mark.parametrize("dout", ["bf16", "f32"])
def test_uniform_random_within_tolerance(din, dout):
    M, N, K = 520, 776, 2064
    A = synth.matrix(M, K, ("uniform", -1.0, 1.0), 19, din)
    B = synth.matrix(K, N, ("uniform", -1.0, 1.0), 20, din)
    C, _ = run_gemm(A, B, din, dout, layout="rcr")
    _check(C, A, B, din, dout, exact=False)


@pytest.mark.parametrize("din", FORMATS)
def test_long_k_random_normal(din):
    # long K: whatever order the tensor core adds in, the fp32 result must
    # stay inside the tolerance
    M, N, K = 256, 256, 32768
    A = synth.matrix(M, K, ("normal", 1.0), 21, din)
    B = synth.matrix(K, N, ("normal", 1.0), 22, din)
    C, _ = run_gemm(A, B, din, "f32", layout="rcr")
    _check(C, A, B, din, "f32", exact=False)


@pytest.mark.parametrize("din", FORMATS)
def test_subnormal_inputs(din):
    # every A entry a subnormal of the format (E4M3: multiples of 2^-9 below
    # 2^-6; E5M2: multiples of 2^-16 below 2^-14), B small integers: the
    # products must not be flushed to zero
    r = np.random.default_rng(23)
    M, N, K = 256, 256, 512
    step, count = (2.0 ** -9, 7) if din == "e4m3" else (2.0 ** -16, 3)
    A = _bits_of(r.integers(1, count + 1, (M, K)) * step * r.choice([-1.0, 1.0], (M, K)), din)
    B = _ints(K, N, 24, din)
    C, _ = run_gemm(A, B, din, "f32", layout="rcr")
    ref, sabs, _ = oracle.gemm(A, B, din)
    assert np.any(ref != 0)
    ok, info = oracle.accept(C, ref, sabs, "f32", exact=True)
    assert ok, info


def test_largest_finite_values():
    # 448 * 448 * K for E4M3, 57344 * 57344 * K for E5M2 (fp32 holds both)
    for din, big in (("e4m3", 448.0), ("e5m2", 57344.0)):
        K = 256
        A = _bits_of(np.full((128, K), big), din)
        B = _bits_of(np.full((K, 128), -big), din)
        C, _ = run_gemm(A, B, din, "f32", layout="rcr")
        assert np.all(C == np.float32(-big * big * K)), din


def test_4096_e4m3_bf16_sampled():
    # the 4096^3 shape in E4M3 with a bf16 output, checked on 4096 sampled
    # outputs plus one whole row and column
    din, M, N, K = "e4m3", 4096, 4096, 4096
    A = synth.matrix(M, K, ("normal", 1.0), 25, din)
    B = synth.matrix(K, N, ("normal", 1.0), 26, din)
    C, cfg = run_gemm(A, B, din, "bf16", layout="rcr")
    r = np.random.default_rng(27)
    rows = np.concatenate([r.integers(0, M, 4096), np.full(N, 1234), np.arange(M)])
    cols = np.concatenate([r.integers(0, N, 4096), np.arange(N), np.full(M, 3071)])
    ref, sabs = oracle.gemm_sampled(A, B, din, rows, cols)
    ok, info = oracle.accept(C[rows, cols], ref, sabs, "bf16", exact=False)
    assert ok, (cfg, info)


def test_binding_gemm_infers_layout_from_strides():
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    M, N, K = 384, 512, 1024
    A_bits = _ints(M, K, 28, "e4m3")
    W_bits = _ints(N, K, 29, "e4m3")  # a weight stored N x K
    A = to_dev(A_bits, "e4m3")
    W = to_dev(W_bits, "e4m3")
    C = tsgemm.gemm(A, W.t(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    _check(from_dev(C, "f32"), A_bits, np.ascontiguousarray(W_bits.T), "e4m3", "f32", exact=True)
    with pytest.raises(tsgemm.TsgemmError):
        tsgemm.gemm(A, W.t().contiguous())  # B stored K x N: not a K-major 8-bit operand
