"""Pins for the fp64 oracle, checked against facts fixed outside it.

Each test ties the oracle to something other than itself: the format
definitions (a golden table), a library conversion, a closed form (identity,
permutation, rank-1, all-ones), brute force in exact rational arithmetic, an
independent library matmul, or an algebraic invariant.  A plausible mistake in
the oracle (a dropped term, a swapped index, a transposed operand, a wrong
rounding rule) fails at least one of them; test_planted_mistakes_are_caught
checks that for a few such mistakes.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import BF16, F16, F32

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "float16_formats.txt")


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------- formats --

def test_decode_golden_table():
    n = 0
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fmt, hexbits, val = line.split()
            got = oracle.lib().oracle_decode(int(hexbits, 16), F16 if fmt == "f16" else BF16)
            if val == "nan":
                assert np.isnan(got), line
            else:
                want = float(val) if val in ("inf", "-inf") else float.fromhex(val)
                assert got == want and np.signbit(got) == np.signbit(want), line
            n += 1
    assert n >= 30


def test_decode_f16_all_patterns_match_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode(bits, F16)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_decode_bf16_all_patterns_are_upper_half_of_fp32():
    bits = np.arange(65536, dtype=np.uint32)
    got = oracle.decode(bits.astype(np.uint16), BF16)
    with np.errstate(invalid="ignore"):
        want = (bits << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_round_f16_matches_numpy_conversion():
    r = _rng(1)
    x = np.concatenate([
        r.standard_normal(200000) * 10.0 ** r.integers(-9, 6, 200000),
        # exact ties between neighbouring binary16 values
        (np.arange(-2048, 2048) + 0.5) * 2.0 ** -10,
        (np.arange(0, 1024) + 0.5) * 2.0 ** -24,      # subnormal ties
        np.array([65504.0, 65519.99, 65520.0, 1e6, -1e6, 0.0, -0.0,
                  2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -26]),
    ])
    got = oracle.round_out(x, F16)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_round_bf16_matches_torch_on_fp32_values():
    r = _rng(2)
    f = (r.standard_normal(200000) * 10.0 ** r.integers(-30, 30, 200000)).astype(np.float32)
    # ties: fp32 values exactly halfway between two bf16 values
    ties = ((np.arange(1, 4096, dtype=np.uint32) << 16) | 0x8000).view(np.float32)
    f = np.concatenate([f, ties, -ties]).astype(np.float32)
    got = oracle.round_out(f.astype(np.float64), BF16)
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_round_bf16_is_a_single_rounding_from_double():
    # 1 + 2^-8 lies exactly halfway between 1 and 1 + 2^-7: ties to even -> 1.
    # 1 + 2^-8 + 2^-30 lies just above the tie -> 1 + 2^-7 (a path through
    # fp32 would lose the 2^-30 and round to 1).
    lib = oracle.lib()
    assert lib.oracle_round16(1.0 + 2.0 ** -8, BF16) == 0x3F80
    assert lib.oracle_round16(1.0 + 2.0 ** -8 + 2.0 ** -30, BF16) == 0x3F81
    assert lib.oracle_round16(1.0 + 3 * 2.0 ** -8, BF16) == 0x3F82  # tie -> even
    assert lib.oracle_round16(-(1.0 + 2.0 ** -8 + 2.0 ** -30), BF16) == 0xBF81
    # overflow boundary: largest finite bf16 is (2 - 2^-7) * 2^127; halfway
    # to 2^128 rounds to infinity
    assert lib.oracle_round16(float.fromhex("0x1.fep+127"), BF16) == 0x7F7F
    assert lib.oracle_round16(float.fromhex("0x1.ffp+127"), BF16) == 0x7F80
    assert lib.oracle_round16(float.fromhex("0x1.fefffffp+127"), BF16) == 0x7F7F
    # smallest subnormal and the tie below it
    assert lib.oracle_round16(2.0 ** -133, BF16) == 0x0001
    assert lib.oracle_round16(2.0 ** -134, BF16) == 0x0000
    assert lib.oracle_round16(2.0 ** -134 * 1.5, BF16) == 0x0001


def test_round32_is_float_conversion():
    x = np.array([1.0 + 2.0 ** -24, 1.0 + 3 * 2.0 ** -24, 16777217.0, -0.1])
    assert np.array_equal(oracle.round_out(x, F32), x.astype(np.float32))


# ------------------------------------------------------------------ GEMM --

def _f16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def _bf16(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _rand_bits(shape, dtype, seed, scale=1.0):
    x = _rng(seed).uniform(-scale, scale, shape)
    return _f16(x) if dtype == F16 else _bf16(x)


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_identity_left_and_right(dtype):
    n = 40
    eye = _f16(np.eye(n)) if dtype == F16 else _bf16(np.eye(n))
    B = _rand_bits((n, 33), dtype, 3)
    ref, sabs, _ = oracle.gemm(eye, B, dtype)
    assert np.array_equal(ref, oracle.decode(B, dtype))
    A = _rand_bits((17, n), dtype, 4)
    ref, sabs, _ = oracle.gemm(A, eye, dtype)
    assert np.array_equal(ref, oracle.decode(A, dtype))
    assert np.array_equal(sabs, np.abs(ref))


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_permutation_left_and_right(dtype):
    r = _rng(5)
    n = 48
    perm = r.permutation(n)
    P = np.zeros((n, n))
    P[np.arange(n), perm] = 1.0
    Pb = _f16(P) if dtype == F16 else _bf16(P)
    B = _rand_bits((n, 24), dtype, 6)
    ref, _, _ = oracle.gemm(Pb, B, dtype)
    # (P B)[i] = B[perm[i]]
    assert np.array_equal(ref, oracle.decode(B, dtype)[perm])
    A = _rand_bits((20, n), dtype, 7)
    ref, _, _ = oracle.gemm(A, Pb, dtype)
    # (A P)[:, perm[i]] = A[:, i]
    want = np.empty_like(ref)
    want[:, perm] = oracle.decode(A, dtype)
    assert np.array_equal(ref, want)


def test_rank_one_closed_form():
    r = _rng(8)
    M, N, K = 37, 29, 300
    u = r.integers(-3, 4, M)
    v = r.integers(-3, 4, N)
    p = r.integers(-2, 3, K)
    q = r.integers(-2, 3, K)
    A = _bf16(np.outer(u, p))
    B = _bf16(np.outer(q, v))
    ref, sabs, _ = oracle.gemm(A, B, BF16)
    pq = int(np.dot(p, q))
    apq = int(np.dot(np.abs(p), np.abs(q)))
    assert np.array_equal(ref, pq * np.outer(u, v).astype(np.float64))
    assert np.array_equal(sabs, apq * np.abs(np.outer(u, v)).astype(np.float64))


@pytest.mark.parametrize("K", [1, 7, 64, 1000])
def test_all_ones_gives_K(K):
    A = _f16(np.ones((5, K)))
    B = _f16(np.ones((K, 6)))
    ref, sabs, _ = oracle.gemm(A, B, F16)
    assert np.all(ref == K) and np.all(sabs == K)


def _exact_products(Ad, Bd):
    M, K = Ad.shape
    N = Bd.shape[1]
    ex = [[sum(Fraction(Ad[i, k]) * Fraction(Bd[k, j]) for k in range(K))
           for j in range(N)] for i in range(M)]
    return ex


@pytest.mark.parametrize("dtype", [F16, BF16])
def test_brute_force_exact_arithmetic_tiny_shapes(dtype):
    seed = 10
    for M in range(1, 6):
        for N in (1, 3, 8):
            for K in (1, 2, 5, 9):
                seed += 1
                A = _rand_bits((M, K), dtype, seed, scale=4.0)
                B = _rand_bits((K, N), dtype, seed + 1000, scale=4.0)
                Ad, Bd = oracle.decode(A, dtype), oracle.decode(B, dtype)
                ref, sabs, _ = oracle.gemm(A, B, dtype)
                ex = _exact_products(Ad, Bd)
                for i in range(M):
                    for j in range(N):
                        bound = K * 2.0 ** -52 * sabs[i, j]
                        assert abs(Fraction(ref[i, j]) - ex[i][j]) <= Fraction(bound)
                        sa = sum(abs(Fraction(Ad[i, k]) * Fraction(Bd[k, j])) for k in range(K))
                        assert abs(Fraction(sabs[i, j]) - sa) <= Fraction(bound)


def test_brute_force_python_loop_exact_on_integers():
    r = _rng(20)
    M, N, K = 9, 11, 70
    a = r.integers(-2, 3, (M, K))
    b = r.integers(-2, 3, (K, N))
    ref, sabs, _ = oracle.gemm(_bf16(a), _bf16(b), BF16)
    for i in range(M):
        for j in range(N):
            s = 0
            t = 0
            for k in range(K):
                s += int(a[i, k]) * int(b[k, j])
                t += abs(int(a[i, k]) * int(b[k, j]))
            assert ref[i, j] == s and sabs[i, j] == t


@pytest.mark.parametrize("shape", [(64, 80, 96), (129, 72, 264), (1, 300, 1), (200, 1, 33)])
def test_against_torch_float64_matmul(shape):
    M, N, K = shape
    A = _rand_bits((M, K), F16, 30 + M)
    B = _rand_bits((K, N), F16, 31 + N)
    Ad = torch.from_numpy(oracle.decode(A, F16))
    Bd = torch.from_numpy(oracle.decode(B, F16))
    ref, sabs, _ = oracle.gemm(A, B, F16)
    want = (Ad @ Bd).numpy()
    wabs = (Ad.abs() @ Bd.abs()).numpy()
    assert np.all(np.abs(ref - want) <= 1e-12 * wabs + 1e-300)
    assert np.all(np.abs(sabs - wabs) <= 1e-12 * wabs + 1e-300)


def test_transpose_invariant_is_bitwise():
    A = _rand_bits((23, 41), BF16, 40)
    B = _rand_bits((41, 17), BF16, 41)
    ref, sabs, _ = oracle.gemm(A, B, BF16)
    refT, sabsT, _ = oracle.gemm(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T), BF16)
    assert np.array_equal(ref, refT.T) and np.array_equal(sabs, sabsT.T)


def test_linearity_in_A_on_integers():
    r = _rng(42)
    a1 = r.integers(-2, 3, (13, 50))
    a2 = r.integers(-2, 3, (13, 50))
    b = r.integers(-2, 3, (50, 19))
    r1, _, _ = oracle.gemm(_bf16(a1), _bf16(b), BF16)
    r2, _, _ = oracle.gemm(_bf16(a2), _bf16(b), BF16)
    r12, _, _ = oracle.gemm(_bf16(a1 + a2), _bf16(b), BF16)
    assert np.array_equal(r12, r1 + r2)


def test_threads_do_not_change_the_result():
    A = _rand_bits((31, 64), F16, 50)
    B = _rand_bits((64, 40), F16, 51)
    r1, s1, _ = oracle.gemm(A, B, F16, nthreads=1)
    r4, s4, used = oracle.gemm(A, B, F16, nthreads=4)
    assert used == 4
    assert np.array_equal(r1, r4) and np.array_equal(s1, s4)


def test_sampled_equals_full_at_positions():
    A = _rand_bits((70, 90), BF16, 60)
    B = _rand_bits((90, 50), BF16, 61)
    ref, sabs, _ = oracle.gemm(A, B, BF16)
    r = _rng(62)
    rows = r.integers(0, 70, 300)
    cols = r.integers(0, 50, 300)
    sr, ss = oracle.gemm_sampled(A, B, BF16, rows, cols)
    assert np.array_equal(sr, ref[rows, cols]) and np.array_equal(ss, sabs[rows, cols])


def test_accept_rule_boundaries():
    ref = np.array([[1.0, 100.0]])
    sabs = np.array([[1.0, 200.0]])
    # bound = 1e-3 * sabs + 1e-5
    C = np.array([[1.0 + 1.0e-3 + 0.5e-5, 100.0 - 0.19]], dtype=np.float32)
    ok, _ = oracle.accept(C, ref, sabs, F32)
    assert ok
    C2 = np.array([[1.0 + 1.2e-3, 100.0]], dtype=np.float32)
    ok, info = oracle.accept(C2, ref, sabs, F32)
    assert not ok and info["mismatches"] == 1
    ok, _ = oracle.accept(np.array([[np.nan, 100.0]], dtype=np.float32), ref, sabs, F32)
    assert not ok
    # exact mode compares bits after rounding the oracle value
    ok, _ = oracle.accept(_bf16([[1.0, 100.0]]), ref, sabs, BF16, exact=True)
    assert ok
    ok, _ = oracle.accept(_bf16([[1.0, 100.5]]), ref, sabs, BF16, exact=True)
    assert not ok


# --------------------------------------------------- planted mistakes --

def _pins_pass(gemm_fn):
    """Run a subset of the GEMM pins against a (possibly mutated) oracle."""
    n = 16
    eye = _bf16(np.eye(n))
    B = _rand_bits((n, 8), BF16, 70)
    A = _rand_bits((8, n), BF16, 71)
    checks = []
    ref = gemm_fn(eye, B)
    checks.append(np.array_equal(ref, oracle.decode(B, BF16)))
    ref = gemm_fn(A, eye)
    checks.append(np.array_equal(ref, oracle.decode(A, BF16)))
    r = _rng(72)
    u, v = r.integers(-3, 4, 5), r.integers(-3, 4, 6)
    p, q = r.integers(-2, 3, 30), r.integers(-2, 3, 30)
    ref = gemm_fn(_bf16(np.outer(u, p)), _bf16(np.outer(q, v)))
    checks.append(np.array_equal(ref, np.dot(p, q) * np.outer(u, v)))
    ones = gemm_fn(_bf16(np.ones((3, 20))), _bf16(np.ones((20, 4))))
    checks.append(np.all(ones == 20))
    perm = r.permutation(n)
    P = np.zeros((n, n))
    P[np.arange(n), perm] = 1.0
    ref = gemm_fn(A, _bf16(P))
    want = np.empty_like(ref)
    want[:, perm] = oracle.decode(A, BF16)
    checks.append(np.array_equal(ref, want))
    return all(checks)


def test_planted_mistakes_are_caught():
    def good(A, B):
        return oracle.gemm(A, B, BF16)[0]

    def drops_last_k(A, B):
        return oracle.gemm(np.ascontiguousarray(A[:, :-1]), np.ascontiguousarray(B[:-1]), BF16)[0]

    def transposes_B(A, B):
        if B.shape[0] == B.shape[1]:
            return oracle.gemm(A, np.ascontiguousarray(B.T), BF16)[0]
        return oracle.gemm(A, B, BF16)[0]

    def flips_sign(A, B):
        return -oracle.gemm(A, B, BF16)[0]

    def wrong_format(A, B):
        return oracle.gemm(A, B, F16)[0]  # decodes bf16 bits as fp16

    assert _pins_pass(good)
    for bad in (drops_last_k, transposes_B, flips_sign, wrong_format):
        assert not _pins_pass(bad), bad.__name__


def test_half_ulp_matches_the_format_spacing():
    # spacing of bf16 numbers in [1, 2) is 2^-7; of fp16 is 2^-10
    assert oracle.half_ulp(1.0, BF16) == 2.0 ** -8
    assert oracle.half_ulp(1.99, BF16) == 2.0 ** -8
    assert oracle.half_ulp(2.0, BF16) == 2.0 ** -7
    assert oracle.half_ulp(1.0, F16) == 2.0 ** -11
    assert oracle.half_ulp(-65504.0, F16) == 16.0
    # subnormal range: fixed spacing 2^-24 (fp16), 2^-133 (bf16)
    assert oracle.half_ulp(2.0 ** -20, F16) == 2.0 ** -25
    assert oracle.half_ulp(0.0, BF16) == 2.0 ** -134
    # neighbouring representable values are two half-ulps apart
    for dt, one_up in ((BF16, 0x3F81), (F16, 0x3C01)):
        gap = oracle.decode(np.array([one_up], dtype=np.uint16), dt)[0] - 1.0
        assert gap == 2 * oracle.half_ulp(1.0, dt)


def test_accept_admits_the_correctly_rounded_16_bit_output():
    # With K small |ref| can approach sabs, where half a bf16 ulp exceeds
    # 1e-3 * sabs; the correctly rounded output must still be accepted and
    # one ulp further must not.
    r = _rng(80)
    ref = r.uniform(-4, 4, 5000)
    sabs = np.abs(ref) * 1.0001
    for dt in (BF16, F16):
        C = oracle.round_out(ref, dt)
        ok, info = oracle.accept(C, ref, sabs, dt)
        assert ok, info
        # move one element far enough that it exceeds 1e-3 * sabs plus half
        # an ulp: 2 bf16 ulps (2^-6 relative) or 8 fp16 ulps (2^-7 relative)
        off = C.copy()
        off[0] = off[0] + (2 if dt == BF16 else 8)
        ok, info = oracle.accept(off, ref, sabs, dt)
        assert not ok and info["mismatches"] == 1


# ------------------------------------------------------------ FP8 formats --

from oracle import E4M3, E5M2  # noqa: E402

GOLDEN8 = os.path.join(os.path.dirname(__file__), "golden", "float8_formats.txt")


def test_decode_fp8_golden_table():
    n = 0
    with open(GOLDEN8) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fmt, hexbits, val = line.split()
            got = oracle.lib().oracle_decode8(int(hexbits, 16), E4M3 if fmt == "e4m3" else E5M2)
            if val == "nan":
                assert np.isnan(got), line
            else:
                want = float(val) if val in ("inf", "-inf") else float.fromhex(val)
                assert got == want and np.signbit(got) == np.signbit(want), line
            n += 1
    assert n >= 24


@pytest.mark.parametrize("code,tdt", [(E4M3, torch.float8_e4m3fn), (E5M2, torch.float8_e5m2)])
def test_decode_fp8_all_patterns_match_torch(code, tdt):
    bits = np.arange(256, dtype=np.uint8)
    got = oracle.decode(bits, code)
    want = torch.from_numpy(bits.copy()).view(tdt).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def _fp8(x, code):
    t = torch.tensor(np.asarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn if code == E4M3 else torch.float8_e5m2).view(torch.uint8).numpy().copy()


@pytest.mark.parametrize("code", [E4M3, E5M2])
def test_fp8_gemm_pins(code):
    r = _rng(90)
    n = 48
    eye = _fp8(np.eye(n), code)
    B = _fp8(r.integers(-6, 7, (n, 20)), code)
    ref, sabs, _ = oracle.gemm(eye, B, code)
    assert np.array_equal(ref, oracle.decode(B, code))
    perm = r.permutation(n)
    P = np.zeros((n, n))
    P[np.arange(n), perm] = 1.0
    A = _fp8(r.integers(-6, 7, (15, n)), code)
    ref, _, _ = oracle.gemm(A, _fp8(P, code), code)
    want = np.empty_like(ref)
    want[:, perm] = oracle.decode(A, code)
    assert np.array_equal(ref, want)
    u, v = r.integers(-3, 4, 9), r.integers(-3, 4, 11)
    p_, q_ = r.integers(-2, 3, 200), r.integers(-2, 3, 200)
    ref, sabs, _ = oracle.gemm(_fp8(np.outer(u, p_), code), _fp8(np.outer(q_, v), code), code)
    assert np.array_equal(ref, np.dot(p_, q_) * np.outer(u, v).astype(np.float64))
    ones, _, _ = oracle.gemm(_fp8(np.ones((3, 77)), code), _fp8(np.ones((77, 5)), code), code)
    assert np.all(ones == 77)


@pytest.mark.parametrize("code", [E4M3, E5M2])
def test_fp8_gemm_against_torch_float64(code):
    r = _rng(91)
    A = _fp8(r.uniform(-3, 3, (40, 96)), code)
    B = _fp8(r.uniform(-3, 3, (96, 56)), code)
    Ad = torch.from_numpy(oracle.decode(A, code))
    Bd = torch.from_numpy(oracle.decode(B, code))
    ref, sabs, _ = oracle.gemm(A, B, code)
    want = (Ad @ Bd).numpy()
    wabs = (Ad.abs() @ Bd.abs()).numpy()
    assert np.all(np.abs(ref - want) <= 1e-12 * wabs + 1e-300)
    rows, cols = r.integers(0, 40, 50), r.integers(0, 56, 50)
    sr, ss = oracle.gemm_sampled(A, B, code, rows, cols)
    assert np.array_equal(sr, ref[rows, cols]) and np.array_equal(ss, sabs[rows, cols])


def test_fp8_brute_force_exact_arithmetic():
    r = _rng(92)
    for code in (E4M3, E5M2):
        A = _fp8(r.uniform(-8, 8, (3, 7)), code)
        B = _fp8(r.uniform(-8, 8, (7, 4)), code)
        Ad, Bd = oracle.decode(A, code), oracle.decode(B, code)
        ref, _, _ = oracle.gemm(A, B, code)
        for i in range(3):
            for j in range(4):
                ex = sum(Fraction(Ad[i, k]) * Fraction(Bd[k, j]) for k in range(7))
                assert Fraction(ref[i, j]) == ex  # few terms: exact in double
