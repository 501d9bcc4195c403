"""fp64 CPU oracle for the tile-level GEMM C = A*B.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only tests/, __graft_entry__.smoke()
and the cpu_baseline / reference legs of bench.py may import this package.
The product path (hierarchical_gemm_gb300) never imports it and shares no
code with it.

The operation is the one the TileLang GEMM skeleton computes ("TileScale 与
TileLang比较", section 核心抽象与编程模型对比): C is cleared, every BK-slice
product of A (M x K, row-major) and B (K x N, row-major) is added into it, and
the result is copied out.  Up to the order of additions this is
C[i][j] = sum_k A[i][k] * B[k][j]; the C library in oracle_gemm.c writes that
sum out in double precision in the order k = 0..K-1.

Inputs and outputs here are numpy arrays of raw bits (uint16 for fp16/bf16,
float32 for fp32 outputs), so the oracle decodes the exact values itself.
"""
import ctypes
import os

import numpy as np

from . import build as _build

F16, BF16, F32, E4M3, E5M2 = 0, 1, 2, 3, 4
_NAMES = {"f16": F16, "fp16": F16, "float16": F16,
          "bf16": BF16, "bfloat16": BF16,
          "f32": F32, "fp32": F32, "float32": F32,
          "e4m3": E4M3, "float8_e4m3fn": E4M3, "e5m2": E5M2, "float8_e5m2": E5M2}
_EIGHT_BIT = (E4M3, E5M2)

_lib = None


def dtype_code(d):
    if isinstance(d, int):
        return d
    return _NAMES[str(d).lower()]


def lib():
    """Load (building first if needed) the oracle's shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        L.oracle_decode.restype = ctypes.c_double
        L.oracle_decode.argtypes = [ctypes.c_uint16, i32]
        L.oracle_round16.restype = ctypes.c_uint16
        L.oracle_round16.argtypes = [ctypes.c_double, i32]
        L.oracle_decode_n.argtypes = [vp, i64, i32, vp]
        L.oracle_round16_n.argtypes = [vp, i64, i32, vp]
        L.oracle_round32_n.argtypes = [vp, i64, vp]
        L.oracle_gemm.restype = i32
        L.oracle_gemm.argtypes = [i64, i64, i64, vp, vp, i32, vp, vp, i32]
        L.oracle_gemm_sampled.argtypes = [i64, i64, i64, vp, vp, i32, i64, vp,
                                          vp, vp, vp]
        L.oracle_default_threads.restype = i32
        L.oracle_decode8.restype = ctypes.c_double
        L.oracle_decode8.argtypes = [ctypes.c_uint8, i32]
        L.oracle_decode8_n.argtypes = [vp, i64, i32, vp]
        L.oracle_gemm8.restype = i32
        L.oracle_gemm8.argtypes = [i64, i64, i64, vp, vp, i32, vp, vp, i32]
        L.oracle_gemm8_sampled.argtypes = [i64, i64, i64, vp, vp, i32, i64, vp,
                                           vp, vp, vp]
        L.oracle_attention.restype = i32
        L.oracle_attention.argtypes = [i64, i64, i64, i64, i64, i64, vp, vp, vp, i32,
                                       ctypes.c_double, i32, vp, vp]
        _lib = L
    return _lib


def _c(a, dt):
    a = np.ascontiguousarray(a, dtype=dt)
    return a, a.ctypes.data


def default_threads():
    return lib().oracle_default_threads()


def decode(bits, dtype):
    """Exact float64 values of an array of 16-bit (or, for E4M3/E5M2, 8-bit)
    float bit patterns."""
    code = dtype_code(dtype)
    if code in _EIGHT_BIT:
        bits, p = _c(bits, np.uint8)
        out = np.empty(bits.shape, dtype=np.float64)
        lib().oracle_decode8_n(p, bits.size, code, out.ctypes.data)
        return out
    bits, p = _c(bits, np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    lib().oracle_decode_n(p, bits.size, code, out.ctypes.data)
    return out


def round_out(x, dtype_out):
    """Round float64 values to the output format, ties to even.

    Returns uint16 bit patterns for f16/bf16 and float32 values for f32.
    """
    x, p = _c(x, np.float64)
    code = dtype_code(dtype_out)
    if code == F32:
        out = np.empty(x.shape, dtype=np.float32)
        lib().oracle_round32_n(p, x.size, out.ctypes.data)
    else:
        out = np.empty(x.shape, dtype=np.uint16)
        lib().oracle_round16_n(p, x.size, code, out.ctypes.data)
    return out


def gemm(A_bits, B_bits, dtype_in, nthreads=0):
    """ref = A*B and sabs = |A|*|B| (elementwise products), both float64.

    A_bits: (M, K), B_bits: (K, N), both row-major bit patterns: uint16 for
    fp16/bf16, uint8 for the FP8 formats E4M3/E5M2.
    Returns (ref, sabs, threads_used).
    """
    code = dtype_code(dtype_in)
    eight = code in _EIGHT_BIT
    A_bits, pa = _c(A_bits, np.uint8 if eight else np.uint16)
    B_bits, pb = _c(B_bits, np.uint8 if eight else np.uint16)
    M, K = A_bits.shape
    K2, N = B_bits.shape
    assert K == K2, "inner dimensions differ"
    ref = np.empty((M, N), dtype=np.float64)
    sabs = np.empty((M, N), dtype=np.float64)
    fn = lib().oracle_gemm8 if eight else lib().oracle_gemm
    used = fn(M, N, K, pa, pb, code, ref.ctypes.data, sabs.ctypes.data, int(nthreads))
    if used < 0:
        raise MemoryError("oracle_gemm could not allocate its decoded B")
    return ref, sabs, used


def gemm_sampled(A_bits, B_bits, dtype_in, rows, cols):
    """ref and sabs at the positions (rows[s], cols[s]) only."""
    code = dtype_code(dtype_in)
    eight = code in _EIGHT_BIT
    A_bits, pa = _c(A_bits, np.uint8 if eight else np.uint16)
    B_bits, pb = _c(B_bits, np.uint8 if eight else np.uint16)
    M, K = A_bits.shape
    K2, N = B_bits.shape
    assert K == K2, "inner dimensions differ"
    rows, pr = _c(rows, np.int64)
    cols, pc = _c(cols, np.int64)
    assert rows.shape == cols.shape
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < M)
    assert cols.size == 0 or (cols.min() >= 0 and cols.max() < N)
    ref = np.empty(rows.shape, dtype=np.float64)
    sabs = np.empty(rows.shape, dtype=np.float64)
    fn = lib().oracle_gemm8_sampled if eight else lib().oracle_gemm_sampled
    fn(M, N, K, pa, pb, code, rows.size, pr, pc, ref.ctypes.data, sabs.ctypes.data)
    return ref, sabs


# Acceptance rule for a GEMM result against the oracle:
#   * exact mode (integer-valued inputs whose fp32 partial sums are all
#     exact): the output must equal the oracle's sum rounded to the output
#     format, bit for bit;
#   * otherwise |C - ref| <= RTOL * sabs + ATOL per element for the fp32
#     accumulated value; a 16-bit output is that value rounded once more
#     (to nearest, ties to even), which may add up to half a unit in the
#     last place of the output format, so for f16/bf16 outputs the bound is
#     RTOL * sabs + ATOL + half_ulp(max(|ref|, |C|)).
RTOL = 1e-3
ATOL = 1e-5

# (fraction bits, smallest normal exponent) of the 16-bit output formats
_FMT = {F16: (10, -14), BF16: (7, -126)}


def half_ulp(x, dtype_out):
    """Half the spacing of the 16-bit format's numbers at |x| (elementwise)."""
    fb, emin = _FMT[dtype_code(dtype_out)]
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, e2 = np.frexp(a)            # a = m * 2^e2, m in [0.5, 1)
    E = np.where(a > 0, np.maximum(e2 - 1, emin), emin)  # subnormals and 0 share emin
    return np.ldexp(1.0, E - fb - 1)


def output_values(C, dtype_out):
    """float64 values of a GEMM output given as raw bits (u16) or float32."""
    code = dtype_code(dtype_out)
    if code == F32:
        return np.asarray(C, dtype=np.float32).astype(np.float64)
    return decode(np.asarray(C).view(np.uint16), code)


def accept(C, ref, sabs, dtype_out, exact=False):
    """Compare an output against the oracle.

    Returns (ok, info) where info holds the worst error and its position.
    """
    code = dtype_code(dtype_out)
    if exact:
        want = round_out(ref, code)
        if code == F32:
            got = np.asarray(C, dtype=np.float32).view(np.uint32)
            want = want.view(np.uint32)
        else:
            got = np.asarray(C).view(np.uint16)
        bad = got != want
        nbad = int(bad.sum())
        info = {"mismatches": nbad}
        if nbad:
            idx = np.argwhere(bad)[0]
            info["first"] = tuple(int(v) for v in idx)
        return nbad == 0, info
    cv = output_values(C, code)
    err = np.abs(cv - ref)
    bound = RTOL * sabs + ATOL
    if code != F32:
        with np.errstate(invalid="ignore"):
            bound = bound + half_ulp(np.fmax(np.abs(ref), np.abs(cv)), code)
    bad = ~(err <= bound)  # NaN counts as bad
    nbad = int(bad.sum())
    ratio = err / bound
    worst = int(np.nanargmax(ratio)) if ratio.size else 0
    info = {"mismatches": nbad,
            "max_err_over_bound": float(np.nanmax(ratio)) if ratio.size else 0.0,
            "worst_index": tuple(int(v) for v in np.unravel_index(worst, ratio.shape))
            if ratio.size else ()}
    return nbad == 0, info


# ------------------------------------------------------------- attention --

def attention(Q_bits, K_bits, V_bits, dtype_in, scale, causal=False):
    """O = softmax(scale * Q K^T) V per (batch, head), and per element
    bound = sum_t w_t |V[t]|, both float64 of shape (B, H, Sq, Dv).

    Q_bits (B, H, Sq, D), K_bits (B, H, Sk, D), V_bits (B, H, Sk, Dv): 16-bit
    bit patterns.  Causal: row i sees keys t <= i + Sk - Sq; a row that sees
    none is zero.  (oracle_attention.c, after the FlashMLA example of the
    TileScale README.)"""
    code = dtype_code(dtype_in)
    Q_bits, pq = _c(Q_bits, np.uint16)
    K_bits, pk = _c(K_bits, np.uint16)
    V_bits, pv = _c(V_bits, np.uint16)
    B, H, Sq, D = Q_bits.shape
    Sk, Dv = K_bits.shape[2], V_bits.shape[3]
    assert K_bits.shape == (B, H, Sk, D) and V_bits.shape == (B, H, Sk, Dv)
    O = np.empty((B, H, Sq, Dv), dtype=np.float64)
    bound = np.empty((B, H, Sq, Dv), dtype=np.float64)
    if lib().oracle_attention(B, H, Sq, Sk, D, Dv, pq, pk, pv, code, float(scale), int(bool(causal)),
                              O.ctypes.data, bound.ctypes.data) != 0:
        raise MemoryError("oracle_attention could not allocate its scratch")
    return O, bound


def mla_decode(Q_bits, Qpe_bits, KV_bits, Kpe_bits, dtype_in, scale):
    """The MLA decode shape of the attention block (the FlashMLA example of
    the TileScale README): per batch b and head h, scores over the latent
    and rotary parts, s[t] = Q[b,h] . KV[b,t] + Q_pe[b,h] . K_pe[b,t], and
    O[b,h] = softmax(scale s) KV[b] -- the latent cache is also the value.
    That is the attention definition above with the query [Q Q_pe], the keys
    [KV K_pe] (576 deep) and the values KV (512 wide), one query row per
    head.  Q_bits (B, H, dim), Qpe_bits (B, H, pe), KV_bits (B, Skv, dim),
    Kpe_bits (B, Skv, pe).  Returns (O, bound) of shape (B, H, dim)."""
    Q_bits = np.asarray(Q_bits)
    B, H, dim = Q_bits.shape
    Skv = np.asarray(KV_bits).shape[1]
    q = np.concatenate([Q_bits, np.asarray(Qpe_bits)], axis=2).reshape(B, 1, H, -1)
    k = np.concatenate([np.asarray(KV_bits), np.asarray(Kpe_bits)], axis=2).reshape(B, 1, Skv, -1)
    v = np.asarray(KV_bits).reshape(B, 1, Skv, dim)
    O, bound = attention(q, k, v, dtype_in, scale, causal=False)
    return O.reshape(B, H, dim), bound.reshape(B, H, dim)


# Acceptance rule for an attention output (derived from the arithmetic of
# the kernel's online softmax): the weights are computed in fp32 and
# rounded once to the 16-bit input format before they multiply V, a
# relative error of at most 2^-9 (bf16) per weight, which moves an output
# element by at most 2^-9 * sum_t w_t |V[t]|; fp32 accumulation, the
# approximate base-2 exponential and the fp32 division add far less.  The
# bound allows twice that, plus half an ulp of the 16-bit output format.
ATTN_RTOL = 2.0 ** -8
ATTN_ATOL = 1e-6


def accept_attention(O, ref, bound, dtype_out):
    code = dtype_code(dtype_out)
    got = output_values(O, code)
    tol = ATTN_RTOL * bound + ATTN_ATOL
    if code != F32:
        tol = tol + half_ulp(np.maximum(np.abs(ref), np.abs(got)), code)
    err = np.abs(got - ref)
    bad = ~(err <= tol)
    info = {"max_err": float(np.nanmax(err)) if err.size else 0.0,
            "max_err_over_bound": float(np.nanmax(err / tol)) if err.size else 0.0,
            "bad": int(bad.sum())}
    if bad.any():
        idx = np.unravel_index(int(np.argmax(np.where(bad, err / tol, -1))), err.shape)
        info["first_bad"] = [int(x) for x in idx]
        info["got"] = float(got[idx])
        info["want"] = float(ref[idx])
    return not bad.any(), info
