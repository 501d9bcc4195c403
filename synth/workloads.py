"""The seeded GEMM workloads: shapes, formats, distributions and seeds.

WORKLOADS holds the five benchmark configurations; EXTRA_WORKLOADS the ones
of the wider rows built on the same kernels (8-bit inputs).  Seeds: A uses
0x7E5A0000 + index, B uses 0x7E5A0000 + index + 0x100.  A (M x K) is
generated before B (K x N), both as logical row-major matrices; `layout`
says how the library is handed them (for "rcr", B is stored transposed,
N x K), which changes no value.
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


# FP8 (E4M3) inputs, bf16 output, operands stored K-major (RCR): the
# 4096^3 and 16384 x 16384 x 8192 shapes of the table above.
EXTRA_WORKLOADS = {
    "gemm_4096_e4m3_rcr": dict(
        index=5, M=4096, N=4096, K=4096, dtype_in="e4m3", dtype_out="bf16",
        dist_a=("normal", 1.0), dist_b=("normal", 1.0),
        exact=False, cluster=None, layout="rcr"),
    "gemm_16384x16384x8192_e4m3_rcr": dict(
        index=6, M=16384, N=16384, K=8192, dtype_in="e4m3", dtype_out="bf16",
        dist_a=("uniform", -1.0, 1.0), dist_b=("uniform", -1.0, 1.0),
        exact=False, cluster=(2, 1), layout="rcr"),
}


# The attention block (softmax(scale Q K^T) V): Q, K, V of shape (B, H, S, D)
# drawn from N(0, 1), scale D^-1/2.  Seeds as above (Q: the A seed, K: the
# B seed, V: the B seed + 0x100).
ATTN_WORKLOADS = {
    "attn_b4h32s4096d128_bf16": dict(
        index=7, B=4, H=32, Sq=4096, Sk=4096, D=128, dtype="bf16", causal=False),
    "attn_b4h32s4096d128_causal_bf16": dict(
        index=8, B=4, H=32, Sq=4096, Sk=4096, D=128, dtype="bf16", causal=True),
    # a smaller case for profiler captures (still 3 x 64 MiB, larger than L2)
    "attn_b2h16s4096d128_bf16": dict(
        index=9, B=2, H=16, Sq=4096, Sk=4096, D=128, dtype="bf16", causal=False),
    # its causal twin, for profiler captures of the causal launch
    "attn_b2h16s4096d128_causal_bf16": dict(
        index=11, B=2, H=16, Sq=4096, Sk=4096, D=128, dtype="bf16", causal=True),
}


# The MLA decode shape (softmax(scale [Q Q_pe] [KV K_pe]^T) KV per batch):
# one query token per sequence, H heads, a latent cache of Skv keys that is
# both key (with its rotary part) and value; entries N(0, 1), scale
# (512 + 64)^-1/2.  Seeds: Q 0x7E5A0000 + index, Q_pe that + 0x300, KV that
# + 0x100, K_pe that + 0x400.
MLA_WORKLOADS = {
    "mla_decode_b64h128s4096_bf16": dict(
        index=10, B=64, H=128, Skv=4096, dim=512, pe_dim=64, dtype="bf16"),
}


def mla_workload(name):
    w = dict(MLA_WORKLOADS[name])
    w["name"] = name
    w["seed_q"] = _SEED_BASE + w["index"]
    w["seed_qpe"] = _SEED_BASE + w["index"] + 0x300
    w["seed_kv"] = _SEED_BASE + w["index"] + 0x100
    w["seed_kpe"] = _SEED_BASE + w["index"] + 0x400
    w["scale"] = float(w["dim"] + w["pe_dim"]) ** -0.5
    # two products per key and head: 576-deep scores, 512-wide values
    w["flops"] = 2 * w["B"] * w["H"] * w["Skv"] * (w["dim"] + w["pe_dim"] + w["dim"])
    # Q, Q_pe, KV, K_pe read once, O written once (16-bit)
    w["bytes"] = 2 * (w["B"] * w["H"] * (w["dim"] + w["pe_dim"]) + w["B"] * w["Skv"] * (w["dim"] + w["pe_dim"])
                      + w["B"] * w["H"] * w["dim"])
    return w


def mla_inputs(w, off=0):
    """Q (B, H, dim), Q_pe (B, H, pe_dim), KV (B, Skv, dim), K_pe (B, Skv,
    pe_dim) bit patterns of an MLA workload, N(0, 1)."""
    from . import matrix
    B, H, S = w["B"], w["H"], w["Skv"]

    def mk(rows, cols, seed):
        return matrix(B * rows, cols, ("normal", 1.0), seed + off, w["dtype"]).reshape(B, rows, cols)
    return (mk(H, w["dim"], w["seed_q"]), mk(H, w["pe_dim"], w["seed_qpe"]),
            mk(S, w["dim"], w["seed_kv"]), mk(S, w["pe_dim"], w["seed_kpe"]))


def attn_workload(name):
    w = dict(ATTN_WORKLOADS[name])
    w["name"] = name
    w["seed_q"] = _SEED_BASE + w["index"]
    w["seed_k"] = _SEED_BASE + w["index"] + 0x100
    w["seed_v"] = _SEED_BASE + w["index"] + 0x200
    # score / weighted-sum pairs a row visits: all keys, or the causal
    # t <= i + Sk - Sq
    Sq, Sk = w["Sq"], w["Sk"]
    if w["causal"]:
        i = np.arange(Sq, dtype=np.int64)
        pairs = int(np.clip(i + Sk - Sq + 1, 0, Sk).sum())
    else:
        pairs = Sq * Sk
    w["flops"] = 4 * w["B"] * w["H"] * pairs * w["D"]
    return w


def workload(name):
    w = dict(WORKLOADS[name] if name in WORKLOADS else EXTRA_WORKLOADS[name])
    w.setdefault("layout", "rrr")
    w["name"] = name
    w["seed_a"] = _SEED_BASE + w["index"]
    w["seed_b"] = _SEED_BASE + w["index"] + 0x100
    w["flops"] = 2 * w["M"] * w["N"] * w["K"]
    return w


def inputs(name, out_a=None, out_b=None):
    """(A_bits, B_bits) numpy arrays (uint16 for 16-bit inputs, uint8 for
    8-bit) of the logical row-major A (M x K) and B (K x N) of a named
    workload."""
    from . import matrix
    w = workload(name)
    A = matrix(w["M"], w["K"], w["dist_a"], w["seed_a"], w["dtype_in"], out=out_a)
    B = matrix(w["K"], w["N"], w["dist_b"], w["seed_b"], w["dtype_in"], out=out_b)
    return A, B


def out_nbytes(dtype_out):
    return 4 if dtype_out == "f32" else 2


def in_nbytes(dtype_in):
    return 1 if dtype_in in ("e4m3", "e5m2") else 2


def stored(A, B, layout):
    """The operands as the library is handed them for `layout`: A as is or
    transposed (K x M), B as is or transposed (N x K), both contiguous."""
    import numpy as np
    lay = {"rrr": 0, "rcr": 1, "crr": 2, "ccr": 3}[layout]
    A_s = np.ascontiguousarray(A.T) if lay & 2 else A
    B_s = np.ascontiguousarray(B.T) if lay & 1 else B
    return A_s, B_s


def out_numpy_dtype(dtype_out):
    return np.float32 if dtype_out == "f32" else np.uint16
