"""Parity of the MLA decode kernel (tsattn_mla_decode) against the fp64 oracle.

O[b, h] = softmax(scale [Q Q_pe][b, h] . [KV K_pe][b, t]) KV[b, t] over the
keys t: 576-deep scores, 512-wide values, one query token per head.  The
cases cover one and several 128-head blocks (and a ragged last one), key
counts that do not fill the last 64-key block, a single key, a wide score
range that makes the running maximum move (the rescale of the partial
output), both 16-bit formats, the L2 prefetch option, the full-size
workload on sampled batches, and an expired bounded wait.  The acceptance
rule is the attention block's (oracle.accept_attention).
"""
import time

import numpy as np
import pytest

import oracle
import synth
from gpu_util import from_dev, to_dev

pytestmark = pytest.mark.gpu

DIM, PE = 512, 64


def _inputs(B, H, S, dtype, seed, sigma=1.0):
    def mk(rows, cols, s):
        return synth.matrix(B * rows, cols, ("normal", sigma), seed + s, dtype).reshape(B, rows, cols)
    return mk(H, DIM, 0), mk(H, PE, 1), mk(S, DIM, 2), mk(S, PE, 3)


def _run(bits, dtype, scale, **kw):
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    q, qpe, kv, kpe = (to_dev(x.reshape(-1, x.shape[-1]), dtype).reshape(x.shape) for x in bits)
    B, H = q.shape[:2]
    O = torch.full((B, H, DIM), float("nan"), dtype=q.dtype, device="cuda")
    tsgemm.mla_decode(q, qpe, kv, kpe, scale=scale, O=O, **kw)
    torch.cuda.synchronize()
    return O


def _check(B, H, S, dtype, seed, scale=None, sigma=1.0, **kw):
    from hierarchical_gemm_gb300 import tsgemm
    bits = _inputs(B, H, S, dtype, seed, sigma)
    scale = (DIM + PE) ** -0.5 if scale is None else scale
    O = _run(bits, dtype, scale, **kw)
    assert tsgemm.attention_status() == 0
    got = from_dev(O.reshape(-1, DIM), dtype).reshape(B, H, DIM)
    ref, bound = oracle.mla_decode(*bits, dtype, scale)
    ok, info = oracle.accept_attention(got, ref, bound, dtype)
    assert ok, info


@pytest.mark.parametrize("B,H,S", [(2, 128, 256), (3, 128, 1000), (1, 64, 130), (2, 200, 64), (1, 128, 1),
                                   (4, 16, 333), (1, 256, 4096)])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_shapes(B, H, S, dtype):
    _check(B, H, S, dtype, seed=0x3A00 + B * 7 + H + S)


def test_wide_score_range_moves_the_maximum():
    # scores spread over tens of base-2 units: the running maximum of most
    # rows grows past the lazy-rescale threshold in later key blocks
    _check(2, 128, 1024, "bf16", seed=0x3B00, scale=0.5)
    _check(1, 128, 777, "f16", seed=0x3B10, scale=0.3)


def test_prefetch_option():
    _check(2, 128, 2000, "bf16", seed=0x3C00, prefetch_blocks=4)


def test_full_size_workload_sampled_batches():
    # the bench workload (B = 64, H = 128, Skv = 4096) in one launch; every
    # head of three batches against the oracle
    from hierarchical_gemm_gb300 import tsgemm
    w = synth.mla_workload("mla_decode_b64h128s4096_bf16")
    bits = synth.mla_inputs(w)
    O = _run(bits, w["dtype"], w["scale"])
    assert tsgemm.attention_status() == 0
    got = from_dev(O.reshape(-1, DIM), "bf16").reshape(w["B"], w["H"], DIM)
    for b in (0, 31, w["B"] - 1):
        sel = [x[b:b + 1] for x in bits]
        ref, bound = oracle.mla_decode(*sel, "bf16", w["scale"])
        ok, info = oracle.accept_attention(got[b:b + 1], ref, bound, "bf16")
        assert ok, (b, info)


def test_expired_wait_reports_timeout_and_the_context_survives():
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    bits = _inputs(2, 128, 512, "bf16", 0x3D00)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    _run(bits, "bf16", 0.05, status=status, debug_flags=tsgemm.DEBUG_SKIP_FIRST_LOAD, timeout_ms=50)
    assert time.time() - t0 < 10.0
    assert int(status.item()) == tsgemm.ERR_TIMEOUT
    _check(2, 128, 512, "bf16", seed=0x3D00)


def test_argument_errors():
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    L = tsgemm.lib
    x = torch.zeros(1 << 20, dtype=torch.bfloat16, device="cuda")
    p = x.data_ptr()
    o = torch.zeros(1 << 20, dtype=torch.bfloat16, device="cuda").data_ptr()
    args = lambda dim=DIM, pe=PE, B=1, H=8, S=8, dt=tsgemm.BF16, pq=p, po=o: (  # noqa: E731
        B, H, S, dim, pe, dt, 0.1, pq, p, p, p, po, None, None)
    assert L.tsattn_mla_decode(*args(dim=256)) == tsgemm.ERR_UNSUPPORTED
    assert L.tsattn_mla_decode(*args(pe=32)) == tsgemm.ERR_UNSUPPORTED
    assert L.tsattn_mla_decode(*args(dt=tsgemm.F32)) == tsgemm.ERR_UNSUPPORTED
    assert L.tsattn_mla_decode(*args(S=0)) == tsgemm.ERR_INVALID_ARG
    assert L.tsattn_mla_decode(*args(pq=p + 2)) == tsgemm.ERR_ALIGNMENT
    assert L.tsattn_mla_decode(*args(po=p)) == tsgemm.ERR_INVALID_ARG  # O overlaps the inputs
    assert L.tsattn_mla_decode(*args()) == tsgemm.OK
    torch.cuda.synchronize()
