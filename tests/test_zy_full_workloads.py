"""Full-output parity of the largest workloads against the fp64 oracle.

Every element of C of the 16384 x 16384 x 8192 GEMM (bf16 and 8-bit E4M3
inputs) and of the 4096^3 E4M3 GEMM, and every output row of the B = 4,
H = 32, S = 4096 attention workloads (causal and not), is compared with the
oracle under the acceptance rules of oracle.accept / accept_attention, in
the launch configuration the benchmark times.  The oracle takes minutes of
host time here, so this file is collected after the other GPU tests: a
failure in it stops nothing else.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import from_dev, run_gemm, to_dev

pytestmark = pytest.mark.gpu

ROW_BLOCK = 2048


def _compare_in_row_blocks(C, A, B, w):
    """oracle.accept on blocks of rows (the oracle's fp64 output of a whole
    16384^2 product would take 4 GB of host memory at once)."""
    M = w["M"]
    worst = 0.0
    for r0 in range(0, M, ROW_BLOCK):
        r1 = min(M, r0 + ROW_BLOCK)
        ref, sabs, _ = oracle.gemm(A[r0:r1], B, w["dtype_in"])
        ok, info = oracle.accept(C[r0:r1], ref, sabs, w["dtype_out"], exact=w["exact"])
        assert ok, (w["name"], r0, info)
        worst = max(worst, info.get("max_err_over_bound", 0.0))
    return worst


@pytest.mark.parametrize("name", ["gemm_16384x16384x8192_bf16", "gemm_16384x16384x8192_e4m3_rcr",
                                  "gemm_4096_e4m3_rcr"])
def test_gemm_workload_every_element(name):
    w = synth.workload(name)
    A, B = synth.inputs(name)
    C, cfg = run_gemm(A, B, w["dtype_in"], w["dtype_out"], layout=w["layout"])
    assert C.shape == (w["M"], w["N"])
    worst = _compare_in_row_blocks(C, A, B, w)
    assert worst <= 1.0


@pytest.mark.parametrize("causal", [False, True])
def test_attention_workload_every_row(causal):
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    name = "attn_b4h32s4096d128_causal_bf16" if causal else "attn_b4h32s4096d128_bf16"
    w = synth.attn_workload(name)
    B, H, S, D = w["B"], w["H"], w["Sq"], w["D"]

    def mk(seed):
        return synth.matrix(B * H * S, D, ("normal", 1.0), seed, "bf16").reshape(B, H, S, D)
    Qb, Kb, Vb = mk(w["seed_q"]), mk(w["seed_k"]), mk(w["seed_v"])
    Q, K, V = (to_dev(x.reshape(-1, D), "bf16").reshape(x.shape) for x in (Qb, Kb, Vb))
    O = torch.full(Q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    tsgemm.attention(Q, K, V, scale=D ** -0.5, causal=causal, O=O)
    torch.cuda.synchronize()
    assert tsgemm.attention_status() == 0
    got = from_dev(O.reshape(-1, D), "bf16").reshape(B, H, S, D)
    # one batch at a time: the oracle's fp64 output and bound of a batch
    # take 2 x 128 MB
    for b in range(B):
        ref, bound = oracle.attention(Qb[b:b + 1], Kb[b:b + 1], Vb[b:b + 1], "bf16", D ** -0.5, causal)
        ok, info = oracle.accept_attention(got[b:b + 1], ref, bound, "bf16")
        assert ok, (name, b, info)
