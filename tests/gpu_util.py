"""Helpers shared by the GPU tests: move 16-bit or 8-bit input bits to the
device, run a plan through the C ABI and bring the output back as raw bits."""
import numpy as np
import torch

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32,
            "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def to_dev(bits, din, device="cuda"):
    if din in ("e4m3", "e5m2"):
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.uint8)).to(device)
    else:
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
    return t.view(TORCH_DT[din])


def from_dev(C, dout):
    c = C.cpu()
    if dout == "f32":
        return c.numpy()
    return c.view(torch.int16).numpy().view(np.uint16)


def run_gemm(A_bits, B_bits, din, dout, device="cuda", repeat=1, layout="rrr", **force):
    """C = A * B through tsgemm; returns (C bits/values, plan config).

    A_bits (M x K) and B_bits (K x N) are the logical operands; for the
    column-major layouts they are handed to the library transposed (A stored
    K x M, B stored N x K)."""
    from hierarchical_gemm_gb300 import tsgemm
    M, K = A_bits.shape
    N = B_bits.shape[1]
    code = tsgemm.layout_code(layout)
    plan = tsgemm.Plan(M, N, K, din, dout, layout=code, **force)
    A_store = np.ascontiguousarray(A_bits.T) if code & 2 else A_bits
    B_store = np.ascontiguousarray(B_bits.T) if code & 1 else B_bits
    A = to_dev(A_store, din, device)
    B = to_dev(B_store, din, device)
    C = torch.full((M, N), float("nan"), dtype=TORCH_DT[dout], device=device)
    outs = []
    for _ in range(repeat):
        plan.run(A, B, C)
        torch.cuda.synchronize()
        st = plan.status()
        assert st == 0, "device status %d (%s)" % (st, tsgemm.status_string(st))
        outs.append(from_dev(C, dout))
    cfg = plan.config
    plan.close()
    return (outs if repeat > 1 else outs[0]), cfg
