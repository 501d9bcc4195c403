"""Split-K and stream-K plans whose CTAs cannot all run at the same time.

The parts of a tile cut along K never wait for one another: whichever part
completes a chunk's set of fp32 partials adds them (in part order) and
stores C.  So a split factor larger than the grid, a stream-K plan on a
small grid, and a plan launched while another kernel holds all but a few
SMs for longer than the device-side wait limit all finish with the exact
result.  Integer inputs make every fp32 sum exact, so results are compared
bit for bit with the oracle.
"""
import ctypes
import os
import subprocess
import time

import numpy as np
import pytest

import oracle
import synth
from gpu_util import TORCH_DT, from_dev, run_gemm, to_dev

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _ints(rows, cols, seed, lo=-2, hi=2):
    return synth.matrix(rows, cols, ("int", lo, hi), seed, "bf16")


def _check_exact(C, A, B, dout):
    ref, sabs, _ = oracle.gemm(A, B, "bf16")
    ok, info = oracle.accept(C, ref, sabs, dout, exact=True)
    assert ok, info


@pytest.mark.parametrize("force", [
    dict(block_m=128, block_n=128, splits=8, grid=2),
    dict(block_m=128, block_n=64, splits=16, grid=1),
    dict(block_m=256, block_n=256, splits=8, grid=2),
    dict(block_m=256, block_n=128, splits=5, grid=4),
])
@pytest.mark.parametrize("dout", ["f32", "bf16"])
def test_split_factor_larger_than_the_grid(force, dout):
    A = _ints(512, 6144, 11)
    B = _ints(6144, 384, 12)
    C, cfg = run_gemm(A, B, "bf16", dout, **force)
    assert cfg["splits"] == force["splits"] and cfg["grid"] == force["grid"]
    _check_exact(C, A, B, dout)


@pytest.mark.parametrize("M,N,K,force", [
    (1024, 1024, 4096, dict(block_m=256, block_n=256, stream_k_tiles=16, grid=4)),
    (1024, 768, 2048, dict(block_m=128, block_n=128, stream_k_tiles=20, grid=3)),
])
def test_stream_k_on_a_small_grid(M, N, K, force):
    A = _ints(M, K, 21)
    B = _ints(K, N, 22)
    C, cfg = run_gemm(A, B, "bf16", "f32", **force)
    assert cfg["stream_k_tiles"] == force["stream_k_tiles"] and cfg["grid"] == force["grid"]
    _check_exact(C, A, B, "f32")


def _filler():
    """The test helper library (tests/filler.cu), built with nvcc on first use."""
    out_dir = os.path.join(HERE, "_build")
    lib = os.path.join(out_dir, "libfiller.so")
    src = os.path.join(HERE, "filler.cu")
    if not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src):
        os.makedirs(out_dir, exist_ok=True)
        tmp = lib + ".%d.tmp" % os.getpid()
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                        "-Xcompiler", "-fPIC", "-o", tmp, src], check=True)
        os.replace(tmp, lib)
    L = ctypes.CDLL(lib)
    L.filler_launch.restype = ctypes.c_int
    L.filler_launch.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_ulonglong, ctypes.c_void_p, ctypes.c_void_p]
    return L


@pytest.mark.parametrize("block_m,free_sms", [(128, 3), (256, 6)])
def test_long_k_beside_a_kernel_holding_most_sms(block_m, free_sms):
    # The long-K workload with every tile split in 4.  A filler kernel holds
    # all but `free_sms` SMs for 1.5 s, longer than the GEMM's 1 s wait limit;
    # fewer parts of a tile than its split factor fit in the free SMs, so a
    # scheme whose parts waited for one another would give up.
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    lib = _filler()
    w = synth.workload("longk_1024x1024x65536_int_f32")
    A_np, B_np = synth.inputs(w["name"])
    A, B = to_dev(A_np, "bf16"), to_dev(B_np, "bf16")
    C = torch.full((w["M"], w["N"]), float("nan"), dtype=torch.float32, device="cuda")
    plan = tsgemm.Plan(w["M"], w["N"], w["K"], "bf16", "f32", block_m=block_m, splits=4, split_tiles=0)
    cfg = plan.config
    assert cfg["splits"] == 4 and cfg["split_tiles"] > 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    done = torch.zeros(1, dtype=torch.int32, device="cuda")
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    blocks = sms - free_sms
    rc = lib.filler_launch(blocks, 200 * 1024, 1_500_000_000, done.data_ptr(), side.cuda_stream)
    assert rc == 0, rc
    time.sleep(0.1)  # the filler's blocks are resident
    t0 = time.time()
    plan.run(A, B, C)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert int(done.item()) == blocks
    st = plan.status()
    assert st == 0, "device status %d (%s)" % (st, tsgemm.status_string(st))
    plan.close()
    _check_exact(from_dev(C, "f32"), A_np, B_np, "f32")
    assert elapsed < 10.0
