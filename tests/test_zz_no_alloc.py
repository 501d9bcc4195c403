"""The split-K GEMM entry point that allocates nothing.

Some callers cannot call cudaMalloc: code running inside another
framework's allocator hooks, plug-ins that are handed their buffers, and
real-time loops that forbid allocation (which can synchronise the device)
after start-up.  tsgemm_run_splitk_noalloc serves them: its split-K scratch
is a fixed device array inside the library.  These tests call it through
the C ABI and check its output against the planned entry point
(tsgemm_plan + tsgemm_run with the same split) and the fp64 oracle, on two
calls in a row that reuse the same scratch array.

This file is collected last so that, if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import TORCH_DT, from_dev, run_gemm, to_dev

pytestmark = pytest.mark.gpu


def _noalloc(A_bits, B_bits, din, dout, splits):
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    M, K = A_bits.shape
    N = B_bits.shape[1]
    A = to_dev(A_bits, din)
    B = to_dev(B_bits, din)
    C = torch.full((M, N), float("nan"), dtype=TORCH_DT[dout], device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    code = tsgemm.lib.tsgemm_run_splitk_noalloc(M, N, K, tsgemm.dtype_code(din), tsgemm.dtype_code(dout),
                                                splits, A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                                status.data_ptr(), stream)
    assert code == tsgemm.OK, tsgemm.status_string(code)
    return A, B, C, status


def test_noalloc_matches_the_planned_entry_point_on_two_calls_in_a_row():
    import torch
    cases = [
        # integer inputs: exact sums, compared bit for bit
        (synth.matrix(333, 2048, ("int", -2, 2), 0xA110C, "bf16"),
         synth.matrix(2048, 776, ("int", -2, 2), 0xA110D, "bf16"), "bf16", "f32", 5, True),
        # real inputs, a different shape and split on the same scratch array
        (synth.matrix(520, 1000, ("uniform", -1.0, 1.0), 0xA110E, "bf16"),
         synth.matrix(1000, 264, ("uniform", -1.0, 1.0), 0xA110F, "bf16"), "bf16", "bf16", 3, False),
    ]
    pending = []
    for A_bits, B_bits, din, dout, splits, exact in cases:
        pending.append((A_bits, B_bits, din, dout, splits, exact) + _noalloc(A_bits, B_bits, din, dout, splits))
    torch.cuda.synchronize()
    for A_bits, B_bits, din, dout, splits, exact, _, _, C, status in pending:
        assert int(status.item()) == 0, "device status %d" % int(status.item())
        got = from_dev(C, dout)
        want, cfg = run_gemm(A_bits, B_bits, din, dout, splits=splits, block_m=128)
        assert cfg["splits"] == splits
        # the same kernel and configuration: the same bits
        assert np.array_equal(got.view(np.uint8), want.view(np.uint8))
        ref, sabs, _ = oracle.gemm(A_bits, B_bits, din)
        ok, info = oracle.accept(got, ref, sabs, dout, exact=exact)
        assert ok, info


def test_noalloc_rejects_problems_beyond_its_scratch():
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    # 4096 x 4096 with every tile split needs 4096 * 4096 * 4 B = 64 MiB of
    # running sums, twice the fixed scratch
    A = torch.zeros((4096, 4096), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((4096, 4096), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((4096, 4096), dtype=torch.bfloat16, device="cuda")
    code = tsgemm.lib.tsgemm_run_splitk_noalloc(4096, 4096, 4096, tsgemm.BF16, tsgemm.BF16, 8,
                                                A.data_ptr(), B.data_ptr(), C.data_ptr(), None,
                                                torch.cuda.current_stream().cuda_stream)
    assert code == tsgemm.ERR_SCRATCH_LIMIT
    assert "scratch" in tsgemm.status_string(code)
    # without a status pointer the call still runs (device timeouts go to
    # the library's own word)
    A_bits = synth.matrix(128, 512, ("int", -2, 2), 1, "bf16")
    B_bits = synth.matrix(512, 128, ("int", -2, 2), 2, "bf16")
    A, B = to_dev(A_bits, "bf16"), to_dev(B_bits, "bf16")
    C = torch.empty((128, 128), dtype=torch.float32, device="cuda")
    code = tsgemm.lib.tsgemm_run_splitk_noalloc(128, 128, 512, tsgemm.BF16, tsgemm.F32, 2,
                                                A.data_ptr(), B.data_ptr(), C.data_ptr(), None,
                                                torch.cuda.current_stream().cuda_stream)
    assert code == tsgemm.OK
    torch.cuda.synchronize()
    ref, sabs, _ = oracle.gemm(A_bits, B_bits, "bf16")
    ok, info = oracle.accept(C.cpu().numpy(), ref, sabs, "f32", exact=True)
    assert ok, info
