"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each with its own
instance of the workload, timing reduced as the max over ranks and the
whole-job value summed over ranks (weak scaling, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import synth
    try:
        r, w, lr = bench.dist_env()
        ms = 1.0 + rank  # rank 1 is slower
        ms_max = bench.max_over_ranks(ms, w)
        value = bench.aggregate_tflops(1e12, ms_max, w)
        wl = synth.workload("gemm_256_f16_f32")
        off = bench.rank_seed_offset(r)
        A = synth.matrix(4, 8, wl["dist_a"], wl["seed_a"] + off, wl["dtype_in"])
        bench.barrier(w)
        q.put((r, w, lr, ms_max, value, A.tobytes()))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_weak_scaling():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=100) for _ in procs]
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    out.sort()
    assert [o[0] for o in out] == [0, 1] and all(o[1] == 2 for o in out)
    assert [o[2] for o in out] == [0, 1]
    # both ranks see the slower rank's time; value counts both ranks' work
    assert all(o[3] == 2.0 for o in out)
    assert all(abs(o[4] - 2 * 1e12 / 2e-3 / 1e12) < 1e-9 for o in out)
    # the ranks ran different instances of the workload
    assert out[0][5] != out[1][5]


def test_single_rank_helpers():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert abs(bench.aggregate_tflops(2e12, 1.0, 1) - 2000.0) < 1e-9
    assert bench.rank_seed_offset(0) == 0


def test_bench_arguments():
    import bench
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 1 and a.impl == "ours"
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])
    a = bench.parse_args(["--impl", "reference", "--steps", "3", "--warmup", "3"])
    assert a.impl == "reference"


def test_peak_choice_follows_the_clock_regime():
    import bench
    peaks, _ = bench.measured_peaks()
    burst, kind_b = bench.bf16_peak({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []})
    assert "burst" in kind_b and burst == float(peaks.get("bf16_tflops", bench.FALLBACK_BF16_TFLOPS))
    # the power cap noted but the clock at its maximum: still the burst figure
    same, kind_s = bench.bf16_peak({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]})
    assert same == burst and "burst" in kind_s
    capped, kind_c = bench.bf16_peak({"sm_mhz": 1518.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]})
    if "bf16_tflops_sustained" in peaks:
        assert "sustained" in kind_c and capped == float(peaks["bf16_tflops_sustained"])
    else:
        assert capped == burst
    assert bench.bf16_peak(None)[0] == burst


def test_roofline_point_picks_the_bound_by_intensity():
    import bench
    peaks, _ = bench.measured_peaks()
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    # the skinny projection: 60.1 GFLOP over 479.2 MB (125 F/B) is HBM-bound
    b, a, p, u, _ = bench.roofline_point(60129542144.0, 479199232, 0.0919, 1912.5, "t")
    assert (b, u, p) == ("hbm", "GB/s", hbm) and abs(a - 479199232 / 0.0919e-3 / 1e9) < 1e-6
    # 4096^3: 1365 F/B, tensor-bound
    b, a, p, u, d = bench.roofline_point(2.0 * 4096 ** 3, 100663296, 0.0886, 1912.5, "t")
    assert (b, u, p, d) == ("tensor", "TFLOP/s", 1912.5, "t") and abs(a - 2.0 * 4096 ** 3 / 0.0886e-3 / 1e12) < 1e-6
