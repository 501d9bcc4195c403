"""The seeded input generator: determinism, the published SplitMix64 stream,
distribution shape and exact quantisation."""
import numpy as np

import synth


def test_splitmix64_matches_scalar_definition():
    # scalar restatement with Python integers (mod 2^64)
    def sm(seed, c):
        x = (seed + (c + 1) * 0x9E3779B97F4A7C15) & (2 ** 64 - 1)
        x = ((x ^ (x >> 30)) * 0xBF58476D1CE4E5B9) & (2 ** 64 - 1)
        x = ((x ^ (x >> 27)) * 0x94D049BB133111EB) & (2 ** 64 - 1)
        return x ^ (x >> 31)
    got = synth.splitmix64(1234567, 5, 20)
    assert [int(v) for v in got] == [sm(1234567, c) for c in range(5, 25)]


def test_splitmix64_known_first_output_for_seed_zero():
    # The first output of SplitMix64 seeded with 0 is 0xE220A8397B1DCDAF
    # (the commonly quoted first value of the published generator).
    assert int(synth.splitmix64(0, 0, 1)[0]) == 0xE220A8397B1DCDAF


def test_chunking_does_not_change_the_stream():
    old = synth._CHUNK
    try:
        a = synth.matrix(33, 77, ("normal", 1.0), 99, "bf16")
        synth._CHUNK = 100
        b = synth.matrix(33, 77, ("normal", 1.0), 99, "bf16")
    finally:
        synth._CHUNK = old
    assert np.array_equal(a, b)


def test_distributions_have_their_moments():
    n = 1 << 20
    u = synth._draw(("uniform", -1.0, 1.0), 7, 0, n)
    assert abs(u.mean()) < 5e-3 and abs(u.var() - 1 / 3) < 5e-3
    assert u.min() >= -1.0 and u.max() < 1.0
    g = synth._draw(("normal", 0.02), 8, 0, n)
    assert abs(g.mean()) < 1e-4 and abs(g.std() - 0.02) < 1e-4
    i = synth._draw(("int", -2, 2), 9, 0, n)
    vals, counts = np.unique(i, return_counts=True)
    assert list(vals) == [-2, -1, 0, 1, 2]
    assert np.all(np.abs(counts / n - 0.2) < 5e-3)


def test_integer_inputs_are_exact_in_both_formats():
    for dt in ("bf16", "f16"):
        m = synth.matrix(64, 64, ("int", -2, 2), 11, dt)
        x = m.view(np.float16).astype(np.float64) if dt == "f16" else \
            (m.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        assert set(np.unique(x)) <= {-2.0, -1.0, 0.0, 1.0, 2.0}


def test_workload_table():
    w = synth.workload("gemm_16384x16384x8192_bf16")
    assert (w["M"], w["N"], w["K"]) == (16384, 16384, 8192)
    assert w["seed_a"] == 0x7E5A0003 and w["seed_b"] == 0x7E5A0103
    assert len(synth.WORKLOADS) == 5
    A, B = synth.inputs("gemm_256_f16_f32")
    assert A.shape == (256, 256) and A.dtype == np.uint16
    A2, _ = synth.inputs("gemm_256_f16_f32")
    assert np.array_equal(A, A2)
