"""Parity of the CUDA path against the fp64 oracle, element by element.

Acceptance (per output element): bit-exact equality with the oracle's sum
rounded to the output format when the inputs are integers whose fp32
partial sums are all exact; otherwise |C - ref| <= 1e-3 * sum_k |a_ik b_kj|
+ 1e-5.  Shapes span several tiles and ragged tails; every tile width,
split factor and output format is exercised, then the five workloads (the
16384 x 16384 x 8192 one on sampled outputs and whole rows/columns).
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import run_gemm

pytestmark = pytest.mark.gpu


def _ints(rows, cols, seed, lo=-2, hi=2, dtype="bf16"):
    return synth.matrix(rows, cols, ("int", lo, hi), seed, dtype)


def _unif(rows, cols, seed, dtype):
    return synth.matrix(rows, cols, ("uniform", -1.0, 1.0), seed, dtype)


def _bits_of(x, dtype):
    return synth.quantise(np.asarray(x, dtype=np.float64), dtype)


def _check(C, A, B, din, dout, exact):
    ref, sabs, _ = oracle.gemm(A, B, din)
    ok, info = oracle.accept(C, ref, sabs, dout, exact=exact)
    assert ok, info


# ------------------------------------------------------------ pin cases --

@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f16", "f32"), ("f16", "f16"), ("bf16", "f32")])
@pytest.mark.parametrize("n", [256, 200])
def test_identity_left(din, dout, n):
    # I * B = B exactly: pins the A-side (K-major) layout and the epilogue.
    eye = _bits_of(np.eye(n), din)
    B = _ints(n, 264, 1, -8, 8, din)
    C, _ = run_gemm(eye, B, din, dout)
    _check(C, eye, B, din, dout, exact=True)


@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f16", "f32")])
@pytest.mark.parametrize("n", [256, 136])
def test_identity_right(din, dout, n):
    # A * I = A exactly: pins the B-side (MN-major) descriptor.
    eye = _bits_of(np.eye(n), din)
    A = _ints(300, n, 2, -8, 8, din)
    C, _ = run_gemm(A, eye, din, dout)
    _check(C, A, eye, din, dout, exact=True)


TILES = [(128, 64), (128, 128), (128, 192), (128, 256), (256, 128), (256, 256)]


@pytest.mark.parametrize("block_m,block_n", TILES)
def test_permutation_both_sides(block_m, block_n):
    r = np.random.default_rng(3)
    n = 384
    perm = r.permutation(n)
    P = np.zeros((n, n))
    P[np.arange(n), perm] = 1.0
    Pb = _bits_of(P, "bf16")
    B = _ints(n, 320, 4, -16, 16)
    C, cfg = run_gemm(Pb, B, "bf16", "bf16", block_m=block_m, block_n=block_n)
    assert (cfg["block_m"], cfg["block_n"]) == (block_m, block_n)
    _check(C, Pb, B, "bf16", "bf16", exact=True)
    A = _ints(256, n, 5, -16, 16)
    C, _ = run_gemm(A, Pb, "bf16", "bf16", block_m=block_m, block_n=block_n)
    _check(C, A, Pb, "bf16", "bf16", exact=True)


@pytest.mark.parametrize("splits", [1, 2, 5])
def test_rank_one_closed_form(splits):
    r = np.random.default_rng(6)
    M, N, K = 260, 392, 1000
    u, v = r.integers(-3, 4, M), r.integers(-3, 4, N)
    p, q = r.integers(-2, 3, K), r.integers(-2, 3, K)
    A = _bits_of(np.outer(u, p), "bf16")
    B = _bits_of(np.outer(q, v), "bf16")
    C, _ = run_gemm(A, B, "bf16", "f32", splits=splits)
    want = (np.dot(p, q) * np.outer(u, v)).astype(np.float32)
    assert np.array_equal(C, want)


@pytest.mark.parametrize("K", [8, 64, 72, 640, 4104])
@pytest.mark.parametrize("splits", [1, 3])
def test_all_ones_counts_every_k_block_once(K, splits):
    if splits > (K + 63) // 64:
        pytest.skip("more splits than K-slices")
    A = _bits_of(np.ones((130, K)), "bf16")
    B = _bits_of(np.ones((K, 136)), "bf16")
    C, _ = run_gemm(A, B, "bf16", "f32", splits=splits)
    assert np.all(C == K)


# --------------------------------------------- random shapes and configs --

SHAPES = [(256, 256, 256), (129, 264, 72), (300, 520, 200), (1, 8, 8), (127, 64, 64),
          (128, 512, 1000), (513, 1032, 328), (64, 1928, 512)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("din,dout", [("bf16", "bf16"), ("f16", "f32"), ("f16", "f16"), ("bf16", "f32")])
def test_random_shapes_default_plan(shape, din, dout):
    M, N, K = shape
    A = _unif(M, K, 10 + M, din)
    B = _unif(K, N, 20 + N, din)
    C, _ = run_gemm(A, B, din, dout)
    _check(C, A, B, din, dout, exact=False)


@pytest.mark.parametrize("block_m,block_n", TILES)
@pytest.mark.parametrize("splits", [1, 2, 7])
@pytest.mark.parametrize("stages", [2, 0])
def test_every_tile_shape_and_split(block_m, block_n, splits, stages):
    M, N, K = 333, 776, 1096
    A = _ints(M, K, 30, dtype="bf16")
    B = _ints(K, N, 31, dtype="bf16")
    force = {"block_m": block_m, "block_n": block_n, "splits": splits}
    if stages:
        force["stages"] = stages
    C, cfg = run_gemm(A, B, "bf16", "f32", **force)
    assert (cfg["block_m"], cfg["block_n"], cfg["splits"]) == (block_m, block_n, splits)
    _check(C, A, B, "bf16", "f32", exact=True)


@pytest.mark.parametrize("block_m,block_n", TILES)
@pytest.mark.parametrize("which", ["one", "all_but_one"])
def test_tail_tiles_split(block_m, block_n, which):
    # Only the last tiles of the schedule are split along K (the tail wave);
    # the others are computed whole, in the same launch.
    M, N, K = 600, 776, 1096
    tiles = -(-M // block_m) * -(-N // block_n)
    st = 1 if which == "one" else tiles - 1
    A = _ints(M, K, 32, dtype="bf16")
    B = _ints(K, N, 33, dtype="bf16")
    C, cfg = run_gemm(A, B, "bf16", "f32", block_m=block_m, block_n=block_n, splits=3, split_tiles=st)
    assert cfg["split_tiles"] == st and cfg["units"] == tiles - st + 3 * st
    _check(C, A, B, "bf16", "f32", exact=True)


LAYOUTS = ["rrr", "rcr", "crr", "ccr"]


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("block_m,block_n", TILES)
def test_layouts_every_tile_shape(layout, block_m, block_n):
    # Operands stored transposed (column-major A: K x M; B: N x K) give the
    # same product; integer inputs make the comparison bit-exact.
    M, N, K = 264, 328, 1096
    A = _ints(M, K, 34, dtype="bf16")
    B = _ints(K, N, 35, dtype="bf16")
    C, cfg = run_gemm(A, B, "bf16", "f32", layout=layout, block_m=block_m, block_n=block_n)
    assert (cfg["block_m"], cfg["block_n"]) == (block_m, block_n)
    _check(C, A, B, "bf16", "f32", exact=True)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_layouts_permutation_pins(layout):
    # P * B and A * P with a permutation P, stored in each layout.
    r = np.random.default_rng(36)
    n = 256
    perm = r.permutation(n)
    P = np.zeros((n, n))
    P[np.arange(n), perm] = 1.0
    Pb = _bits_of(P, "f16")
    B = _ints(n, 200, 37, -16, 16, "f16")
    C, _ = run_gemm(Pb, B, "f16", "f16", layout=layout)
    _check(C, Pb, B, "f16", "f16", exact=True)
    A = _ints(136, n, 38, -16, 16, "f16")
    C, _ = run_gemm(A, Pb, "f16", "f16", layout=layout)
    _check(C, A, Pb, "f16", "f16", exact=True)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("splits", [1, 3])
def test_layouts_random_real_inputs(layout, splits):
    M, N, K = 520, 776, 2048
    A = _unif(M, K, 39, "bf16")
    B = _unif(K, N, 40, "bf16")
    C, _ = run_gemm(A, B, "bf16", "bf16", layout=layout, splits=splits)
    _check(C, A, B, "bf16", "bf16", exact=False)


@pytest.mark.parametrize("block_m,grid", [(128, 2), (128, 3), (256, 4), (256, 6)])
def test_persistent_loop_with_small_grid(block_m, grid):
    # Few CTAs walk many units: exercises ring-phase and accumulator-phase
    # wrap-around over many tiles.
    A = _ints(640, 512, 40)
    B = _ints(512, 1024, 41)
    C, cfg = run_gemm(A, B, "bf16", "bf16", grid=grid, block_m=block_m, block_n=128, splits=2)
    assert cfg["grid"] == grid
    _check(C, A, B, "bf16", "bf16", exact=True)


@pytest.mark.parametrize("M", [1, 128, 200, 257, 511])
def test_pair_tiles_with_ragged_rows(M):
    # A pair tile whose second CTA has few or no valid rows.
    A = _unif(M, 192, 45 + M, "bf16")
    B = _unif(192, 264, 46, "bf16")
    C, cfg = run_gemm(A, B, "bf16", "bf16", block_m=256, block_n=256)
    assert cfg["block_m"] == 256
    _check(C, A, B, "bf16", "bf16", exact=False)


@pytest.mark.parametrize("group_m", [1, 3, 16])
@pytest.mark.parametrize("block_m,block_n", [(128, 64), (256, 128)])
def test_raster_groups(group_m, block_m, block_n):
    A = _unif(700, 256, 50, "bf16")
    B = _unif(256, 1280, 51, "bf16")
    C, _ = run_gemm(A, B, "bf16", "bf16", group_m=group_m, block_m=block_m, block_n=block_n)
    _check(C, A, B, "bf16", "bf16", exact=False)


def test_fp16_subnormal_inputs():
    # Many A entries are fp16 subnormals; their exact products must reach
    # the fp32 accumulator (a flush to zero would show up here).
    r = np.random.default_rng(60)
    a = r.integers(1, 1024, (256, 512)) * 2.0 ** -24 * r.choice([-1, 1], (256, 512))
    A = _bits_of(a, "f16")
    B = _bits_of(r.integers(-4, 5, (512, 256)) * 64.0, "f16")
    C, _ = run_gemm(A, B, "f16", "f32")
    _check(C, A, B, "f16", "f32", exact=True)


def test_runs_are_bitwise_reproducible():
    A = _unif(512, 512, 70, "bf16")
    B = _unif(512, 768, 71, "bf16")
    outs, _ = run_gemm(A, B, "bf16", "f32", splits=4, repeat=3)
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_large_m_narrow_n():
    A = _ints(70001, 64, 80)
    B = _ints(64, 8, 81)
    C, _ = run_gemm(A, B, "bf16", "bf16")
    _check(C, A, B, "bf16", "bf16", exact=True)


def test_host_pointer_is_rejected_before_launch():
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    plan = tsgemm.Plan(128, 128, 128, "bf16", "bf16")
    A = torch.zeros((128, 128), dtype=torch.bfloat16)  # host memory
    B = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(tsgemm.TsgemmError) as e:
        plan.run(A, B, C)
    assert e.value.status == tsgemm.ERR_INVALID_ARG
    with pytest.raises(tsgemm.TsgemmError) as e:
        plan.run(B, B, B)  # C aliases A and B
    assert e.value.status == tsgemm.ERR_INVALID_ARG
    with pytest.raises(tsgemm.TsgemmError) as e:
        plan.run(B.view(-1)[1:].data_ptr(), B, C)  # 2-byte offset
    assert e.value.status == tsgemm.ERR_ALIGNMENT
    plan.close()


# -------------------------------------------------------- the workloads --

def _workload_case(name, **force):
    w = synth.workload(name)
    A, B = synth.inputs(name)
    C, cfg = run_gemm(A, B, w["dtype_in"], w["dtype_out"], **force)
    return w, A, B, C, cfg


@pytest.mark.parametrize("name", ["gemm_256_f16_f32", "gemm_4096_bf16",
                                  "skinny_128x28672x8192_bf16", "longk_1024x1024x65536_int_f32"])
def test_workload_full_compare(name):
    w, A, B, C, _ = _workload_case(name)
    _check(C, A, B, w["dtype_in"], w["dtype_out"], exact=w["exact"])


@pytest.mark.parametrize("name", ["gemm_4096_bf16", "longk_1024x1024x65536_int_f32"])
def test_workload_full_compare_one_sm_tiles(name):
    w, A, B, C, cfg = _workload_case(name, block_m=128)
    assert cfg["block_m"] == 128
    _check(C, A, B, w["dtype_in"], w["dtype_out"], exact=w["exact"])


def test_workload_16384x16384x8192_sampled():
    w, A, B, C, _ = _workload_case("gemm_16384x16384x8192_bf16")
    r = np.random.default_rng(90)
    M, N = w["M"], w["N"]
    rows = np.concatenate([r.integers(0, M, 8192), np.repeat([0, M - 1, 12345], N)])
    cols = np.concatenate([r.integers(0, N, 8192), np.tile(np.arange(N), 3)])
    # every tile's corner elements
    tr = np.arange(0, M, 128)
    tc = np.arange(0, N, 256)
    for dr, dc in [(0, 0), (127, 255), (0, 255), (127, 0)]:
        g = np.array(np.meshgrid(tr + dr, tc + dc, indexing="ij")).reshape(2, -1)
        rows = np.concatenate([rows, g[0]])
        cols = np.concatenate([cols, g[1]])
    ref, sabs = oracle.gemm_sampled(A, B, w["dtype_in"], rows, cols)
    ok, info = oracle.accept(C[rows, cols], ref, sabs, w["dtype_out"])
    assert ok, info
