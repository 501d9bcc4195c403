"""Parity of the attention block (softmax(scale Q K^T) V on tcgen05) with
the fp64 oracle, element by element, under the acceptance rule derived
from the kernel's arithmetic (oracle.accept_attention)."""
import time

import numpy as np
import pytest

import oracle
import synth
from gpu_util import TORCH_DT, from_dev, to_dev

pytestmark = pytest.mark.gpu

D = 128


def _tensor(shape, seed, dt, dist=("normal", 1.0)):
    n = int(np.prod(shape))
    return synth.matrix(n // D, D, dist, seed, dt).reshape(shape)


def _run(Qb, Kb, Vb, dt, scale, causal, **kw):
    from hierarchical_gemm_gb300 import tsgemm
    import torch
    Q, K, V = (to_dev(x.reshape(-1, D), dt).reshape(x.shape) for x in (Qb, Kb, Vb))
    O = torch.full(Q.shape, float("nan"), dtype=TORCH_DT[dt], device="cuda")
    tsgemm.attention(Q, K, V, scale=scale, causal=causal, O=O, **kw)
    torch.cuda.synchronize()
    st = tsgemm.attention_status()
    return from_dev(O.reshape(-1, D), dt).reshape(Qb.shape), st


def _check(shape_q, shape_k, dt, causal, scale=D ** -0.5, seed=0, dist=("normal", 1.0)):
    Qb = _tensor(shape_q, 70 + seed, dt, dist)
    Kb = _tensor(shape_k, 71 + seed, dt, dist)
    Vb = _tensor(shape_k, 72 + seed, dt)
    O, st = _run(Qb, Kb, Vb, dt, scale, causal)
    assert st == 0
    ref, bound = oracle.attention(Qb, Kb, Vb, dt, scale, causal)
    ok, info = oracle.accept_attention(O, ref, bound, dt)
    assert ok, info
    return O, ref


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("B,H,Sq,Sk", [(1, 1, 128, 128), (2, 3, 256, 384), (1, 2, 200, 333), (1, 2, 384, 384)])
def test_shapes(dt, causal, B, H, Sq, Sk):
    if causal and Sq > Sk:
        pytest.skip("covered by test_causal_rows_without_keys")
    _check((B, H, Sq, D), (B, H, Sk, D), dt, causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Sq,Sk", [(600, 600), (1000, 777), (641, 1024), (700, 650), (513, 1)])
def test_query_ranges_across_tiles(causal, Sq, Sk):
    # query ranges that end inside a 128-row tile, inside the second tile
    # of a CTA, or with a CTA's second tile wholly past the last row; more
    # queries than keys; a single key
    _check((1, 2, Sq, D), (1, 2, Sk, D), "bf16", causal, seed=50 + Sq + Sk)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Sk", [64, 320, 448])
def test_key_half_past_the_end(causal, Sk):
    # each 128-key block is split between two softmax halves with their own
    # maxima and accumulators; here the last block's second half (Sk = 64,
    # 320) or part of it (448 = 3 x 128 + 64) holds no key, so that half
    # keeps a maximum of -inf for that block (or for the whole row)
    _check((1, 2, 192, D), (1, 2, Sk, D), "bf16", causal, seed=60 + Sk)


def test_key_halves_with_far_apart_maxima():
    # the second half of every 128-key block holds keys scaled up, so its
    # running maximum sits far above the first half's and the final combine
    # scales the first half's sum and output down by a large factor
    B, H, Sq, Sk = 1, 2, 256, 512
    Qb = _tensor((B, H, Sq, D), 91, "bf16")
    k = oracle.decode(_tensor((B, H, Sk, D), 92, "bf16"), "bf16")
    k *= np.where((np.arange(Sk) % 128) >= 64, 6.0, 1.0)[None, None, :, None]
    Kb = synth.quantise(k, "bf16")
    Vb = _tensor((B, H, Sk, D), 93, "bf16")
    for causal in (False, True):
        O, st = _run(Qb, Kb, Vb, "bf16", 0.125, causal)
        assert st == 0
        ref, bound = oracle.attention(Qb, Kb, Vb, "bf16", 0.125, causal)
        ok, info = oracle.accept_attention(O, ref, bound, "bf16")
        assert ok, (causal, info)


def test_causal_rows_without_keys():
    # more queries than keys: the first Sq - Sk rows see no key and are zero
    O, ref = _check((1, 1, 300, D), (1, 1, 200, D), "bf16", True)
    assert np.all(O[0, 0, :100] == 0)


def test_causal_fewer_queries_than_keys():
    _check((1, 2, 128, D), (1, 2, 320, D), "bf16", True)


def test_growing_scores_exercise_the_rescale():
    # keys grow in magnitude along the sequence, so a row's maximum keeps
    # rising block after block and the output accumulator is rescaled
    B, H, Sq, Sk = 1, 2, 256, 1024
    Qb = _tensor((B, H, Sq, D), 80, "bf16")
    k = oracle.decode(_tensor((B, H, Sk, D), 81, "bf16"), "bf16")
    k *= (1.0 + np.arange(Sk) / 128.0)[None, None, :, None]
    Kb = synth.quantise(k, "bf16")
    Vb = _tensor((B, H, Sk, D), 82, "bf16")
    O, st = _run(Qb, Kb, Vb, "bf16", 0.25, False)
    assert st == 0
    ref, bound = oracle.attention(Qb, Kb, Vb, "bf16", 0.25, False)
    ok, info = oracle.accept_attention(O, ref, bound, "bf16")
    assert ok, info


def test_larger_causal_and_repeatable_bits():
    Qb = _tensor((2, 4, 1024, D), 83, "bf16")
    Kb = _tensor((2, 4, 1024, D), 84, "bf16")
    Vb = _tensor((2, 4, 1024, D), 85, "bf16")
    O1, _ = _run(Qb, Kb, Vb, "bf16", D ** -0.5, True)
    O2, _ = _run(Qb, Kb, Vb, "bf16", D ** -0.5, True)
    assert np.array_equal(O1, O2)
    ref, bound = oracle.attention(Qb, Kb, Vb, "bf16", D ** -0.5, True)
    ok, info = oracle.accept_attention(O1, ref, bound, "bf16")
    assert ok, info


def test_causal_chunks_with_a_ragged_last_chunk():
    # the causal launch runs in chunks of (batch, head)s that share about
    # 8 MiB of K and V (eight at Sk = 2048); nine of them leave a last chunk
    # of one, and 1900 query rows a ragged last tile in every head
    _check((3, 3, 1900, D), (3, 3, 2048, D), "bf16", True, seed=30)


def test_uniform_queries_average_the_values():
    # Q = 0: every visible key weighs the same
    Qb = synth.quantise(np.zeros((1, 1, 256, D)), "bf16")
    Kb = _tensor((1, 1, 512, D), 86, "bf16")
    Vb = _tensor((1, 1, 512, D), 87, "bf16")
    O, _ = _run(Qb, Kb, Vb, "bf16", 1.0, False)
    want = oracle.decode(Vb, "bf16").mean(axis=2)
    got = oracle.decode(O, "bf16")
    assert np.all(np.abs(got - want[:, :, None]) <= 2.0 ** -7 * np.abs(want[:, :, None]) + 1e-3)


def test_expired_wait_reports_timeout_and_the_context_survives():
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    Qb = _tensor((1, 2, 256, D), 88, "bf16")
    Kb = _tensor((1, 2, 256, D), 89, "bf16")
    Vb = _tensor((1, 2, 256, D), 90, "bf16")
    Q, K, V = (to_dev(x.reshape(-1, D), "bf16").reshape(x.shape) for x in (Qb, Kb, Vb))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    tsgemm.attention(Q, K, V, status=status, debug_flags=tsgemm.DEBUG_SKIP_FIRST_LOAD, timeout_ms=50)
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    assert int(status.item()) == tsgemm.ERR_TIMEOUT
    _check((1, 2, 256, D), (1, 2, 256, D), "bf16", False, seed=18)


def test_wide_score_range_underflows_weights():
    # a large scale spreads a row's scores over hundreds of base-2 units:
    # most weights underflow to zero, a few dominate
    _check((1, 2, 256, D), (1, 2, 640, D), "bf16", False, scale=6.0, seed=30)
    _check((1, 2, 256, D), (1, 2, 640, D), "f16", True, scale=6.0, seed=31)


def test_tiny_scale_weights_near_one():
    _check((1, 2, 256, D), (1, 2, 512, D), "f16", False, scale=1e-3, seed=32)


@pytest.mark.parametrize("causal", [False, True])
def test_full_size_workload_sampled_rows(causal):
    # the B = 4, H = 32, S = 4096 workload in the launch the benchmark
    # times; sampled 128-row windows (whole query tiles, a window across
    # two tiles, the last rows) of three heads against the oracle
    import torch
    from hierarchical_gemm_gb300 import tsgemm
    name = "attn_b4h32s4096d128_causal_bf16" if causal else "attn_b4h32s4096d128_bf16"
    w = synth.attn_workload(name)
    B, H, S = w["B"], w["H"], w["Sq"]

    def mk(seed):
        return synth.matrix(B * H * S, D, ("normal", 1.0), seed, "bf16").reshape(B, H, S, D)
    Qb, Kb, Vb = mk(w["seed_q"]), mk(w["seed_k"]), mk(w["seed_v"])
    Q, K, V = (to_dev(x.reshape(-1, D), "bf16").reshape(x.shape) for x in (Qb, Kb, Vb))
    O = torch.full(Q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    tsgemm.attention(Q, K, V, scale=D ** -0.5, causal=causal, O=O)
    torch.cuda.synchronize()
    assert tsgemm.attention_status() == 0
    for b, h in ((0, 0), (1, 17), (B - 1, H - 1)):
        Ob = from_dev(O[b, h].contiguous(), "bf16")
        for r0 in (0, 128, 2048 + 64, S - 128):
            r1 = r0 + 128
            kv = r1 if causal else S
            q = np.ascontiguousarray(Qb[b:b + 1, h:h + 1, r0:r1])
            k = np.ascontiguousarray(Kb[b:b + 1, h:h + 1, :kv])
            v = np.ascontiguousarray(Vb[b:b + 1, h:h + 1, :kv])
            ref, bound = oracle.attention(q, k, v, "bf16", D ** -0.5, causal)
            ok, info = oracle.accept_attention(Ob[r0:r1][None, None], ref, bound, "bf16")
            assert ok, (b, h, r0, info)


@pytest.mark.parametrize("causal", [False, True])
def test_single_query_row(causal):
    # decode-like: one query row per (batch, head); the query tile holds
    # one valid row (causal: the row is the last query, so it sees every
    # key)
    _check((2, 4, 1, D), (2, 4, 1000, D), "bf16", causal, seed=40)


def test_many_keys_with_a_ragged_tail():
    _check((1, 2, 256, D), (1, 2, 4097, D), "f16", False, seed=41)
    _check((1, 2, 256, D), (1, 2, 4097, D), "bf16", True, seed=42)
