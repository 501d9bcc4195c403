"""Pins of the attention oracle (CPU only): closed forms, invariants and a
library routine (torch's scaled-dot-product attention in float64)."""
import numpy as np
import pytest
import torch

import oracle
import synth


def _bits(x, dt="bf16"):
    return synth.quantise(np.asarray(x, dtype=np.float64), dt)


def _rand(shape, seed, dt="bf16", sigma=1.0):
    n = int(np.prod(shape))
    return synth.matrix(1, n, ("normal", sigma), seed, dt).reshape(shape)


def _vals(bits, dt="bf16"):
    return oracle.decode(bits, dt)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_against_torch_sdpa_float64(causal, dt):
    B, H, Sq, Sk, D, Dv = 2, 3, 9, 9 if causal else 13, 16, 8
    Q, K, V = _rand((B, H, Sq, D), 1, dt), _rand((B, H, Sk, D), 2, dt), _rand((B, H, Sk, Dv), 3, dt)
    scale = 0.3
    O, bound = oracle.attention(Q, K, V, dt, scale, causal)
    q, k, v = (torch.from_numpy(_vals(x, dt)) for x in (Q, K, V))
    want = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=scale).numpy()
    assert np.allclose(O, want, rtol=1e-12, atol=1e-13)
    assert np.all(bound >= np.abs(O) - 1e-15)


def test_zero_queries_average_the_values():
    B, H, Sq, Sk, D, Dv = 1, 2, 4, 6, 8, 5
    Q = _bits(np.zeros((B, H, Sq, D)))
    K, V = _rand((B, H, Sk, D), 4), _rand((B, H, Sk, Dv), 5)
    O, _ = oracle.attention(Q, K, V, "bf16", 1.0, False)
    want = _vals(V).mean(axis=2, keepdims=True)
    assert np.allclose(O, np.broadcast_to(want, O.shape), rtol=0, atol=1e-15)
    # with the causal mask, row i averages the first i + 1 values (Sq = Sk)
    Q6 = _bits(np.zeros((B, H, Sk, D)))
    O, _ = oracle.attention(Q6, K, V, "bf16", 1.0, True)
    vals = _vals(V)
    for i in range(Sk):
        assert np.allclose(O[:, :, i], vals[:, :, :i + 1].mean(axis=2), rtol=0, atol=1e-15)


def test_constant_values_pass_through():
    B, H, Sq, Sk, D, Dv = 1, 1, 5, 7, 8, 4
    Q, K = _rand((B, H, Sq, D), 6), _rand((B, H, Sk, D), 7)
    V = _bits(np.broadcast_to(np.array([1.5, -2.0, 0.25, 3.0]), (B, H, Sk, Dv)))
    O, bound = oracle.attention(Q, K, V, "bf16", 0.7, False)
    assert np.allclose(O, [1.5, -2.0, 0.25, 3.0], rtol=0, atol=1e-14)
    assert np.allclose(bound, [1.5, 2.0, 0.25, 3.0], rtol=0, atol=1e-14)


def test_one_hot_selects_a_value_row():
    # key t is 8 * e_t and query i is 8 * e_{p(i)}: scaled scores differ by
    # 64 * scale = 64, so row i's weight sits on key p(i) within e^-64
    D = Sk = 8
    perm = np.random.default_rng(8).permutation(Sk)
    K = _bits(8 * np.eye(D)[None, None])
    Q = _bits(8 * np.eye(D)[perm][None, None])
    V = _rand((1, 1, Sk, 6), 9)
    O, _ = oracle.attention(Q, K, V, "bf16", 1.0, False)
    assert np.allclose(O[0, 0], _vals(V)[0, 0][perm], rtol=1e-20, atol=1e-25)


def test_key_permutation_and_shift_invariance():
    B, H, Sq, Sk, D, Dv = 1, 2, 6, 10, 8, 4
    Q = _bits(np.random.default_rng(10).integers(-2, 3, (B, H, Sq, D)))
    K = _bits(np.random.default_rng(11).integers(-2, 3, (B, H, Sk, D)))
    V = _rand((B, H, Sk, Dv), 12)
    O, _ = oracle.attention(Q, K, V, "bf16", 0.25, False)
    perm = np.random.default_rng(13).permutation(Sk)
    O2, _ = oracle.attention(Q, K[:, :, perm], V[:, :, perm], "bf16", 0.25, False)
    assert np.allclose(O, O2, rtol=1e-14, atol=1e-15)
    # adding the same vector c to every key adds q . c to every score of a row
    c = np.array([1, -1, 2, 0, 0, 1, -2, 1])
    K3 = _bits(_vals(K) + c)
    O3, _ = oracle.attention(Q, K3, V, "bf16", 0.25, False)
    assert np.allclose(O, O3, rtol=1e-13, atol=1e-14)


def test_causal_edges():
    B, H, S, D, Dv = 1, 1, 7, 8, 3
    Q, K, V = _rand((B, H, S, D), 14), _rand((B, H, S, D), 15), _rand((B, H, S, Dv), 16)
    O, _ = oracle.attention(Q, K, V, "bf16", 0.5, True)
    Of, _ = oracle.attention(Q, K, V, "bf16", 0.5, False)
    assert np.array_equal(O[0, 0, 0], _vals(V)[0, 0, 0])  # row 0 sees key 0 only
    assert np.allclose(O[0, 0, -1], Of[0, 0, -1], rtol=1e-15, atol=0)  # the last row sees all keys
    # more queries than keys: the first Sq - Sk rows see nothing and are zero
    Qb = _rand((B, H, 9, D), 17)
    O, bound = oracle.attention(Qb, K, V, "bf16", 0.5, True)
    assert np.all(O[0, 0, :2] == 0) and np.all(bound[0, 0, :2] == 0)
    assert np.array_equal(O[0, 0, 2], _vals(V)[0, 0, 0])


def test_acceptance_rule_catches_a_perturbation():
    B, H, Sq, Sk, D, Dv = 1, 1, 4, 6, 8, 4
    Q, K, V = _rand((B, H, Sq, D), 18), _rand((B, H, Sk, D), 19), _rand((B, H, Sk, Dv), 20)
    O, bound = oracle.attention(Q, K, V, "bf16", 0.5, False)
    ok, _ = oracle.accept_attention(O.astype(np.float32), O, bound, "f32")
    assert ok
    bad = O.copy()
    bad[0, 0, 1, 2] += 0.02 * bound[0, 0, 1, 2] + 1e-3
    ok, info = oracle.accept_attention(bad.astype(np.float32), O, bound, "f32")
    assert not ok and info["first_bad"] == [0, 0, 1, 2]


# ------------------------------------------------------------ MLA decode --

def test_mla_decode_matches_float64_torch():
    # The MLA decode shape against torch's float64 arithmetic written out
    # from the definition: scores over the latent and rotary parts, the
    # softmax over keys, and the latent cache as the values.
    import torch
    B, H, S, dim, pe = 2, 5, 37, 16, 8
    r = np.random.default_rng(12)
    q, qpe, kv, kpe = (synth.quantise(r.standard_normal(shape), "bf16")
                       for shape in ((B, H, dim), (B, H, pe), (B, S, dim), (B, S, pe)))
    scale = 0.37
    O, bound = oracle.mla_decode(q, qpe, kv, kpe, "bf16", scale)

    def t(x):
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    s = scale * (t(q) @ t(kv).transpose(1, 2) + t(qpe) @ t(kpe).transpose(1, 2))  # (B, H, S)
    w = torch.softmax(s, dim=-1)
    ref = w @ t(kv)
    mag = w @ t(kv).abs()
    assert np.allclose(O, ref.numpy(), rtol=1e-12, atol=1e-13)
    assert np.allclose(bound, mag.numpy(), rtol=1e-12, atol=1e-13)
    # the rotary part counts: dropping it changes the result
    O0, _ = oracle.mla_decode(q, np.zeros_like(qpe), kv, kpe, "bf16", scale)
    assert not np.allclose(O0, O, rtol=1e-6, atol=1e-9)
