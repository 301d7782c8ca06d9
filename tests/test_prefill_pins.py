"""Pins of the prefill oracle (causal ReLU^2 attention of a full layer over a prompt).

The prefill of T tokens is pinned against things other than its own loop: every row equals
the (separately pinned) single-token decode at that row's context length; a closed form with
one surviving key; causality (future keys and values never reach a row); the last rows of a
longer prefill equal a shorter prefill; scale invariance at c = 0."""
import numpy as np
import pytest

import gen
import oracle

D = 128


def _inputs(seed, G, T, n):
    q = gen.normal_bf16(gen.stream(seed, gen.ROLE_IID, 7, 0, 0), (G, T, D))
    K = gen.normal_bf16(gen.stream(seed, gen.ROLE_IID, 8, 0, 0), (n, D))
    V = gen.normal_bf16(gen.stream(seed, gen.ROLE_IID, 9, 0, 0), (n, D))
    return q, K, V


@pytest.mark.parametrize("G,T,n", [(4, 1, 1), (4, 7, 7), (4, 5, 40), (8, 33, 200)])
@pytest.mark.parametrize("alpha,c", [(1.0, 1.0), (0.3, 0.0)])
def test_every_row_is_the_decode_at_its_context(G, T, n, alpha, c):
    q, K, V = _inputs(1, G, T, n)
    out = oracle.prefill(q, K, V, alpha=alpha, c=c)
    for t in range(T):
        p = n - T + t
        ref, _, _, _ = oracle.full_decode(q[:, t], K[:p + 1], V[:p + 1], alpha=alpha, c=c)
        np.testing.assert_allclose(out[:, t], ref, rtol=1e-12, atol=1e-12)


def test_one_surviving_key_closed_form():
    # every key points against the query except key 3, which is the query itself: that key
    # scores alpha * D (up to eps) and is the only one with weight
    rng = np.random.default_rng(4)
    qv = rng.standard_normal(D)
    n, T = 9, 2
    K = np.tile(-qv, (n, 1))
    K[3] = qv
    V = rng.standard_normal((n, D))
    q = np.tile(qv, (1, T, 1))
    alpha, c, eps = 0.5, 2.0, 1e-6
    out = oracle.prefill(q, K, V, alpha=alpha, c=c, eps=eps)
    ms = np.mean(qv * qv)
    s = alpha * D * ms / (ms + eps)
    w = s * s
    for t in range(T):
        np.testing.assert_allclose(out[0, t], w / (c + w) * V[3], rtol=1e-12)


def test_future_keys_never_reach_a_row():
    G, T, n = 4, 12, 30
    q, K, V = _inputs(2, G, T, n)
    out = oracle.prefill(q, K, V)
    K2 = gen.bf16_to_f32(K).astype(np.float64)
    V2 = gen.bf16_to_f32(V).astype(np.float64)
    rng = np.random.default_rng(5)
    cut = n - T + 5  # rows of tokens 0..5 see keys <= cut
    K2[cut + 1:] = rng.standard_normal(K2[cut + 1:].shape) * 10
    V2[cut + 1:] = np.nan
    out2 = oracle.prefill(q, K2, V2)
    np.testing.assert_array_equal(out[:, :6], out2[:, :6])
    assert np.isnan(out2[:, 6:]).any()


def test_last_rows_match_a_shorter_prefill():
    G, T, n = 4, 20, 64
    q, K, V = _inputs(3, G, T, n)
    full = oracle.prefill(q, K, V)
    tail = oracle.prefill(q[:, T - 6:], K, V)
    np.testing.assert_array_equal(full[:, T - 6:], tail)


def test_scale_invariance_at_c_zero():
    G, T, n = 4, 6, 50
    q, K, V = _inputs(6, G, T, n)
    a = oracle.prefill(q, K, V, alpha=1.0, c=0.0)
    b = oracle.prefill(q, K, V, alpha=1.0 / 128, c=0.0)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_batch_layout_matches_units():
    B, Hq, Hkv, T, n, ncap = 2, 8, 2, 5, 21, 24
    rng = np.random.default_rng(7)
    q = rng.standard_normal((B, Hq, T, D))
    K = rng.standard_normal((B, Hkv, ncap, D))
    V = rng.standard_normal((B, Hkv, ncap, D))
    out = oracle.prefill_batch(q, K, V, n)
    G = Hq // Hkv
    for b in range(B):
        for g in range(Hkv):
            ref = oracle.prefill(q[b, g * G:(g + 1) * G], K[b, g, :n], V[b, g, :n])
            np.testing.assert_array_equal(out[b, g * G:(g + 1) * G], ref)
