"""Pins that tie the fp64 oracle to what "The Architecture of Embla 1" and the
mathematics fix, without re-running the oracle's own formulas.

Each test names the passage it follows.  The kinds of evidence used:
closed forms on constructed inputs, invariants, special cases that reduce to a
library routine (torch's scaled_dot_product_attention in fp64), statistics the
page reports, and brute force on tiny inputs.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import gen
import oracle

D = 128


def _basis(i, D=D):
    e = np.zeros(D)
    e[i] = 1.0
    return e


def sdpa64(q, K, V, tau):
    """Softmax attention of G queries over n keys via torch's library routine (fp64)."""
    qt = torch.from_numpy(np.asarray(q, dtype=np.float64))[None, :, None, :]    # [1, G, 1, D]
    G = qt.shape[1]
    Kt = torch.from_numpy(np.asarray(K, dtype=np.float64))[None, None].expand(1, G, -1, -1)
    Vt = torch.from_numpy(np.asarray(V, dtype=np.float64))[None, None].expand(1, G, -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=tau)
    return o[0, :, 0, :].numpy()


# ----------------------------------------------------------------------------- full layer
# "Sevren Sparse Attention learns to be sparse": scores of RMS-normalised q and k,
# weight ReLU(s)^2, weighted sum of values over (constant + sum of weights).

@pytest.mark.parametrize("alpha", [1.0, 1.0 / 128, 3.7])
def test_score_is_D_times_cosine_when_eps_is_zero(alpha):
    # RMS normalisation makes qhat . khat = D * cos(q, k) exactly when eps = 0.
    rng = np.random.default_rng(1)
    q = rng.standard_normal((4, D)) * rng.uniform(0.1, 10, (4, 1))
    K = rng.standard_normal((64, D)) * rng.uniform(0.1, 10, (64, 1))
    s = oracle.full_scores(q, K, alpha=alpha, eps=0.0)
    cos = (q @ K.T) / np.linalg.norm(q, axis=1)[:, None] / np.linalg.norm(K, axis=1)[None, :]
    np.testing.assert_allclose(s, alpha * D * cos, rtol=1e-12, atol=1e-12)


def test_eps_enters_the_mean_square():
    # q = beta e_0, k = gamma e_0 (D = 4): qhat.khat = beta*gamma / (sqrt(beta^2/D+eps) sqrt(gamma^2/D+eps)).
    Dd, beta, gamma, eps, alpha = 4, 0.2, 0.5, 0.01, 1.5
    q = (beta * _basis(0, Dd))[None]
    K = (gamma * _basis(0, Dd))[None]
    s = oracle.full_scores(q, K, alpha=alpha, eps=eps)[0, 0]
    expect = alpha * beta * gamma / (math.sqrt(beta ** 2 / Dd + eps) * math.sqrt(gamma ** 2 / Dd + eps))
    assert s == pytest.approx(expect, rel=1e-14)


def _single_survivor_unit(beta=0.3, gamma=2.0, rho=1.5, n=50, seed=3):
    """Group of 4 heads q_h = beta e_h; key 0 = gamma e_0 (positive for head 0 only,
    exactly zero score for heads 1-3); every other key scores below zero for all heads."""
    rng = np.random.default_rng(seed)
    q = np.stack([beta * _basis(h) for h in range(4)])
    K = np.zeros((n, D))
    K[0] = gamma * _basis(0)
    for j in range(1, n):
        K[j, :4] = -rho * rng.uniform(0.5, 1.5, 4)
        K[j, 4:] = rng.standard_normal(D - 4)
    V = rng.standard_normal((n, D))
    return q, K, V


@pytest.mark.parametrize("c", [1.0, 0.25])
@pytest.mark.parametrize("eps", [1e-6, 0.05])
def test_single_survivor_closed_form(c, eps):
    beta, gamma, alpha = 0.3, 2.0, 0.7
    q, K, V = _single_survivor_unit(beta, gamma)
    out, sigma, n_surv, n_zero = oracle.full_decode(q, K, V, alpha=alpha, c=c, eps=eps)
    s = alpha * beta * gamma / (math.sqrt(beta ** 2 / D + eps) * math.sqrt(gamma ** 2 / D + eps))
    w = s * s
    np.testing.assert_allclose(out[0], w / (c + w) * V[0], rtol=1e-12, atol=1e-15)
    assert np.all(out[1:] == 0.0)             # heads 1-3 weigh every key zero (score 0 or below)
    assert n_surv == 1
    assert sigma[0] == np.float32(s)
    assert np.all(sigma[1:] < 0)
    assert list(n_zero) == [49, 50, 50, 50]


def test_single_survivor_c0_returns_its_value():
    q, K, V = _single_survivor_unit()
    out, _, _, _ = oracle.full_decode(q, K, V, alpha=1.0, c=0.0, eps=1e-6)
    np.testing.assert_allclose(out[0], V[0], rtol=1e-14, atol=1e-15)
    assert np.all(out[1:] == 0.0)             # nothing survives: the stated 0/0 reading


def test_identical_keys_closed_form():
    # n copies of one key positive for every head: out_h = n w_h / (c + n w_h) * mean(v).
    rng = np.random.default_rng(5)
    q = np.abs(rng.standard_normal((4, D)))
    k = np.abs(rng.standard_normal(D))
    n, c, alpha, eps = 37, 2.0, 0.05, 1e-6
    K = np.tile(k, (n, 1))
    V = rng.standard_normal((n, D))
    out, _, n_surv, _ = oracle.full_decode(q, K, V, alpha=alpha, c=c, eps=eps)
    rq = 1 / np.sqrt((q ** 2).mean(1) + eps)
    rk = 1 / np.sqrt((k ** 2).mean() + eps)
    s = alpha * (q @ k) * rq * rk
    w = s ** 2
    expect = (n * w / (c + n * w))[:, None] * V.mean(0)[None, :]
    np.testing.assert_allclose(out, expect, rtol=1e-12, atol=1e-15)
    assert n_surv == n


def test_weights_exactly_zero_iff_score_nonpositive_and_never_negative():
    # With V = identity rows (n <= D), out_h[j] = w_hj / (c + sum w): the weights themselves.
    rng = np.random.default_rng(7)
    n = 96
    q = rng.standard_normal((4, D))
    q[0] = 0.0
    q[0, :2] = 1.0                       # head 0 reads dims 0 and 1 only
    K = rng.standard_normal((n, D))
    K[:8, 1] = -K[:8, 0]                 # keys 0-7 score exactly 0 for head 0
    V = np.eye(n, D)
    c = 1.0
    out, _, _, n_zero = oracle.full_decode(q, K, V, alpha=1.0, c=c, eps=0.0)
    s = D * (q @ K.T) / np.linalg.norm(q, axis=1)[:, None] / np.linalg.norm(K, axis=1)[None]
    assert np.all(s[0, :8] == 0.0)
    W = out[:, :n]
    assert np.all(W >= 0.0)
    for h in range(4):
        S = W[h].sum()
        w = W[h] * c / (1 - S)             # recover the weights from out_h
        zero = w == 0.0
        assert np.array_equal(zero, s[h] <= 0)
        np.testing.assert_allclose(w[~zero], s[h][~zero] ** 2, rtol=1e-9)
        assert n_zero[h] == zero.sum()


def test_v_rows_of_zero_weight_keys_are_never_used():
    # "Skipping V": a key whose weight is zero for every head of the group needs no value.
    rng = np.random.default_rng(11)
    q = rng.standard_normal((4, D))
    K = rng.standard_normal((300, D))
    V = rng.standard_normal((300, D))
    out, sigma, n_surv, _ = oracle.full_decode(q, K, V)
    dead = sigma <= 0
    assert 0 < dead.sum() < 300 and n_surv == (~dead).sum()
    V2 = V.copy()
    V2[dead] = rng.standard_normal((dead.sum(), D)) * 1e6
    out2, _, _, _ = oracle.full_decode(q, K, V2)
    assert np.array_equal(out, out2)
    V3 = V.copy()
    V3[np.flatnonzero(~dead)[0]] += 1.0
    out3, _, _, _ = oracle.full_decode(q, K, V3)
    assert not np.array_equal(out, out3)


def test_about_half_the_weights_are_zero_at_random_directions():
    # With q and k in random directions a score is positive or negative with equal odds,
    # so half the weights vanish (the page measured 50.8% at initialisation).  iid N(0,1)
    # bf16 q and k: the zero
    # fraction over all (head, key) pairs lies inside a 5-sigma binomial band around 1/2.
    zeros = total = 0
    for unit in range(4):
        q, K, V = gen.iid_unit(seed=123, G=4, D=D, n=4096, unit=unit)
        _, _, _, n_zero = oracle.full_decode(q, K, V)
        zeros += int(n_zero.sum())
        total += 4 * 4096
    # scores of the 4 heads on one key are independent given random q directions; the band
    # is widened by sqrt(4) to allow for the shared key.
    sd = math.sqrt(total * 0.25) * 2
    assert abs(zeros - total / 2) < 5 * sd


def test_scale_and_permutation_invariances():
    rng = np.random.default_rng(13)
    q = rng.standard_normal((4, D))
    K = rng.standard_normal((200, D))
    V = rng.standard_normal((200, D))
    base, _, _, _ = oracle.full_decode(q, K, V, alpha=1.0, c=0.0, eps=0.0)
    # c = 0: the output does not depend on the score scale alpha
    o2, _, _, _ = oracle.full_decode(q, K, V, alpha=5.3, c=0.0, eps=0.0)
    np.testing.assert_allclose(o2, base, rtol=1e-12, atol=1e-14)
    # eps = 0: scaling any key by a positive factor changes nothing (RMS normalisation)
    lam = rng.uniform(0.01, 100, (200, 1))
    o3, _, _, _ = oracle.full_decode(q, K * lam, V, alpha=1.0, c=0.0, eps=0.0)
    np.testing.assert_allclose(o3, base, rtol=1e-11, atol=1e-14)
    # keys form a set: permuting (k_j, v_j) pairs leaves the output unchanged
    perm = rng.permutation(200)
    o4, sig4, _, _ = oracle.full_decode(q, K[perm], V[perm], alpha=1.0, c=0.0, eps=0.0)
    np.testing.assert_allclose(o4, base, rtol=1e-12, atol=1e-14)
    # the output is linear in V
    V2 = rng.standard_normal((200, D))
    oa, _, _, _ = oracle.full_decode(q, K, V2, alpha=1.0, c=1.0)
    ob, _, _, _ = oracle.full_decode(q, K, V, alpha=1.0, c=1.0)
    oc, _, _, _ = oracle.full_decode(q, K, V + 2.0 * V2, alpha=1.0, c=1.0)
    np.testing.assert_allclose(oc, ob + 2.0 * oa, rtol=1e-10, atol=1e-13)


def test_query_heads_map_to_kv_head_h_div_G():
    # 16 query heads, 4 KV heads: head h reads KV head h // 4.  Unit (b, g) holds one key
    # equal to e_{h*} with h* = 4g + (g+b) % 4; query head h is e_h, so only head h* of
    # that unit sees a positive score (and every other head scores it 0 -> zero weight).
    B, Hq, Hkv, n = 2, 16, 4, 5
    q = np.zeros((B, Hq, D))
    for b in range(B):
        for h in range(Hq):
            q[b, h] = _basis(h) * (1.0 + 0.1 * h)
    K = np.zeros((B, Hkv, n, D))
    V = np.zeros((B, Hkv, n, D))
    hot = {}
    rng = np.random.default_rng(17)
    for b in range(B):
        for g in range(Hkv):
            hstar = 4 * g + (g + b) % 4
            hot[(b, g)] = hstar
            K[b, g, 0] = _basis(hstar)
            for j in range(1, n):
                K[b, g, j, :16] = -rng.uniform(0.5, 1.0, 16)
                K[b, g, j, 16:] = rng.standard_normal(D - 16)
            V[b, g] = rng.standard_normal((n, D))
    out, sigma, n_surv = oracle.full_decode_batch(q, K, V, n, alpha=1.0, c=0.0, eps=0.0)
    assert np.all(n_surv == 1)
    for b in range(B):
        for h in range(Hq):
            g = h // 4
            if hot[(b, g)] == h:
                np.testing.assert_allclose(out[b, h], V[b, g, 0], rtol=1e-14)
            else:
                assert np.all(out[b, h] == 0.0)


@pytest.mark.parametrize("pattern,frac", [("bernoulli", 0.5), ("subset", 0.05), ("runs", 0.05),
                                          ("subset", 0.01)])
def test_survivor_count_matches_the_generators_construction(pattern, frac):
    # The generator builds each key so that all heads of its group score it with the
    # target sign; the oracle's survivor count must equal the number of +1 targets.
    fl = gen.make_full_layer(seed=21, layer=0, B=1, Hq=16, Hkv=4, D=D, n=4096, pattern=pattern,
                             frac=frac)
    _, sigma, n_surv = oracle.full_decode_batch(fl.q, fl.K, fl.V, fl.n)
    assert np.array_equal(n_surv, fl.n_pos)
    assert np.array_equal(sigma > 0, fl.targets > 0)


@pytest.mark.parametrize("G,pattern,frac", [(4, "subset", 0.05), (4, "subset", 0.01),
                                            (8, "subset", 0.2), (4, "runs", 0.05)])
def test_generator_keeps_a_gap_at_every_top_k_boundary(G, pattern, frac):
    # Both readings of the selection (the group's score and each head's own) need a clear
    # boundary between the 1024th and 1025th candidate, or fp32 rounding could pick either.
    # Checked here with plain numpy cosines of the stored bf16 keys, not the oracle.
    n, gap = 4096, 2e-3
    fl = gen.make_full_layer(seed=31 + G, layer=0, B=2, Hq=16, Hkv=16 // G, D=D, n=n,
                             pattern=pattern, frac=frac, gap=gap)
    for b in range(2):
        for g in range(16 // G):
            q = gen.bf16_to_f32(fl.q[b, g * G:(g + 1) * G]).astype(np.float64)
            K = gen.bf16_to_f32(fl.K[b, g, :n - 128]).astype(np.float64)
            cos = (q @ K.T) / np.outer(np.linalg.norm(q, axis=1), np.linalg.norm(K, axis=1))
            for row in list(D * cos) + [D * cos.max(axis=0)]:
                top = np.sort(row)[::-1]
                assert top[1023] - top[1024] >= gap


def test_head_scores_batch_is_each_heads_score_and_their_max_is_sigma():
    # Per-head scores (the per-query-head reading of the selection): with eps 0 each is
    # alpha * D * cos(q_h, k_j) (numpy cosines), rounded to fp32; the maximum over a
    # group's heads is the group's selection score, bit for bit (rounding is monotone).
    fl = gen.make_full_layer(seed=5, layer=0, B=2, Hq=16, Hkv=4, D=D, n=700, pattern="bernoulli",
                             frac=0.3, n_cap=703)
    hs = oracle.head_scores_batch(fl.q, fl.K, fl.n, alpha=0.5, eps=0.0)
    assert np.isnan(hs[..., fl.n:]).all()
    _, sigma, _ = oracle.full_decode_batch(fl.q, fl.K, fl.V, fl.n, alpha=0.5, eps=0.0)
    for b in range(2):
        for h in range(16):
            q = gen.bf16_to_f32(fl.q[b, h]).astype(np.float64)
            K = gen.bf16_to_f32(fl.K[b, h // 4, :fl.n]).astype(np.float64)
            cos = K @ q / (np.linalg.norm(K, axis=1) * np.linalg.norm(q))
            np.testing.assert_allclose(hs[b, h, :fl.n], 0.5 * D * cos, rtol=1e-6, atol=1e-6)
        grp = hs[b, :, :fl.n].reshape(4, 4, fl.n).max(axis=1)
        assert np.array_equal(grp, sigma[b, :, :fl.n])


# ----------------------------------------------------------------------------- selection
# "Three kinds of attention", Sparse: top 1,024 keys by the full layer's score (whether or
# not they survived ReLU^2), together with the newest 128 keys.

def test_selection_is_every_key_up_to_topk_plus_recent():
    rng = np.random.default_rng(1)
    for n in (1, 7, 128, 129, 1000, 1151, 1152):
        idx = oracle.select_topk(rng.standard_normal(n).astype(np.float32))
        assert np.array_equal(idx, np.arange(n))


def test_selection_closed_forms():
    n = 5000
    dec = -np.arange(n, dtype=np.float32)                  # earliest keys score highest
    idx = oracle.select_topk(dec)
    assert np.array_equal(idx, np.r_[np.arange(1024), np.arange(n - 128, n)])
    inc = np.arange(n, dtype=np.float32)                   # latest candidates score highest
    idx = oracle.select_topk(inc)
    assert np.array_equal(idx, np.arange(n - 128 - 1024, n))
    flat = np.full(n, 0.5, dtype=np.float32)               # all tied: smaller index wins
    idx = oracle.select_topk(flat)
    assert np.array_equal(idx, np.r_[np.arange(1024), np.arange(n - 128, n)])
    # recent keys are always in, even when they score lowest of all
    low_recent = np.ones(n, dtype=np.float32)
    low_recent[-128:] = -1e30
    assert np.array_equal(oracle.select_topk(low_recent)[-128:], np.arange(n - 128, n))


def _dominates(sig, a, b):
    return sig[a] > sig[b] or (sig[a] == sig[b] and a < b)


def test_selection_dominance_property_random_with_ties():
    rng = np.random.default_rng(2)
    n = 6000
    sig = np.round(rng.standard_normal(n), 2).astype(np.float32)   # many exact ties
    idx = oracle.select_topk(sig)
    assert len(idx) == 1152 and np.all(np.diff(idx) > 0)
    sel = np.zeros(n, bool)
    sel[idx] = True
    assert sel[-128:].all()
    cand = np.arange(n - 128)
    chosen, rest = cand[sel[:n - 128]], cand[~sel[:n - 128]]
    assert len(chosen) == 1024
    # weakest chosen (lowest score, largest index among equals) beats the best of the rest
    worst = min(chosen, key=lambda j: (sig[j], -j))
    best = max(rest, key=lambda j: (sig[j], -j))
    assert _dominates(sig, worst, best)


def test_selection_spills_below_zero_when_few_survive():
    # fewer than 1,024 positive scores: all of them are kept, the rest are the keys
    # scored just below zero.
    rng = np.random.default_rng(3)
    n = 8000
    sig = -np.abs(rng.standard_normal(n)).astype(np.float32)
    pos = rng.choice(n - 128, 300, replace=False)
    sig[pos] = np.abs(sig[pos]) + 0.1
    idx = oracle.select_topk(sig)
    sel = set(idx.tolist())
    assert set(pos.tolist()) <= sel
    neg_chosen = [j for j in idx if j < n - 128 and sig[j] <= 0]
    assert len(neg_chosen) == 724
    neg_rest = [j for j in range(n - 128) if j not in sel]
    assert min(sig[neg_chosen]) >= max(sig[neg_rest])


def test_selection_brute_force_tiny():
    # Brute force: among all topk-subsets of the candidates, exactly one has every member
    # dominating every non-member; the oracle must return it.
    rng = np.random.default_rng(4)
    for trial in range(20):
        n, topk, recent = 14, 5, 3
        sig = rng.integers(-3, 4, n).astype(np.float32)     # small ints: many ties
        cand = range(n - recent)
        good = [S for S in itertools.combinations(cand, topk)
                if all(_dominates(sig, a, b) for a in S for b in cand if b not in S)]
        assert len(good) == 1
        expect = sorted(good[0] + tuple(range(n - recent, n)))
        assert oracle.select_topk(sig, topk=topk, recent=recent).tolist() == expect


# ----------------------------------------------------------------------------- sparse layer
# "Three kinds of attention", Sparse: its own softmax over the selection, no position.

def test_sparse_equals_full_softmax_when_context_fits_the_selection():
    rng = np.random.default_rng(5)
    for n in (1, 100, 1152):
        q = rng.standard_normal((4, D))
        K = rng.standard_normal((n, D))
        V = rng.standard_normal((n, D))
        idx = oracle.select_topk(rng.standard_normal(n).astype(np.float32))
        tau = 1 / math.sqrt(D)
        np.testing.assert_allclose(oracle.sparse_decode(q, K, V, idx, tau), sdpa64(q, K, V, tau),
                                   rtol=1e-10, atol=1e-12)


def test_sparse_gathers_the_selected_rows():
    rng = np.random.default_rng(6)
    n = 3000
    q = rng.standard_normal((4, D))
    K = rng.standard_normal((n, D))
    V = rng.standard_normal((n, D))
    idx = np.sort(rng.choice(n, 1152, replace=False)).astype(np.int32)
    tau = 0.3
    np.testing.assert_allclose(oracle.sparse_decode(q, K, V, idx, tau),
                               sdpa64(q, K[idx], V[idx], tau), rtol=1e-10, atol=1e-12)


def test_sparse_weights_are_never_zero():
    # The sparse layer's softmax leaves no selected key at exactly zero weight: even a key
    # far below the dominant one still moves the output when its value moves.
    rng = np.random.default_rng(7)
    n = 40
    q = np.zeros((1, D))
    q[0, 0] = 1.0
    K = rng.standard_normal((n, D)) * 0.1
    K[3, 0] = 30.0                                  # dominant key (score gap ~ 30)
    V = rng.standard_normal((n, D))
    idx = np.arange(n, dtype=np.int32)
    base = oracle.sparse_decode(q, K, V, idx, tau=1.0)
    np.testing.assert_allclose(base[0], V[3], atol=1e-11)
    for i in range(n):
        if i == 3:
            continue
        V2 = V.copy()
        V2[i] += 1e6
        assert not np.array_equal(oracle.sparse_decode(q, K, V2, idx, tau=1.0), base)
    # equal scores (q = 0): the mean of the selected values
    np.testing.assert_allclose(oracle.sparse_decode(np.zeros((2, D)), K, V, idx[5:20]),
                               np.tile(V[5:20].mean(0), (2, 1)), rtol=1e-12, atol=1e-15)


# ----------------------------------------------------------------------------- window layer
# "Three kinds of attention", Sliding window: softmax over a window of the newest 128 keys,
# positions encoded by rotary embedding (adjacent pairs).

def _rotate_complex(x, pos, base):
    """RoPE written as complex multiplication: (x_2i + i x_2i+1) * exp(i pos base^(-2i/D))."""
    Dd = x.shape[-1]
    z = x[..., 0::2] + 1j * x[..., 1::2]
    ang = np.asarray(pos, dtype=np.float64)[..., None] * base ** (-np.arange(0, Dd, 2) / Dd)
    r = z * np.exp(1j * ang)
    out = np.empty_like(x)
    out[..., 0::2] = r.real
    out[..., 1::2] = r.imag
    return out


def test_window_at_position_zero_returns_the_only_value():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((4, D))
    Kw = np.full((128, D), np.nan)
    Vw = np.full((128, D), np.nan)
    Kw[0] = rng.standard_normal(D)
    Vw[0] = rng.standard_normal(D)
    out = oracle.window_decode(q, Kw, Vw, pos=0)
    assert np.array_equal(out, np.tile(Vw[0], (4, 1)))


@pytest.mark.parametrize("pos", [127, 128, 1000, 65535])
def test_window_matches_softmax_of_complex_rotated_query(pos):
    rng = np.random.default_rng(9)
    q = rng.standard_normal((4, D))
    Kw = rng.standard_normal((128, D))
    Vw = rng.standard_normal((128, D))
    tau = 1 / math.sqrt(D)
    expect = sdpa64(_rotate_complex(q, pos, 10000.0), Kw, Vw, tau)
    np.testing.assert_allclose(oracle.window_decode(q, Kw, Vw, pos, 10000.0, tau), expect,
                               rtol=1e-9, atol=1e-11)


def test_window_depends_only_on_relative_positions():
    # Keys rotated at their own positions, query at pos: shifting every position by the
    # same amount leaves the scores, and so the output, unchanged.
    rng = np.random.default_rng(10)
    W, base = 128, 10000.0
    q = rng.standard_normal((4, D))
    raw_k = rng.standard_normal((W, D))
    Vr = rng.standard_normal((W, D))
    outs = []
    for pos in (500, 777, 4096 + 3):
        positions = np.arange(pos - W + 1, pos + 1)
        Kw = np.empty((W, D))
        Vw = np.empty((W, D))
        Kw[positions % W] = _rotate_complex(raw_k, positions, base)
        Vw[positions % W] = Vr
        outs.append(oracle.window_decode(q, Kw, Vw, pos, base))
    np.testing.assert_allclose(outs[1], outs[0], rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(outs[2], outs[0], rtol=1e-9, atol=1e-11)


def test_window_reads_only_filled_slots_early_on():
    rng = np.random.default_rng(11)
    q = rng.standard_normal((4, D))
    Kw = np.full((128, D), np.nan)
    Vw = np.full((128, D), np.nan)
    pos = 40
    Kw[:pos + 1] = rng.standard_normal((pos + 1, D))
    Vw[:pos + 1] = rng.standard_normal((pos + 1, D))
    out = oracle.window_decode(q, Kw, Vw, pos)
    expect = sdpa64(_rotate_complex(q, pos, 10000.0), Kw[:pos + 1], Vw[:pos + 1], 1 / math.sqrt(D))
    np.testing.assert_allclose(out, expect, rtol=1e-9, atol=1e-11)


def test_window_rotation_frequencies_closed_form():
    # D = 4: pair 0 turns by pos, pair 1 by pos * base^(-1/2).  Two keys, one per pair axis.
    Dd, pos, base = 4, 3, 10000.0
    q = np.array([[1.0, 0.0, 0.0, 0.0], [0.0, 0.0, 1.0, 0.0]])
    Kw = np.array([[0.0, 1.0, 0.0, 0.0], [0.0, 0.0, 0.0, 1.0], [1.0, 0.0, 0.0, 0.0],
                   [0.0, 0.0, 1.0, 0.0]])
    Vw = np.eye(4)
    out = oracle.window_decode(q, Kw, Vw, pos, base, tau=1.0)
    # head 0: q_rot = (cos 3, sin 3, 0, 0): scores (sin 3, 0, cos 3, 0)
    z0 = np.array([math.sin(3), 0.0, math.cos(3), 0.0])
    t = pos * base ** -0.5
    z1 = np.array([0.0, math.sin(t), 0.0, math.cos(t)])    # head 1: q_rot = (0, 0, cos t, sin t)
    for h, z in enumerate((z0, z1)):
        p = np.exp(z - z.max())
        np.testing.assert_allclose(out[h], p / p.sum(), rtol=1e-13)


# ----------------------------------------------------------------------------- V-read accounting
# "Skipping V": a value row is needed exactly when sigma_j > 0; the page's kernel decides it
# for groups of 8 keys.  The accounting counts needed keys and needed chunks.

def test_skip_stats_degenerate_chunk_sizes():
    rng = np.random.default_rng(40)
    sig = rng.standard_normal((2, 3, 1000)).astype(np.float32)
    keys1, chunks1 = oracle.skip_stats_batch(sig, 1000, 1)
    assert np.array_equal(keys1, chunks1)                       # a chunk of one key is the key
    assert np.array_equal(keys1, (sig > 0).sum(-1))
    keysn, chunksn = oracle.skip_stats_batch(sig, 1000, 4096)  # one chunk holds everything
    assert np.array_equal(chunksn, (keysn > 0).astype(np.int64))
    zero = np.full((1, 1, 64), -1.0, dtype=np.float32)
    assert oracle.skip_stats_batch(zero, 64, 8) == (np.zeros((1, 1)), np.zeros((1, 1)))


@pytest.mark.parametrize("p,chunk", [(8, 8), (16, 8), (40, 8), (2, 8), (4, 16), (1, 8)])
def test_skip_stats_periodic_survivors(p, chunk):
    # survivors at every p-th key: when p >= chunk each one has a chunk of its own; when p
    # divides the chunk every chunk holds chunk / p of them
    n = 4096
    sig = np.where(np.arange(n) % p == 0, 1.0, -1.0).astype(np.float32)[None, None]
    keys, chunks = oracle.skip_stats_batch(sig, n, chunk)
    multiples = (n + p - 1) // p
    assert keys[0, 0] == multiples
    if p >= chunk:
        assert chunks[0, 0] == multiples
    else:
        assert chunk % p == 0 and chunks[0, 0] == n // chunk


@pytest.mark.parametrize("f", [0.01, 0.05, 0.2])
def test_skip_stats_independent_survivors_binomial(f):
    # keys survive independently with probability f: a chunk of 8 is needed with
    # probability 1 - (1 - f)^8, independently of the others
    n, units = 1 << 16, 8
    rng = np.random.default_rng(int(f * 1000))
    sig = np.where(rng.random((1, units, n)) < f, 1.0, -1.0).astype(np.float32)
    _, chunks = oracle.skip_stats_batch(sig, n, 8)
    m = units * n // 8
    pr = 1.0 - (1.0 - f) ** 8
    mean, sd = m * pr, math.sqrt(m * pr * (1 - pr))
    assert abs(chunks.sum() - mean) < 5 * sd


def test_skip_stats_keys_needed_equals_survivor_count():
    fl = gen.make_full_layer(seed=41, layer=0, B=2, Hq=16, Hkv=4, D=128, n=3000,
                             pattern="subset", frac=0.1)
    _, sig, n_surv = oracle.full_decode_batch(fl.q, fl.K, fl.V, fl.n)
    keys, chunks = oracle.skip_stats_batch(sig, fl.n, 8)
    assert np.array_equal(keys, n_surv)
    assert (chunks * 8 >= keys).all() and (chunks <= keys).all()


# ----------------------------------------------------------------------------- 8-bit caches
# E4M3 as the OCP 8-bit float format defines it: largest finite 448 (S.1111.110), smallest
# normal 2^-6, smallest subnormal 2^-9, no infinities, S.1111.111 NaN.

def test_e4m3_table_fixed_points():
    t = oracle.e4m3_table()
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert t[0x08] == 2.0 ** -6 and t[0x01] == 2.0 ** -9 and t[0x07] == 7 * 2.0 ** -9
    assert t[0x38] == 1.0 and t[0xB8] == -1.0 and t[0x00] == 0.0 and t[0x80] == 0.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    pos = t[:0x7F]
    assert (np.diff(pos) > 0).all()                      # codes 0..126 increase strictly
    assert np.array_equal(t[0x80:0xFF], -pos)            # negatives mirror the positives


def test_e4m3_encoder_rounds_to_nearest_even():
    # the generator's encoder against this decoder: the nearest code, ties to the even one
    t = oracle.e4m3_table()
    grid = t[:0x7F]
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(4000) * 10, (grid[1:] + grid[:-1]) / 2,
                        rng.uniform(0, 2.0 ** -6, 500)])
    codes = gen.e4m3_encode(x)
    dec = t[codes]
    a = np.minimum(np.abs(x), 448.0)
    # distance to the chosen code is the smallest distance to any code
    best = np.abs(grid[None, :] - a[:, None]).min(axis=1)
    assert np.allclose(np.abs(np.abs(dec) - a), best, atol=0, rtol=0)
    ties = np.isclose(np.abs(grid[None, :] - a[:, None]), best[:, None], rtol=0, atol=0).sum(1) == 2
    assert (codes[ties] % 2 == 0).all()                  # ties go to the even mantissa
    assert (gen.e4m3_encode(np.array([1e9, -1e9])) == [0x7E, 0xFE]).all()


def test_e4m3_full_layer_matches_bf16_path_on_the_decoded_cache():
    # the full layer reads the decoded cache: same survivors as the construction targets,
    # and the oracle on decoded values is the oracle of the bf16 path on those values
    fl = gen.make_full_layer(seed=42, layer=0, B=1, Hq=16, Hkv=2, D=128, n=2000,
                             pattern="subset", frac=0.1, kv="e4m3")
    Kd = oracle.dequant_e4m3(fl.K, fl.Ks)
    Vd = oracle.dequant_e4m3(fl.V, fl.Vs)
    out, sig, ns = oracle.full_decode_batch(fl.q, Kd, Vd, fl.n)
    assert np.array_equal(ns, fl.n_pos)
    assert np.isfinite(out).all()
    # scaling a key row (its scale) does not change the normalised score
    Ks2 = fl.Ks.copy(); Ks2[0, 0, :fl.n] *= 3.0
    _, sig2, _ = oracle.full_decode_batch(fl.q, oracle.dequant_e4m3(fl.K, Ks2), Vd, fl.n,
                                          eps=0.0)
    _, sig0, _ = oracle.full_decode_batch(fl.q, Kd, Vd, fl.n, eps=0.0)
    assert np.allclose(sig2[0, 0, :fl.n], sig0[0, 0, :fl.n], rtol=1e-6, atol=1e-6)
