"""Parity at the benchmark's full sizes, in the launch configuration the benchmark times
(alpha 1, c 1, eps 1e-6, top 1024 + recent 128, tau 1/sqrt(D), the same shapes).

Every unit is checked against properties that hold at any size (survivor counts equal the
generator's construction, histogram = counts of the scores' top bits, selection size,
order, recent keys and the top-k boundary); sampled units are recomputed one by one by the
fp64 oracle and compared element by element."""
import numpy as np
import pytest
import torch

import gen
import oracle
import relu_sparse_kv_gb300 as E
from helpers import assert_close, order_key_np, to_dev

pytestmark = pytest.mark.gpu

TOPK, RECENT = 1024, 128


def _run_layer(fl):
    B, Hq, D = fl.q.shape
    Hkv, ncap = fl.K.shape[1], fl.K.shape[2]
    shape = E.Shape(B, Hq, Hkv, D, fl.n, ncap)
    q, K, V = to_dev(fl.q), to_dev(fl.K), to_dev(fl.V)
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    ns = torch.full((B, Hkv), -1, dtype=torch.int32, device="cuda")
    sel = torch.full((B, Hkv, ncap), float("nan"), device="cuda")
    hist = torch.full((B, Hkv, E.HIST_BINS), -1, dtype=torch.int32, device="cuda")
    E.embla_full_decode(shape, q, K, V, out, ns, sel, hist, alpha=1.0, c=1.0, eps=1e-6)
    res = dict(out=out, n_surv=ns, sel=sel, hist=hist, sparse=[])
    if fl.sparse_q:
        idx = torch.full((B, Hkv, TOPK + RECENT), -7, dtype=torch.int32, device="cuda")
        cnt = torch.full((B, Hkv), -1, dtype=torch.int32, device="cuda")
        E.embla_select_topk(shape, sel, hist, idx, cnt, TOPK, RECENT)
        for qs in fl.sparse_q:
            so = torch.full((B, Hq, D), float("nan"), device="cuda")
            E.embla_sparse_decode(shape, to_dev(qs), K, V, idx, cnt, so)
            res["sparse"].append(so)
        res.update(idx=idx, count=cnt)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0
    del q, K, V
    return {k: (v.cpu().numpy() if torch.is_tensor(v) else [x.cpu().numpy() for x in v])
            for k, v in res.items()}


def _check_every_unit(fl, r):
    n = fl.n
    assert np.array_equal(r["n_surv"], fl.n_pos)
    sel = r["sel"][:, :, :n]
    assert np.isfinite(r["out"]).all()
    assert np.array_equal(sel > 0, fl.targets > 0)
    hist = r["hist"].view(np.uint32)
    B, Hkv = r["n_surv"].shape
    for b in range(B):
        for g in range(Hkv):
            assert np.array_equal(hist[b, g], np.bincount(order_key_np(sel[b, g]) >> 21,
                                                          minlength=E.HIST_BINS))
    if not fl.sparse_q:
        return
    want = min(n, TOPK + RECENT)
    assert (r["count"] == want).all()
    for b in range(B):
        for g in range(Hkv):
            ix = r["idx"][b, g, :want]
            assert (np.diff(ix) > 0).all() and ix[0] >= 0 and ix[-1] < n
            if n > TOPK + RECENT:
                assert np.array_equal(ix[-RECENT:], np.arange(n - RECENT, n))
                cand = sel[b, g, :n - RECENT]
                chosen = np.zeros(n - RECENT, dtype=bool)
                chosen[ix[:-RECENT]] = True
                assert cand[chosen].min() > cand[~chosen].max()
    for so in r["sparse"]:
        assert np.isfinite(so).all()


def _check_sampled_units(fl, r, units):
    n = fl.n
    G = fl.q.shape[1] // fl.K.shape[1]
    for b, g in units:
        hs = slice(g * G, (g + 1) * G)
        K, V = fl.K[b, g, :n], fl.V[b, g, :n]
        out, sig, ns, _ = oracle.full_decode(fl.q[b, hs], K, V, alpha=1.0, c=1.0, eps=1e-6)
        assert r["n_surv"][b, g] == ns
        assert_close(r["out"][b, hs], out, what=f"full output unit ({b},{g})")
        assert_close(r["sel"][b, g, :n], sig, atol=1e-4, rtol=1e-5, what=f"sigma ({b},{g})")
        if not fl.sparse_q:
            continue
        idx = oracle.select_topk(sig, TOPK, RECENT)
        cnt = r["count"][b, g]
        assert np.array_equal(r["idx"][b, g, :cnt], idx), f"selection of unit ({b},{g})"
        for qs, so in zip(fl.sparse_q, r["sparse"]):
            ref = oracle.sparse_decode(qs[b, hs], K, V, idx)
            assert_close(so[b, hs], ref, what=f"sparse output unit ({b},{g})")


def _units(B, Hkv, extra=()):
    picks = {(0, 0), (B - 1, Hkv - 1), (B // 2, 1 % Hkv), (B // 3, Hkv // 2)}
    picks.update(extra)
    return sorted(picks)


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_full_size_workload(cfg):
    fl = next(gen.config_full_layers(cfg, seed=0))
    r = _run_layer(fl)
    _check_every_unit(fl, r)
    B, Hkv = fl.q.shape[0], fl.K.shape[1]
    # the mixed-sparsity batch: one sequence of every survivor fraction
    extra = [(b, b % Hkv) for b in range(4)] if cfg == 4 else []
    if cfg == 3:
        extra = [(0, g) for g in range(Hkv)]
    _check_sampled_units(fl, r, _units(B, Hkv, extra))


def test_full_size_whole_attention_step_block():
    """The whole-step workload: one of its full layers with the sparse layers that reuse its
    selection (sampled), and every window layer of the step in full."""
    cfg = 5
    layers = gen.config_full_layers(cfg, seed=0)
    fl = next(layers)
    if not fl.sparse_q:
        fl = next(layers)
    r = _run_layer(fl)
    _check_every_unit(fl, r)
    B, Hkv = fl.q.shape[0], fl.K.shape[1]
    _check_sampled_units(fl, r, _units(B, Hkv))
    del fl, r
    for wl in gen.config_window_layers(cfg, seed=0):
        B, Hq, D = wl.q.shape
        Hkv, W = wl.K.shape[1], wl.K.shape[2]
        out = torch.full((B, Hq, D), float("nan"), device="cuda")
        E.embla_window_decode(E.Shape(B, Hq, Hkv, D, 0, 0), to_dev(wl.q), to_dev(wl.K),
                              to_dev(wl.V), wl.pos, out)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), oracle.window_decode_batch(wl.q, wl.K, wl.V, wl.pos),
                     what="window output")


@pytest.mark.parametrize("cfg", [7, 8])
def test_full_size_prefill(cfg):
    """The prefill workloads at full size (one sequence, a whole prompt of 8192 / 32768
    tokens, 16 query heads): every output finite, and sampled rows of every head against the
    oracle's single-token decode at that row's context (the prefill oracle's pinned
    equivalent)."""
    q, K, V = gen.config_prefill(cfg, seed=0)
    B, Hq, T, D = q.shape
    Hkv, n = K.shape[1], K.shape[2]
    shape = E.Shape(B, Hq, Hkv, D, n, n)
    out = torch.full((B, Hq, T, D), float("nan"), device="cuda")
    E.embla_prefill(shape, to_dev(q), to_dev(K), to_dev(V), out)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0
    out = out.cpu().numpy()
    assert np.isfinite(out).all()
    G = Hq // Hkv
    rows = sorted({0, 1, 127, 128, 129, T // 3, T // 2 + 5, T - 129, T - 2, T - 1})
    for t in rows:
        p = n - T + t
        for g in range(Hkv):
            ref, _, _, _ = oracle.full_decode(q[0, g * G:(g + 1) * G, t], K[0, g, :p + 1],
                                              V[0, g, :p + 1], alpha=1.0, c=1.0, eps=1e-6)
            assert_close(out[0, g * G:(g + 1) * G, t], ref, what=f"prefill row {t} group {g}")


def test_full_size_per_head_selection():
    """The benchmarked workload with a selection per query head: per-head scores and
    histograms of every unit, selections of sampled heads bit-exact on the scores ranked,
    their sparse outputs against the oracle."""
    fl = next(gen.config_full_layers(10, seed=0))
    B, Hq, D = fl.q.shape
    Hkv, n = fl.K.shape[1], fl.n
    G = Hq // Hkv
    shape = E.Shape(B, Hq, Hkv, D, n, n)
    q, K, V = to_dev(fl.q), to_dev(fl.K), to_dev(fl.V)
    out = torch.empty(B, Hq, D, device="cuda")
    ns = torch.empty(B, Hkv, dtype=torch.int32, device="cuda")
    hs = torch.full((B, Hq, n), float("nan"), device="cuda")
    hh = torch.empty(B, Hq, E.HIST_BINS, dtype=torch.int32, device="cuda")
    E.embla_full_decode_head_scores(shape, q, K, V, out, ns, hs, hh)
    idx = torch.full((B, Hq, TOPK + RECENT), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, Hq), -1, dtype=torch.int32, device="cuda")
    E.embla_select_topk_per_head(shape, hs, hh, idx, cnt, TOPK, RECENT)
    sparse = []
    for qs in fl.sparse_q:
        so = torch.full((B, Hq, D), float("nan"), device="cuda")
        E.embla_sparse_decode_per_head(shape, to_dev(qs), K, V, idx, cnt, so)
        sparse.append(so)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0
    assert np.array_equal(ns.cpu().numpy(), fl.n_pos)
    hs, hh = hs.cpu().numpy(), hh.cpu().numpy().view(np.uint32)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    sparse = [so.cpu().numpy() for so in sparse]
    assert (cnt == TOPK + RECENT).all()
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(hh[b, h], np.bincount(order_key_np(hs[b, h]) >> 21,
                                                        minlength=E.HIST_BINS))
    for b, h in [(0, 0), (B - 1, Hq - 1), (3, 5), (5, 10)]:
        g = h // G
        s = oracle.full_scores(fl.q[b, g * G:(g + 1) * G], fl.K[b, g, :n])[h - g * G]
        assert_close(hs[b, h], s, atol=1e-4, rtol=1e-5, what=f"scores of head ({b},{h})")
        ref_idx = oracle.select_topk(hs[b, h], TOPK, RECENT)
        assert np.array_equal(idx[b, h], ref_idx), f"selection of head ({b},{h})"
        for qs, so in zip(fl.sparse_q, sparse):
            ref = oracle.sparse_decode(qs[b, h:h + 1], fl.K[b, g, :n], fl.V[b, g, :n], ref_idx)
            assert_close(so[b, h:h + 1], ref, what=f"sparse output of head ({b},{h})")
