"""Parity at the benchmark's full sizes, in the launch configuration the benchmark times
(alpha 1, c 1, eps 1e-6, top 1024 + recent 128, tau 1/sqrt(D), the same shapes).

Every unit of every full layer is recomputed by the fp64 oracle and compared element by
element: survivor counts and selections bit-exact (the selection ranked on the oracle's own
fp32 scores, never the kernel's), outputs and scores within tolerance.  Properties that
hold at any size (counts equal the generator's construction, the histogram counts the
scores' top bits) are checked on the GPU's results as well."""
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


def _check_layer(fl, r, Kf=None, Vf=None):
    """Every unit of one full layer (and its sparse layers) against the oracle.  Kf, Vf: the
    caches as float64 (the decoded rows for 8-bit caches)."""
    n = fl.n
    Kf = oracle.f64(fl.K) if Kf is None else Kf
    Vf = oracle.f64(fl.V) if Vf is None else Vf
    # invariants of the GPU's own results
    assert np.array_equal(r["n_surv"], fl.n_pos)
    sel = r["sel"][:, :, :n]
    assert np.array_equal(sel > 0, fl.targets > 0)
    hist = r["hist"].view(np.uint32)
    B, Hkv = r["n_surv"].shape
    for b in range(B):
        for g in range(Hkv):
            assert np.array_equal(hist[b, g], np.bincount(order_key_np(sel[b, g]) >> 21,
                                                          minlength=E.HIST_BINS))
    # the oracle, every unit
    out, sig, ns = oracle.full_decode_batch(fl.q, Kf, Vf, n, alpha=1.0, c=1.0, eps=1e-6)
    assert np.array_equal(r["n_surv"], ns)
    assert_close(r["out"], out, what="full output")
    assert_close(sel, sig[:, :, :n], atol=1e-4, rtol=1e-5, what="sigma")
    if not fl.sparse_q:
        return
    idx, cnt = oracle.select_topk_batch(sig, n, TOPK, RECENT)
    assert np.array_equal(r["count"], cnt)
    for b in range(B):
        for g in range(Hkv):
            c = cnt[b, g]
            assert np.array_equal(r["idx"][b, g, :c], idx[b, g, :c]), f"selection ({b},{g})"
    for qs, so in zip(fl.sparse_q, r["sparse"]):
        assert_close(so, oracle.sparse_decode_batch(qs, Kf, Vf, idx, cnt), what="sparse output")


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_full_size_workload(cfg):
    fl = next(gen.config_full_layers(cfg, seed=0))
    _check_layer(fl, _run_layer(fl))


def test_full_size_whole_attention_step():
    """The whole-step workload: all five full layers with the sparse layers that reuse their
    selections, and every window layer of the step, each unit against the oracle."""
    cfg = 5
    for fl in gen.config_full_layers(cfg, seed=0):
        _check_layer(fl, _run_layer(fl))
        del fl
    for wl in gen.config_window_layers(cfg, seed=0):
        B, Hq, D = wl.q.shape
        Hkv, W = wl.K.shape[1], wl.K.shape[2]
        out = torch.full((B, Hq, D), float("nan"), device="cuda")
        E.embla_window_decode(E.Shape(B, Hq, Hkv, D, 0, 0), to_dev(wl.q), to_dev(wl.K),
                              to_dev(wl.V), wl.pos, out)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), oracle.window_decode_batch(wl.q, wl.K, wl.V, wl.pos),
                     what="window output")


def test_full_size_prefill_every_row():
    """The 8192-token prompt (one sequence, 16 query heads) at full size: every output row
    of every head against the prefill oracle."""
    q, K, V = gen.config_prefill(7, seed=0)
    B, Hq, T, D = q.shape
    Hkv, n = K.shape[1], K.shape[2]
    shape = E.Shape(B, Hq, Hkv, D, n, n)
    out = torch.full((B, Hq, T, D), float("nan"), device="cuda")
    E.embla_prefill(shape, to_dev(q), to_dev(K), to_dev(V), out)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0
    assert_close(out.cpu().numpy(), oracle.prefill_batch(q, K, V, n), what="prefill output")


def test_full_size_prefill_32k_rows():
    """The 32768-token prompt: every output finite, and 48 rows spread over the prompt (its
    first and last tiles, tile edges and rows in between) of every head against the oracle's
    single-token decode at that row's context (the prefill oracle's pinned equivalent)."""
    q, K, V = gen.config_prefill(8, seed=0)
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
    rng = np.random.default_rng(8)
    rows = {0, 1, 2, 7, 127, 128, 129, 255, 256, T // 3, T // 2 + 5, T - 129, T - 128, T - 2, T - 1}
    rows.update(int(x) for x in rng.integers(0, T, 48 - len(rows)))
    Kf, Vf = oracle.f64(K[0]), oracle.f64(V[0])
    for t in sorted(rows):
        p = n - T + t
        for g in range(Hkv):
            ref, _, _, _ = oracle.full_decode(q[0, g * G:(g + 1) * G, t], Kf[g, :p + 1],
                                              Vf[g, :p + 1], alpha=1.0, c=1.0, eps=1e-6)
            assert_close(out[0, g * G:(g + 1) * G, t], ref, what=f"prefill output row {t}")


def test_full_size_per_head_selection():
    """The benchmarked workload with a selection per query head: every head's scores,
    histogram, selection (bit-exact against the top-k of the oracle's own scores rounded to
    fp32) and sparse outputs."""
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
    del q, K, V
    out, ns = out.cpu().numpy(), ns.cpu().numpy()
    hs, hh = hs.cpu().numpy(), hh.cpu().numpy().view(np.uint32)
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    sparse = [so.cpu().numpy() for so in sparse]

    Kf, Vf = oracle.f64(fl.K), oracle.f64(fl.V)
    ref_out, _, ref_ns = oracle.full_decode_batch(fl.q, Kf, Vf, n)
    assert np.array_equal(ns, ref_ns) and np.array_equal(ns, fl.n_pos)
    assert_close(out, ref_out, what="full output")
    ref_hs = oracle.head_scores_batch(fl.q, Kf, n)
    assert_close(hs, ref_hs, atol=1e-4, rtol=1e-5, what="per-head scores")
    ref_idx, ref_cnt = oracle.select_topk_batch(ref_hs, n, TOPK, RECENT)
    assert np.array_equal(cnt, ref_cnt) and (cnt == TOPK + RECENT).all()
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(hh[b, h], np.bincount(order_key_np(hs[b, h]) >> 21,
                                                        minlength=E.HIST_BINS))
            assert np.array_equal(idx[b, h], ref_idx[b, h]), f"selection of head ({b},{h})"
    for b in range(B):
        for h in range(Hq):
            g = h // G
            for qs, so in zip(fl.sparse_q, sparse):
                ref = oracle.sparse_decode(qs[b, h:h + 1], Kf[b, g, :n], Vf[b, g, :n],
                                           ref_idx[b, h])
                assert_close(so[b, h:h + 1], ref, what="per-head sparse output")
