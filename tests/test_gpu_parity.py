"""GPU parity against the fp64 oracle, through the C ABI.

Bars: surviving-key counts and selected index sets bit-exact; outputs within
|gpu - oracle| <= 2e-3 + 1e-2 |oracle| (bf16 inputs, fp32 accumulation).
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import relu_sparse_kv_gb300 as E
from helpers import FullRun, assert_close, order_key_np, to_dev

pytestmark = pytest.mark.gpu

D = 128


def _layer(B, Hq, Hkv, n, pattern="subset", frac=0.05, n_cap=None, seed=1, sparse=(1,)):
    return gen.make_full_layer(seed=seed, layer=0, B=B, Hq=Hq, Hkv=Hkv, D=D, n=n,
                               pattern=pattern, frac=frac, n_cap=n_cap, sparse_layers=sparse)


def _check_full(fl, run, alpha=1.0, c=1.0, eps=1e-6):
    ref_out, ref_sig, ref_ns = oracle.full_decode_batch(fl.q, fl.K, fl.V, fl.n, alpha=alpha, c=c,
                                                        eps=eps)
    ns = run.n_surv.cpu().numpy()
    assert np.array_equal(ns, ref_ns), (ns, ref_ns)
    assert np.array_equal(ns, fl.n_pos)
    assert_close(run.out.cpu().numpy(), ref_out, what="full output, small")
    sel = run.sel.cpu().numpy()[:, :, :fl.n]
    assert_close(sel, ref_sig[:, :, :fl.n], atol=1e-4 * max(alpha, 1e-3), rtol=1e-5, what="sigma")
    assert np.array_equal(sel > 0, ref_sig[:, :, :fl.n] > 0)
    # histogram: counts of the top 11 bits of the GPU's own scores
    hist = run.hist.cpu().numpy().view(np.uint32)
    for b in range(sel.shape[0]):
        for g in range(sel.shape[1]):
            expect = np.bincount(order_key_np(sel[b, g]) >> 21, minlength=E.HIST_BINS)
            assert np.array_equal(hist[b, g], expect)
    return ref_sig


@pytest.mark.parametrize("n", [1, 7, 127, 128, 129, 1000, 1152, 1153, 2048, 4099])
def test_full_and_select_small_contexts(n):
    fl = _layer(2, 16, 4, n, pattern="bernoulli", frac=0.3)
    run = FullRun(fl)
    ref_sig = _check_full(fl, run)
    ref_idx, ref_cnt = oracle.select_topk_batch(ref_sig, fl.n)
    cnt = run.count.cpu().numpy()
    assert np.array_equal(cnt, ref_cnt)
    idx = run.idx.cpu().numpy()
    for b in range(2):
        for g in range(4):
            assert np.array_equal(idx[b, g, :cnt[b, g]], ref_idx[b, g, :ref_cnt[b, g]])
    ref_sp = oracle.sparse_decode_batch(fl.sparse_q[0], fl.K, fl.V, ref_idx, ref_cnt)
    assert_close(run.sparse(fl.sparse_q[0]), ref_sp, what="sparse output, small contexts")


@pytest.mark.parametrize("G", [4, 8])
@pytest.mark.parametrize("alpha,c", [(1.0, 1.0), (1.0, 0.0), (1.0 / 128, 1.0), (1.0 / 128, 0.0)])
def test_full_scalars_and_group_sizes(G, alpha, c):
    Hkv = 2 if G == 8 else 4
    fl = _layer(3, G * Hkv, Hkv, 3000, pattern="subset", frac=0.2, seed=5)
    run = FullRun(fl, alpha=alpha, c=c)
    _check_full(fl, run, alpha=alpha, c=c)


def test_padding_rows_past_context_are_never_read():
    # rows n..n_cap-1 of K and V hold NaN; none may reach any output
    fl = _layer(2, 16, 4, 2500, pattern="subset", frac=0.1, n_cap=2700, seed=7)
    run = FullRun(fl)
    ref_sig = _check_full(fl, run)
    assert np.isfinite(run.out.cpu().numpy()).all()
    ref_idx, ref_cnt = oracle.select_topk_batch(ref_sig, fl.n)
    assert np.array_equal(run.idx.cpu().numpy(), ref_idx)


@pytest.mark.parametrize("B,n", [(1, 64 * 128), (5, 3 * 128 + 5), (40, 300)])
def test_full_many_units_and_split_boundaries(B, n):
    # shapes whose tiles split across CTAs at unit boundaries in different ways
    fl = _layer(B, 16, 4, n, pattern="runs" if n > 2000 else "subset", frac=0.05, seed=B)
    run = FullRun(fl)
    _check_full(fl, run)


@pytest.mark.parametrize("tiles_per_cta,n_short", [(70, 77), (110, 50)])
def test_full_pieces_over_units_of_mixed_survival(tiles_per_cta, n_short):
    # shares long enough that each CTA takes three or five pieces spread over the batch;
    # sequences whose keys survive at 50 / 20 / 5 / 1 %, ragged last tiles
    B, Hkv = 5, 4
    tu = -(-tiles_per_cta * E.embla_device_sm_count() // (B * Hkv))
    fl = _layer(B, 16, Hkv, tu * 128 - n_short, pattern="subset", frac=[0.5, 0.2, 0.05, 0.01],
                seed=23)
    run = FullRun(fl)
    _check_full(fl, run)


def _fused(run, topk=1024, recent=128):
    """The decode with its selection in one call, on the inputs of a FullRun."""
    r = dict(out=torch.full_like(run.out, float("nan")), n_surv=torch.full_like(run.n_surv, -1),
             sel=torch.full_like(run.sel, float("nan")), hist=torch.full_like(run.hist, -1),
             idx=torch.full_like(run.idx, -7), count=torch.full_like(run.count, -1))
    E.embla_full_decode_select(run.shape, run.q, run.K, run.V, r["out"], r["n_surv"], r["sel"],
                               r["hist"], r["idx"], r["count"], topk=topk, recent=recent)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0
    return r


def _assert_same_as_two_calls(run, r, n):
    assert torch.equal(r["out"], run.out) and torch.equal(r["n_surv"], run.n_surv)
    assert torch.equal(r["sel"][..., :n], run.sel[..., :n]) and torch.equal(r["hist"], run.hist)
    assert torch.equal(r["count"], run.count)
    cnt = run.count.cpu().numpy()
    idx_a, idx_b = r["idx"].cpu().numpy(), run.idx.cpu().numpy()
    for b in range(cnt.shape[0]):
        for g in range(cnt.shape[1]):
            assert np.array_equal(idx_a[b, g, :cnt[b, g]], idx_b[b, g, :cnt[b, g]])


@pytest.mark.parametrize("B,Hkv,n,frac", [
    (2, 4, 3000, 0.2),                         # one selection CTA per unit
    (1, 4, 70001, 0.05),                       # clusters of selection CTAs per unit
    (5, 4, 532 * 128 - 77, [0.5, 0.2, 0.05, 0.01]),  # several pieces per decode CTA
    (1, 1, 600001, 0.05),                      # the long-context selection (workspace)
    (2, 4, 700, 0.3),                          # every key selected
])
def test_full_decode_select_matches_the_two_calls(B, Hkv, n, frac):
    fl = _layer(B, 4 * Hkv, Hkv, n, pattern="subset", frac=frac, seed=31, sparse=())
    run = FullRun(fl)
    _assert_same_as_two_calls(run, _fused(run), fl.n)


def test_full_decode_select_then_sparse_layers_are_repeatable():
    # the output is finished beside the selection: the sparse layer after the call must see
    # the finished selection every time
    fl = _layer(8, 16, 4, 32768, pattern="subset", frac=0.05, seed=37, sparse=(1,))
    run = FullRun(fl)
    ref_sp = run.sparse(fl.sparse_q[0])
    qs = to_dev(fl.sparse_q[0])
    r = _fused(run)
    sp_out = torch.empty_like(run.out)
    for _ in range(20):
        E.embla_full_decode_select(run.shape, run.q, run.K, run.V, r["out"], r["n_surv"], r["sel"],
                                   r["hist"], r["idx"], r["count"])
        E.embla_sparse_decode(run.shape, qs, run.K, run.V, r["idx"], r["count"], sp_out)
        torch.cuda.synchronize()
        assert np.array_equal(sp_out.cpu().numpy(), ref_sp)
    _assert_same_as_two_calls(run, r, fl.n)
    assert E.embla_device_check() == 0


@pytest.mark.parametrize("B,n,frac", [(8, 32768, 0.05), (16, 8192, 0.5),
                                      (32, 16384, [0.5, 0.2, 0.05, 0.01])])
def test_full_decode_is_repeatable(B, n, frac):
    # pipeline races show up as a tile scored from the wrong buffer now and then: every
    # call must give the same bits (the combine sums in a fixed order)
    fl = _layer(B, 16, 4, n, pattern="subset", frac=frac, seed=17, sparse=())
    shape = E.Shape(B, 16, 4, D, fl.n, fl.K.shape[2])
    q, K, V = to_dev(fl.q), to_dev(fl.K), to_dev(fl.V)
    out = torch.empty(B, 16, D, device="cuda")
    ns = torch.empty(B, 4, dtype=torch.int32, device="cuda")
    sel = torch.empty(B, 4, fl.K.shape[2], device="cuda")
    hist = torch.empty(B, 4, E.HIST_BINS, dtype=torch.int32, device="cuda")
    want = torch.from_numpy(fl.n_pos.astype(np.int32)).cuda()
    E.embla_full_decode(shape, q, K, V, out, ns, sel, hist)
    torch.cuda.synchronize()
    out0, sel0, hist0 = out.clone(), sel.clone(), hist.clone()
    for _ in range(40):
        E.embla_full_decode(shape, q, K, V, out, ns, sel, hist)
        torch.cuda.synchronize()
        assert torch.equal(ns, want)
        assert torch.equal(out, out0) and torch.equal(sel[..., :fl.n], sel0[..., :fl.n])
        assert torch.equal(hist, hist0)
    assert E.embla_device_check() == 0


def test_zero_context_gives_zero_output():
    B, Hq, Hkv = 2, 16, 4
    shape = E.Shape(B, Hq, Hkv, D, 0, 16)
    q = torch.randn(B, Hq, D, device="cuda").to(torch.bfloat16)
    K = torch.zeros(B, Hkv, 16, D, device="cuda", dtype=torch.bfloat16)
    out = torch.full((B, Hq, D), 7.0, device="cuda")
    ns = torch.full((B, Hkv), 9, dtype=torch.int32, device="cuda")
    E.embla_full_decode(shape, q, K, K, out, ns)
    torch.cuda.synchronize()
    assert (out == 0).all() and (ns == 0).all()


def test_spill_below_zero_and_dense_selection():
    # per-sequence positive fractions 0.5 / 0.2 / 0.05 / 0.01: more and fewer than 1,024
    # survivors; the selection then takes keys scored just below zero
    fl = _layer(4, 16, 4, 16384, pattern="subset", frac=[0.5, 0.2, 0.05, 0.01], seed=11)
    run = FullRun(fl)
    ref_sig = _check_full(fl, run)
    ref_idx, ref_cnt = oracle.select_topk_batch(ref_sig, fl.n)
    assert np.array_equal(run.count.cpu().numpy(), ref_cnt)
    assert np.array_equal(run.idx.cpu().numpy(), ref_idx)
    assert_close(run.sparse(fl.sparse_q[0]),
                 oracle.sparse_decode_batch(fl.sparse_q[0], fl.K, fl.V, ref_idx, ref_cnt),
                 what="sparse output, spill below zero")


def test_select_handles_a_crowded_boundary_bin():
    # all candidate scores equal except a few: the boundary bin holds thousands of keys,
    # which exercises the radix passes before the shared-memory sort
    B, Hkv, n = 1, 4, 20000
    shape = E.Shape(B, 16, Hkv, D, n, n)
    rng = np.random.default_rng(3)
    sig = np.full((B, Hkv, n), 0.75, dtype=np.float32)
    sig[0, 1, rng.choice(n, 50, replace=False)] = 2.0
    sig[0, 2] = rng.integers(0, 3, n).astype(np.float32) * 0.5
    sel = torch.from_numpy(sig).cuda()
    hist = np.stack([[np.bincount(order_key_np(sig[0, g]) >> 21, minlength=E.HIST_BINS)
                      for g in range(Hkv)]]).astype(np.int32)
    hist_t = torch.from_numpy(hist).cuda()
    idx = torch.full((B, Hkv, 1152), -1, dtype=torch.int32, device="cuda")
    cnt = torch.empty(B, Hkv, dtype=torch.int32, device="cuda")
    E.embla_select_topk(shape, sel, hist_t, idx, cnt)
    torch.cuda.synchronize()
    ref_idx, ref_cnt = oracle.select_topk_batch(sig, n)
    assert np.array_equal(cnt.cpu().numpy(), ref_cnt)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)


def _select_case(sig, n, ncap):
    """Run the selection on given scores (rows of ncap, the first n used) and compare."""
    B, Hkv = sig.shape[:2]
    shape = E.Shape(B, 16, Hkv, D, n, ncap)
    hist = np.stack([[np.bincount(order_key_np(sig[b, g, :n]) >> 21, minlength=E.HIST_BINS)
                      for g in range(Hkv)] for b in range(B)]).astype(np.int32)
    idx = torch.full((B, Hkv, 1152), -1, dtype=torch.int32, device="cuda")
    cnt = torch.empty(B, Hkv, dtype=torch.int32, device="cuda")
    E.embla_select_topk(shape, torch.from_numpy(sig).cuda(), torch.from_numpy(hist).cuda(), idx, cnt)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0
    ref_idx, ref_cnt = oracle.select_topk_batch(sig, n)
    assert np.array_equal(cnt.cpu().numpy(), ref_cnt)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)


@pytest.mark.parametrize("n,ncap", [(524288, 524288), (524289, 524291), (300000, 300000),
                                    (262144, 262144), (50001, 50003), (4097, 4098),
                                    (1153, 1157)])
def test_select_long_and_unaligned_rows(n, ncap):
    # the largest context one cluster holds in shared memory, one past it (the streaming
    # kernel), two passes per CTA, and row strides that start every unit's scores at a
    # different 4-byte phase
    rng = np.random.default_rng(n)
    B, Hkv = 2, 4
    sig = rng.standard_normal((B, Hkv, ncap)).astype(np.float32)
    sig[:, :, n:] = np.nan
    sig[0, 3, :n] = np.round(sig[0, 3, :n] * 4) / 4  # many exact ties
    _select_case(sig, n, ncap)


@pytest.mark.parametrize("topk,recent", [(0, 128), (1024, 0), (1, 1), (300, 2000), (5000, 50)])
@pytest.mark.parametrize("n", [20000, 100000])
def test_select_other_topk_and_recent(topk, recent, n):
    # sizes other than 1024 + 128: no top-k, no recent keys, more recent keys than threads,
    # more candidates than one list holds; one CTA per unit (20000) and clusters (100000)
    rng = np.random.default_rng(topk + 7 * recent + n)
    B, Hkv = 2, 4
    sig = rng.standard_normal((B, Hkv, n)).astype(np.float32)
    sig[1, 2] = np.round(sig[1, 2] * 2) / 2  # many exact ties
    shape = E.Shape(B, 16, Hkv, D, n, n)
    hist = np.stack([[np.bincount(order_key_np(sig[b, g]) >> 21, minlength=E.HIST_BINS)
                      for g in range(Hkv)] for b in range(B)]).astype(np.int32)
    stride = max(topk + recent, 1)
    idx = torch.full((B, Hkv, stride), -1, dtype=torch.int32, device="cuda")
    cnt = torch.empty(B, Hkv, dtype=torch.int32, device="cuda")
    E.embla_select_topk(shape, torch.from_numpy(sig).cuda(), torch.from_numpy(hist).cuda(), idx, cnt,
                        topk, recent)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0
    idx, cnt = idx.cpu().numpy(), cnt.cpu().numpy()
    for b in range(B):
        for g in range(Hkv):
            ref = oracle.select_topk(sig[b, g], topk, recent)
            assert cnt[b, g] == len(ref)
            assert np.array_equal(idx[b, g, :cnt[b, g]], ref)


@pytest.mark.parametrize("chunk", [1, 2, 8, 32, 64, 1024])
@pytest.mark.parametrize("n,ncap", [(5000, 5000), (4099, 4103), (33, 40), (1, 1)])
def test_skip_stats(chunk, n, ncap):
    rng = np.random.default_rng(n + chunk)
    B, Hkv = 3, 4
    sig = rng.standard_normal((B, Hkv, ncap)).astype(np.float32)
    sig[0, 0] = -1.0                                      # nothing needed
    sig[1, 1] = np.where(rng.random(ncap) < 0.01, 1.0, -1.0)
    sig[2, 3, n:] = 5.0                                    # past the context: not counted
    shape = E.Shape(B, 16, Hkv, D, n, ncap)
    keys = torch.full((B, Hkv), -1, dtype=torch.int32, device="cuda")
    chunks = torch.full((B, Hkv), -1, dtype=torch.int32, device="cuda")
    E.embla_skip_stats(shape, torch.from_numpy(sig).cuda(), keys, chunks, chunk=chunk)
    torch.cuda.synchronize()
    rk, rc = oracle.skip_stats_batch(sig, n, chunk)
    assert np.array_equal(keys.cpu().numpy(), rk)
    assert np.array_equal(chunks.cpu().numpy(), rc)


def test_skip_stats_of_a_full_layer_match_its_survivors():
    fl = _layer(2, 16, 4, 20000, pattern="runs", frac=0.05, seed=19, sparse=())
    run = FullRun(fl, with_select=False)
    keys = torch.empty(2, 4, dtype=torch.int32, device="cuda")
    chunks = torch.empty(2, 4, dtype=torch.int32, device="cuda")
    E.embla_skip_stats(run.shape, run.sel, keys, chunks, chunk=8)
    torch.cuda.synchronize()
    assert np.array_equal(keys.cpu().numpy(), fl.n_pos)
    _, rc = oracle.skip_stats_batch(run.sel.cpu().numpy(), fl.n, 8)
    assert np.array_equal(chunks.cpu().numpy(), rc)


@pytest.mark.parametrize("pos", [0, 5, 126, 127, 128, 1000, 65535])
@pytest.mark.parametrize("G", [4, 8])
def test_window_decode(pos, G):
    Hkv = 4 if G == 4 else 2
    wl = gen.make_window_layer(seed=2, layer=3, B=3, Hq=G * Hkv, Hkv=Hkv, D=D, W=128, pos=pos)
    shape = E.Shape(3, G * Hkv, Hkv, D, 0, 0)
    out = torch.full((3, G * Hkv, D), float("nan"), device="cuda")
    E.embla_window_decode(shape, to_dev(wl.q), to_dev(wl.K), to_dev(wl.V), pos, out)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), oracle.window_decode_batch(wl.q, wl.K, wl.V, pos), what="window output, small")


def test_sparse_decode_with_arbitrary_indices_and_counts():
    B, Hq, Hkv, n = 2, 16, 4, 5000
    rng = np.random.default_rng(9)
    q = gen.normal_bf16(11, (B, Hq, D))
    K = gen.normal_bf16(12, (B, Hkv, n, D))
    V = gen.normal_bf16(13, (B, Hkv, n, D))
    stride = 1152
    idx = np.zeros((B, Hkv, stride), dtype=np.int32)
    cnt = np.array([[0, 1, 500, 1152], [37, 129, 1000, 1151]], dtype=np.int64)
    for b in range(B):
        for g in range(Hkv):
            idx[b, g, :cnt[b, g]] = np.sort(rng.choice(n, cnt[b, g], replace=False))
    shape = E.Shape(B, Hq, Hkv, D, n, n)
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    E.embla_sparse_decode(shape, to_dev(q), to_dev(K), to_dev(V), torch.from_numpy(idx).cuda(),
                          torch.from_numpy(cnt.astype(np.int32)).cuda(), out, tau=0.1)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0
    ref = oracle.sparse_decode_batch(q, K, V, idx, cnt, tau=0.1)
    got = out.cpu().numpy()
    assert np.all(got[0, 0:4] == 0.0)  # count 0: zero output
    assert_close(got, ref, what="sparse output, arbitrary indices tau 0.1")


@pytest.mark.parametrize("B,Hq,Hkv", [(8, 16, 4), (9, 16, 4), (16, 16, 2), (19, 16, 2),
                                      (10, 16, 4), (20, 16, 4), (40, 16, 4), (80, 16, 4),
                                      (40, 16, 2), (90, 16, 2)])
def test_sparse_decode_cluster_sizes(B, Hq, Hkv):
    # 32 .. 320 units: the launch spreads a unit over 8, 4, 2 or 1 CTAs to stay one wave
    # (on 152 SMs: 32 .. 38 units take four 18-warp CTAs per unit, 40 .. 76 two)
    n, stride = 1400, 1152
    rng = np.random.default_rng(B * 7 + Hkv)
    q = gen.normal_bf16(21, (B, Hq, D))
    K = gen.normal_bf16(22, (B, Hkv, n, D))
    V = gen.normal_bf16(23, (B, Hkv, n, D))
    cnt = rng.integers(0, stride + 1, size=(B, Hkv)).astype(np.int64)
    idx = np.zeros((B, Hkv, stride), dtype=np.int32)
    for b in range(B):
        for g in range(Hkv):
            idx[b, g, :cnt[b, g]] = np.sort(rng.choice(n, cnt[b, g], replace=False))
    shape = E.Shape(B, Hq, Hkv, D, n, n)
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    E.embla_sparse_decode(shape, to_dev(q), to_dev(K), to_dev(V), torch.from_numpy(idx).cuda(),
                          torch.from_numpy(cnt.astype(np.int32)).cuda(), out)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0
    assert_close(out.cpu().numpy(), oracle.sparse_decode_batch(q, K, V, idx, cnt), what="sparse output, cluster shapes")


def test_out_of_range_index_is_skipped_and_flagged():
    B, Hq, Hkv, n = 1, 16, 4, 300
    q = gen.normal_bf16(21, (B, Hq, D))
    K = gen.normal_bf16(22, (B, Hkv, n, D))
    V = gen.normal_bf16(23, (B, Hkv, n, D))
    idx = np.tile(np.arange(8, dtype=np.int32), (B, Hkv, 1))
    idx[0, 2, 3] = n + 5
    cnt = np.full((B, Hkv), 8, dtype=np.int32)
    shape = E.Shape(B, Hq, Hkv, D, n, n)
    out = torch.empty((B, Hq, D), device="cuda")
    E.embla_device_check(clear=True)
    E.embla_sparse_decode(shape, to_dev(q), to_dev(K), to_dev(V), torch.from_numpy(idx).cuda(),
                          torch.from_numpy(cnt).cuda(), out)
    assert E.embla_device_check(clear=True) & 1
    assert E.embla_device_check(clear=True) == 0
    good = np.array([0, 1, 2, 4, 5, 6, 7], dtype=np.int32)
    ref = oracle.sparse_decode(q[0, 8:12], K[0, 2], V[0, 2], good)
    assert_close(out.cpu().numpy()[0, 8:12], ref, what="sparse output, out-of-range index skipped")


def test_timed_out_wait_is_flagged_and_the_context_stays_usable():
    """The bounded-wait error path: a wait that nothing completes gives up after its limit,
    sets bit 1 of the check word and returns; the next calls run normally.  A wait that is
    completed sets nothing."""
    import time
    E.embla_device_check(clear=True)
    E.embla_self_test_wait_limit(1000, arrive=True)
    assert E.embla_device_check(clear=True) == 0
    t0 = time.perf_counter()
    E.embla_self_test_wait_limit(2000)
    flags = E.embla_device_check(clear=True)
    waited = time.perf_counter() - t0
    assert flags == 2
    assert 0.002 <= waited < 5.0
    assert E.embla_device_check(clear=True) == 0
    # the context is intact: a full layer and its selection still match the oracle
    fl = _layer(1, 16, 4, 3000, pattern="bernoulli", frac=0.3)
    run = FullRun(fl)
    ref_sig = _check_full(fl, run)
    ref_idx, ref_cnt = oracle.select_topk_batch(ref_sig, fl.n)
    assert np.array_equal(run.count.cpu().numpy(), ref_cnt)
    assert E.embla_device_check(clear=True) == 0
