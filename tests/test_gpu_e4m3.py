"""8-bit (E4M3) caches on the GPU against the fp64 oracle on the decoded rows, through the
C ABI.

The oracle decodes every code exactly (scale * value, in fp64) and runs the same
full-layer, selection and sparse-layer definitions as for bf16 caches.  Bars: surviving-key
counts and selected index sets bit-exact (the generator keeps every decoded key's scores a
margin away from zero and the top-k boundary a gap away from its neighbour); outputs within
|gpu - oracle| <= 2e-3 + 1e-2 |oracle|; sigma within 1e-4 + 1e-5 |sigma|.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import relu_sparse_kv_gb300 as E
from helpers import assert_close, order_key_np, to_dev

pytestmark = pytest.mark.gpu

D = 128


def _layer(B, Hq, Hkv, n, pattern="subset", frac=0.05, n_cap=None, seed=1, sparse=(1,)):
    return gen.make_full_layer(seed=seed, layer=0, B=B, Hq=Hq, Hkv=Hkv, D=D, n=n,
                               pattern=pattern, frac=frac, n_cap=n_cap, sparse_layers=sparse,
                               kv="e4m3")


def _dev8(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class Run8:
    """Full layer over the 8-bit caches of one generated layer."""

    def __init__(self, fl, alpha=1.0, c=1.0, eps=1e-6, with_sel=True):
        B, Hq, _ = fl.q.shape
        Hkv, ncap = fl.K.shape[1], fl.K.shape[2]
        self.shape = E.Shape(B, Hq, Hkv, D, fl.n, ncap)
        self.q = to_dev(fl.q)
        self.K8, self.Ks = _dev8(fl.K), _dev8(fl.Ks)
        self.V8, self.Vs = _dev8(fl.V), _dev8(fl.Vs)
        self.out = torch.full((B, Hq, D), float("nan"), device="cuda")
        self.n_surv = torch.full((B, Hkv), -1, dtype=torch.int32, device="cuda")
        self.sel = self.hist = None
        if with_sel:
            self.sel = torch.full((B, Hkv, ncap), float("nan"), device="cuda")
            self.hist = torch.full((B, Hkv, E.HIST_BINS), -1, dtype=torch.int32, device="cuda")
        E.embla_full_decode_e4m3(self.shape, self.q, self.K8, self.Ks, self.V8, self.Vs, self.out,
                                 self.n_surv, self.sel, self.hist, alpha=alpha, c=c, eps=eps)
        torch.cuda.synchronize()
        assert E.embla_device_check() == 0

    def select(self, topk=1024, recent=128):
        B, Hkv = self.n_surv.shape
        self.idx = torch.full((B, Hkv, topk + recent), -7, dtype=torch.int32, device="cuda")
        self.count = torch.full((B, Hkv), -1, dtype=torch.int32, device="cuda")
        E.embla_select_topk(self.shape, self.sel, self.hist, self.idx, self.count, topk, recent)
        torch.cuda.synchronize()
        return self.idx.cpu().numpy(), self.count.cpu().numpy()

    def sparse(self, q_sparse, tau=None):
        out = torch.full(tuple(q_sparse.shape), float("nan"), device="cuda")
        E.embla_sparse_decode_e4m3(self.shape, to_dev(q_sparse), self.K8, self.Ks, self.V8, self.Vs,
                                   self.idx, self.count, out, tau=tau)
        torch.cuda.synchronize()
        assert E.embla_device_check() == 0
        return out.cpu().numpy()


def _decoded(fl):
    return (oracle.dequant_e4m3(fl.K[:, :, :fl.n], fl.Ks[:, :, :fl.n]),
            oracle.dequant_e4m3(fl.V[:, :, :fl.n], fl.Vs[:, :, :fl.n]))


def _check(fl, run, alpha=1.0, c=1.0, eps=1e-6):
    Kd, Vd = _decoded(fl)
    ref_out, ref_sig, ref_ns = oracle.full_decode_batch(fl.q, Kd, Vd, fl.n, alpha=alpha, c=c,
                                                        eps=eps)
    ns = run.n_surv.cpu().numpy()
    assert np.array_equal(ns, ref_ns), (ns, ref_ns)
    assert np.array_equal(ns, fl.n_pos)
    assert_close(run.out.cpu().numpy(), ref_out, what="8-bit full output, small")
    if run.sel is None:
        return ref_sig
    sel = run.sel.cpu().numpy()[:, :, :fl.n]
    assert_close(sel, ref_sig[:, :, :fl.n], atol=1e-4 * max(alpha, 1e-3), rtol=1e-5, what="sigma")
    assert np.array_equal(sel > 0, ref_sig[:, :, :fl.n] > 0)
    hist = run.hist.cpu().numpy().view(np.uint32)
    for b in range(sel.shape[0]):
        for g in range(sel.shape[1]):
            expect = np.bincount(order_key_np(sel[b, g]) >> 21, minlength=E.HIST_BINS)
            assert np.array_equal(hist[b, g], expect)
    return ref_sig


@pytest.mark.parametrize("n", [1, 7, 127, 128, 129, 1000, 1153, 4099])
@pytest.mark.parametrize("G", [4, 8])
def test_e4m3_full_select_sparse_small_contexts(n, G):
    Hkv = 4 if G == 4 else 2
    n_cap = (n + 3) // 4 * 4
    fl = _layer(2, G * Hkv, Hkv, n, pattern="bernoulli", frac=0.3, n_cap=n_cap, seed=3 + G)
    run = Run8(fl)
    ref_sig = _check(fl, run)
    ref_idx, ref_cnt = oracle.select_topk_batch(ref_sig, fl.n)
    idx, cnt = run.select()
    assert np.array_equal(cnt, ref_cnt)
    for b in range(2):
        for g in range(Hkv):
            assert np.array_equal(idx[b, g, :cnt[b, g]], ref_idx[b, g, :ref_cnt[b, g]])
    Kd, Vd = _decoded(fl)
    ref_sp = oracle.sparse_decode_batch(fl.sparse_q[0], Kd, Vd, ref_idx, ref_cnt)
    assert_close(run.sparse(fl.sparse_q[0]), ref_sp, what="sparse output")


@pytest.mark.parametrize("alpha,c", [(1.0, 0.0), (1.0 / 128, 1.0)])
def test_e4m3_full_scalars(alpha, c):
    fl = _layer(3, 16, 2, 3000, pattern="subset", frac=0.2, seed=5)
    _check(fl, Run8(fl, alpha=alpha, c=c), alpha=alpha, c=c)


def test_e4m3_padding_rows_are_never_read():
    # rows n..n_cap-1 hold NaN codes and NaN scales; none may reach any output
    fl = _layer(2, 16, 4, 2500, frac=0.1, n_cap=2700, seed=7)
    run = Run8(fl)
    _check(fl, run)
    assert np.isfinite(run.out.cpu().numpy()).all()


@pytest.mark.parametrize("B,n", [(1, 70001), (5, 3 * 128 + 5), (40, 300)])
def test_e4m3_full_many_units_and_split_boundaries(B, n):
    n_cap = (n + 3) // 4 * 4
    fl = _layer(B, 16, 2, n, pattern="runs" if n > 2000 else "subset", frac=0.05, seed=B,
                n_cap=n_cap)
    _check(fl, Run8(fl))


@pytest.mark.parametrize("B,n", [(2, 3000), (8, 32768)])
def test_e4m3_full_decode_select_matches_the_two_calls(B, n):
    fl = _layer(B, 16, 2, n, frac=0.05, seed=41, sparse=())
    run = Run8(fl)
    idx, cnt = run.select()
    Hq, Hkv, ncap = 16, 2, fl.K.shape[2]
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    ns = torch.full((B, Hkv), -1, dtype=torch.int32, device="cuda")
    sel = torch.full((B, Hkv, ncap), float("nan"), device="cuda")
    hist = torch.full((B, Hkv, E.HIST_BINS), -1, dtype=torch.int32, device="cuda")
    idx2 = torch.full((B, Hkv, 1152), -7, dtype=torch.int32, device="cuda")
    cnt2 = torch.full((B, Hkv), -1, dtype=torch.int32, device="cuda")
    E.embla_full_decode_e4m3_select(run.shape, run.q, run.K8, run.Ks, run.V8, run.Vs, out, ns, sel,
                                    hist, idx2, cnt2)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0
    assert torch.equal(out, run.out) and torch.equal(ns, run.n_surv)
    assert torch.equal(sel[..., :fl.n], run.sel[..., :fl.n]) and torch.equal(hist, run.hist)
    assert np.array_equal(cnt2.cpu().numpy(), cnt)
    i2 = idx2.cpu().numpy()
    for b in range(B):
        for g in range(Hkv):
            assert np.array_equal(i2[b, g, :cnt[b, g]], idx[b, g, :cnt[b, g]])


def test_e4m3_without_selection_outputs():
    fl = _layer(4, 32, 4, 2000, frac=0.1, seed=9)
    run = Run8(fl, with_sel=False)
    _check(fl, run)


def test_e4m3_is_repeatable():
    fl = _layer(8, 16, 2, 20000, frac=0.05, seed=17, sparse=())
    run = Run8(fl)
    out0, sel0, hist0 = run.out.clone(), run.sel.clone(), run.hist.clone()
    for _ in range(20):
        E.embla_full_decode_e4m3(run.shape, run.q, run.K8, run.Ks, run.V8, run.Vs, run.out,
                                 run.n_surv, run.sel, run.hist)
        torch.cuda.synchronize()
        assert torch.equal(run.out, out0) and torch.equal(run.sel[..., :fl.n], sel0[..., :fl.n])
        assert torch.equal(run.hist, hist0)
    assert E.embla_device_check() == 0


def test_e4m3_long_tile_streams_are_repeatable():
    """About 108 tiles per CTA (32 sequences of 32768 keys over 2 KV heads): every
    accumulator buffer, norm slot and survivor slot goes round many times, so a wait that
    could pass on a stale phase would show up as a device flag or a changed output."""
    fl = _layer(32, 16, 2, 32768, frac=0.05, seed=23, sparse=())
    run = Run8(fl)
    ns = run.n_surv.cpu().numpy()
    assert np.array_equal(ns, fl.n_pos)
    out0, sel0, hist0 = run.out.clone(), run.sel.clone(), run.hist.clone()
    for _ in range(30):
        E.embla_full_decode_e4m3(run.shape, run.q, run.K8, run.Ks, run.V8, run.Vs, run.out,
                                 run.n_surv, run.sel, run.hist)
        torch.cuda.synchronize()
        assert E.embla_device_check() == 0
        assert torch.equal(run.out, out0) and torch.equal(run.sel, sel0)
        assert torch.equal(run.hist, hist0)
    # sampled units against the oracle
    for b, g in ((0, 0), (31, 1), (17, 0)):
        Kd = oracle.dequant_e4m3(fl.K[b:b + 1, g:g + 1], fl.Ks[b:b + 1, g:g + 1])
        Vd = oracle.dequant_e4m3(fl.V[b:b + 1, g:g + 1], fl.Vs[b:b + 1, g:g + 1])
        ref_out, ref_sig, _ = oracle.full_decode_batch(fl.q[b:b + 1, 8 * g:8 * g + 8], Kd, Vd,
                                                       fl.n)
        assert_close(run.out[b, 8 * g:8 * g + 8].cpu().numpy(), ref_out[0], what="8-bit full output, long tile streams")
        assert_close(run.sel[b, g, :fl.n].cpu().numpy(), ref_sig[0, 0, :fl.n], atol=1e-4, rtol=1e-5,
                     what="sigma")


def test_e4m3_rejects_bad_arguments():
    fl = _layer(1, 16, 2, 256, seed=2)
    run = Run8(fl)
    bad = E.Shape(1, 16, 2, D, 256, 258)   # cache_stride not a multiple of 4
    K8 = torch.zeros(1, 2, 258, D, dtype=torch.uint8, device="cuda")
    Ks = torch.ones(1, 2, 258, device="cuda")
    with pytest.raises(E.EmblaError) as err:
        E.embla_full_decode_e4m3(bad, run.q, K8, Ks, K8, Ks, run.out, run.n_surv)
    assert err.value.status == 1


def test_e4m3_full_size_workload():
    """The GQA-8 8-bit workload at full size (8 sequences, 32768 keys, 16 query and 2 KV
    heads): every unit's survivor count, signs and histogram, and every unit's outputs,
    scores, selection (ranked on the oracle's own scores) and sparse outputs against the
    oracle on the decoded rows."""
    fl = next(gen.config_full_layers(6, seed=0))
    run = Run8(fl)
    B, Hkv, n = fl.q.shape[0], fl.K.shape[1], fl.n
    assert np.array_equal(run.n_surv.cpu().numpy(), fl.n_pos)
    sel = run.sel.cpu().numpy()[:, :, :n]
    assert np.array_equal(sel > 0, fl.targets > 0)
    hist = run.hist.cpu().numpy().view(np.uint32)
    for b in range(B):
        for g in range(Hkv):
            assert np.array_equal(hist[b, g], np.bincount(order_key_np(sel[b, g]) >> 21,
                                                          minlength=E.HIST_BINS))
    topk, recent = 1024, 128
    idx, cnt = run.select(topk, recent)
    sparse = [run.sparse(qs) for qs in fl.sparse_q]
    Kd = oracle.dequant_e4m3(fl.K[:, :, :n], fl.Ks[:, :, :n])
    Vd = oracle.dequant_e4m3(fl.V[:, :, :n], fl.Vs[:, :, :n])
    o, sig, ns = oracle.full_decode_batch(fl.q, Kd, Vd, n, alpha=1.0, c=1.0, eps=1e-6)
    assert np.array_equal(run.n_surv.cpu().numpy(), ns)
    assert_close(run.out.cpu().numpy(), o, what="8-bit full output")
    assert_close(sel, sig, atol=1e-4, rtol=1e-5, what="8-bit sigma")
    ref_idx, ref_cnt = oracle.select_topk_batch(sig, n, topk, recent)
    assert np.array_equal(cnt, ref_cnt) and (cnt == topk + recent).all()
    assert np.array_equal(idx, ref_idx)
    for qs, so in zip(fl.sparse_q, sparse):
        assert_close(so, oracle.sparse_decode_batch(qs, Kd, Vd, ref_idx, ref_cnt),
                     what="8-bit sparse output")


@pytest.mark.parametrize("cnt_fill", ["short", "zero", "bad_index"])
def test_e4m3_sparse_counts_and_bad_indices(cnt_fill):
    """Counts below the index stride read only the listed rows; a unit with count 0 gives
    zeros; an index outside [0, n) is skipped and flagged (device check)."""
    fl = _layer(2, 16, 2, 3000, frac=0.1, seed=21)
    run = Run8(fl)
    idx, cnt = run.select()
    Kd, Vd = _decoded(fl)
    if cnt_fill == "short":
        cnt = np.array([[500, 17], [1, 1152]], dtype=np.int32)
    elif cnt_fill == "zero":
        cnt = np.array([[0, 1152], [1152, 0]], dtype=np.int32)
    else:
        idx = idx.copy()
        idx[0, 1, 5] = 3000       # == n: outside
    run.count = torch.from_numpy(cnt).cuda()
    run.idx = torch.from_numpy(np.ascontiguousarray(idx)).cuda()
    out = torch.full((2, 16, D), float("nan"), device="cuda")
    E.embla_sparse_decode_e4m3(run.shape, to_dev(fl.sparse_q[0]), run.K8, run.Ks, run.V8, run.Vs,
                               run.idx, run.count, out)
    torch.cuda.synchronize()
    flags = E.embla_device_check(clear=True)
    out = out.cpu().numpy()
    if cnt_fill == "bad_index":
        assert flags != 0
        keep = np.ones(idx.shape[2], dtype=bool)
        keep[5] = False
        ref = oracle.sparse_decode(fl.sparse_q[0][0, 8:16], Kd[0, 1], Vd[0, 1], idx[0, 1][keep])
        assert_close(out[0, 8:16], ref, what="sparse output without the bad row")
        return
    assert flags == 0
    for b in range(2):
        for g in range(2):
            hs = slice(8 * g, 8 * g + 8)
            c = int(cnt[b, g])
            if c == 0:
                assert (out[b, hs] == 0).all()
            else:
                ref = oracle.sparse_decode(fl.sparse_q[0][b, hs], Kd[b, g], Vd[b, g], idx[b, g, :c])
                assert_close(out[b, hs], ref, what=f"sparse ({b},{g}) count {c}")
