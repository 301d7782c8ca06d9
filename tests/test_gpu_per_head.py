"""Selection per query head (the other reading of which score the selection ranks) on the
GPU against the fp64 oracle, through the C ABI.

Each head's scores are compared with the oracle's s_hj; each head's selection must equal the
oracle's top-k + recent over the oracle's own scores rounded to fp32, bit for bit (the
generator keeps a gap at every head's top-k boundary, so fp32 rounding cannot move a key
across it); each head's sparse output is compared with the oracle's softmax over that head's
rows."""
import numpy as np
import pytest
import torch

import gen
import oracle
import relu_sparse_kv_gb300 as E
from helpers import assert_close, order_key_np, to_dev

pytestmark = pytest.mark.gpu

D, TOPK, RECENT = 128, 1024, 128


@pytest.mark.parametrize("B,Hq,Hkv,n", [(2, 16, 4, 1000), (2, 16, 4, 3000), (1, 16, 2, 40000),
                                        (3, 32, 4, 5000),
                                        (5, 16, 4, 532 * 128 - 77)])  # several pieces per CTA
def test_per_head_selection_and_sparse(B, Hq, Hkv, n):
    fl = gen.make_full_layer(seed=n + B, layer=0, B=B, Hq=Hq, Hkv=Hkv, D=D, n=n, pattern="subset",
                             frac=0.1, sparse_layers=(1,))
    ncap = fl.K.shape[2]
    shape = E.Shape(B, Hq, Hkv, D, n, ncap)
    q, K, V = to_dev(fl.q), to_dev(fl.K), to_dev(fl.V)
    out = torch.empty(B, Hq, D, device="cuda")
    ns = torch.empty(B, Hkv, dtype=torch.int32, device="cuda")
    hs = torch.full((B, Hq, ncap), float("nan"), device="cuda")
    hh = torch.full((B, Hq, E.HIST_BINS), -1, dtype=torch.int32, device="cuda")
    E.embla_full_decode_head_scores(shape, q, K, V, out, ns, hs, hh)
    idx = torch.full((B, Hq, TOPK + RECENT), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, Hq), -1, dtype=torch.int32, device="cuda")
    E.embla_select_topk_per_head(shape, hs, hh, idx, cnt, TOPK, RECENT)
    so = torch.full((B, Hq, D), float("nan"), device="cuda")
    E.embla_sparse_decode_per_head(shape, to_dev(fl.sparse_q[0]), K, V, idx, cnt, so)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0

    ref_out, _, ref_ns = oracle.full_decode_batch(fl.q, fl.K, fl.V, n)
    assert np.array_equal(ns.cpu().numpy(), ref_ns)
    assert_close(out.cpu().numpy(), ref_out, what="full output")
    hs, hh = hs.cpu().numpy()[:, :, :n], hh.cpu().numpy().view(np.uint32)
    idx, cnt, so = idx.cpu().numpy(), cnt.cpu().numpy(), so.cpu().numpy()
    G = Hq // Hkv
    want = min(n, TOPK + RECENT)
    assert (cnt == want).all()
    for b in range(B):
        for g in range(Hkv):
            s = oracle.full_scores(fl.q[b, g * G:(g + 1) * G], fl.K[b, g, :n])
            for hl in range(G):
                h = g * G + hl
                assert_close(hs[b, h], s[hl], atol=1e-4, rtol=1e-5, what=f"scores of head {h}")
                assert np.array_equal(hh[b, h], np.bincount(order_key_np(hs[b, h]) >> 21,
                                                            minlength=E.HIST_BINS))
                ref_idx = oracle.select_topk(s[hl].astype(np.float32), TOPK, RECENT)
                assert np.array_equal(idx[b, h, :want], ref_idx), f"selection of head {h}"
                ref = oracle.sparse_decode(fl.sparse_q[0][b, h:h + 1], fl.K[b, g, :n],
                                           fl.V[b, g, :n], ref_idx)
                assert_close(so[b, h:h + 1], ref, what=f"sparse output of head {h}")


def test_identical_heads_select_like_the_group():
    """When every head of a group has the same query, its own scores are the group's and
    the per-head selection equals the shared one."""
    B, Hq, Hkv, n = 1, 16, 4, 6000
    fl = gen.make_full_layer(seed=3, layer=0, B=B, Hq=Hq, Hkv=Hkv, D=D, n=n, pattern="subset",
                             frac=0.05)
    G = Hq // Hkv
    qsame = np.repeat(fl.q[:, ::G], G, axis=1)
    shape = E.Shape(B, Hq, Hkv, D, n, n)
    q, K, V = to_dev(qsame), to_dev(fl.K), to_dev(fl.V)
    out = torch.empty(B, Hq, D, device="cuda")
    ns = torch.empty(B, Hkv, dtype=torch.int32, device="cuda")
    hs = torch.empty(B, Hq, n, device="cuda")
    hh = torch.empty(B, Hq, E.HIST_BINS, dtype=torch.int32, device="cuda")
    E.embla_full_decode_head_scores(shape, q, K, V, out, ns, hs, hh)
    sel = torch.empty(B, Hkv, n, device="cuda")
    hist = torch.empty(B, Hkv, E.HIST_BINS, dtype=torch.int32, device="cuda")
    E.embla_full_decode(shape, q, K, V, out, ns, sel, hist)
    idx_h = torch.empty(B, Hq, TOPK + RECENT, dtype=torch.int32, device="cuda")
    cnt_h = torch.empty(B, Hq, dtype=torch.int32, device="cuda")
    E.embla_select_topk_per_head(shape, hs, hh, idx_h, cnt_h)
    idx_g = torch.empty(B, Hkv, TOPK + RECENT, dtype=torch.int32, device="cuda")
    cnt_g = torch.empty(B, Hkv, dtype=torch.int32, device="cuda")
    E.embla_select_topk(shape, sel, hist, idx_g, cnt_g)
    torch.cuda.synchronize()
    idx_h, idx_g = idx_h.cpu().numpy(), idx_g.cpu().numpy()
    for h in range(Hq):
        assert np.array_equal(idx_h[0, h], idx_g[0, h // G])
