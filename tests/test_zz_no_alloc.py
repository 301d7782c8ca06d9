"""embla_full_decode_static_scratch: the full-layer decode on the library's fixed device
scratch, called through the C ABI, against embla_full_decode with a caller workspace.

The file name sorts last, so a run that stops at its first failure has run every other
test before this one.  Nothing here depends on that order: the first call on a device looks
up the scratch's device address, and every call in this file is a plain call outside any
stream capture (no test in the suite captures a graph), so the look-up works whichever test
makes it, alone in a fresh process or after the rest of the suite."""
import gc

import pytest
import torch

import gen
import relu_sparse_kv_gb300 as E
from helpers import assert_close, to_dev

pytestmark = pytest.mark.gpu


def _layer(seed, B, Hq, n, n_cap=None, pattern="bernoulli", frac=0.05):
    return gen.make_full_layer(seed=seed, layer=0, B=B, Hq=Hq, Hkv=4, D=128, n=n, pattern=pattern,
                               frac=frac, n_cap=n_cap)


def _buffers(shape):
    B, Hq, Hkv, D, ncap = (shape.batch, shape.n_q_heads, shape.n_kv_heads, shape.head_dim,
                           shape.cache_stride)
    return (torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda"),
            torch.full((B, Hkv), -1, dtype=torch.int32, device="cuda"),
            torch.full((B, Hkv, ncap), float("nan"), dtype=torch.float32, device="cuda"),
            torch.full((B, Hkv, E.HIST_BINS), -1, dtype=torch.int32, device="cuda"))


def _compare(shape, q, K, V, with_sel, alpha=1.0, c=1.0):
    out0, ns0, sel0, hist0 = _buffers(shape)
    sel_args = (sel0, hist0) if with_sel else (None, None)
    E.embla_full_decode(shape, q, K, V, out0, ns0, *sel_args, alpha=alpha, c=c)
    runs = [_buffers(shape) for _ in range(2)]
    gc.collect()  # tensors left over from earlier tests are freed now, not during the calls
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    # two calls in a row on one stream: the second reuses the scratch the first left behind
    for out, ns, sel, hist in runs:
        E.embla_full_decode_static_scratch(shape, q, K, V, out, ns,
                                           *((sel, hist) if with_sel else (None, None)),
                                           alpha=alpha, c=c)
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() <= before  # nothing was allocated by the calls
    assert E.embla_device_check() == 0
    n = shape.ctx_len
    for out, ns, sel, hist in runs:
        assert_close(out.cpu().numpy(), out0.cpu().numpy(), what="static-scratch output")
        assert torch.equal(ns, ns0)
        if with_sel:
            assert torch.equal(sel[..., :n], sel0[..., :n])
            assert torch.equal(hist, hist0)


@pytest.mark.parametrize("B,Hq,n,with_sel", [
    (4, 16, 5000, True),     # units split over several CTAs: their records are combined
    (2, 32, 1153, True),     # G = 8, ragged last tile
    (8, 16, 300, False),     # without the selection outputs
    (1, 16, 70001, True),    # one unit over every CTA
])
def test_static_scratch_matches_workspace_call(B, Hq, n, with_sel):
    fl = _layer(11 + n, B, Hq, n, n_cap=n + 64)
    shape = E.Shape(B, Hq, 4, 128, fl.n, fl.K.shape[2])
    _compare(shape, to_dev(fl.q), to_dev(fl.K), to_dev(fl.V), with_sel, alpha=0.7, c=0.5)


def test_static_scratch_takes_fewer_pieces_when_the_records_do_not_fit():
    """1300 units of 12 tiles: on 152 SMs the usual split cuts each CTA's 102 tiles into five
    pieces, whose records need more than the fixed scratch; the static call takes three
    pieces instead (its partial sums are grouped differently: the output agrees to within
    rounding, the counts, scores and histogram exactly)."""
    B, Hq, n = 325, 16, 1536
    fl = _layer(29, B, Hq, n, pattern="subset")
    shape = E.Shape(B, Hq, 4, 128, fl.n, fl.K.shape[2])
    if E.embla_device_sm_count() == 152:
        assert E.embla_full_decode_workspace_size(shape) > E.FULL_DECODE_SCRATCH_BYTES
    _compare(shape, to_dev(fl.q), to_dev(fl.K), to_dev(fl.V), True)


def test_static_scratch_size_limit():
    """The largest batch whose workspace fits the fixed scratch runs and matches; one more
    sequence is refused with 'workspace too small' and leaves the outputs untouched."""
    Hq, n = 16, 1
    fits = lambda b: E.embla_full_decode_workspace_size(E.Shape(b, Hq, 4, 128, n, n)) \
        <= E.FULL_DECODE_SCRATCH_BYTES
    lo, hi = 1, 1
    while fits(hi):
        lo, hi = hi, hi * 2
    while hi - lo > 1:
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if fits(mid) else (lo, mid)
    assert fits(lo) and not fits(lo + 1)

    g = torch.Generator().manual_seed(5)
    def inputs(b):
        q = torch.randn(b, Hq, 128, generator=g).to(torch.bfloat16).cuda()
        K = torch.randn(b, 4, n, 128, generator=g).to(torch.bfloat16).cuda()
        V = torch.randn(b, 4, n, 128, generator=g).to(torch.bfloat16).cuda()
        return q, K, V

    shape = E.Shape(lo, Hq, 4, 128, n, n)
    _compare(shape, *inputs(lo), with_sel=True)

    big = E.Shape(lo + 1, Hq, 4, 128, n, n)
    q, K, V = inputs(lo + 1)
    out, ns, sel, hist = _buffers(big)
    with pytest.raises(E.EmblaError) as err:
        E.embla_full_decode_static_scratch(big, q, K, V, out, ns, sel, hist)
    assert err.value.status == 3
    torch.cuda.synchronize()
    assert torch.isnan(out).all() and (ns == -1).all()
