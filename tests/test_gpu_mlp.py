"""ReLU^2 MLP at batch 1 on the GPU against the fp64 oracle, through the C ABI.

Bars: the live-neuron count bit-exact; y within 2e-3 + 1e-2 |y| element-wise (bf16 weights
and token, fp32 sums); the down-projection rows of dead neurons never read (NaN there
leaves y finite and bit-identical)."""
import numpy as np
import pytest
import torch

import gen
import oracle
import relu_sparse_kv_gb300 as E
from helpers import assert_close, to_dev

pytestmark = pytest.mark.gpu


def _run(x, wu, wd):
    d, f = x.shape[0], wu.shape[0]
    y = torch.full((d,), float("nan"), device="cuda")
    nl = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    E.embla_relu2_mlp(to_dev(x), to_dev(wu), to_dev(wd), y, nl)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0
    return y.cpu().numpy(), int(nl.item())


@pytest.mark.parametrize("d,f,live", [(512, 1, 1.0), (512, 100, 0.3), (1024, 1500, 0.05),
                                      (2048, 8192, 0.22), (2048, 3000, 0.0), (2048, 700, 1.0),
                                      (1024, 60001, 0.1)])
def test_mlp_matches_oracle(d, f, live):
    x, wu, wd, mask = gen.make_mlp(d + f, d, f, live)
    y, nl = _run(x, wu, wd)
    ref, _, ref_nl = oracle.relu2_mlp(gen.bf16_to_f32(x), gen.bf16_to_f32(wu), gen.bf16_to_f32(wd))
    assert nl == ref_nl == int(mask.sum())
    assert_close(y, ref, what="mlp output")


def test_dead_rows_are_never_read():
    d, f = 2048, 4000
    x, wu, wd, mask = gen.make_mlp(77, d, f, 0.22)
    y, _ = _run(x, wu, wd)
    wd2 = wd.copy()
    wd2[~mask] = gen.BF16_NAN
    y2, _ = _run(x, wu, wd2)
    assert np.isfinite(y2).all()
    assert np.array_equal(y, y2)


def test_mlp_is_repeatable_and_rejects():
    x, wu, wd, _ = gen.make_mlp(5, 1024, 5000, 0.2)
    y0, _ = _run(x, wu, wd)
    for _ in range(5):
        y, _ = _run(x, wu, wd)
        assert np.array_equal(y, y0)
    xb = torch.zeros(768, dtype=torch.bfloat16, device="cuda")
    wb = torch.zeros(10, 768, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(E.EmblaError) as err:
        E.embla_relu2_mlp(xb, wb, wb, torch.empty(768, device="cuda"),
                          torch.empty(1, dtype=torch.int32, device="cuda"))
    assert err.value.status == 2   # width 768 is not built
