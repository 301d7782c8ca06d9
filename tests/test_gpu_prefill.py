"""Full-layer prefill (causal ReLU^2 attention over a prompt) on the GPU against the fp64
oracle, through the C ABI.

Bar: |gpu - oracle| <= 2e-3 + 1e-2 |oracle| element-wise (bf16 inputs, fp32 accumulation;
the weights enter the value product as bf16 hi + lo, about 16 bits)."""
import numpy as np
import pytest
import torch

import gen
import oracle
import relu_sparse_kv_gb300 as E
from helpers import assert_close, to_dev

pytestmark = pytest.mark.gpu

D = 128


def _case(seed, B, Hq, Hkv, n, T, ncap=None, nan_pad=True):
    ncap = n if ncap is None else ncap
    q = gen.normal_bf16(gen.stream(seed, gen.ROLE_IID, 11, 0, 0), (B, Hq, T, D))
    K = np.full((B, Hkv, ncap, D), gen.BF16_NAN if nan_pad else 0, dtype=np.uint16)
    V = np.full((B, Hkv, ncap, D), gen.BF16_NAN if nan_pad else 0, dtype=np.uint16)
    K[:, :, :n] = gen.normal_bf16(gen.stream(seed, gen.ROLE_IID, 12, 0, 0), (B, Hkv, n, D))
    V[:, :, :n] = gen.normal_bf16(gen.stream(seed, gen.ROLE_IID, 13, 0, 0), (B, Hkv, n, D))
    return q, K, V


def _run(q, K, V, n, alpha=1.0, c=1.0, eps=1e-6):
    B, Hq, T, _ = q.shape
    Hkv, ncap = K.shape[1], K.shape[2]
    shape = E.Shape(B, Hq, Hkv, D, n, ncap)
    out = torch.full((B, Hq, T, D), float("nan"), device="cuda")
    E.embla_prefill(shape, to_dev(q), to_dev(K), to_dev(V), out, alpha=alpha, c=c, eps=eps)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0
    return out.cpu().numpy()


@pytest.mark.parametrize("B,Hq,Hkv,n,T", [
    (1, 16, 4, 1, 1),        # one token, one key
    (1, 16, 4, 7, 7),        # a short prompt, no prefix
    (1, 16, 4, 300, 300),    # three query tiles, ragged, masked diagonal tiles
    (2, 16, 4, 1000, 200),   # a prefix of 800 keys (not a multiple of 128)
    (1, 16, 2, 513, 129),    # G = 8, one query row past a tile
    (2, 16, 4, 1280, 1280),  # ten full tiles
])
def test_prefill_matches_oracle(B, Hq, Hkv, n, T):
    q, K, V = _case(B * 7 + n, B, Hq, Hkv, n, T, ncap=n + 40)
    out = _run(q, K, V, n)
    assert np.isfinite(out).all()
    ref = oracle.prefill_batch(q, K, V, n)
    assert_close(out, ref, what="prefill output")


def test_prefill_output_only_16_byte_aligned():
    """An output base that is 16- but not 32-byte aligned takes the 16-byte stores; the
    results are the same and nothing is written outside the output."""
    B, Hq, Hkv, n, T = 1, 16, 4, 700, 300
    q, K, V = _case(5, B, Hq, Hkv, n, T)
    shape = E.Shape(B, Hq, Hkv, D, n, n)
    size = B * Hq * T * D
    buf = torch.full((size + 16,), 7.0, device="cuda")
    out = buf[4:4 + size].view(B, Hq, T, D)  # base 16 bytes past a 32-byte boundary
    assert out.data_ptr() % 32 == 16
    E.embla_prefill(shape, to_dev(q), to_dev(K), to_dev(V), out)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0
    assert (buf[:4] == 7.0).all() and (buf[4 + size:] == 7.0).all()
    assert_close(out.cpu().numpy(), oracle.prefill_batch(q, K, V, n), what="prefill output")


@pytest.mark.parametrize("alpha,c", [(1.0 / 128, 0.0), (0.5, 2.0), (3.0, 0.0)])
def test_prefill_scalars(alpha, c):
    q, K, V = _case(3, 1, 16, 4, 700, 400)
    out = _run(q, K, V, 700, alpha=alpha, c=c)
    assert_close(out, oracle.prefill_batch(q, K, V, 700, alpha=alpha, c=c), what="prefill output")


def test_prefill_last_row_is_the_decode():
    """The prompt's last token sees the whole cache: its row equals the full-layer decode."""
    n = 900
    q, K, V = _case(5, 1, 16, 4, n, 256, ncap=n)
    out = _run(q, K, V, n)
    shape = E.Shape(1, 16, 4, D, n, n)
    dec = torch.empty(1, 16, D, device="cuda")
    ns = torch.empty(1, 4, dtype=torch.int32, device="cuda")
    E.embla_full_decode(shape, to_dev(np.ascontiguousarray(q[:, :, -1])), to_dev(K), to_dev(V), dec, ns)
    torch.cuda.synchronize()
    assert_close(out[:, :, -1], dec.cpu().numpy(), what="last prefill row vs decode")


def test_prefill_empty_prompt_and_rejects():
    q, K, V = _case(9, 1, 16, 4, 64, 0)
    shape = E.Shape(1, 16, 4, D, 64, 64)
    out = torch.empty(1, 16, 0, D, device="cuda")
    E.embla_prefill(shape, to_dev(q), to_dev(K), to_dev(V), out)  # nothing to do
    torch.cuda.synchronize()
    q2 = torch.zeros(1, 16, 65, D, dtype=torch.bfloat16, device="cuda")
    out2 = torch.empty(1, 16, 65, D, device="cuda")
    with pytest.raises(E.EmblaError) as err:   # more prompt tokens than keys
        E.embla_prefill(shape, q2, to_dev(K), to_dev(V), out2)
    assert err.value.status == 1
