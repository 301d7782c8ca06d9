"""embla_append_kv / embla_append_kv_e4m3: the decode step's token written into row `pos` of
every plane of the caches, against the same rows written by PyTorch indexing; every other
row stays as it was."""
import pytest
import torch

import relu_sparse_kv_gb300 as E

pytestmark = pytest.mark.gpu
D = 128


@pytest.mark.parametrize("B,Hkv,ncap,pos", [(2, 4, 300, 0), (3, 2, 1037, 517), (8, 4, 32768, 32767)])
def test_append_bf16_rows(B, Hkv, ncap, pos):
    g = torch.Generator(device="cuda").manual_seed(B * 1000 + pos)
    shape = E.Shape(B, 4 * Hkv, Hkv, D, pos + 1, ncap)
    K = torch.randn(B, Hkv, ncap, D, device="cuda", generator=g).to(torch.bfloat16)
    V = torch.randn(B, Hkv, ncap, D, device="cuda", generator=g).to(torch.bfloat16)
    kr = torch.randn(B, Hkv, D, device="cuda", generator=g).to(torch.bfloat16)
    vr = torch.randn(B, Hkv, D, device="cuda", generator=g).to(torch.bfloat16)
    Kw, Vw = K.clone(), V.clone()
    Kw[:, :, pos] = kr
    Vw[:, :, pos] = vr
    E.embla_append_kv(shape, pos, kr, vr, K, V)
    torch.cuda.synchronize()
    assert torch.equal(K, Kw) and torch.equal(V, Vw)


@pytest.mark.parametrize("B,Hkv,ncap,pos,offset", [
    (2, 2, 300, 7, 0),       # 16-byte pieces for the codes, 4-byte ones for the scales
    (3, 2, 1037, 1036, 0),   # an odd cache stride: the scale planes are 4-byte aligned only
    (2, 2, 64, 5, 1),        # code rows one byte off a 16-byte boundary: byte copies
])
def test_append_e4m3_rows_and_scales(B, Hkv, ncap, pos, offset):
    g = torch.Generator(device="cuda").manual_seed(17 + pos)
    shape = E.Shape(B, 8 * Hkv, Hkv, D, pos + 1, ncap)
    rnd = lambda *s: torch.randint(0, 256, s, device="cuda", generator=g, dtype=torch.int32).to(torch.uint8)
    K8, V8 = rnd(B, Hkv, ncap, D), rnd(B, Hkv, ncap, D)
    Ks = torch.rand(B, Hkv, ncap, device="cuda", generator=g)
    Vs = torch.rand(B, Hkv, ncap, device="cuda", generator=g)
    # the packed rows, optionally starting one byte into a buffer
    buf = rnd(2 * B * Hkv * D + offset)
    kr = buf[offset:offset + B * Hkv * D].view(B, Hkv, D)
    vr = buf[offset + B * Hkv * D:offset + 2 * B * Hkv * D].view(B, Hkv, D)
    ksr = torch.rand(B, Hkv, device="cuda", generator=g)
    vsr = torch.rand(B, Hkv, device="cuda", generator=g)
    want = [t.clone() for t in (K8, Ks, V8, Vs)]
    want[0][:, :, pos] = kr
    want[1][:, :, pos] = ksr
    want[2][:, :, pos] = vr
    want[3][:, :, pos] = vsr
    E.embla_append_kv_e4m3(shape, pos, kr, ksr, vr, vsr, K8, Ks, V8, Vs)
    torch.cuda.synchronize()
    for got, w in zip((K8, Ks, V8, Vs), want):
        assert torch.equal(got, w)


def test_append_then_decode_sees_the_row():
    # the appended row is read by the full-layer call right after it on the same stream
    B, Hkv, n = 2, 4, 1000
    g = torch.Generator(device="cuda").manual_seed(3)
    shape = E.Shape(B, 4 * Hkv, Hkv, D, n, n)
    q = torch.randn(B, 4 * Hkv, D, device="cuda", generator=g).to(torch.bfloat16)
    K = torch.randn(B, Hkv, n, D, device="cuda", generator=g).to(torch.bfloat16)
    V = torch.randn(B, Hkv, n, D, device="cuda", generator=g).to(torch.bfloat16)
    kr = torch.randn(B, Hkv, D, device="cuda", generator=g).to(torch.bfloat16)
    vr = torch.randn(B, Hkv, D, device="cuda", generator=g).to(torch.bfloat16)
    out_a = torch.empty(B, 4 * Hkv, D, device="cuda")
    out_b = torch.empty_like(out_a)
    ns_a = torch.empty(B, Hkv, dtype=torch.int32, device="cuda")
    ns_b = torch.empty_like(ns_a)
    K2, V2 = K.clone(), V.clone()
    K2[:, :, n - 1] = kr
    V2[:, :, n - 1] = vr
    torch.cuda.synchronize()
    E.embla_full_decode(shape, q, K2, V2, out_b, ns_b)
    for _ in range(5):
        E.embla_append_kv(shape, n - 1, kr, vr, K, V)
        E.embla_full_decode(shape, q, K, V, out_a, ns_a)
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_b) and torch.equal(ns_a, ns_b)
        K[:, :, n - 1] = 0
        V[:, :, n - 1] = 0
    assert E.embla_device_check() == 0
