"""CPU-side checks of the C ABI: the library loads without a GPU, exports every symbol the
header declares, and rejects bad arguments before touching the device.  Also the host-side
work split of the full-layer decode, compiled from its header with g++."""
import ctypes
import os
import re
import subprocess

import pytest

import relu_sparse_kv_gb300 as E
from relu_sparse_kv_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "embla_attn.h")


@pytest.fixture(scope="module")
def lib():
    B.build()
    return E.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(embla_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 11
    out = subprocess.run(["nm", "-D", "--defined-only", E.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (embla_[a-z0-9_]+)", out))
    assert set(names) <= exported, set(names) - exported
    for n in names:
        getattr(lib, n)


def test_status_strings(lib):
    for code in range(6):
        assert lib.embla_status_string(code)
    assert lib.embla_status_string(99) == b"unknown status"


def _shape(**kw):
    d = dict(batch=1, n_q_heads=16, n_kv_heads=4, head_dim=128, ctx_len=4096, cache_stride=4096)
    d.update(kw)
    return E._Shape(**d)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), 2),              # unsupported head_dim
    (dict(n_q_heads=12, n_kv_heads=4), 2),  # G = 3
    (dict(n_q_heads=16, n_kv_heads=3), 1),  # Hq % Hkv != 0
    (dict(cache_stride=100), 1),         # stride < n
    (dict(ctx_len=-1), 1),
    (dict(batch=-1), 1),
])
def test_shape_validation_without_gpu(lib, kw, status):
    s = _shape(**kw)
    st = lib.embla_full_decode(ctypes.byref(s), None, None, None, 1.0, 1.0, 1e-6, None, None,
                               None, None, None, 0, None)
    assert st == status


def test_scalar_and_pointer_validation_without_gpu(lib):
    s = _shape()
    f = lib.embla_full_decode
    assert f(None, None, None, None, 1.0, 1.0, 1e-6, None, None, None, None, None, 0, None) == 1
    assert f(ctypes.byref(s), None, None, None, -1.0, 1.0, 1e-6, None, None, None, None, None, 0, None) == 1
    assert f(ctypes.byref(s), None, None, None, 1.0, -1.0, 1e-6, None, None, None, None, None, 0, None) == 1
    assert f(ctypes.byref(s), None, None, None, 1.0, 1.0, float("nan"), None, None, None, None, None, 0, None) == 1
    assert f(ctypes.byref(s), None, None, None, 1.0, 1.0, 1e-6, None, None, None, None, None, 0, None) == 1
    sel = lib.embla_select_topk
    assert sel(ctypes.byref(s), None, None, 1024, 128, None, 1000, None, None, 0, None) == 1  # stride
    assert sel(ctypes.byref(s), None, None, -1, 128, None, 1152, None, None, 0, None) == 1
    sp = lib.embla_sparse_decode
    assert sp(ctypes.byref(s), None, None, None, None, 1152, None, float("inf"), None, None, 0, None) == 1
    w = lib.embla_window_decode
    assert w(ctypes.byref(s), None, None, None, 0, 5, 10000.0, 0.1, None, None, 0, None) == 1
    assert w(ctypes.byref(s), None, None, None, 128, -1, 10000.0, 0.1, None, None, 0, None) == 1
    assert w(ctypes.byref(s), None, None, None, 128, 5, 0.0, 0.1, None, None, 0, None) == 1
    # the decode with its selection: the selection's arguments are checked with the rest
    fs = lib.embla_full_decode_select
    a = [ctypes.c_void_p(256 * (k + 1)) for k in range(8)]  # aligned, never dereferenced
    base = [ctypes.byref(s), a[0], a[1], a[2], 1.0, 1.0, 1e-6, a[3], a[4], a[5], a[6]]
    assert fs(*base, 1024, 128, a[7], 1000, a[7], a[7], 1 << 20, None) == 1   # stride < topk + recent
    assert fs(*base, -1, 128, a[7], 1152, a[7], a[7], 1 << 20, None) == 1
    assert fs(*base, 1024, 128, None, 1152, a[7], a[7], 1 << 20, None) == 1    # no idx
    assert fs(*base, 1024, 128, a[7], 1152, ctypes.c_void_p(260), a[7], 1 << 20, None) == 1  # count unaligned
    nosel = base[:9] + [None, None]
    assert fs(*nosel, 1024, 128, a[7], 1152, a[7], a[7], 1 << 20, None) == 1  # scores required
    # the token's rows into the caches: the position must lie inside the cache
    ap = lib.embla_append_kv
    assert ap(ctypes.byref(s), -1, a[0], a[1], a[2], a[3], None) == 1
    assert ap(ctypes.byref(s), 4096, a[0], a[1], a[2], a[3], None) == 1  # pos == cache_stride
    assert ap(ctypes.byref(s), 5, None, a[1], a[2], a[3], None) == 1
    assert lib.embla_append_kv_e4m3(ctypes.byref(s), 5, a[0], a[1], a[2], a[3], a[4], a[5],
                                    a[6], None, None) == 1
    # the token's rows into the caches: the position must lie inside the cache
    ap = lib.embla_append_kv
    assert ap(ctypes.byref(s), -1, a[0], a[1], a[2], a[3], None) == 1
    assert ap(ctypes.byref(s), 4096, a[0], a[1], a[2], a[3], None) == 1  # pos == cache_stride
    assert ap(ctypes.byref(s), 5, None, a[1], a[2], a[3], None) == 1
    assert lib.embla_append_kv_e4m3(ctypes.byref(s), 5, a[0], a[1], a[2], a[3], a[4], a[5],
                                    a[6], None, None) == 1
    st = lib.embla_self_test_wait_limit
    assert st(0, 0, None) == 1  # a limit of 0 or above one second is refused before any launch
    assert st(1000001, 0, None) == 1


def test_empty_batch_is_a_no_op(lib):
    s = _shape(batch=0)
    assert lib.embla_full_decode(ctypes.byref(s), None, None, None, 1.0, 1.0, 1e-6, None, None,
                                 None, None, None, 0, None) == 0
    assert lib.embla_sparse_decode(ctypes.byref(s), None, None, None, None, 1152, None, 0.1,
                                   None, None, 0, None) == 0
    assert lib.embla_append_kv(ctypes.byref(s), 0, None, None, None, None, None) == 0
    assert lib.embla_append_kv(ctypes.byref(s), 0, None, None, None, None, None) == 0
    assert lib.embla_full_decode_select(ctypes.byref(s), None, None, None, 1.0, 1.0, 1e-6, None,
                                        None, None, None, 1024, 128, None, 1152, None, None, 0,
                                        None) == 0


HARNESS = r"""
#include <cstdio>
#include "internal.h"
using namespace embla;
int main() {
  // every tile belongs to exactly one piece; CTA c takes pieces c, c + P, ...; the stretch
  // of unit u inside piece q uses slot q+u, which no other (piece, unit) pair uses; the
  // combine's [q0, q1] range lists exactly the pieces that touch u
  static int slot_user[400];
  for (int mp = 1; mp <= 5; mp += 2)
    for (int sms = 1; sms <= 20; ++sms)
      for (long units = 1; units <= 9; ++units)
        for (long n = 0; n <= 2600; n += 97) {
          FullSplit sp = full_split(units, n, sms, mp);
          long T = sp.tiles, P = sp.ctas, Q = sp.pieces, TU = sp.tiles_per_unit;
          if (T == 0) { if (P != 0) return 1; continue; }
          if (P < 1 || P > T || P > sms) return 2;
          if (Q % P != 0) return 9;
          long K = Q / P;
          if (K < 1 || K > mp || K % 2 == 0 || Q > T) return 10;
          if (K > 1 && T / P / K < kMinPieceTiles) return 12;
          for (int i = 0; i < 400; ++i) slot_user[i] = -1;
          for (long q = 0; q < Q; ++q) {
            long b = split_piece_start(q, T, Q), e = split_piece_start(q + 1, T, Q);
            if (e <= b) return 3;
            for (long t = b; t < e; ++t) {
              if (split_piece_of_tile(t, T, Q) != q) return 4;
              long u = t / TU, slot = q + u;
              if (slot >= Q + units) return 5;
              if (slot_user[slot] != -1 && slot_user[slot] != (int)(q * 1000 + u)) return 6;
              slot_user[slot] = (int)(q * 1000 + u);
            }
          }
          if (split_piece_start(0, T, Q) != 0 || split_piece_start(Q, T, Q) != T) return 7;
          for (long u = 0; u < units; ++u) {
            long q0 = split_piece_of_tile(u * TU, T, Q);
            long q1 = split_piece_of_tile(u * TU + TU - 1, T, Q);
            if (q1 - q0 + 1 > (TU * Q + T - 1) / T + 1) return 11;
            for (long q = 0; q < Q; ++q) {
              long b = split_piece_start(q, T, Q), e = split_piece_start(q + 1, T, Q);
              bool touches = b < (u + 1) * TU && e > u * TU;
              if (touches != (q >= q0 && q <= q1)) return 8;
            }
          }
        }
  // the decode workloads' splits on 152 SMs: B 8 x 4 KV heads at 32k keys keeps one piece
  // per CTA; B 32 x 4 at 16k keys (108 tiles a CTA) takes five
  if (full_split(32, 32768, 152).pieces != 152) return 13;
  if (full_split(128, 16384, 152).pieces != 5 * 152) return 14;
  std::puts("ok");
  return 0;
}
"""


def test_full_decode_work_split_host_logic(tmp_path):
    src = tmp_path / "split.cpp"
    src.write_text(HARNESS)
    exe = tmp_path / "split"
    cuda_inc = "/usr/local/cuda/include"
    r = subprocess.run(["g++", "-std=c++17", "-O1", "-I" + B.CSRC, "-I" + cuda_inc, str(src),
                        os.path.join(B.BUILD, "full_decode.o"), os.path.join(B.BUILD, "select.o"),
                        "-o", str(exe),
                        "-L/usr/local/cuda/lib64", "-lcudart_static", "-ldl", "-lpthread",
                        "-lrt"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout)


def test_static_scratch_size_matches_header():
    text = open(HEADER).read()
    m = re.search(r"#define EMBLA_FULL_DECODE_SCRATCH_BYTES \(\(size_t\)(\d+) << (\d+)\)", text)
    assert m, "scratch size define not found"
    assert int(m.group(1)) << int(m.group(2)) == E.FULL_DECODE_SCRATCH_BYTES
