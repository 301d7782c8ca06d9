"""fp64 CPU oracle for Embla 1 long-context decode attention (ctypes wrapper over oracle.c).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module.  The CUDA library never
calls it and it never calls the CUDA library.

Functions accept bf16 bit patterns (``np.uint16``), which are widened exactly,
or any float array, which is converted to float64.  Layouts:

  q        [B, Hq, D]          (per unit: [G, D])
  K, V     [B, Hkv, ncap, D]   (per unit: [n, D])
  sigma32  [B, Hkv, ncap]      fp32 selection scores
  idx      [B, Hkv, topk+recent] int32, ascending

What each function computes, with the passage of "The Architecture of
Embla 1" it follows, is stated in oracle.c.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (plain gcc, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-std=c99", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i, i64, d, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        sig = {
            "oracle_full_scores": [i, i, i64, vp, vp, i64, d, d, vp],
            "oracle_full_decode": [i, i, i64, vp, vp, i64, vp, i64, d, d, d, vp, vp, vp, vp],
            "oracle_select_topk": [i64, vp, i64, i64, vp, vp],
            "oracle_sparse_decode": [i, i, i64, vp, vp, i64, vp, i64, vp, d, vp],
            "oracle_window_decode": [i, i, i64, i64, vp, vp, vp, d, d, vp],
            "oracle_full_decode_batch": [i, i, i, i, i64, i64, vp, vp, vp, d, d, d, vp, vp, vp],
            "oracle_select_topk_batch": [i, i, i64, i64, vp, i64, i64, vp, i64, vp],
            "oracle_sparse_decode_batch": [i, i, i, i, i64, vp, vp, vp, vp, i64, vp, d, vp],
            "oracle_window_decode_batch": [i, i, i, i, i64, i64, vp, vp, vp, d, d, vp],
            "oracle_skip_stats": [i64, vp, i64, vp, vp],
            "oracle_prefill": [i, i, i64, i64, vp, vp, i64, vp, i64, d, d, d, vp],
            "oracle_relu2_mlp": [i64, i64, vp, vp, vp, vp, vp, vp],
            "oracle_prefill_batch": [i, i, i, i, i64, i64, i64, vp, vp, vp, d, d, d, vp],
            "oracle_skip_stats_batch": [i, i, i64, i64, vp, i64, vp, vp],
            "oracle_head_scores_batch": [i, i, i, i, i64, i64, vp, vp, d, d, vp],
        }
        for name, args in sig.items():
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = args
        lib.oracle_set_threads.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def set_threads(n: int) -> int:
    """Threads the batched functions use from now on; returns the previous count."""
    return int(_load().oracle_set_threads(int(n)))


def f64(a) -> np.ndarray:
    """bf16 bits (uint16) widened exactly, or any numeric array, as C-contiguous float64."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        a = (a.astype(np.uint32) << 16).view(np.float32)
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a) -> int:
    return a.ctypes.data if a is not None else None


def _ok(r: int, name: str):
    if r != 0:
        raise ValueError(f"{name}: bad arguments")


# ----------------------------------------------------------------------------- one unit

def full_scores(q, K, alpha=1.0, eps=1e-6) -> np.ndarray:
    """s[h, j] = alpha * qhat_h . khat_j for one unit (q: [G, D], K: [n, D])."""
    q, K = f64(q), f64(K)
    G, D = q.shape
    n = K.shape[0]
    s = np.empty((G, n), dtype=np.float64)
    _ok(_load().oracle_full_scores(G, D, n, _p(q), _p(K), D, alpha, eps, _p(s)), "full_scores")
    return s


def full_decode(q, K, V, alpha=1.0, c=1.0, eps=1e-6):
    """One unit's full layer: returns (out [G, D], sigma32 [n], n_surv, n_zero [G])."""
    q, K, V = f64(q), f64(K), f64(V)
    G, D = q.shape
    n = K.shape[0]
    out = np.empty((G, D), dtype=np.float64)
    sigma = np.empty(n, dtype=np.float32)
    ns = np.zeros(1, dtype=np.int64)
    nz = np.zeros(G, dtype=np.int64)
    _ok(_load().oracle_full_decode(G, D, n, _p(q), _p(K), D, _p(V), D, alpha, c, eps, _p(out),
                                   _p(sigma), _p(ns), _p(nz)), "full_decode")
    return out, sigma, int(ns[0]), nz


def select_topk(sigma32, topk=1024, recent=128):
    """One unit's selection: ascending int32 indices."""
    s = np.ascontiguousarray(sigma32, dtype=np.float32)
    n = s.shape[0]
    idx = np.empty(max(min(n, topk + recent), 1), dtype=np.int32)
    cnt = np.zeros(1, dtype=np.int64)
    _ok(_load().oracle_select_topk(n, _p(s), topk, recent, _p(idx), _p(cnt)), "select_topk")
    return idx[:int(cnt[0])]


def sparse_decode(q, K, V, idx, tau=None):
    """One unit's sparse layer over the selected rows idx (q: [G, D], K/V: [n, D])."""
    q, K, V = f64(q), f64(K), f64(V)
    G, D = q.shape
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    tau = 1.0 / np.sqrt(D) if tau is None else tau
    out = np.empty((G, D), dtype=np.float64)
    _ok(_load().oracle_sparse_decode(G, D, idx.shape[0], _p(q), _p(K), D, _p(V), D, _p(idx), tau,
                                     _p(out)), "sparse_decode")
    return out


def window_decode(q, Kw, Vw, pos, base=10000.0, tau=None):
    """One unit's window layer (q: [G, D], Kw/Vw: [W, D] ring)."""
    q, Kw, Vw = f64(q), f64(Kw), f64(Vw)
    G, D = q.shape
    W = Kw.shape[0]
    tau = 1.0 / np.sqrt(D) if tau is None else tau
    out = np.empty((G, D), dtype=np.float64)
    _ok(_load().oracle_window_decode(G, D, W, pos, _p(q), _p(Kw), _p(Vw), base, tau, _p(out)),
        "window_decode")
    return out


# ----------------------------------------------------------------------------- batched

def full_decode_batch(q, K, V, n, alpha=1.0, c=1.0, eps=1e-6, want_sigma=True):
    """All units: returns (out [B, Hq, D], sigma32 [B, Hkv, ncap] or None, n_surv [B, Hkv])."""
    q, K, V = f64(q), f64(K), f64(V)
    B, Hq, D = q.shape
    Hkv, ncap = K.shape[1], K.shape[2]
    out = np.empty((B, Hq, D), dtype=np.float64)
    sigma = np.full((B, Hkv, ncap), np.nan, dtype=np.float32) if want_sigma else None
    ns = np.zeros((B, Hkv), dtype=np.int64)
    _ok(_load().oracle_full_decode_batch(B, Hq, Hkv, D, n, ncap, _p(q), _p(K), _p(V), alpha, c,
                                         eps, _p(out), _p(sigma), _p(ns)), "full_decode_batch")
    return out, sigma, ns


def head_scores_batch(q, K, n, alpha=1.0, eps=1e-6):
    """Every query head's own scores s_hj rounded to fp32: [B, Hq, ncap] (NaN at j >= n)."""
    q, K = f64(q), f64(K)
    B, Hq, D = q.shape
    Hkv, ncap = K.shape[1], K.shape[2]
    s = np.full((B, Hq, ncap), np.nan, dtype=np.float32)
    _ok(_load().oracle_head_scores_batch(B, Hq, Hkv, D, n, ncap, _p(q), _p(K), alpha, eps, _p(s)),
        "head_scores_batch")
    return s


def select_topk_batch(sigma32, n, topk=1024, recent=128):
    """All units: returns (idx [B, Hkv, topk+recent] int32 (-1 past count), count [B, Hkv])."""
    s = np.ascontiguousarray(sigma32, dtype=np.float32)
    B, Hkv, ncap = s.shape
    stride = topk + recent
    idx = np.full((B, Hkv, stride), -1, dtype=np.int32)
    cnt = np.zeros((B, Hkv), dtype=np.int64)
    _ok(_load().oracle_select_topk_batch(B, Hkv, n, ncap, _p(s), topk, recent, _p(idx), stride,
                                         _p(cnt)), "select_topk_batch")
    return idx, cnt


def prefill(q, K, V, alpha=1.0, c=1.0, eps=1e-6):
    """One unit's causal prefill: q [G, T, D] (the last T of the n keys' tokens), K and V
    [n, D]; returns out [G, T, D]."""
    q, K, V = f64(q), f64(K), f64(V)
    G, T, D = q.shape
    n = K.shape[0]
    out = np.empty((G, T, D), dtype=np.float64)
    _ok(_load().oracle_prefill(G, D, n, T, _p(q), _p(K), D, _p(V), D, alpha, c, eps, _p(out)),
        "prefill")
    return out


def prefill_batch(q, K, V, n, alpha=1.0, c=1.0, eps=1e-6):
    """All units: q [B, Hq, T, D], K and V [B, Hkv, ncap, D] (keys 0..n-1 valid)."""
    q, K, V = f64(q), f64(K), f64(V)
    B, Hq, T, D = q.shape
    Hkv, ncap = K.shape[1], K.shape[2]
    out = np.empty((B, Hq, T, D), dtype=np.float64)
    _ok(_load().oracle_prefill_batch(B, Hq, Hkv, D, n, T, ncap, _p(q), _p(K), _p(V), alpha, c,
                                     eps, _p(out)), "prefill_batch")
    return out


def relu2_mlp(x, w_up, w_down):
    """One token through a ReLU^2 MLP: x [d], w_up and w_down [f, d] (row i = neuron i).
    Returns (y [d], h [f], n_live)."""
    x, w_up, w_down = f64(x), f64(w_up), f64(w_down)
    f, d = w_up.shape
    h = np.empty(f, dtype=np.float64)
    y = np.empty(d, dtype=np.float64)
    nl = np.zeros(1, dtype=np.int64)
    _ok(_load().oracle_relu2_mlp(d, f, _p(x), _p(w_up), _p(w_down), _p(h), _p(y), _p(nl)),
        "relu2_mlp")
    return y, h, int(nl[0])


def e4m3_table() -> np.ndarray:
    """The 256 values of an 8-bit E4M3 code (no infinities): sign, 4 exponent bits with bias
    7, 3 mantissa bits; exponent field 0 is subnormal, m * 2^-9; S.1111.111 is NaN."""
    v = np.empty(256, dtype=np.float64)
    for b in range(256):
        e, m = (b >> 3) & 15, b & 7
        if e == 15 and m == 7:
            x = np.nan
        elif e == 0:
            x = m * 2.0 ** -9
        else:
            x = (1.0 + m / 8.0) * 2.0 ** (e - 7)
        v[b] = -x if b & 0x80 else x
    return v


def dequant_e4m3(codes, scales) -> np.ndarray:
    """float64 values scale * code of an 8-bit cache [..., n, D] with scales [..., n]."""
    t = e4m3_table()
    return t[np.asarray(codes, dtype=np.uint8)] * np.asarray(scales, dtype=np.float64)[..., None]


def skip_stats_batch(sigma32, n, chunk=8):
    """All units: (keys_needed [B, Hkv], chunks_needed [B, Hkv]) -- keys j < n with
    sigma > 0, and chunks of `chunk` keys holding at least one of them."""
    s = np.ascontiguousarray(sigma32, dtype=np.float32)
    B, Hkv, ncap = s.shape
    keys = np.zeros((B, Hkv), dtype=np.int64)
    chunks = np.zeros((B, Hkv), dtype=np.int64)
    _ok(_load().oracle_skip_stats_batch(B, Hkv, n, ncap, _p(s), chunk, _p(keys), _p(chunks)),
        "skip_stats_batch")
    return keys, chunks


def sparse_decode_batch(q, K, V, idx, count, tau=None):
    q, K, V = f64(q), f64(K), f64(V)
    B, Hq, D = q.shape
    Hkv, ncap = K.shape[1], K.shape[2]
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    count = np.ascontiguousarray(count, dtype=np.int64)
    tau = 1.0 / np.sqrt(D) if tau is None else tau
    out = np.empty((B, Hq, D), dtype=np.float64)
    _ok(_load().oracle_sparse_decode_batch(B, Hq, Hkv, D, ncap, _p(q), _p(K), _p(V), _p(idx),
                                           idx.shape[-1], _p(count), tau, _p(out)),
        "sparse_decode_batch")
    return out


def window_decode_batch(q, Kw, Vw, pos, base=10000.0, tau=None):
    q, Kw, Vw = f64(q), f64(Kw), f64(Vw)
    B, Hq, D = q.shape
    Hkv, W = Kw.shape[1], Kw.shape[2]
    tau = 1.0 / np.sqrt(D) if tau is None else tau
    out = np.empty((B, Hq, D), dtype=np.float64)
    _ok(_load().oracle_window_decode_batch(B, Hq, Hkv, D, W, pos, _p(q), _p(Kw), _p(Vw), base, tau,
                                           _p(out)), "window_decode_batch")
    return out
