"""Seeded synthetic workloads for long-context decode attention.

Thin wrapper over ``gen.c`` (counter-based SplitMix64 + Box-Muller, and the
sign-control construction described there).  Both the CUDA path's tests and
the oracle draw their inputs from here; this module computes nothing of the
attention method itself.

All tensors come back as numpy arrays; bf16 values are carried as their
uint16 bit patterns (numpy has no bf16 type).

Shapes follow the decode layout used throughout the repository:
  q        [B, Hq, D]            one decode query per sequence
  K, V     [B, Hkv, n_cap, D]    cache rows; rows >= n are padding (NaN)
  targets  [B, Hkv, n]           +1 where the key was built to score > 0
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "libgen.so")
_lib = None

BF16_NAN = 0x7FC0

# stream roles
ROLE_Q_FULL, ROLE_K, ROLE_V, ROLE_T, ROLE_Q_SPARSE = 1, 2, 3, 4, 5
ROLE_K_WIN, ROLE_V_WIN, ROLE_Q_WIN, ROLE_IID = 6, 7, 8, 9
ROLE_Q_PRE, ROLE_K_PRE, ROLE_V_PRE = 10, 11, 12
ROLE_MLP_X, ROLE_MLP_UP, ROLE_MLP_DOWN, ROLE_MLP_LIVE = 13, 14, 15, 16


def build(force: bool = False) -> str:
    """Compile gen.c into libgen.so next to it (plain gcc, OpenMP)."""
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
        u64, i64, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        lib.gen_substream.restype = u64
        lib.gen_substream.argtypes = [u64, u64, u64]
        lib.gen_normal_bf16.restype = None
        lib.gen_normal_bf16.argtypes = [u64, i64, i64, vp]
        lib.gen_targets.restype = i64
        lib.gen_targets.argtypes = [u64, i64, ctypes.c_int, ctypes.c_double, i64, vp]
        lib.gen_signed_keys.restype = i64
        lib.gen_signed_keys.argtypes = [u64, ctypes.c_int, ctypes.c_int, i64, vp, vp, i64, i64,
                                        ctypes.c_double, ctypes.c_double, ctypes.c_int, i64, vp]
        lib.gen_signed_keys_e4m3.restype = i64
        lib.gen_signed_keys_e4m3.argtypes = [u64, ctypes.c_int, ctypes.c_int, i64, vp, vp, i64,
                                             i64, ctypes.c_double, ctypes.c_double, ctypes.c_int,
                                             i64, vp, vp]
        lib.gen_normal_e4m3.restype = None
        lib.gen_normal_e4m3.argtypes = [u64, i64, ctypes.c_int, vp, vp]
        lib.gen_e4m3_encode.restype = None
        lib.gen_e4m3_encode.argtypes = [vp, i64, vp]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def stream(seed: int, role: int, layer: int = 0, b: int = 0, head: int = 0) -> int:
    lib = _load()
    mask = (1 << 64) - 1
    s = lib.gen_substream(seed & mask, role & mask, layer & mask)
    return lib.gen_substream(s, b & mask, head & mask)


def normal_bf16(strm: int, shape, start: int = 0) -> np.ndarray:
    """N(0,1) numbers start, start+1, ... of a stream, rounded to bf16 bits."""
    out = np.empty(int(np.prod(shape)), dtype=np.uint16)
    _load().gen_normal_bf16(strm, start, out.size, _ptr(out))
    return out.reshape(shape)


def targets(strm: int, n: int, pattern: str, frac: float, run_len: int = 64) -> np.ndarray:
    """Target signs for n keys: 'bernoulli', 'subset' (exact count) or 'runs'."""
    kind = {"bernoulli": 0, "subset": 1, "runs": 2}[pattern]
    t = np.empty(n, dtype=np.int8)
    r = _load().gen_targets(strm, n, kind, float(frac), run_len, _ptr(t))
    if r < 0:
        raise ValueError("gen_targets: bad arguments")
    return t


def signed_keys(strm: int, q_group: np.ndarray, t: np.ndarray, n_cand: int, topk: int = 1024,
                margin: float = 2e-3, gap: float = 2e-3, max_attempts: int = 64,
                max_gap_iters: int = 100000) -> np.ndarray:
    """Keys whose raw score with every query row of the group has sign t[j].

    margin: every head satisfies t*D*cos(q_h, k) >= margin after bf16 rounding.
    gap:    when n_cand > topk, the topk-th and (topk+1)-th largest values of
            max_h D*cos(q_h, k_j) over j < n_cand differ by at least gap, and so do
            those of every head's own D*cos(q_h, k_j).
    """
    q_group = np.ascontiguousarray(q_group, dtype=np.uint16)
    G, D = q_group.shape
    t = np.ascontiguousarray(t, dtype=np.int8)
    n = t.shape[0]
    K = np.empty((n, D), dtype=np.uint16)
    r = _load().gen_signed_keys(strm, G, D, n, _ptr(q_group), _ptr(t), n_cand, topk, margin, gap,
                                max_attempts, max_gap_iters, _ptr(K))
    if r < 0:
        raise RuntimeError(f"gen_signed_keys failed with code {r}")
    return K


def signed_keys_e4m3(strm: int, q_group: np.ndarray, t: np.ndarray, n_cand: int,
                     topk: int = 1024, margin: float = 2e-3, gap: float = 2e-3,
                     max_attempts: int = 64, max_gap_iters: int = 100000):
    """signed_keys stored as 8-bit E4M3 codes with one float32 scale per key: (K8, Ks).
    The signs, margins and the top-k gap hold for the decoded keys scale * code."""
    q_group = np.ascontiguousarray(q_group, dtype=np.uint16)
    G, D = q_group.shape
    t = np.ascontiguousarray(t, dtype=np.int8)
    n = t.shape[0]
    K8 = np.empty((n, D), dtype=np.uint8)
    Ks = np.empty(n, dtype=np.float32)
    r = _load().gen_signed_keys_e4m3(strm, G, D, n, _ptr(q_group), _ptr(t), n_cand, topk, margin,
                                     gap, max_attempts, max_gap_iters, _ptr(K8), _ptr(Ks))
    if r < 0:
        raise RuntimeError(f"gen_signed_keys_e4m3 failed with code {r}")
    return K8, Ks


def normal_e4m3(strm: int, rows: int, D: int):
    """rows x D standard normals in 8-bit E4M3 codes with one scale per row: (codes, scales)."""
    out = np.empty((rows, D), dtype=np.uint8)
    sc = np.empty(rows, dtype=np.float32)
    _load().gen_normal_e4m3(strm, rows, D, _ptr(out), _ptr(sc))
    return out, sc


def e4m3_encode(x) -> np.ndarray:
    """Round to 8-bit E4M3 codes (nearest, ties to even; saturating at 448)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().gen_e4m3_encode(_ptr(x), x.size, _ptr(out))
    return out


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (a.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 bits (round to nearest even)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(np.asarray(a, dtype=np.float32))
    r[nan] = BF16_NAN
    return r


# ----------------------------------------------------------------------------- workloads

@dataclass
class FullLayer:
    """Inputs of one full (ReLU^2) layer: its query, its cache and the signs built in."""
    layer: int
    q: np.ndarray          # [B, Hq, D] bf16 bits
    K: np.ndarray          # [B, Hkv, n_cap, D] bf16 bits
    V: np.ndarray          # [B, Hkv, n_cap, D] bf16 bits
    targets: np.ndarray    # [B, Hkv, n] int8
    n: int
    sparse_q: list = field(default_factory=list)   # per sparse layer: [B, Hq, D] bf16 bits
    sparse_layers: list = field(default_factory=list)
    kv: str = "bf16"       # "e4m3": K and V hold 8-bit codes, Ks and Vs their scales
    Ks: np.ndarray | None = None  # [B, Hkv, n_cap] float32
    Vs: np.ndarray | None = None

    @property
    def n_pos(self) -> np.ndarray:
        return (self.targets > 0).sum(axis=-1)


@dataclass
class WindowLayer:
    layer: int
    q: np.ndarray          # [B, Hq, D]
    K: np.ndarray          # [B, Hkv, W, D] ring, already rotated at each slot's position
    V: np.ndarray          # [B, Hkv, W, D]
    pos: int


def make_full_layer(seed: int, layer: int, B: int, Hq: int, Hkv: int, D: int, n: int,
                    pattern: str, frac, run_len: int = 64, n_cap: int | None = None,
                    topk: int = 1024, recent: int = 128, margin: float = 2e-3,
                    gap: float = 2e-3, sparse_layers=(), kv: str = "bf16") -> FullLayer:
    """One full layer's query and sign-controlled cache (plus sparse-layer queries).

    frac may be a scalar or a per-sequence list (cycled over the batch).  kv "e4m3"
    stores K and V as 8-bit codes with a float32 scale per (token, KV head).
    """
    n_cap = n if n_cap is None else n_cap
    assert n_cap >= n and Hq % Hkv == 0 and kv in ("bf16", "e4m3")
    G = Hq // Hkv
    q = normal_bf16(stream(seed, ROLE_Q_FULL, layer), (B, Hq, D))
    if kv == "e4m3":
        K = np.full((B, Hkv, n_cap, D), 0x7F, dtype=np.uint8)
        V = np.full((B, Hkv, n_cap, D), 0x7F, dtype=np.uint8)
        Ks = np.full((B, Hkv, n_cap), np.nan, dtype=np.float32)
        Vs = np.full((B, Hkv, n_cap), np.nan, dtype=np.float32)
    else:
        K = np.full((B, Hkv, n_cap, D), BF16_NAN, dtype=np.uint16)
        V = np.full((B, Hkv, n_cap, D), BF16_NAN, dtype=np.uint16)
        Ks = Vs = None
    T = np.empty((B, Hkv, n), dtype=np.int8)
    fr = list(frac) if isinstance(frac, (list, tuple)) else [frac]
    n_cand = n - recent if n > topk + recent else 0
    for b in range(B):
        f_b = fr[b % len(fr)]
        for g in range(Hkv):
            T[b, g] = targets(stream(seed, ROLE_T, layer, b, g), n, pattern, f_b, run_len)
            if kv == "e4m3":
                K[b, g, :n], Ks[b, g, :n] = signed_keys_e4m3(
                    stream(seed, ROLE_K, layer, b, g), q[b, g * G:(g + 1) * G], T[b, g], n_cand,
                    topk, margin, gap)
                V[b, g, :n], Vs[b, g, :n] = normal_e4m3(stream(seed, ROLE_V, layer, b, g), n, D)
            else:
                K[b, g, :n] = signed_keys(stream(seed, ROLE_K, layer, b, g),
                                          q[b, g * G:(g + 1) * G], T[b, g], n_cand, topk,
                                          margin, gap)
                V[b, g, :n] = normal_bf16(stream(seed, ROLE_V, layer, b, g), (n, D))
    fl = FullLayer(layer=layer, q=q, K=K, V=V, targets=T, n=n, kv=kv, Ks=Ks, Vs=Vs)
    for sl in sparse_layers:
        fl.sparse_layers.append(sl)
        fl.sparse_q.append(normal_bf16(stream(seed, ROLE_Q_SPARSE, sl), (B, Hq, D)))
    return fl


def make_window_layer(seed: int, layer: int, B: int, Hq: int, Hkv: int, D: int, W: int,
                      pos: int) -> WindowLayer:
    q = normal_bf16(stream(seed, ROLE_Q_WIN, layer), (B, Hq, D))
    K = normal_bf16(stream(seed, ROLE_K_WIN, layer), (B, Hkv, W, D))
    V = normal_bf16(stream(seed, ROLE_V_WIN, layer), (B, Hkv, W, D))
    return WindowLayer(layer=layer, q=q, K=K, V=V, pos=pos)


def iid_unit(seed: int, G: int, D: int, n: int, unit: int = 0):
    """Plain N(0,1) q (G x D), K and V (n x D) with no sign control."""
    q = normal_bf16(stream(seed, ROLE_IID, 0, unit, 0), (G, D))
    K = normal_bf16(stream(seed, ROLE_IID, 1, unit, 0), (n, D))
    V = normal_bf16(stream(seed, ROLE_IID, 2, unit, 0), (n, D))
    return q, K, V


# The workloads: batch, context, heads and the survivor structure each one is built with.
EMBLA_FULL_LAYERS = (7, 16, 20, 24, 28)
EMBLA_SPARSE_OF = {7: (), 16: (17, 18, 19), 20: (21, 22, 23), 24: (25, 26, 27), 28: (29, 30, 31)}
EMBLA_WINDOW_LAYERS = tuple(l for l in range(16) if l != 7)

CONFIGS = {
    1: dict(name="tiny-full+sparse-b1-n2k", B=1, n=2048, pattern="bernoulli", frac=0.5,
            sparse=(1,)),
    2: dict(name="full+select+3sparse-b8-n32k-f0.05", B=8, n=32768, pattern="subset", frac=0.05,
            sparse=(1, 2, 3)),
    3: dict(name="full+select+3sparse-b1-n128k-bursty64", B=1, n=131072, pattern="runs",
            frac=0.05, sparse=(1, 2, 3)),
    4: dict(name="full+select+sparse-b32-n16k-mixed", B=32, n=16384, pattern="subset",
            frac=[0.5, 0.2, 0.05, 0.01], sparse=(1,)),
    5: dict(name="embla-attention-step-b16-n64k", B=16, n=65536, pattern="subset", frac=0.05,
            sparse=None),
    # Embla 1's own head shape: 8 query heads per KV head, K and V in 8 bits
    6: dict(name="gqa8-e4m3-full+select+3sparse-b8-n32k-f0.05", B=8, n=32768, pattern="subset",
            frac=0.05, sparse=(1, 2, 3), Hq=16, Hkv=2, kv="e4m3"),
    # prefill of a full layer: a whole prompt of T tokens, causal (no prefix)
    7: dict(name="prefill-b1-n8k", kind="prefill", B=1, n=8192, T=8192),
    8: dict(name="prefill-b1-n32k", kind="prefill", B=1, n=32768, T=32768),
    # a ReLU^2 MLP at batch 1 with 22 % of its neurons firing (the page reports 78 % of the
    # down-projection bytes saved)
    9: dict(name="relu2-mlp-b1-d2048-f8192-live0.22", kind="mlp", d=2048, f=8192, live=0.22),
    # the benchmarked workload with a selection per query head instead of per KV head
    10: dict(name="per-head-select-full+3sparse-b8-n32k-f0.05", B=8, n=32768, pattern="subset",
             frac=0.05, sparse=(1, 2, 3), select="per_head"),
}
HQ, HKV, HEAD_DIM, WINDOW, ROPE_BASE = 16, 4, 128, 128, 10000.0


def make_prefill(seed: int, B: int, Hq: int, Hkv: int, n: int, T: int, D: int = 128):
    """A full layer's prompt: queries [B, Hq, T, D] of the last T of n cached keys, and the
    caches [B, Hkv, n, D]; all N(0, 1) in bf16 (untrained statistics: about half the weights
    are zero)."""
    q = normal_bf16(stream(seed, ROLE_Q_PRE), (B, Hq, T, D))
    K = normal_bf16(stream(seed, ROLE_K_PRE), (B, Hkv, n, D))
    V = normal_bf16(stream(seed, ROLE_V_PRE), (B, Hkv, n, D))
    return q, K, V


def config_prefill(cfg: int, seed: int = 0, B: int | None = None, n: int | None = None):
    c = CONFIGS[cfg]
    B = c["B"] if B is None else B
    n = c["n"] if n is None else n
    T = min(c["T"], n)
    return make_prefill(seed, B, c.get("Hq", HQ), c.get("Hkv", HKV), n, T)


def make_mlp(seed: int, d: int, f: int, live: float, margin: float = 1e-2):
    """One token and a ReLU^2 MLP whose neurons fire for exactly round(live * f) of them:
    x [d] ~ N(0, 1); w_up [f, d] rows ~ N(0, I/d), each moved along x so that x . w_i has
    the chosen sign with |x . w_i| >= margin |x| after bf16 rounding; w_down [f, d] ~
    N(0, I/f).  Returns bf16 bit patterns (x, w_up, w_down) and the live mask."""
    x = normal_bf16(stream(seed, ROLE_MLP_X), (d,))
    xf = bf16_to_f32(x).astype(np.float64)
    W = bf16_to_f32(normal_bf16(stream(seed, ROLE_MLP_UP), (f, d))).astype(np.float64) / np.sqrt(d)
    n_live = int(round(live * f))
    perm = np.random.default_rng(stream(seed, ROLE_MLP_LIVE)).permutation(f)
    t = -np.ones(f)
    t[perm[:n_live]] = 1.0
    xx = float(xf @ xf)
    floor = margin * np.sqrt(xx)
    Wb = None
    for _ in range(8):
        c = W @ xf
        target = t * np.maximum(np.abs(c), floor)
        W = W + np.outer((target - c) / xx, xf)
        Wb = f32_to_bf16(W.astype(np.float32))
        got = bf16_to_f32(Wb).astype(np.float64) @ xf
        if np.all(got * t >= 0.5 * floor):
            break
        floor *= 2.0
    else:
        raise RuntimeError("make_mlp: sign control did not converge")
    w_down = normal_bf16(stream(seed, ROLE_MLP_DOWN), (f, d))
    w_down = f32_to_bf16((bf16_to_f32(w_down) / np.float32(np.sqrt(f))).astype(np.float32))
    return x, Wb, w_down, t > 0


def config_mlp(cfg: int, seed: int = 0):
    c = CONFIGS[cfg]
    return make_mlp(seed, c["d"], c["f"], c["live"])


def config_full_layers(cfg: int, seed: int = 0, B: int | None = None, n: int | None = None,
                       n_cap: int | None = None):
    """Yield the full layers of a configuration one at a time (config 5 yields five)."""
    c = CONFIGS[cfg]
    B = c["B"] if B is None else B
    n = c["n"] if n is None else n
    if cfg == 5:
        for layer in EMBLA_FULL_LAYERS:
            yield make_full_layer(seed, layer, B, HQ, HKV, HEAD_DIM, n, c["pattern"], c["frac"],
                                  n_cap=n_cap, sparse_layers=EMBLA_SPARSE_OF[layer])
    else:
        yield make_full_layer(seed, 0, B, c.get("Hq", HQ), c.get("Hkv", HKV), HEAD_DIM, n,
                              c["pattern"], c["frac"], n_cap=n_cap, sparse_layers=c["sparse"],
                              kv=c.get("kv", "bf16"))


def config_window_layers(cfg: int, seed: int = 0, B: int | None = None, n: int | None = None):
    c = CONFIGS[cfg]
    if cfg != 5:
        return
    B = c["B"] if B is None else B
    n = c["n"] if n is None else n
    for layer in EMBLA_WINDOW_LAYERS:
        yield make_window_layer(seed, layer, B, HQ, HKV, HEAD_DIM, WINDOW, pos=n - 1)
