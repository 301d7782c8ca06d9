"""Python binding of libembla_attn.so: decode attention for the Embla 1 layer types
on one GB300 (sm_103a).

Argument marshalling only.  Every function here checks tensor dtypes, devices and
contiguity, then calls the C entry point of the same name with raw device pointers and
the current CUDA stream; all arithmetic runs in the library's CUDA kernels.  There is
no CPU path: if the library was not built, importing the binding's functions raises.

Tensors (torch, on the current CUDA device, C-contiguous):
  q              bf16  [B, Hq, D]
  k_cache/v_cache bf16 [B, Hkv, cache_stride, D]
  k_codes/v_codes uint8 [B, Hkv, cache_stride, D]  (E4M3 codes, *_e4m3 calls)
  k_scales/v_scales fp32 [B, Hkv, cache_stride]    (one scale per token and KV head)
  out            fp32  [B, Hq, D]
  n_surv, count  int32 [B, Hkv]
  sel_scores     fp32  [B, Hkv, cache_stride]
  sel_hist       int32 [B, Hkv, 2048]  (holds uint32 counts)
  idx            int32 [B, Hkv, idx_stride]
  workspace      uint8 (any shape), at least the *_workspace_size result
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libembla_attn.so")
HIST_BINS = 2048
FULL_DECODE_SCRATCH_BYTES = 4 << 20  # EMBLA_FULL_DECODE_SCRATCH_BYTES in the C header

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace too small",
          4: "CUDA error", 5: "device-side check failed"}


class EmblaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {STATUS.get(status, status)} (status {status})")
        self.status = status


class _Shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("ctx_len", ctypes.c_int64), ("cache_stride", ctypes.c_int64)]


@dataclass(frozen=True)
class Shape:
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ctx_len: int
    cache_stride: int

    def c(self) -> _Shape:
        return _Shape(self.batch, self.n_q_heads, self.n_kv_heads, self.head_dim, self.ctx_len,
                      self.cache_stride)

    @property
    def units(self) -> int:
        return self.batch * self.n_kv_heads


_lib = None


def library() -> ctypes.CDLL:
    """Load libembla_attn.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run relu_sparse_kv_gb300.build.build() "
                               "(or __graft_entry__.build()) first")
        lib = ctypes.CDLL(LIB_PATH)
        P, i32, i64, f32, sz, vp = (ctypes.POINTER(_Shape), ctypes.c_int32, ctypes.c_int64,
                                    ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p)
        sigs = {
            "embla_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "embla_device_sm_count": (ctypes.c_int, []),
            "embla_full_decode_workspace_size": (sz, [P]),
            "embla_full_decode": (ctypes.c_int, [P, vp, vp, vp, f32, f32, f32, vp, vp, vp, vp, vp,
                                                 sz, vp]),
            "embla_full_decode_e4m3": (ctypes.c_int, [P, vp, vp, vp, vp, vp, f32, f32, f32, vp,
                                                       vp, vp, vp, vp, sz, vp]),
            "embla_sparse_decode_e4m3": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, i32, vp,
                                                         f32, vp, vp, sz, vp]),
            "embla_prefill_workspace_size": (sz, [P]),
            "embla_prefill": (ctypes.c_int, [P, i64, vp, vp, vp, f32, f32, f32, vp, vp, sz, vp]),
            "embla_relu2_mlp_workspace_size": (sz, [i64, i64]),
            "embla_relu2_mlp": (ctypes.c_int, [i64, i64, vp, vp, vp, vp, vp, vp, sz, vp]),
            "embla_full_decode_head_scores": (ctypes.c_int, [P, vp, vp, vp, f32, f32, f32, vp, vp,
                                                              vp, vp, vp, sz, vp]),
            "embla_select_topk_per_head_workspace_size": (sz, [P, i32, i32]),
            "embla_select_topk_per_head": (ctypes.c_int, [P, vp, vp, i32, i32, vp, i32, vp, vp, sz,
                                                           vp]),
            "embla_sparse_decode_per_head": (ctypes.c_int, [P, vp, vp, vp, vp, i32, vp, f32, vp, vp,
                                                             sz, vp]),
            "embla_full_decode_static_scratch": (ctypes.c_int, [P, vp, vp, vp, f32, f32, f32,
                                                                vp, vp, vp, vp, vp]),
            "embla_append_kv": (ctypes.c_int, [P, i64, vp, vp, vp, vp, vp]),
            "embla_append_kv_e4m3": (ctypes.c_int, [P, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "embla_full_decode_select_workspace_size": (sz, [P, i32, i32]),
            "embla_full_decode_select": (ctypes.c_int, [P, vp, vp, vp, f32, f32, f32, vp, vp, vp,
                                                        vp, i32, i32, vp, i32, vp, vp, sz, vp]),
            "embla_full_decode_e4m3_select": (ctypes.c_int, [P, vp, vp, vp, vp, vp, f32, f32, f32,
                                                             vp, vp, vp, vp, i32, i32, vp, i32,
                                                             vp, vp, sz, vp]),
            "embla_select_topk_workspace_size": (sz, [P, i32, i32]),
            "embla_select_topk": (ctypes.c_int, [P, vp, vp, i32, i32, vp, i32, vp, vp, sz, vp]),
            "embla_sparse_decode_workspace_size": (sz, [P, i32]),
            "embla_sparse_decode": (ctypes.c_int, [P, vp, vp, vp, vp, i32, vp, f32, vp, vp, sz,
                                                   vp]),
            "embla_window_decode_workspace_size": (sz, [P, i32]),
            "embla_window_decode": (ctypes.c_int, [P, vp, vp, vp, i32, i64, f32, f32, vp, vp, sz,
                                                   vp]),
            "embla_skip_stats": (ctypes.c_int, [P, vp, i32, vp, vp, vp]),
            "embla_device_check": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int,
                                                  vp]),
            "embla_self_test_wait_limit": (ctypes.c_int, [ctypes.c_uint32, ctypes.c_int, vp]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(t, dtype, shape, name, allow_none=False):
    if t is None:
        if allow_none:
            return
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def _call(name, *args):
    st = getattr(library(), name)(*args)
    if st != 0:
        raise EmblaError(name, st)


def _workspace(nbytes: int, workspace, device):
    if workspace is None:
        return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise EmblaError("workspace", 3)
    return workspace


# ----------------------------------------------------------------------------- sizes

def embla_full_decode_workspace_size(shape: Shape) -> int:
    return library().embla_full_decode_workspace_size(ctypes.byref(shape.c()))


def embla_select_topk_workspace_size(shape: Shape, topk: int = 1024, recent: int = 128) -> int:
    return library().embla_select_topk_workspace_size(ctypes.byref(shape.c()), topk, recent)


def embla_sparse_decode_workspace_size(shape: Shape, idx_stride: int) -> int:
    return library().embla_sparse_decode_workspace_size(ctypes.byref(shape.c()), idx_stride)


def embla_device_sm_count() -> int:
    return library().embla_device_sm_count()


# ----------------------------------------------------------------------------- calls

def embla_full_decode(shape: Shape, q, k_cache, v_cache, out, n_surv, sel_scores=None,
                      sel_hist=None, alpha: float = 1.0, c: float = 1.0, eps: float = 1e-6,
                      workspace=None, stream=None):
    B, Hq, Hkv, D, ncap = shape.batch, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, \
        shape.cache_stride
    _check(q, torch.bfloat16, (B, Hq, D), "q")
    _check(k_cache, torch.bfloat16, (B, Hkv, ncap, D), "k_cache")
    _check(v_cache, torch.bfloat16, (B, Hkv, ncap, D), "v_cache")
    _check(out, torch.float32, (B, Hq, D), "out")
    _check(n_surv, torch.int32, (B, Hkv), "n_surv")
    _check(sel_scores, torch.float32, (B, Hkv, ncap), "sel_scores", allow_none=True)
    _check(sel_hist, torch.int32, (B, Hkv, HIST_BINS), "sel_hist", allow_none=True)
    ws = _workspace(embla_full_decode_workspace_size(shape), workspace, q.device)
    _call("embla_full_decode", ctypes.byref(shape.c()), _ptr(q), _ptr(k_cache), _ptr(v_cache),
          alpha, c, eps, _ptr(out), _ptr(n_surv), _ptr(sel_scores), _ptr(sel_hist), _ptr(ws),
          ws.numel() * ws.element_size(), _stream(stream))


def embla_full_decode_e4m3(shape: Shape, q, k_codes, k_scales, v_codes, v_scales, out, n_surv,
                           sel_scores=None, sel_hist=None, alpha: float = 1.0, c: float = 1.0,
                           eps: float = 1e-6, workspace=None, stream=None):
    """embla_full_decode over 8-bit caches: E4M3 codes (uint8 [B, Hkv, cache_stride, D]) with
    one fp32 scale per (token, KV head) (float32 [B, Hkv, cache_stride]); row j stands for
    scale * decode(codes).  cache_stride must be a multiple of 4."""
    B, Hq, Hkv, D, ncap = shape.batch, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, \
        shape.cache_stride
    _check(q, torch.bfloat16, (B, Hq, D), "q")
    _check(k_codes, torch.uint8, (B, Hkv, ncap, D), "k_codes")
    _check(k_scales, torch.float32, (B, Hkv, ncap), "k_scales")
    _check(v_codes, torch.uint8, (B, Hkv, ncap, D), "v_codes")
    _check(v_scales, torch.float32, (B, Hkv, ncap), "v_scales")
    _check(out, torch.float32, (B, Hq, D), "out")
    _check(n_surv, torch.int32, (B, Hkv), "n_surv")
    _check(sel_scores, torch.float32, (B, Hkv, ncap), "sel_scores", allow_none=True)
    _check(sel_hist, torch.int32, (B, Hkv, HIST_BINS), "sel_hist", allow_none=True)
    ws = _workspace(embla_full_decode_workspace_size(shape), workspace, q.device)
    _call("embla_full_decode_e4m3", ctypes.byref(shape.c()), _ptr(q), _ptr(k_codes),
          _ptr(k_scales), _ptr(v_codes), _ptr(v_scales), alpha, c, eps, _ptr(out), _ptr(n_surv),
          _ptr(sel_scores), _ptr(sel_hist), _ptr(ws), ws.numel() * ws.element_size(),
          _stream(stream))


def embla_full_decode_static_scratch(shape: Shape, q, k_cache, v_cache, out, n_surv,
                                     sel_scores=None, sel_hist=None, alpha: float = 1.0,
                                     c: float = 1.0, eps: float = 1e-6, stream=None):
    """embla_full_decode on the library's fixed per-device scratch: for callers that may not
    allocate device memory while decoding.  Neither this wrapper nor the library allocates;
    shapes needing more than FULL_DECODE_SCRATCH_BYTES of scratch raise EmblaError
    (workspace too small).  Calls that can overlap on one device share the scratch and race."""
    B, Hq, Hkv, D, ncap = shape.batch, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, \
        shape.cache_stride
    _check(q, torch.bfloat16, (B, Hq, D), "q")
    _check(k_cache, torch.bfloat16, (B, Hkv, ncap, D), "k_cache")
    _check(v_cache, torch.bfloat16, (B, Hkv, ncap, D), "v_cache")
    _check(out, torch.float32, (B, Hq, D), "out")
    _check(n_surv, torch.int32, (B, Hkv), "n_surv")
    _check(sel_scores, torch.float32, (B, Hkv, ncap), "sel_scores", allow_none=True)
    _check(sel_hist, torch.int32, (B, Hkv, HIST_BINS), "sel_hist", allow_none=True)
    _call("embla_full_decode_static_scratch", ctypes.byref(shape.c()), _ptr(q), _ptr(k_cache),
          _ptr(v_cache), alpha, c, eps, _ptr(out), _ptr(n_surv), _ptr(sel_scores),
          _ptr(sel_hist), _stream(stream))


def embla_select_topk(shape: Shape, sel_scores, sel_hist, idx, count, topk: int = 1024,
                      recent: int = 128, workspace=None, stream=None):
    B, Hkv, ncap = shape.batch, shape.n_kv_heads, shape.cache_stride
    _check(sel_scores, torch.float32, (B, Hkv, ncap), "sel_scores")
    _check(sel_hist, torch.int32, (B, Hkv, HIST_BINS), "sel_hist")
    _check(idx, torch.int32, None, "idx")
    if idx.dim() != 3 or tuple(idx.shape[:2]) != (B, Hkv):
        raise ValueError("idx must be [B, Hkv, idx_stride]")
    _check(count, torch.int32, (B, Hkv), "count")
    ws = _workspace(embla_select_topk_workspace_size(shape, topk, recent), workspace,
                    sel_scores.device)
    _call("embla_select_topk", ctypes.byref(shape.c()), _ptr(sel_scores), _ptr(sel_hist), topk,
          recent, _ptr(idx), idx.shape[2], _ptr(count), _ptr(ws), ws.numel() * ws.element_size(),
          _stream(stream))


def embla_append_kv(shape: Shape, pos: int, k_rows, v_rows, k_cache, v_cache, stream=None):
    """Write one token's K and V rows (bf16 [B, Hkv, D]) into row `pos` of every plane of the
    caches (bf16 [B, Hkv, cache_stride, D])."""
    B, Hkv, D, ncap = shape.batch, shape.n_kv_heads, shape.head_dim, shape.cache_stride
    _check(k_rows, torch.bfloat16, (B, Hkv, D), "k_rows")
    _check(v_rows, torch.bfloat16, (B, Hkv, D), "v_rows")
    _check(k_cache, torch.bfloat16, (B, Hkv, ncap, D), "k_cache")
    _check(v_cache, torch.bfloat16, (B, Hkv, ncap, D), "v_cache")
    _call("embla_append_kv", ctypes.byref(shape.c()), pos, _ptr(k_rows), _ptr(v_rows),
          _ptr(k_cache), _ptr(v_cache), _stream(stream))


def embla_append_kv_e4m3(shape: Shape, pos: int, k_code_rows, k_scale_rows, v_code_rows,
                         v_scale_rows, k_codes, k_scales, v_codes, v_scales, stream=None):
    """embla_append_kv for 8-bit caches: the token's E4M3 codes (uint8 [B, Hkv, D]) and scales
    (float32 [B, Hkv]) into row `pos` of the codes and scale arrays."""
    B, Hkv, D, ncap = shape.batch, shape.n_kv_heads, shape.head_dim, shape.cache_stride
    _check(k_code_rows, torch.uint8, (B, Hkv, D), "k_code_rows")
    _check(v_code_rows, torch.uint8, (B, Hkv, D), "v_code_rows")
    _check(k_scale_rows, torch.float32, (B, Hkv), "k_scale_rows")
    _check(v_scale_rows, torch.float32, (B, Hkv), "v_scale_rows")
    _check(k_codes, torch.uint8, (B, Hkv, ncap, D), "k_codes")
    _check(v_codes, torch.uint8, (B, Hkv, ncap, D), "v_codes")
    _check(k_scales, torch.float32, (B, Hkv, ncap), "k_scales")
    _check(v_scales, torch.float32, (B, Hkv, ncap), "v_scales")
    _call("embla_append_kv_e4m3", ctypes.byref(shape.c()), pos, _ptr(k_code_rows),
          _ptr(k_scale_rows), _ptr(v_code_rows), _ptr(v_scale_rows), _ptr(k_codes),
          _ptr(k_scales), _ptr(v_codes), _ptr(v_scales), _stream(stream))


def embla_full_decode_select_workspace_size(shape: Shape, topk: int = 1024, recent: int = 128) -> int:
    return library().embla_full_decode_select_workspace_size(ctypes.byref(shape.c()), topk, recent)


def _check_select_outputs(shape: Shape, idx, count):
    B, Hkv = shape.batch, shape.n_kv_heads
    _check(idx, torch.int32, None, "idx")
    if idx.dim() != 3 or tuple(idx.shape[:2]) != (B, Hkv):
        raise ValueError("idx must be [B, Hkv, idx_stride]")
    _check(count, torch.int32, (B, Hkv), "count")


def embla_full_decode_select(shape: Shape, q, k_cache, v_cache, out, n_surv, sel_scores, sel_hist,
                             idx, count, topk: int = 1024, recent: int = 128, alpha: float = 1.0,
                             c: float = 1.0, eps: float = 1e-6, workspace=None, stream=None):
    """embla_full_decode with sel_scores and sel_hist, then embla_select_topk on them, in one
    call (the selection starts as soon as the scores are complete)."""
    B, Hq, Hkv, D, ncap = shape.batch, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, \
        shape.cache_stride
    _check(q, torch.bfloat16, (B, Hq, D), "q")
    _check(k_cache, torch.bfloat16, (B, Hkv, ncap, D), "k_cache")
    _check(v_cache, torch.bfloat16, (B, Hkv, ncap, D), "v_cache")
    _check(out, torch.float32, (B, Hq, D), "out")
    _check(n_surv, torch.int32, (B, Hkv), "n_surv")
    _check(sel_scores, torch.float32, (B, Hkv, ncap), "sel_scores")
    _check(sel_hist, torch.int32, (B, Hkv, HIST_BINS), "sel_hist")
    _check_select_outputs(shape, idx, count)
    ws = _workspace(embla_full_decode_select_workspace_size(shape, topk, recent), workspace,
                    q.device)
    _call("embla_full_decode_select", ctypes.byref(shape.c()), _ptr(q), _ptr(k_cache),
          _ptr(v_cache), alpha, c, eps, _ptr(out), _ptr(n_surv), _ptr(sel_scores),
          _ptr(sel_hist), topk, recent, _ptr(idx), idx.shape[2], _ptr(count), _ptr(ws),
          ws.numel() * ws.element_size(), _stream(stream))


def embla_full_decode_e4m3_select(shape: Shape, q, k_codes, k_scales, v_codes, v_scales, out,
                                  n_surv, sel_scores, sel_hist, idx, count, topk: int = 1024,
                                  recent: int = 128, alpha: float = 1.0, c: float = 1.0,
                                  eps: float = 1e-6, workspace=None, stream=None):
    """embla_full_decode_e4m3 with its selection, as embla_full_decode_select."""
    B, Hq, Hkv, D, ncap = shape.batch, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, \
        shape.cache_stride
    _check(q, torch.bfloat16, (B, Hq, D), "q")
    _check(k_codes, torch.uint8, (B, Hkv, ncap, D), "k_codes")
    _check(k_scales, torch.float32, (B, Hkv, ncap), "k_scales")
    _check(v_codes, torch.uint8, (B, Hkv, ncap, D), "v_codes")
    _check(v_scales, torch.float32, (B, Hkv, ncap), "v_scales")
    _check(out, torch.float32, (B, Hq, D), "out")
    _check(n_surv, torch.int32, (B, Hkv), "n_surv")
    _check(sel_scores, torch.float32, (B, Hkv, ncap), "sel_scores")
    _check(sel_hist, torch.int32, (B, Hkv, HIST_BINS), "sel_hist")
    _check_select_outputs(shape, idx, count)
    ws = _workspace(embla_full_decode_select_workspace_size(shape, topk, recent), workspace,
                    q.device)
    _call("embla_full_decode_e4m3_select", ctypes.byref(shape.c()), _ptr(q), _ptr(k_codes),
          _ptr(k_scales), _ptr(v_codes), _ptr(v_scales), alpha, c, eps, _ptr(out), _ptr(n_surv),
          _ptr(sel_scores), _ptr(sel_hist), topk, recent, _ptr(idx), idx.shape[2], _ptr(count),
          _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


def embla_sparse_decode(shape: Shape, q, k_cache, v_cache, idx, count, out, tau: float | None = None,
                        workspace=None, stream=None):
    B, Hq, Hkv, D, ncap = shape.batch, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, \
        shape.cache_stride
    _check(q, torch.bfloat16, (B, Hq, D), "q")
    _check(k_cache, torch.bfloat16, (B, Hkv, ncap, D), "k_cache")
    _check(v_cache, torch.bfloat16, (B, Hkv, ncap, D), "v_cache")
    _check(idx, torch.int32, None, "idx")
    if idx.dim() != 3 or tuple(idx.shape[:2]) != (B, Hkv):
        raise ValueError("idx must be [B, Hkv, idx_stride]")
    _check(count, torch.int32, (B, Hkv), "count")
    _check(out, torch.float32, (B, Hq, D), "out")
    tau = D ** -0.5 if tau is None else tau
    ws = _workspace(embla_sparse_decode_workspace_size(shape, idx.shape[2]), workspace, q.device)
    _call("embla_sparse_decode", ctypes.byref(shape.c()), _ptr(q), _ptr(k_cache), _ptr(v_cache),
          _ptr(idx), idx.shape[2], _ptr(count), tau, _ptr(out), _ptr(ws),
          ws.numel() * ws.element_size(), _stream(stream))


def embla_sparse_decode_e4m3(shape: Shape, q, k_codes, k_scales, v_codes, v_scales, idx, count,
                             out, tau: float | None = None, workspace=None, stream=None):
    """embla_sparse_decode over the full layer's 8-bit caches (as for embla_full_decode_e4m3)."""
    B, Hq, Hkv, D, ncap = shape.batch, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, \
        shape.cache_stride
    _check(q, torch.bfloat16, (B, Hq, D), "q")
    _check(k_codes, torch.uint8, (B, Hkv, ncap, D), "k_codes")
    _check(k_scales, torch.float32, (B, Hkv, ncap), "k_scales")
    _check(v_codes, torch.uint8, (B, Hkv, ncap, D), "v_codes")
    _check(v_scales, torch.float32, (B, Hkv, ncap), "v_scales")
    _check(idx, torch.int32, None, "idx")
    if idx.dim() != 3 or tuple(idx.shape[:2]) != (B, Hkv):
        raise ValueError("idx must be [B, Hkv, idx_stride]")
    _check(count, torch.int32, (B, Hkv), "count")
    _check(out, torch.float32, (B, Hq, D), "out")
    tau = D ** -0.5 if tau is None else tau
    ws = _workspace(embla_sparse_decode_workspace_size(shape, idx.shape[2]), workspace, q.device)
    _call("embla_sparse_decode_e4m3", ctypes.byref(shape.c()), _ptr(q), _ptr(k_codes),
          _ptr(k_scales), _ptr(v_codes), _ptr(v_scales), _ptr(idx), idx.shape[2], _ptr(count),
          tau, _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


def embla_prefill_workspace_size(shape: Shape) -> int:
    return library().embla_prefill_workspace_size(ctypes.byref(shape.c()))


def embla_prefill(shape: Shape, q, k_cache, v_cache, out, alpha: float = 1.0, c: float = 1.0,
                  eps: float = 1e-6, workspace=None, stream=None):
    """Causal full-layer attention over the prompt: q bf16 [B, Hq, T, D] holds the queries of
    the last T of the ctx_len cached keys; out fp32 [B, Hq, T, D]."""
    B, Hq, Hkv, D, ncap = shape.batch, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, \
        shape.cache_stride
    _check(q, torch.bfloat16, None, "q")
    if q.dim() != 4 or tuple(q.shape[:2]) != (B, Hq) or q.shape[3] != D:
        raise ValueError("q must be [B, Hq, T, D]")
    T = q.shape[2]
    _check(k_cache, torch.bfloat16, (B, Hkv, ncap, D), "k_cache")
    _check(v_cache, torch.bfloat16, (B, Hkv, ncap, D), "v_cache")
    _check(out, torch.float32, (B, Hq, T, D), "out")
    ws = _workspace(embla_prefill_workspace_size(shape), workspace, q.device)
    _call("embla_prefill", ctypes.byref(shape.c()), T, _ptr(q), _ptr(k_cache), _ptr(v_cache),
          alpha, c, eps, _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


def embla_relu2_mlp_workspace_size(d: int, f: int) -> int:
    return library().embla_relu2_mlp_workspace_size(d, f)


def embla_relu2_mlp(x, w_up, w_down, y, n_live, workspace=None, stream=None):
    """One token through a ReLU^2 MLP: x bf16 [d], w_up and w_down bf16 [f, d] (row i =
    neuron i), y fp32 [d], n_live int32 [1] (neurons that fired)."""
    _check(x, torch.bfloat16, None, "x")
    if x.dim() != 1:
        raise ValueError("x must be [d]")
    d = x.shape[0]
    _check(w_up, torch.bfloat16, None, "w_up")
    if w_up.dim() != 2 or w_up.shape[1] != d:
        raise ValueError("w_up must be [f, d]")
    f = w_up.shape[0]
    _check(w_down, torch.bfloat16, (f, d), "w_down")
    _check(y, torch.float32, (d,), "y")
    _check(n_live, torch.int32, (1,), "n_live")
    ws = _workspace(embla_relu2_mlp_workspace_size(d, f), workspace, x.device)
    _call("embla_relu2_mlp", d, f, _ptr(x), _ptr(w_up), _ptr(w_down), _ptr(y), _ptr(n_live),
          _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


def embla_full_decode_head_scores(shape: Shape, q, k_cache, v_cache, out, n_surv, head_scores,
                                  head_hist, alpha: float = 1.0, c: float = 1.0, eps: float = 1e-6,
                                  workspace=None, stream=None):
    """embla_full_decode writing every query head's own scores: head_scores fp32
    [B, Hq, cache_stride], head_hist int32 [B, Hq, 2048]."""
    B, Hq, Hkv, D, ncap = shape.batch, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, \
        shape.cache_stride
    _check(q, torch.bfloat16, (B, Hq, D), "q")
    _check(k_cache, torch.bfloat16, (B, Hkv, ncap, D), "k_cache")
    _check(v_cache, torch.bfloat16, (B, Hkv, ncap, D), "v_cache")
    _check(out, torch.float32, (B, Hq, D), "out")
    _check(n_surv, torch.int32, (B, Hkv), "n_surv")
    _check(head_scores, torch.float32, (B, Hq, ncap), "head_scores")
    _check(head_hist, torch.int32, (B, Hq, HIST_BINS), "head_hist")
    ws = _workspace(embla_full_decode_workspace_size(shape), workspace, q.device)
    _call("embla_full_decode_head_scores", ctypes.byref(shape.c()), _ptr(q), _ptr(k_cache),
          _ptr(v_cache), alpha, c, eps, _ptr(out), _ptr(n_surv), _ptr(head_scores),
          _ptr(head_hist), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))


def embla_select_topk_per_head(shape: Shape, head_scores, head_hist, idx, count, topk: int = 1024,
                               recent: int = 128, workspace=None, stream=None):
    """Each query head's own top-k + recent: idx int32 [B, Hq, stride], count int32 [B, Hq]."""
    B, Hq, ncap = shape.batch, shape.n_q_heads, shape.cache_stride
    _check(head_scores, torch.float32, (B, Hq, ncap), "head_scores")
    _check(head_hist, torch.int32, (B, Hq, HIST_BINS), "head_hist")
    _check(idx, torch.int32, None, "idx")
    if idx.dim() != 3 or tuple(idx.shape[:2]) != (B, Hq):
        raise ValueError("idx must be [B, Hq, idx_stride]")
    _check(count, torch.int32, (B, Hq), "count")
    nbytes = library().embla_select_topk_per_head_workspace_size(ctypes.byref(shape.c()), topk,
                                                                 recent)
    ws = _workspace(nbytes, workspace, head_scores.device)
    _call("embla_select_topk_per_head", ctypes.byref(shape.c()), _ptr(head_scores),
          _ptr(head_hist), topk, recent, _ptr(idx), idx.shape[2], _ptr(count), _ptr(ws),
          ws.numel() * ws.element_size(), _stream(stream))


def embla_sparse_decode_per_head(shape: Shape, q, k_cache, v_cache, idx, count, out,
                                 tau: float | None = None, workspace=None, stream=None):
    """embla_sparse_decode where query head h reads its own selection idx[b, h]."""
    B, Hq, Hkv, D, ncap = shape.batch, shape.n_q_heads, shape.n_kv_heads, shape.head_dim, \
        shape.cache_stride
    _check(q, torch.bfloat16, (B, Hq, D), "q")
    _check(k_cache, torch.bfloat16, (B, Hkv, ncap, D), "k_cache")
    _check(v_cache, torch.bfloat16, (B, Hkv, ncap, D), "v_cache")
    _check(idx, torch.int32, None, "idx")
    if idx.dim() != 3 or tuple(idx.shape[:2]) != (B, Hq):
        raise ValueError("idx must be [B, Hq, idx_stride]")
    _check(count, torch.int32, (B, Hq), "count")
    _check(out, torch.float32, (B, Hq, D), "out")
    tau = D ** -0.5 if tau is None else tau
    ws = _workspace(embla_sparse_decode_workspace_size(shape, idx.shape[2]), workspace, q.device)
    _call("embla_sparse_decode_per_head", ctypes.byref(shape.c()), _ptr(q), _ptr(k_cache),
          _ptr(v_cache), _ptr(idx), idx.shape[2], _ptr(count), tau, _ptr(out), _ptr(ws),
          ws.numel() * ws.element_size(), _stream(stream))


def embla_window_decode(shape: Shape, q, k_win, v_win, pos: int, out, window: int = 128,
                        rope_base: float = 10000.0, tau: float | None = None, stream=None):
    B, Hq, Hkv, D = shape.batch, shape.n_q_heads, shape.n_kv_heads, shape.head_dim
    _check(q, torch.bfloat16, (B, Hq, D), "q")
    _check(k_win, torch.bfloat16, (B, Hkv, window, D), "k_win")
    _check(v_win, torch.bfloat16, (B, Hkv, window, D), "v_win")
    _check(out, torch.float32, (B, Hq, D), "out")
    tau = D ** -0.5 if tau is None else tau
    _call("embla_window_decode", ctypes.byref(shape.c()), _ptr(q), _ptr(k_win), _ptr(v_win),
          window, pos, rope_base, tau, _ptr(out), None, 0, _stream(stream))


def embla_skip_stats(shape: Shape, sel_scores, keys_needed, chunks_needed, chunk: int = 8,
                     stream=None):
    """Per unit: keys whose V row is needed (sigma > 0) and chunks of `chunk` keys that
    hold at least one of them."""
    B, Hkv, ncap = shape.batch, shape.n_kv_heads, shape.cache_stride
    _check(sel_scores, torch.float32, (B, Hkv, ncap), "sel_scores")
    _check(keys_needed, torch.int32, (B, Hkv), "keys_needed")
    _check(chunks_needed, torch.int32, (B, Hkv), "chunks_needed")
    _call("embla_skip_stats", ctypes.byref(shape.c()), _ptr(sel_scores), chunk, _ptr(keys_needed),
          _ptr(chunks_needed), _stream(stream))


def embla_self_test_wait_limit(limit_us: int, arrive: bool = False, stream=None):
    """Run the bounded-wait error path on the device (see the header): a wait that nothing
    completes gives up after limit_us and sets bit 1 of the check word."""
    _call("embla_self_test_wait_limit", limit_us, 1 if arrive else 0, _stream(stream))


def embla_device_check(clear: bool = True, stream=None) -> int:
    """Synchronise and return the device-side check flags (bit 0: index range, bit 1: wait timeout)."""
    flags = ctypes.c_uint32(0)
    library().embla_device_check(ctypes.byref(flags), 1 if clear else 0, _stream(stream))
    return flags.value
