"""Shared test plumbing: moving generator arrays to the GPU and running the library."""
import numpy as np
import torch

import relu_sparse_kv_gb300 as E

ATOL, RTOL = 2e-3, 1e-2

# Worst share of the tolerance used per comparison kind: max |gpu - ref| / (atol + rtol |ref|)
# (1.0 is the limit).  Filled by assert_close, printed at the end of the run.
MARGINS = {}


def to_dev(a, dev="cuda"):
    """bf16 bit patterns (uint16 numpy) -> torch bf16 on the device."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def assert_close(gpu, ref, atol=ATOL, rtol=RTOL, what="output"):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    err = np.abs(gpu - ref)
    lim = atol + rtol * np.abs(ref)
    if err.size:
        use = float(np.nanmax(np.where(np.isnan(err), np.inf, err / lim)))
        key = what.split(" unit")[0].split(" of head")[0].split(" row")[0]
        MARGINS[key] = max(MARGINS.get(key, 0.0), use)
    bad = ~(err <= lim)
    assert not bad.any(), (f"{what}: {int(bad.sum())}/{bad.size} out of tolerance; "
                           f"max abs err {np.nanmax(err):.3e}")


class FullRun:
    """Full layer + selection on the GPU for one generated layer."""

    def __init__(self, fl, n_cap=None, alpha=1.0, c=1.0, eps=1e-6, topk=1024, recent=128,
                 with_select=True):
        B, Hq, D = fl.q.shape
        Hkv, ncap = fl.K.shape[1], fl.K.shape[2]
        self.shape = E.Shape(B, Hq, Hkv, D, fl.n, ncap)
        dev = "cuda"
        self.q, self.K, self.V = to_dev(fl.q), to_dev(fl.K), to_dev(fl.V)
        self.out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=dev)
        self.n_surv = torch.full((B, Hkv), -1, dtype=torch.int32, device=dev)
        self.sel = torch.full((B, Hkv, ncap), float("nan"), dtype=torch.float32, device=dev)
        self.hist = torch.full((B, Hkv, E.HIST_BINS), -1, dtype=torch.int32, device=dev)
        E.embla_full_decode(self.shape, self.q, self.K, self.V, self.out, self.n_surv, self.sel,
                            self.hist, alpha=alpha, c=c, eps=eps)
        self.stride = topk + recent
        if with_select:
            self.idx = torch.full((B, Hkv, self.stride), -7, dtype=torch.int32, device=dev)
            self.count = torch.full((B, Hkv), -1, dtype=torch.int32, device=dev)
            E.embla_select_topk(self.shape, self.sel, self.hist, self.idx, self.count, topk=topk,
                                recent=recent)
        torch.cuda.synchronize()
        assert E.embla_device_check() == 0

    def sparse(self, q_sparse, tau=None):
        B, Hq, D = q_sparse.shape
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        E.embla_sparse_decode(self.shape, to_dev(q_sparse), self.K, self.V, self.idx, self.count,
                              out, tau=tau)
        torch.cuda.synchronize()
        assert E.embla_device_check() == 0
        return out.cpu().numpy()


def order_key_np(x):
    """Order-preserving uint32 key of float32 values (-0 folded onto +0)."""
    x = np.where(x == 0, np.float32(0), x).astype(np.float32)
    b = x.view(np.uint32)
    return np.where(b & 0x80000000, ~b, b | 0x80000000).astype(np.uint32)
