"""Decode-attention benchmark for the Embla 1 layer types on GB300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl reference]

One step is one decode token for every sequence of the batch through the whole hot
path of the workload: the full (ReLU^2) layer, its top-1024 + recent-128 selection
and the sparse layers that reuse it (and, for the whole-model workload, every window
layer).  Default workload: batch 8, context 32,768, 16 query / 4 KV heads, head_dim
128, 5% of keys scoring above zero, three sparse layers.

The timed steps replay CUDA graphs of the library's C-ABI calls on device-resident
inputs.  Prints one JSON line (rank 0).  --impl reference times the fp64 CPU oracle
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attention tokens/s and needed-byte HBM GB/s (% of roofline) at 32k–128k"
MLP_METRIC = "ReLU^2 MLP batch-1 tokens/s and needed-byte HBM GB/s (% of roofline)"
PREFILL_METRIC = "full-layer prefill tokens/s (causal ReLU^2 attention over the prompt) and TFLOP/s (% of bf16 tensor peak)"
ROW_BYTES = 128 * 2          # one bf16 key or value row (head_dim 128)
ROW_BYTES_E4M3 = 128 + 4     # one 8-bit row (E4M3 codes) and its fp32 scale
TOPK, RECENT = 1024, 128
L2_BYTES = 129 * 10**6       # GB300 L2


def replicas_for(step_bytes: int) -> int:
    """Copies of the caches that the timed steps rotate through, so a step's cache rows
    were last touched at least 1.5 L2 sizes of other reads ago (1 when a step alone
    reads that much)."""
    if step_bytes >= 1.5 * L2_BYTES:
        return 1
    return 1 + -(-int(1.5 * L2_BYTES) // max(1, step_bytes))


def row_bytes(kv: str) -> int:
    return ROW_BYTES_E4M3 if kv == "e4m3" else ROW_BYTES


# ----------------------------------------------------------------------------- accounting

def state_bytes(c: int, batch: int, bytes_per_elem: int, d_kv: int, tokens: int, layers: int) -> int:
    """Cache state M_state = c * B * b * d_kv * L_kv * n_ret (c = 2 for separate K and V)."""
    return c * batch * bytes_per_elem * d_kv * tokens * layers


def full_layer_needed_bytes(units: int, n: int, total_survivors: int, kv: str = "bf16") -> int:
    """Bytes a full layer must read: every K row, and the V rows of surviving keys only
    (8-bit caches: each row's scale with it)."""
    return units * n * row_bytes(kv) + total_survivors * row_bytes(kv)


def sparse_layer_needed_bytes(total_selected: int, kv: str = "bf16") -> int:
    """Bytes a sparse layer must read: the selected K and V rows."""
    return 2 * total_selected * row_bytes(kv)


def window_layer_needed_bytes(units: int, valid_rows: int) -> int:
    return 2 * units * valid_rows * ROW_BYTES


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _traffic_from_profile(workload_key: str, src_digest: str):
    """DRAM bytes per launch of the full-layer kernel, as an ncu capture measured them
    (profiles/full_decode_traffic.json: one record per workload with the digest of the
    kernel source it was taken on).  None when no record matches the current source."""
    path = os.path.join(ROOT, "profiles", "full_decode_traffic.json")
    try:
        with open(path) as f:
            records = json.load(f)["records"]
    except (OSError, ValueError, KeyError):
        return None
    for rec in records:
        if rec.get("workload") == workload_key and rec.get("src") == src_digest:
            return float(rec["bytes_per_launch"])
    return None


def _kernel_digest() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ("full_decode.cu", "ptx.cuh", "internal.h"):
        with open(os.path.join(ROOT, "relu_sparse_kv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(device_index)], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = _dt.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        window = [r for r in rows if t0 - 0.15 <= r[0] <= t1 + 0.15] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in window for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in window),
                "sm_max_mhz": max(r[2] for r in window), "reasons": reasons,
                "samples": len(window)}


# ----------------------------------------------------------------------------- workload

def workload_name(cfg, batch=None, ctx=None) -> str:
    if batch is None and ctx is None:
        return cfg["name"]
    return cfg["name"] + f" (overridden: batch {batch}, ctx {ctx})"


def prefill_flops(B: int, Hq: int, n: int, T: int) -> float:
    """Algorithmic flops of a causal prefill: Q K^T and P V once each over the (query, key)
    pairs with key <= query position, 2 flops per multiply-add, D = 128."""
    pairs = T * (n - T) + T * (T + 1) / 2
    return 4.0 * 128 * pairs * B * Hq


def static_config(cfg_id: int, batch=None, ctx=None) -> dict:
    """The workload's description, the same on both arms."""
    import gen
    cfg = gen.CONFIGS[cfg_id]
    if cfg.get("kind") == "mlp":
        return {"workload": cfg["name"], "batch": 1, "width": cfg["d"], "neurons": cfg["f"],
                "live_fraction": cfg["live"], "weights": "bf16", "accumulate": "f32"}
    if cfg.get("kind") == "prefill":
        n = cfg["n"] if ctx is None else ctx
        return {"workload": workload_name(cfg, batch, ctx),
                "batch": cfg["B"] if batch is None else batch, "ctx_len": n,
                "prompt_tokens": min(cfg["T"], n), "q_heads": cfg.get("Hq", gen.HQ),
                "kv_heads": cfg.get("Hkv", gen.HKV), "head_dim": gen.HEAD_DIM,
                "kv_cache": "bf16", "causal": True, "accumulate": "f32"}
    if cfg_id == 5:
        fulls = [len(gen.EMBLA_SPARSE_OF[layer]) for layer in gen.EMBLA_FULL_LAYERS]
        wins = list(gen.EMBLA_WINDOW_LAYERS)
    else:
        fulls, wins = [len(cfg["sparse"])], []
    return {"workload": workload_name(cfg, batch, ctx),
            "batch": cfg["B"] if batch is None else batch,
            "ctx_len": cfg["n"] if ctx is None else ctx,
            "q_heads": cfg.get("Hq", gen.HQ), "kv_heads": cfg.get("Hkv", gen.HKV),
            "head_dim": gen.HEAD_DIM, "kv_cache": cfg.get("kv", "bf16"),
            "full_layers": len(fulls), "sparse_layers": sum(fulls),
            "window_layers": len(wins), "accumulate": "f32"}


def omp_threads() -> int:
    """Threads the oracle's OpenMP loops use on this host."""
    env = os.environ.get("OMP_NUM_THREADS")
    if env and env.split(",")[0].strip().isdigit():
        return int(env.split(",")[0])
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def load_workload(cfg: int, seed: int = 0, batch=None, ctx=None):
    import gen
    fls = list(gen.config_full_layers(cfg, seed=seed, B=batch, n=ctx))
    wls = list(gen.config_window_layers(cfg, seed=seed, B=batch, n=ctx))
    return fls, wls


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _graph_events_work(torch, stream) -> bool:
    """Whether timing events can be recorded inside a captured CUDA graph (PyTorch's
    external events) and read back after a replay."""
    try:
        a = torch.cuda.Event(enable_timing=True, external=True)
        b = torch.cuda.Event(enable_timing=True, external=True)
        x = torch.zeros(1024, device=stream.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                a.record(stream)
                x.add_(1.0)
                b.record(stream)
            g.replay()
        torch.cuda.synchronize()
        return a.elapsed_time(b) >= 0.0
    except Exception:
        return False


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of every rank's x (x itself on one rank).  The timed regions of all ranks
    are bracketed by barriers, so the slowest rank's time is the job's time."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, batch: int, seconds_per_step: float) -> float:
    """Weak scaling: every rank decodes its own batch of `batch` sequences per step, so the
    job's tokens/s is world * batch over the slowest rank's step time."""
    return world * batch / seconds_per_step


def _oracle_kv(oracle, fl):
    """The layer's caches as float64 for the oracle (8-bit caches decoded: scale * code)."""
    if fl.kv == "e4m3":
        return oracle.dequant_e4m3(fl.K, fl.Ks), oracle.dequant_e4m3(fl.V, fl.Vs)
    return oracle.f64(fl.K), oracle.f64(fl.V)


def run_reference(args):
    """The fp64 CPU oracle on a bounded sample: every layer of the step for a few sequences."""
    world, rank, _ = _dist()
    if rank != 0:
        return 0
    import numpy as np
    import gen
    import oracle

    cfg = gen.CONFIGS[args.config]
    if cfg.get("kind") == "prefill":
        return run_reference_prefill(args, cfg)
    if cfg.get("kind") == "mlp":
        return run_reference_mlp(args, cfg)
    cores = omp_threads()
    oracle.set_threads(cores)
    if args.config == 5:
        # the whole-model step: every layer of the step for one of its sixteen sequences
        sample_b = 1
        fls = list(gen.config_full_layers(args.config, seed=0, B=sample_b))
        wls = list(gen.config_window_layers(args.config, seed=0, B=sample_b))
        prep = []
        for fl in fls:
            K, V = _oracle_kv(oracle, fl)
            prep.append((oracle.f64(fl.q), K, V, [oracle.f64(qs) for qs in fl.sparse_q], fl.n))
        wprep = [(oracle.f64(w.q), oracle.f64(w.K), oracle.f64(w.V), w.pos) for w in wls]
        sample = f"{sample_b} of {cfg['B']} sequences, every layer of the step"
    else:
        # the same work as the GPU step: the whole batch, every layer of the step
        sample_b = cfg["B"]
        prep = [_oracle_step_inputs(args.config, sample_b)]
        wprep = []
        sample = f"all {sample_b} sequences, every layer of the step"

    def step():
        for p in prep:
            _oracle_layer_step(*p)
        for q, K, V, pos in wprep:
            oracle.window_decode_batch(q, K, V, pos)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = sample_b * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": static_config(args.config),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def prefill_oracle_sample(cfg_id: int, rows: int):
    """The oracle's prefill of the last `rows` prompt tokens of sequence 0 (every head): those
    rows see the most keys, so their rate is the slowest the oracle runs."""
    import gen
    import oracle
    q, K, V = gen.config_prefill(cfg_id, seed=0, B=1)
    n = K.shape[2]
    qs = oracle.f64(q[:, :, -rows:])
    Kd, Vd = oracle.f64(K), oracle.f64(V)

    def run():
        oracle.prefill_batch(qs, Kd, Vd, n)
    return run


def run_reference_prefill(args, cfg):
    import gen
    rows = 8
    run = prefill_oracle_sample(args.config, rows)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = rows * args.steps / dt
    line = {
        "impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": static_config(args.config),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": omp_threads(),
                         "kind": "oracle",
                         "sample": f"the last {rows} prompt tokens of sequence 0, every head"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def cpu_baseline_prefill(cfg_id: int, budget_s: float = 12.0):
    rows = 8
    run = prefill_oracle_sample(cfg_id, rows)
    reps = 0
    t0 = time.perf_counter()
    while True:
        run()
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": rows * reps / dt, "unit": "tokens/s", "cores": omp_threads(), "kind": "oracle",
            "sample": f"{reps} pass(es) over the last {rows} prompt tokens of sequence 0 (the rows "
                      "with the most keys), every head", "seconds": round(dt, 2)}


def bench_prefill(args, cfg):
    """One step = one embla_prefill call over the whole prompt of every sequence."""
    import numpy as np
    import torch
    import gen
    import relu_sparse_kv_gb300 as E

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    q_h, K_h, V_h = gen.config_prefill(args.config, seed=rank, B=args.batch, n=args.ctx)
    B, Hq, T, D = q_h.shape
    Hkv, n = K_h.shape[1], K_h.shape[2]

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    shape = E.Shape(B, Hq, Hkv, D, n, n)
    step_bytes = (q_h.size + K_h.size + V_h.size) * 2 + B * Hq * T * D * 4
    n_rep = replicas_for(step_bytes)
    reps = [dict(q=bf(q_h), K=bf(K_h), V=bf(V_h), out=torch.empty(B, Hq, T, D, device=dev))]
    for _ in range(n_rep - 1):
        reps.append({k: v.clone() for k, v in reps[0].items()})
    ws = torch.empty(max(16, E.embla_prefill_workspace_size(shape)), dtype=torch.uint8, device=dev)

    def call(r):
        E.embla_prefill(shape, r["q"], r["K"], r["V"], r["out"], alpha=1.0, c=1.0, eps=1e-6,
                        workspace=ws)

    for r in reps:
        call(r)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0
    stream = torch.cuda.Stream(device=dev)
    graphs = []
    with torch.cuda.stream(stream):
        for r in reps:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                call(r)
            graphs.append(g)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % n_rep].replay()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        t_wall0 = time.time()
        for i in range(args.steps):
            ev[i][0].record(stream)
            graphs[i % n_rep].replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop(t_wall0, t_wall1)
    ms = ev[0][0].elapsed_time(ev[-1][1])
    call_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    assert E.embla_device_check() == 0
    ms = max_over_ranks(ms, world, dev)
    ms_per_step = ms / args.steps
    value = world * B * T / (ms_per_step * 1e-3)

    e2e = None
    if args.e2e_steps > 0:
        h_q = reps[0]["q"].cpu().pin_memory()
        h_out = torch.empty_like(reps[0]["out"], device="cpu").pin_memory()
        h2d = h_q.numel() * h_q.element_size()
        d2h = h_out.numel() * h_out.element_size()

        def e2e_step(k):
            r = reps[k % n_rep]
            r["q"].copy_(h_q, non_blocking=True)
            call(r)
            h_out.copy_(r["out"], non_blocking=True)
            torch.cuda.current_stream().synchronize()

        for k in range(3):
            e2e_step(k)
        steps = max(3, min(args.e2e_steps, 20))
        t0 = time.perf_counter()
        for k in range(steps):
            e2e_step(k)
        dt = max_over_ranks(time.perf_counter() - t0, world, dev)
        e2e = {"value": world * B * T / (dt / steps), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": steps,
               "inputs": "per-step queries from pinned host memory, outputs back to host; the "
                         "KV caches stay resident in HBM"}

    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    peak = peaks.get("bf16_tflops_sustained")
    peak_src = "measured bf16_tflops_sustained (MEASURED_PEAKS.json; the timed region is a long run of back-to-back calls)"
    if not peak:
        peak, peak_src = 1700.0, "fallback 1.7 PFLOP/s sustained"
    flops = prefill_flops(B, Hq, n, T)
    ach = flops / (call_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": "prefill_kernel (one embla_prefill call: key-norm kernel + attention kernel)",
                "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s", "frac": round(ach / peak, 4),
                "peak_source": peak_src, "traffic": None, "algorithmic_flops_per_launch": flops,
                "launch_ms": round(call_ms, 5)}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_prefill(args.config)
    line = {
        "metric": PREFILL_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {**static_config(args.config, args.batch, args.ctx),
                   "launch": "one CUDA graph per call; events around each replay",
                   "l2": (f"not flushed: the steps rotate through {n_rep} copies of q, K, V and out "
                          f"({step_bytes / 1e6:.0f} MB each)" if n_rep > 1 else
                          f"not flushed: inputs and output larger than L2 ({step_bytes / 1e6:.0f} MB)")},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": 2 * args.steps, "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def mlp_oracle_step(cfg_id: int):
    import gen
    import oracle
    x, wu, wd, _ = gen.config_mlp(cfg_id, seed=0)
    xf, wuf, wdf = oracle.f64(x), oracle.f64(wu), oracle.f64(wd)

    def run():
        oracle.relu2_mlp(xf, wuf, wdf)
    return run


def run_reference_mlp(args, cfg):
    run = mlp_oracle_step(args.config)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = args.steps / dt
    line = {
        "impl": "reference", "metric": MLP_METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": static_config(args.config),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": "the whole token (one thread: the oracle's MLP is one loop)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


MLP_LAYERS = 32  # calls per CUDA graph: the MLPs of a 32-layer decoder, one after another


def bench_mlp(args, cfg):
    """One step = one embla_relu2_mlp call: one token through one MLP.  The calls run in CUDA
    graphs of MLP_LAYERS consecutive calls (one per layer of a decoder step, each on its own
    copy of the weights in turn), as a model's decode step launches them; the time of a call
    in a graph of its own is reported beside it."""
    import numpy as np
    import torch
    import gen
    import relu_sparse_kv_gb300 as E

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    x_h, wu_h, wd_h, mask = gen.config_mlp(args.config, seed=rank)
    d, f = x_h.shape[0], wu_h.shape[0]

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    n_live = int(mask.sum())
    needed = f * d * 2 + n_live * d * 2 + d * 2 + d * 4
    n_rep = replicas_for(needed)
    reps = [dict(x=bf(x_h), wu=bf(wu_h), wd=bf(wd_h), y=torch.empty(d, device=dev),
                 nl=torch.empty(1, dtype=torch.int32, device=dev))]
    for _ in range(n_rep - 1):
        reps.append({k: v.clone() for k, v in reps[0].items()})
    ws = torch.empty(max(16, E.embla_relu2_mlp_workspace_size(d, f)), dtype=torch.uint8, device=dev)

    def call(r):
        E.embla_relu2_mlp(r["x"], r["wu"], r["wd"], r["y"], r["nl"], workspace=ws)

    for r in reps:
        call(r)
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0
    assert int(reps[0]["nl"].item()) == n_live
    stream = torch.cuda.Stream(device=dev)

    def capture(ncalls, first):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(ncalls):
                call(reps[(first + i) % n_rep])
        return g

    # the timed steps: K // MLP_LAYERS replays of a graph of MLP_LAYERS calls, then one graph
    # of the K % MLP_LAYERS calls left; a graph of a single call for comparison
    full_n, rem_n = divmod(args.steps, MLP_LAYERS)
    with torch.cuda.stream(stream):
        g_layers = capture(MLP_LAYERS, 0)
        g_rem = capture(rem_n, MLP_LAYERS) if rem_n else None
        g_one = [capture(1, k) for k in range(n_rep)]
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    with torch.cuda.stream(stream):
        for i in range(max(1, args.warmup // MLP_LAYERS)):
            g_layers.replay()
        for i in range(args.warmup):
            g_one[i % n_rep].replay()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        t_wall0 = time.time()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for i in range(full_n):
            g_layers.replay()
        if g_rem is not None:
            g_rem.replay()
        end.record(stream)
        torch.cuda.synchronize()
        t_wall1 = time.time()
        one = []
        for i in range(2 * n_rep):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g_one[i % n_rep].replay()
            b.record(stream)
            one.append((a, b))
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop(t_wall0, t_wall1)
    ms = max_over_ranks(start.elapsed_time(end), world, dev)
    ms_per_step = ms / args.steps
    call_ms = ms_per_step
    one_call_us = statistics.median(a.elapsed_time(b) for a, b in one) * 1e3
    value = world / (ms_per_step * 1e-3)
    e2e = None
    if args.e2e_steps > 0:
        h_x = reps[0]["x"].cpu().pin_memory()
        h_y = torch.empty(d, device="cpu").pin_memory()

        def e2e_step(k):
            r = reps[k % n_rep]
            r["x"].copy_(h_x, non_blocking=True)
            call(r)
            h_y.copy_(r["y"], non_blocking=True)
            torch.cuda.current_stream().synchronize()

        for k in range(3):
            e2e_step(k)
        t0 = time.perf_counter()
        for k in range(args.e2e_steps):
            e2e_step(k)
        dt_eager = max_over_ranks(time.perf_counter() - t0, world, dev)
        # the same step as one CUDA graph (copy in, call, copy out), then a host synchronise
        e2e_graphs = []
        with torch.cuda.stream(stream):
            for k in range(n_rep):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    r = reps[k]
                    r["x"].copy_(h_x, non_blocking=True)
                    call(r)
                    h_y.copy_(r["y"], non_blocking=True)
                e2e_graphs.append(g)
            for k in range(3):
                e2e_graphs[k % n_rep].replay()
                stream.synchronize()
            t0 = time.perf_counter()
            for k in range(args.e2e_steps):
                e2e_graphs[k % n_rep].replay()
                stream.synchronize()
            dt = max_over_ranks(time.perf_counter() - t0, world, dev)
        e2e = {"value": world * args.e2e_steps / dt, "unit": "tokens/s",
               "h2d_bytes_per_step": d * 2, "d2h_bytes_per_step": d * 4, "steps": args.e2e_steps,
               "launch": "per step one CUDA graph of the copy in, the public API call and the copy "
                         "out, then a host synchronise",
               "eager_value": world * args.e2e_steps / dt_eager,
               "eager_launch": "the public API called from Python per step, copies issued eagerly, "
                               "then a host synchronise",
               "inputs": "the token from pinned host memory, y back to host; weights resident"}
    peak, peak_src = _peaks()
    ach = needed / (call_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": "relu2_mlp_kernel (one embla_relu2_mlp call: fused kernel + combine, "
                                          "the average call of the timed graphs)",
                "achieved": round(ach, 1), "peak": peak, "unit": "GB/s", "frac": round(ach / peak, 4),
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback 6.8 TB/s",
                "traffic": None, "algorithmic_bytes_per_launch": needed, "launch_ms": round(call_ms, 5)}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        run = mlp_oracle_step(args.config)
        reps_cpu, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < 5.0:
            run()
            reps_cpu += 1
        dt = time.perf_counter() - t0
        cpu = {"value": reps_cpu / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"{reps_cpu} whole tokens (the oracle's MLP is one loop on one thread)",
               "seconds": round(dt, 2)}
    line = {
        "metric": MLP_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {**static_config(args.config),
                   "launch": f"CUDA graphs of {MLP_LAYERS} consecutive calls (one per layer of a decoder "
                             f"step), events around the timed region; ms_per_step = its time / steps",
                   "one_call_graph_us": round(one_call_us, 2),
                   "one_call_graph": "median time of one call in a CUDA graph of its own (events around "
                                     "each replay): mostly the graph's launch",
                   "l2": f"not flushed: the steps rotate through {n_rep} copies of the weights",
                   "needed_bytes_per_step": needed,
                   "needed_gbs": round(needed / (ms_per_step * 1e-3) / 1e9, 1),
                   "live_neurons": n_live,
                   "down_projection_bytes_skipped": round(1.0 - n_live / f, 5)},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": 2 * args.steps, "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def _oracle_step_inputs(cfg_id: int, B: int):
    """One full layer of a workload (the first of config 5) widened for the oracle once:
    (q, K, V, sparse queries, n)."""
    import gen
    import oracle
    fl = next(gen.config_full_layers(cfg_id, seed=0, B=B))
    K, V = _oracle_kv(oracle, fl)
    return oracle.f64(fl.q), K, V, [oracle.f64(x) for x in fl.sparse_q], fl.n


def _oracle_layer_step(q, K, V, qss, n):
    """The oracle as it stands over one full layer of the batch: full layer, selection and
    the sparse layers that reuse it."""
    import oracle
    _, sig, _ = oracle.full_decode_batch(q, K, V, n)
    if qss:
        idx, cnt = oracle.select_topk_batch(sig, n)
        for qs in qss:
            oracle.sparse_decode_batch(qs, K, V, idx, cnt)


def _time_passes(fn, budget_s: float):
    reps, t0 = 0, time.perf_counter()
    while True:
        fn()
        reps += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return reps, time.perf_counter() - t0


def cpu_baseline(cfg_id: int, budget_s: float = 8.0):
    """The oracle as it stands, on this host's cores, over the whole batch of one full layer
    step (full + selection + its sparse layers), repeated for ~budget_s: once with every
    core (OpenMP over the (sequence, KV head) units) and once on a single thread."""
    import gen
    import oracle

    cfg = gen.CONFIGS[cfg_id]
    B = cfg["B"] if cfg_id != 5 else 1
    inp = _oracle_step_inputs(cfg_id, B)
    cores = omp_threads()
    oracle.set_threads(cores)
    reps, dt = _time_passes(lambda: _oracle_layer_step(*inp), budget_s)
    prev = oracle.set_threads(1)
    reps1, dt1 = _time_passes(lambda: _oracle_layer_step(*inp), budget_s)
    oracle.set_threads(prev)
    what = (f"full layer + selection + {len(inp[3])} sparse layer(s) over {B} sequence(s)"
            + (" (one of the five full-layer blocks)" if cfg_id == 5 else ""))
    return {"value": B * reps / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} pass(es) of {what}", "seconds": round(dt, 2),
            "single_thread": {"value": B * reps1 / dt1, "unit": "tokens/s", "cores": 1,
                              "sample": f"{reps1} pass(es) of the same", "seconds": round(dt1, 2)}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch (profiling)")
    ap.add_argument("--ctx", type=int, default=None, help="override the workload's context (profiling)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch
    import gen
    import relu_sparse_kv_gb300 as E

    if gen.CONFIGS[args.config].get("kind") == "prefill":
        return bench_prefill(args, gen.CONFIGS[args.config])
    if gen.CONFIGS[args.config].get("kind") == "mlp":
        return bench_mlp(args, gen.CONFIGS[args.config])
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    cfg = gen.CONFIGS[args.config]
    fls, wls = load_workload(args.config, seed=rank, batch=args.batch, ctx=args.ctx)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    def to_dev_raw(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    per_head = cfg.get("select") == "per_head"
    layers = []
    for fl in fls:
        B, Hq, D = fl.q.shape
        Hkv, ncap = fl.K.shape[1], fl.K.shape[2]
        shape = E.Shape(B, Hq, Hkv, D, fl.n, ncap)
        if fl.kv == "e4m3":
            L = dict(fl=fl, shape=shape, q=to_dev(fl.q), K=to_dev_raw(fl.K), V=to_dev_raw(fl.V),
                     Ks=to_dev_raw(fl.Ks), Vs=to_dev_raw(fl.Vs), qs=[to_dev(x) for x in fl.sparse_q])
        else:
            L = dict(fl=fl, shape=shape, q=to_dev(fl.q), K=to_dev(fl.K), V=to_dev(fl.V),
                     qs=[to_dev(x) for x in fl.sparse_q])
        L["out"] = torch.empty(B, Hq, D, dtype=torch.float32, device=dev)
        L["per_head"] = per_head
        L["n_surv"] = torch.empty(B, Hkv, dtype=torch.int32, device=dev)
        need_sel = len(fl.sparse_q) > 0
        Hs = Hq if per_head else Hkv  # units of the selection
        L["sel"] = torch.empty(B, Hs, ncap, dtype=torch.float32, device=dev) if need_sel else None
        L["hist"] = torch.empty(B, Hs, E.HIST_BINS, dtype=torch.int32, device=dev) if need_sel else None
        L["idx"] = torch.empty(B, Hs, TOPK + RECENT, dtype=torch.int32, device=dev)
        L["count"] = torch.empty(B, Hs, dtype=torch.int32, device=dev)
        L["souts"] = [torch.empty(B, Hq, D, dtype=torch.float32, device=dev) for _ in fl.sparse_q]
        L["ws_full"] = torch.empty(E.embla_full_decode_workspace_size(shape), dtype=torch.uint8, device=dev)
        L["ws_sel"] = torch.empty(max(16, E.embla_select_topk_workspace_size(shape) * (Hq // Hkv if per_head else 1)),
                                  dtype=torch.uint8, device=dev)
        L["ws_sp"] = torch.empty(max(16, E.embla_sparse_decode_workspace_size(shape, TOPK + RECENT)),
                                 dtype=torch.uint8, device=dev)
        layers.append(L)
    wins = []
    for wl in wls:
        B, Hq, D = wl.q.shape
        Hkv, W = wl.K.shape[1], wl.K.shape[2]
        wins.append(dict(wl=wl, shape=E.Shape(B, Hq, Hkv, D, 0, 0), q=to_dev(wl.q), K=to_dev(wl.K),
                         V=to_dev(wl.V), out=torch.empty(B, Hq, D, dtype=torch.float32, device=dev)))

    # Every per-step input (the queries and the appended token's K/V rows) lives in one device
    # buffer and every output in another, so a step moves its inputs with one host->device
    # copy and its results with one device->host copy.
    for L in layers:
        n_last = L["fl"].n - 1
        L["krow"] = L["K"][:, :, n_last].clone()
        L["vrow"] = L["V"][:, :, n_last].clone()
        if "Ks" in L:
            L["ksrow"] = L["Ks"][:, :, n_last].clone()
            L["vsrow"] = L["Vs"][:, :, n_last].clone()

    def rehome(refs):
        """Move each (container, key) tensor into one contiguous device buffer (256-byte
        aligned slots) and put the view back; returns the buffer."""
        sizes = [((c[k].numel() * c[k].element_size()) + 255) // 256 * 256 for c, k in refs]
        arena = torch.empty(max(256, sum(sizes)), dtype=torch.uint8, device=dev)
        off = 0
        for (c, k), sz in zip(refs, sizes):
            t = c[k]
            v = arena[off:off + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
            v.copy_(t)
            c[k] = v
            off += sz
        return arena

    in_refs, out_refs = [], []
    for L in layers:
        in_refs += [(L, "q"), (L, "krow"), (L, "vrow")] + [(L["qs"], i) for i in range(len(L["qs"]))]
        if "Ks" in L:
            in_refs += [(L, "ksrow"), (L, "vsrow")]
        out_refs += [(L, "out"), (L, "n_surv")] + [(L["souts"], i) for i in range(len(L["souts"]))]
    for w in wins:
        in_refs.append((w, "q"))
        out_refs.append((w, "out"))
    arena_in, arena_out = rehome(in_refs), rehome(out_refs)

    def full_call(L):
        if L["per_head"]:
            E.embla_full_decode_head_scores(L["shape"], L["q"], L["K"], L["V"], L["out"], L["n_surv"],
                                            L["sel"], L["hist"], alpha=1.0, c=1.0, eps=1e-6,
                                            workspace=L["ws_full"])
            return
        if "Ks" in L:
            E.embla_full_decode_e4m3(L["shape"], L["q"], L["K"], L["Ks"], L["V"], L["Vs"], L["out"],
                                     L["n_surv"], L["sel"], L["hist"], alpha=1.0, c=1.0, eps=1e-6,
                                     workspace=L["ws_full"])
            return
        E.embla_full_decode(L["shape"], L["q"], L["K"], L["V"], L["out"], L["n_surv"], L["sel"],
                            L["hist"], alpha=1.0, c=1.0, eps=1e-6, workspace=L["ws_full"])

    def rest_calls(L):
        if not L["qs"]:
            return
        if L["per_head"]:
            E.embla_select_topk_per_head(L["shape"], L["sel"], L["hist"], L["idx"], L["count"], TOPK,
                                         RECENT, workspace=L["ws_sel"])
            for qs, so in zip(L["qs"], L["souts"]):
                E.embla_sparse_decode_per_head(L["shape"], qs, L["K"], L["V"], L["idx"], L["count"],
                                               so, workspace=L["ws_sp"])
            return
        E.embla_select_topk(L["shape"], L["sel"], L["hist"], L["idx"], L["count"], TOPK, RECENT,
                            workspace=L["ws_sel"])
        for qs, so in zip(L["qs"], L["souts"]):
            if "Ks" in L:
                E.embla_sparse_decode_e4m3(L["shape"], qs, L["K"], L["Ks"], L["V"], L["Vs"],
                                           L["idx"], L["count"], so, workspace=L["ws_sp"])
            else:
                E.embla_sparse_decode(L["shape"], qs, L["K"], L["V"], L["idx"], L["count"], so,
                                      workspace=L["ws_sp"])

    def window_calls():
        for w in wins:
            E.embla_window_decode(w["shape"], w["q"], w["K"], w["V"], w["wl"].pos, w["out"])

    # eager pass: sets kernel attributes and fills the library's per-device caches
    for L in layers:
        full_call(L)
        rest_calls(L)
    window_calls()
    torch.cuda.synchronize()
    assert E.embla_device_check() == 0

    # caches smaller than L2: the steps rotate through copies of them (identical contents)
    step_read = sum(full_layer_needed_bytes(L["shape"].units, L["fl"].n, 0, L["fl"].kv) *
                    (1 + 2 * len(L["qs"]) * TOPK // max(1, L["fl"].n)) for L in layers)
    n_rep = replicas_for(step_read)
    reps = [layers]
    for _ in range(n_rep - 1):
        copies = []
        for L in layers:
            Lr = dict(L)
            for key in ("K", "V", "Ks", "Vs"):
                if key in L:
                    Lr[key] = L[key].clone()
            copies.append(Lr)
        reps.append(copies)
    for copies in reps[1:]:
        for L in copies:
            full_call(L)
            rest_calls(L)
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=dev)
    nl = len(layers)
    in_graph_events = _graph_events_work(torch, stream)

    def capture(body):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            body()
        return g

    if in_graph_events:
        # one graph per timed step (a decode step is one graph launch), with the events
        # around each full-layer call recorded inside it
        ev = [(torch.cuda.Event(enable_timing=True, external=True),
               torch.cuda.Event(enable_timing=True, external=True)) for _ in range(args.steps * nl)]

        side = torch.cuda.Stream(device=dev)

        def step_body(i):
            # the events around a full-layer call are recorded on a side branch of the graph
            # (it forks after the work before the call, and after the call), so every kernel
            # stays directly chained to the one before it: the start event fires when the
            # work before the call has finished, the end event when the call has, and their
            # difference is the call's share of the step
            def body():
                for li, L in enumerate(reps[(i or 0) % n_rep]):
                    if i is not None:
                        side.wait_stream(stream)
                        ev[i * nl + li][0].record(side)
                    full_call(L)
                    if i is not None:
                        side.wait_stream(stream)
                        ev[i * nl + li][1].record(side)
                    rest_calls(L)
                window_calls()
                if i is not None:
                    stream.wait_stream(side)
            return body

        with torch.cuda.stream(stream):
            g_warm = capture(step_body(None))
            g_steps = [capture(step_body(i)) for i in range(args.steps)]

        def step(timed_i=None):
            (g_warm if timed_i is None else g_steps[timed_i]).replay()
    else:
        # graphs: one per full-layer call (timed alone for the roofline) and one for the rest
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps * nl)]
        with torch.cuda.stream(stream):
            g_full = [[capture(lambda L=L: full_call(L)) for L in Ls] for Ls in reps]
            g_rest = [[capture(lambda L=L: rest_calls(L)) for L in Ls] for Ls in reps]
            g_win = capture(window_calls) if wins else None

        def step(timed_i=None):
            r = (timed_i or 0) % n_rep
            for li, (gf, gr) in enumerate(zip(g_full[r], g_rest[r])):
                if timed_i is not None:
                    ev[timed_i * nl + li][0].record(stream)
                gf.replay()
                if timed_i is not None:
                    ev[timed_i * nl + li][1].record(stream)
                gr.replay()
            if g_win is not None:
                g_win.replay()
    torch.cuda.synchronize()

    # accounting from this rank's own results
    n_surv_tot = [int(L["n_surv"].sum().item()) for L in layers]
    sel_tot = [int(L["count"].sum().item()) if L["qs"] else 0 for L in layers]
    full_bytes = [full_layer_needed_bytes(L["shape"].units, L["fl"].n, s, L["fl"].kv)
                  for L, s in zip(layers, n_surv_tot)]
    # a block's first sparse layer reads its selected rows from HBM; the block's later sparse
    # layers read the same rows right after it, from L2, so they are counted apart
    sparse_first = sum(sparse_layer_needed_bytes(s, L["fl"].kv)
                       for L, s in zip(layers, sel_tot) if L["qs"])
    sparse_rereads = sum((len(L["qs"]) - 1) * sparse_layer_needed_bytes(s, L["fl"].kv)
                         for L, s in zip(layers, sel_tot) if L["qs"])
    win_bytes = sum(window_layer_needed_bytes(w["shape"].units, min(w["wl"].pos + 1, w["wl"].K.shape[2]))
                    for w in wins)
    needed = sum(full_bytes) + sparse_first + win_bytes
    keys_total = sum(L["shape"].units * L["fl"].n for L in layers)
    skipped_v = 1.0 - sum(n_surv_tot) / max(1, keys_total)
    # the same V reads counted at the page's granularity (8-key chunks)
    chunk_rows = 0
    for L in layers:
        if L["sel"] is None or L["per_head"]:
            # no group scores to count chunks on (per-head scores rank differently)
            chunk_rows += L["shape"].units * L["fl"].n
            continue
        kn = torch.empty(L["shape"].batch, L["shape"].n_kv_heads, dtype=torch.int32, device=dev)
        cn = torch.empty_like(kn)
        E.embla_skip_stats(L["shape"], L["sel"], kn, cn, chunk=8)
        chunk_rows += min(int(cn.sum().item()) * 8, L["shape"].units * L["fl"].n)
    skipped_v_chunk8 = None if per_head else 1.0 - chunk_rows / max(1, keys_total)
    batch = layers[0]["shape"].batch
    # kernels of this library per step: per full layer a zeroing kernel and the decode
    # kernel, one selection kernel and one kernel per sparse layer, one window kernel per
    # window layer
    launches_per_step = 0
    for L in layers:
        # zeroing, decode and combining kernels (+ the per-head score histograms)
        launches_per_step += 4 if L["per_head"] else 3
        if L["qs"]:
            launches_per_step += 1 + len(L["qs"])
    launches_per_step += len(wins)

    clocks = ClockSampler(local)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_wall0 = time.time()
        start.record(stream)
        for i in range(args.steps):
            step(i)
        end.record(stream)
        torch.cuda.synchronize()
        t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop(t_wall0, t_wall1)
    ms = start.elapsed_time(end)
    full_ms = [statistics.mean(ev[i * nl + li][0].elapsed_time(ev[i * nl + li][1])
                               for i in range(args.steps)) for li in range(nl)]
    assert E.embla_device_check() == 0
    ms = max_over_ranks(ms, world, dev)
    ms_per_step = ms / args.steps
    value = job_throughput(world, batch, ms_per_step * 1e-3)

    # end to end through the public Python API, host buffers, copies inside the timed region
    e2e = None
    if args.e2e_steps > 0:
        n = layers[0]["fl"].n
        h_in = torch.empty(arena_in.numel(), dtype=torch.uint8).pin_memory()
        h_in.copy_(arena_in)
        h_res = torch.empty(arena_out.numel(), dtype=torch.uint8).pin_memory()
        h2d, d2h = arena_in.numel(), arena_out.numel()

        def e2e_body(k):
            arena_in.copy_(h_in, non_blocking=True)  # every query and appended row: one copy
            for L in reps[k % n_rep]:
                # the appended token's rows into the caches (a kernel of the library's)
                if "Ks" in L:
                    E.embla_append_kv_e4m3(L["shape"], n - 1, L["krow"], L["ksrow"], L["vrow"],
                                           L["vsrow"], L["K"], L["Ks"], L["V"], L["Vs"])
                else:
                    E.embla_append_kv(L["shape"], n - 1, L["krow"], L["vrow"], L["K"], L["V"])
                full_call(L)
                rest_calls(L)
            window_calls()
            h_res.copy_(arena_out, non_blocking=True)  # every output: one copy

        def e2e_eager(k):
            e2e_body(k)
            torch.cuda.current_stream().synchronize()

        # the same calls and copies captured once per cache copy: a step is one graph launch
        # (host->device copies, every kernel, device->host copies) and a host synchronise
        e2e_stream = torch.cuda.Stream(device=dev)
        e2e_graphs = []
        with torch.cuda.stream(e2e_stream):
            for r in range(n_rep):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=e2e_stream):
                    e2e_body(r)
                e2e_graphs.append(g)
        torch.cuda.synchronize()

        def e2e_graph(k):
            e2e_graphs[k % n_rep].replay()
            e2e_stream.synchronize()

        rates = {}
        for name, fn in (("eager", e2e_eager), ("graph", e2e_graph)):
            with torch.cuda.stream(e2e_stream):
                for k in range(3):
                    fn(k)
                if world > 1:
                    torch.distributed.barrier()
                t0 = time.perf_counter()
                for k in range(args.e2e_steps):
                    fn(k)
                dt = time.perf_counter() - t0
            dt = max_over_ranks(dt, world, dev)
            rates[name] = job_throughput(world, batch, dt / args.e2e_steps)
        e2e = {"value": rates["graph"], "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": args.e2e_steps,
               "launch": "per step one CUDA graph of the public API calls with the copies in it, "
                         "then a host synchronise",
               "eager_value": rates["eager"],
               "eager_launch": "the public API called from Python per step, copies issued "
                               "eagerly, then a host synchronise",
               "inputs": "per step, one copy of every query and the appended token's K/V rows "
                         "from pinned host memory (then written into the caches by embla_append_kv) and "
                         "one copy of every output back; the KV caches stay resident in HBM"}

    # one sparse layer (the first of the first block): its marginal cost after a write of twice
    # the L2 size (its rows come from HBM), and right after itself (its rows in L2)
    sparse_alone = None
    Lsp = next((L for L in layers if L["qs"]), None)
    if Lsp is not None:
        def sparse_one(L=Lsp):
            qs, so = L["qs"][0], L["souts"][0]
            if L["per_head"]:
                E.embla_sparse_decode_per_head(L["shape"], qs, L["K"], L["V"], L["idx"], L["count"],
                                               so, workspace=L["ws_sp"])
            elif "Ks" in L:
                E.embla_sparse_decode_e4m3(L["shape"], qs, L["K"], L["Ks"], L["V"], L["Vs"],
                                           L["idx"], L["count"], so, workspace=L["ws_sp"])
            else:
                E.embla_sparse_decode(L["shape"], qs, L["K"], L["V"], L["idx"], L["count"], so,
                                      workspace=L["ws_sp"])
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

        def graph_ms(body, reps=30):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                with torch.cuda.graph(g, stream=stream):
                    body()
                g.replay()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(reps):
                    g.replay()
                e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / reps

        # marginal cost in a graph: (flush, call) - (flush) and (call, call) - (call)
        cold_ms = graph_ms(lambda: (flush.fill_(1.0), sparse_one())) - graph_ms(lambda: flush.fill_(1.0))
        warm_ms = graph_ms(lambda: (sparse_one(), sparse_one())) - graph_ms(sparse_one)
        del flush
        sp_bytes = sparse_layer_needed_bytes(sel_tot[layers.index(Lsp)], Lsp["fl"].kv)
        sparse_alone = {"bytes": sp_bytes,
                        "cold_l2_us": round(cold_ms * 1e3, 2),
                        "cold_l2_gbs": round(sp_bytes / (cold_ms * 1e-3) / 1e9, 1),
                        "warm_l2_us": round(warm_ms * 1e3, 2),
                        "how": "marginal cost of one sparse-layer call in a CUDA graph: after a "
                               "write of twice the L2 size (cold: graph of the write and the call "
                               "minus graph of the write) and right after the same call (warm)"}

    peak, peak_src = _peaks()
    wl_key = workload_name(cfg, args.batch, args.ctx).replace(" ", "_")
    achieved = [fb / (fm * 1e-3) / 1e9 for fb, fm in zip(full_bytes, full_ms)]
    ach = statistics.mean(achieved)
    roofline = {"bound": "hbm", "kernel": "full_decode_kernel (one embla_full_decode call: zeroing, decode and combining kernels)",
                "achieved": round(ach, 1), "peak": peak, "unit": "GB/s", "frac": round(ach / peak, 4),
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback 6.8 TB/s",
                "traffic": _traffic_from_profile(wl_key, _kernel_digest()),
                "algorithmic_bytes_per_launch": full_bytes[0],
                "launch_ms": round(statistics.mean(full_ms), 5)}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.config)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if layers[0]["fl"].kv == "e4m3" else "bf16",
        "data": "synthetic",
        "config": {**static_config(args.config, args.batch, args.ctx),
                   "launch": ("one CUDA graph per step; events inside it around each full-layer call, "
                              "on a side branch that forks before and after the call (the kernels stay "
                              "chained): the call's share of the step"
                              if in_graph_events else
                              "two CUDA graphs per full layer (its call, then the rest); events between them"),
                   "l2": ("not flushed: inputs larger than L2 (each full layer's K cache is "
                          f"{keys_total * row_bytes(layers[0]['fl'].kv) // len(layers) / 1e6:.0f} MB)"
                          if n_rep == 1 else
                          f"not flushed: the steps rotate through {n_rep} copies of the caches "
                          f"({step_read / 1e6:.0f} MB read per step, smaller than L2), so each "
                          f"step's rows were last read {(n_rep - 1) * step_read / 1e6:.0f} MB of "
                          "other reads earlier"),
                   "needed_bytes_per_step": needed,
                   "needed_bytes": "HBM: every full layer's K rows and surviving V rows, each "
                                   "block's first sparse layer's selected K and V rows, the "
                                   "window rows",
                   "needed_gbs": round(needed / (ms_per_step * 1e-3) / 1e9, 1),
                   "needed_frac_of_peak": round(needed / (ms_per_step * 1e-3) / 1e9 / peak, 4),
                   "sparse_reread_bytes_per_step": sparse_rereads,
                   "sparse_reread": "the same selected rows read again by a block's later "
                                    "sparse layers right after its first (from L2; not in "
                                    "needed_bytes_per_step)",
                   "sparse_layer_alone": sparse_alone,
                   "skipped_v_fraction": round(skipped_v, 5),
                   "skipped_v_fraction_8key_chunks": None if skipped_v_chunk8 is None else round(skipped_v_chunk8, 5),
                   "selection": "per query head" if per_head else "per KV head (group max)"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps, "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
