#!/usr/bin/env python
"""Benchmark of the masked second-order HLA forward (and the decode step and the
backward pass) on GB300.

Prints ONE JSON line (rank 0).  A step is one hla_forward_chunked call over one
batch of the workload (all hot-path stages: chunk products, segment summaries,
exclusive scan, outputs, final-state export), inputs resident in HBM.  Timing:
W eager warm-up steps, then K steps replayed from CUDA graphs, bracketed by
CUDA events on the launching stream (barrier + synchronize on both sides, max
over ranks).  The steps cycle over enough input sets that the bytes touched
between reuses exceed the 129 MB L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Multi-GPU: the path does not shard (every (b,h) pair is independent), so N ranks
run N independent replicas ("replicas only"); value = tokens of all ranks / max time.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from causal_prefix_scan_gb300 import workloads as W  # noqa: E402

METRIC = "masked 2nd-order HLA forward tokens/s and % roofline on 1 GB300"


def metric_for(w) -> str:
    if getattr(w, "unmasked", False):
        return METRIC.replace("masked", "unmasked", 1)
    if getattr(w, "asymmetric", False):
        return METRIC.replace("masked 2nd-order HLA", "masked asymmetric 2nd-order HLA (AHLA)", 1)
    return METRIC
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
CSRC = os.path.join(ROOT, "causal_prefix_scan_gb300", "csrc")
# source file of each forward kernel (its hash keys the committed DRAM traffic)
FWD_KERNEL_SRCS = {"fwd_ws2_kernel": "hla_fwd_ws2.cuh", "fwd_ws_kernel": "hla_fwd_ws.cuh",
                   "fwd_tc_kernel": "hla_fwd_tc.cuh", "fwd_simt_kernel": "hla_fwd_simt.cu"}
DECODE_KERNEL_SRC = os.path.join(ROOT, "causal_prefix_scan_gb300", "csrc", "hla_decode.cu")
BWD_KERNEL_SRC = os.path.join(ROOT, "causal_prefix_scan_gb300", "csrc", "hla_bwd_simt.cuh")
BWD_METRIC = "masked 2nd-order HLA backward (dq, dk, dv) tokens/s and % roofline on 1 GB300"
FWD3_KERNEL_SRC = os.path.join(ROOT, "causal_prefix_scan_gb300", "csrc", "hla_fwd3_simt.cuh")
FWD3_METRIC = "masked 3rd-order HLA forward tokens/s and % roofline on 1 GB300"
FWD3_DISPATCH_SRC = os.path.join(ROOT, "causal_prefix_scan_gb300", "csrc", "hla_fwd3_simt.cu")
FWD3_TC_KERNEL_SRC = os.path.join(ROOT, "causal_prefix_scan_gb300", "csrc", "hla_fwd3_tc.cu")
BWD_NORM_SRC = os.path.join(ROOT, "causal_prefix_scan_gb300", "csrc", "hla_bwd_norm.cu")
BWD_NORM_TC_SRC = os.path.join(ROOT, "causal_prefix_scan_gb300", "csrc", "hla_bwd_norm_tc.cu")
NORM_UNIT_WIDTH = 16  # width of the unit-value tile of the normalised backward
BWD_TC_KERNEL_SRC = os.path.join(ROOT, "causal_prefix_scan_gb300", "csrc", "hla_bwd_tc.cu")
SCAN_TC_SRC = os.path.join(ROOT, "causal_prefix_scan_gb300", "csrc", "hla_scan_tc.cu")
# fp32 FMA peak of the CUDA cores: 152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz (maximum SM clock)
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2070e6 / 1e12


# ----------------------------------------------------------------- arithmetic
def alg_flops_per_token_head(w: W.Workload) -> float:
    """Masked: c(3d+dv) + 4d^2 + 6 d dv + 2 d^2 dv / c; unmasked (no X = S C - G):
    c(3d+dv) + 4d^2 + 4 d dv; triangular products at half."""
    c, d, dv = w.chunk, w.d, w.dv
    if w.unmasked:
        return c * (3 * d + dv) + 4 * d * d + 4 * d * dv
    if w.asymmetric:  # A, A-tilde V, A-tilde Z at half; Q P_p, Q E_p, P, E updates; R update
        return c * (d + 2 * dv) + 8 * d * dv + 2 * d * d
    return c * (3 * d + dv) + 4 * d * d + 6 * d * dv + 2 * d * d * dv / c


def alg_bytes_per_launch(w: W.Workload, with_state: bool = True) -> float:
    """q read and o written once per token-head, k and v read once per token and
    key/value head, the final state written once per (b,h): S, C, m, G, h (masked)
    or S, C, m (unmasked)."""
    s = 2 if w.dtype == "bf16" else 4
    qo = (w.d + w.dv) * s * w.token_heads
    kv = (w.d + w.dv) * s * w.B * w.kv_heads * w.n
    per_pair = w.d * w.d + w.d * w.dv + w.d if w.unmasked else w.d * w.d + 2 * w.d * w.dv + 2 * w.d
    state = per_pair * 4 if with_state else 0
    return qo + kv + w.B * w.H * state


def bwd_flops_per_token_head(w: W.Workload) -> dict:
    """Algorithmic flops per token-head of each backward kernel (an FMA is 2 flops;
    triangular chunk products counted at half).  Local sums: A~, P, A~K, P^T Q at
    half, and the six d x d / d x dv sums; scan: S_p Cq and Lam W per chunk; gradients:
    A~, P, B, M and the products A~K, P^T Q, P U, B K, A~^T dU, B^T Q, M^T G at half,
    Q S_p, V Lam^T, G X_p^T, dU S_p, K (Om + Om^T), U Lam in full."""
    c, d, dv = w.chunk, w.d, w.dv
    return {"bwd_local_kernel": 3 * c * d + c * dv + 4 * d * d + 8 * d * dv,
            "bwd_scan_kernel": 4 * d * d * dv / c,
            "bwd_grad_kernel": 9 * c * d + 2 * c * dv + 6 * d * d + 6 * d * dv}


def norm_tc(w: W.Workload) -> bool:
    """The ratio-normalised backward runs on the tensor cores (bf16, d = dv = chunk = 64)."""
    return w.normalize and w.dtype == "bf16" and w.d == w.dv == w.chunk == 64


def bwd_norm_tc_flops_per_token_head(w: W.Workload) -> dict:
    """Algorithmic flops per token-head of the three phases of the tensor-core
    normalised backward (an FMA is 2 flops, triangular chunk products at half; the
    unit column's d-vectors and the hi/lo split's extra products are not counted).
    Forward and local sums: A~, A~K twice, M, P^T Q at half (c d each), M V and P at
    half (c dv each), S_loc, Q S_p, O_loc (2 d^2 each), C_q, X_loc, Q X_p, L_loc, W
    (2 d dv each), S_p C_q per chunk; scan: Lam W per chunk; gradients as for the
    unnormalised backward."""
    c, d, dv = w.chunk, w.d, w.dv
    return {"bwd_norm_tc_forward_local": 6 * c * d + 2 * c * dv + 6 * d * d + 10 * d * dv + 2 * d * d * dv / c,
            "bwd_norm_tc_scan": 2 * d * d * dv / c,
            "bwd_norm_tc_grad_kernel": 9 * c * d + 2 * c * dv + 6 * d * d + 6 * d * dv}


def bwd_bytes_per_step(w: W.Workload) -> float:
    """q, k, v and dout read once, dq, dk, dv written once."""
    s = 2 if w.dtype == "bf16" else 4
    return w.token_heads * (3 * w.d + 3 * w.dv) * s


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"]))}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS, bf16_tflops_sustained=1700.0), "fallback"


def file_hash(path: str) -> str:
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def traffic_for(kernel: str, workload: str, src: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[kernel][workload]
        if e.get("source_sha256_16") == file_hash(src):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", self.gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.15)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.06)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def gpu_selector(dev_index: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    if vis:
        return vis.split(",")[dev_index]
    return str(dev_index)


# ----------------------------------------------------------------- dist
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world):
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        return dist
    return None


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ----------------------------------------------------------------- oracle timing
def oracle_rate(w: W.Workload, x, batch_rows: int, n_tokens: int, nthreads: int):
    """Time the fp64 oracle on the first `batch_rows` rows (all heads) over the first
    `n_tokens` tokens; returns (seconds, tokens)."""
    import oracle
    sl = lambda a: np.ascontiguousarray(a[:batch_rows, :, :n_tokens], dtype=np.float64)
    q, k, v = sl(x["q"]), sl(x["k"]), sl(x["v"])
    g = None if x["gamma"] is None else np.asarray(x["gamma"], np.float64)
    oracle.build()
    t0 = time.perf_counter()
    oracle.forward(q, k, v, gamma=g, normalize=w.normalize, eps=w.eps, want_state=True, nthreads=nthreads,
                   unmasked=w.unmasked, asymmetric=w.asymmetric)
    return time.perf_counter() - t0, batch_rows * n_tokens


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline_forward(w: W.Workload, x):
    """The oracle on the whole workload when that takes at most ~20 s, else on its
    first batch rows (all heads, all tokens) sized to ~20 s."""
    cores = cpu_threads()
    rows = max(1, min(w.B, -(-cores // w.H)))
    secs, toks = oracle_rate(w, x, rows, w.n, min(cores, rows * w.H))
    if rows < w.B:
        more = int(rows * 20.0 / max(secs, 1e-9))
        rows = max(rows, min(w.B, more))
        if rows > max(1, -(-cores // w.H)):
            secs, toks = oracle_rate(w, x, rows, w.n, min(cores, rows * w.H))
    used = min(cores, rows * w.H)
    reps = 1
    if secs < 5.0:  # a quick sample is repeated to about 10 s for a stable rate
        reps = max(2, min(500, int(10.0 / max(secs, 1e-9))))
        secs = (secs + sum(oracle_rate(w, x, rows, w.n, used)[0] for _ in range(reps - 1))) / reps
    return {"value": toks / secs, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"fp64 serial recurrence over {rows} of {w.B} batch row(s) x {w.H} heads x {w.n} tokens "
                      f"of the same inputs, threads over (b,h); mean of {reps} run(s)", "seconds": secs}


def oracle_bwd_rate(x, g, batch_rows: int, n_tokens: int, nthreads: int, w: W.Workload | None = None):
    import oracle
    sl = lambda a: np.ascontiguousarray(a[:batch_rows, :, :n_tokens], dtype=np.float64)
    gam = None if x["gamma"] is None else np.asarray(x["gamma"], np.float64)
    norm = dict(normalize=True, eps=w.eps) if w is not None and w.normalize else {}
    oracle.build()
    t0 = time.perf_counter()
    oracle.backward(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(g), gam, nthreads=nthreads, **norm)
    return time.perf_counter() - t0, batch_rows * n_tokens


def cpu_baseline_backward(w: W.Workload, x, g):
    """The oracle's gradient on the first batch rows (all heads, all tokens), repeated
    to about 10 s."""
    cores = cpu_threads()
    rows = max(1, min(w.B, -(-cores // w.H)))
    used = min(cores, rows * w.H)
    secs, toks = oracle_bwd_rate(x, g, rows, w.n, used, w)
    reps = max(1, min(500, int(10.0 / max(secs, 1e-9))))
    if reps > 1:
        secs = (secs + sum(oracle_bwd_rate(x, g, rows, w.n, used, w)[0] for _ in range(reps - 1))) / reps
    return {"value": toks / secs, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"fp64 reverse-mode recurrence over {rows} of {w.B} batch row(s) x {w.H} heads x {w.n} "
                      f"tokens of the same inputs, threads over (b,h); mean of {reps} run(s)", "seconds": secs}


def oracle3_rate(x, batch_rows: int, n_tokens: int, nthreads: int):
    import oracle
    sl = lambda a: np.ascontiguousarray(a[:batch_rows, :, :n_tokens], dtype=np.float64)
    oracle.build()
    t0 = time.perf_counter()
    oracle.forward3(sl(x["q"]), sl(x["k"]), sl(x["v"]), nthreads=nthreads)
    return time.perf_counter() - t0, batch_rows * n_tokens


def cpu_baseline_third(w: W.Workload, x):
    """The third-order oracle (serial recurrence) on the first batch rows, all heads and
    tokens, repeated to about 10 s."""
    cores = cpu_threads()
    rows = max(1, min(w.B, -(-cores // w.H)))
    used = min(cores, rows * w.H)
    secs, toks = oracle3_rate(x, rows, w.n, used)
    reps = max(1, min(500, int(10.0 / max(secs, 1e-9))))
    if reps > 1:
        secs = (secs + sum(oracle3_rate(x, rows, w.n, used)[0] for _ in range(reps - 1))) / reps
    return {"value": toks / secs, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"fp64 serial third-order recurrence over {rows} of {w.B} batch row(s) x {w.H} heads x {w.n} "
                      f"tokens of the same inputs, threads over (b,h); mean of {reps} run(s)", "seconds": secs}


def time_e2e(e2e_steps, Ke, stream, s_up, s_down, dist) -> float:
    """Milliseconds (max over ranks) for Ke end-to-end steps.  The steps are captured in
    CUDA graphs of up to 50 steps and replayed, so that the host's per-call overhead does
    not pace the pipeline; every step still uploads its inputs from pinned host memory,
    makes the library call and reads its result back."""
    import torch
    R = min(Ke, 50)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            s_up.wait_stream(stream)   # fork the copy streams from the capture stream
            s_down.wait_stream(stream)
            e2e_steps(n)               # joins them back before it returns
        return g

    torch.cuda.synchronize()
    g_main = capture(R)
    g_rem = capture(Ke % R) if Ke % R else None
    with torch.cuda.stream(stream):
        g_main.replay()  # untimed warm replay
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(Ke // R):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
    stream.synchronize()
    barrier(dist)
    return max_over_ranks(dist, e0.elapsed_time(e1))


# ----------------------------------------------------------------- forward bench
def workload_by_name(name: str):
    if name in W.WORKLOADS:
        return W.WORKLOADS[name]
    if name == W.DECODE.name:
        return W.DECODE
    if name == W.DECODE3.name:
        return W.DECODE3
    raise SystemExit(f"unknown workload {name}; choose from {list(W.WORKLOADS) + [W.DECODE.name, W.DECODE3.name]}")


def config_dict(w: W.Workload, nsets: int, set_bytes: int, world: int):
    variant = "normalised" if w.normalize else ("decay" if w.decay else "unnormalised")
    variant = ("unmasked " if w.unmasked else ("asymmetric " if w.asymmetric else "masked ")) + variant
    return {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.kv_heads, "n": w.n, "d": w.d, "dv": w.dv,
            "chunk": w.chunk,
            "variant": variant, "inputs": f"q,k {w.qk}, v N(0,1), seed {w.seed}",
            "l2": f"inputs larger than L2: {nsets} rotating input sets, {nsets * set_bytes / 2**20:.0f} MiB",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def bench_forward(args, w: W.Workload, rank, world, local, dist):
    import torch
    import causal_prefix_scan_gb300 as hla
    from causal_prefix_scan_gb300 import _build
    _build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    x = W.make_inputs(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    host = {k: torch.from_numpy(x[k]).to(tdt).pin_memory() for k in ("q", "k", "v")}
    gamma = torch.from_numpy(x["gamma"]).to(dev) if x["gamma"] is not None else None
    esz = 2 if w.dtype == "bf16" else 4
    set_bytes = (w.token_heads + w.B * w.kv_heads * w.n) * (w.d + w.dv) * esz  # q, o and k, v
    nsets = max(1, min(16, -(-2 * L2_BYTES // set_bytes)))
    sets = []
    for _ in range(nsets):
        q, k, v = (host[n].to(dev, non_blocking=True) for n in ("q", "k", "v"))
        o = torch.empty(q.shape[:3] + (w.dv,), dtype=tdt, device=dev)
        sets.append((q, k, v, o))
    params = hla.make_params(sets[0][0], sets[0][2], w.chunk, gamma, w.normalize, w.eps, w.unmasked, w.asymmetric)
    ws_bytes = hla.hla_forward_workspace_size(params)
    ws = hla.new_workspace(ws_bytes, dev)
    st = hla.State.empty(w.B * w.H, w.d, w.dv, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(i, s=None):
        q, k, v, o = sets[i % nsets]
        hla.hla_forward_chunked(params, q, k, v, o, None, st, ws, ws_bytes, s or stream)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    hla.hla_sync_status(stream)

    # graphs of R steps (+ a remainder graph) replayed to make exactly K steps
    K = args.steps
    R = min(K, max(nsets, 50))
    graphs = []

    def capture(nsteps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="thread_local"):
            for i in range(nsteps):
                step(i, torch.cuda.current_stream())
        return g

    g_main = capture(R)
    reps = K // R
    g_rem = capture(K % R) if K % R else None
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        g_main.replay()  # untimed warm replay
    stream.synchronize()
    hla.hla_sync_status(stream)

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(gpu_selector(local)) as clk, torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            g_main.replay()
        if g_rem is not None:
            g_rem.replay()
        ev1.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    barrier(dist)
    hla.hla_sync_status(stream)
    t_ms = ev0.elapsed_time(ev1)
    t_max = max_over_ranks(dist, t_ms)
    ms_per_step = t_max / K
    value = world * w.tokens * K / (t_max / 1e3)

    # ---- end to end: host buffers, copies inside the timed region.  Every step
    # copies its q, k, v from pinned host memory and reads its o back; as a
    # streaming caller would, step i+1's upload and step i-1's download run on
    # their own streams while step i computes (two device buffer sets).
    Ke = min(K, 200)
    o_host = [torch.empty(sets[0][3].shape, dtype=tdt).pin_memory() for _ in range(2)]
    bufs = [sets[b % nsets] for b in range(2)] if nsets >= 2 else \
        [sets[0], tuple(torch.empty_like(t) for t in sets[0])]
    s_up, s_down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {kk: [torch.cuda.Event() for _ in range(2)] for kk in ("up", "fwd", "down")}

    def e2e_steps(n):
        for i in range(n):
            b = i % 2
            q, k, v, o = bufs[b]
            if i >= 2:
                s_up.wait_event(ev["fwd"][b])       # step i-2 has finished reading buffer b
            with torch.cuda.stream(s_up):
                q.copy_(host["q"], non_blocking=True); k.copy_(host["k"], non_blocking=True)
                v.copy_(host["v"], non_blocking=True)
            ev["up"][b].record(s_up)
            stream.wait_event(ev["up"][b])
            if i >= 2:
                stream.wait_event(ev["down"][b])    # o of step i-2 has been read back
            hla.hla_forward_chunked(params, q, k, v, o, None, st, ws, ws_bytes, stream)
            ev["fwd"][b].record(stream)
            s_down.wait_event(ev["fwd"][b])
            with torch.cuda.stream(s_down):
                o_host[b].copy_(o, non_blocking=True)
            ev["down"][b].record(s_down)
        stream.wait_stream(s_up)
        stream.wait_stream(s_down)

    te = time_e2e(e2e_steps, Ke, stream, s_up, s_down, dist)
    hla.hla_sync_status(stream)
    e2e = {"value": world * w.tokens * Ke / (te / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": int(sum(host[n].numel() * host[n].element_size() for n in ("q", "k", "v"))),
           "d2h_bytes_per_step": int(o_host[0].numel() * o_host[0].element_size()), "steps": Ke,
           "overlap": "upload of step i+1 and download of step i-1 on their own streams during step i",
           "replay": "CUDA graphs of up to 50 such steps (uploads, library calls, downloads and their "
                     "cross-stream order captured), replayed back to back"}

    # ---- roofline of the (only) kernel of the step, as the library names it
    fwd_kernel = hla.hla_forward_kernel(params)
    peaks, peak_kind = load_peaks()
    bytes_launch = alg_bytes_per_launch(w)
    flops_launch = alg_flops_per_token_head(w) * w.token_heads
    t_launch = ms_per_step / 1e3
    t_hbm = bytes_launch / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops_launch / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        ach, peak, unit, bound = bytes_launch / t_launch / 1e9, peaks["hbm_gbs"], "GB/s", "hbm"
    else:
        ach, peak, unit, bound = flops_launch / t_launch / 1e12, peaks["bf16_tflops"], "TFLOP/s", "tensor"
    roofline = {"bound": bound, "achieved": ach, "peak": peak, "unit": unit, "frac": ach / peak,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback",
                "traffic": traffic_for(fwd_kernel, w.name, os.path.join(CSRC, FWD_KERNEL_SRCS[fwd_kernel])),
                "kernel": fwd_kernel,
                "alg_bytes_per_launch": bytes_launch, "alg_flops_per_launch": flops_launch,
                "tensor_frac": (flops_launch / t_launch / 1e12) / peaks["bf16_tflops"],
                "roofline_time_us": max(t_hbm, t_tc) * 1e6, "launch_time_us": t_launch * 1e6}
    line = {"metric": metric_for(w), "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": config_dict(w, nsets, set_bytes, world), "roofline": roofline,
            "e2e": e2e, "gpu_launches": K, "clocks": clk.summary(),
            "token_heads_per_s": world * w.token_heads * K / (t_max / 1e3)}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_forward(w, x)
    return line


# ----------------------------------------------------------------- multi-kernel benches
def fwd3_flops_per_token_head(w: W.Workload) -> dict:
    """Algorithmic fp32 flops per token-head of each third-order kernel (an FMA is 2
    flops; triangular chunk products at half).  Local sums: A~, A~K, A~V at half and
    K^T K, Q^T Q, U^T Q, K^T V, U^T W, Q^T W; scan: S^Q P, S^K X, M^KQ P per chunk;
    outputs: A~, A~K, A~V, Q U^T, M W at half and Q S^K, Q P, Q T in full."""
    c, d, dv = w.chunk, w.d, w.dv
    return {"fwd3_local_kernel": c * (2 * d + dv) + 6 * d * d + 6 * d * dv,
            "fwd3_scan_kernel": 6 * d * d * dv / c,
            "fwd3_out_kernel": c * (3 * d + 2 * dv) + 2 * d * d + 4 * d * dv}


def is_backward(w) -> bool:
    return isinstance(w, W.Workload) and w.name.startswith("bwd_")


def is_third(w) -> bool:
    return isinstance(w, W.Workload) and w.name.startswith("fwd3_")


def launches_per_step(w: W.Workload) -> int:
    """Kernels of one library call: three for the backward or third order (four, the
    tensor-core scans counted as their own launches, are reported per phase); the
    normalised backward adds the input widening (bf16), the unit values, two forwards,
    the upstream gradients, a second backward and the sums."""
    if not (is_backward(w) and w.normalize):
        return 3
    if norm_tc(w):  # local sums, S prefix, increments, X/Y prefix, outputs, Lam suffix, increments, Om suffix, gradients
        return 9 + (2 if w.kv_heads != w.H else 0)
    bf = w.dtype == "bf16"
    split = norm_segments(w) > 1  # two forwards and a segment scan per part instead of one forward
    forwards = (4 + 2 + (1 if w.decay else 0)) if split else 2
    return (4 if bf else 0) + 1 + forwards + 1 + 3 + 3 + (3 if bf else 2)


def norm_segments(w: W.Workload) -> int:
    """Segments per sequence of the normalised backward's fp32 forwards: the library's
    rule (a power of two up to 16 dividing n into pieces of at least one chunk, with
    B H P at most 608; 1 with shared key/value heads)."""
    if w.kv_heads != w.H:
        return 1
    P = 1
    while P < 16 and w.n % (2 * P) == 0 and w.n // (2 * P) >= w.chunk and w.B * w.H * 2 * P <= 4 * 152:
        P *= 2
    return P


def bench_phased(args, w: W.Workload, rank, world, local, dist):
    """The backward pass or the third-order forward: a step is one library call
    (three kernels: local sums, scan over chunks, per-chunk results) over the whole
    batch.  Steps are launched eagerly with events at the phase boundaries (the
    *_traced entry points), so every kernel's duration is measured inside the timed
    region."""
    import torch
    import causal_prefix_scan_gb300 as hla
    from causal_prefix_scan_gb300 import _build
    _build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    bwd = is_backward(w)
    x = W.make_inputs(w)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    in_names = ("q", "k", "v", "dout") if bwd else ("q", "k", "v")
    host = {k: torch.from_numpy(x[k]).to(tdt).pin_memory() for k in ("q", "k", "v")}
    gout = None
    if bwd:
        gout = W.make_dout(w)
        host["dout"] = torch.from_numpy(gout).to(tdt).pin_memory()
    gamma = torch.from_numpy(x["gamma"]).to(dev) if x["gamma"] is not None else None
    esz = 2 if w.dtype == "bf16" else 4
    set_bytes = w.token_heads * ((3 * w.d + 3 * w.dv) if bwd else (2 * w.d + 2 * w.dv)) * esz
    nsets = max(2, min(16, -(-2 * L2_BYTES // set_bytes)))
    sets = []
    for _ in range(nsets):
        ins = tuple(host[n].to(dev, non_blocking=True) for n in in_names)
        outs = (torch.empty_like(ins[0]), torch.empty_like(ins[1]), torch.empty_like(ins[2])) if bwd else \
            (torch.empty(ins[0].shape[:3] + (w.dv,), dtype=tdt, device=dev),)
        sets.append((ins, outs))
    if bwd and w.normalize and norm_tc(w):
        params = hla.make_params(sets[0][0][0], sets[0][0][2], w.chunk, gamma, True, w.eps)
        ws_bytes = hla.hla_backward_workspace_size(params)
        fl = bwd_norm_tc_flops_per_token_head(w)
        names = tuple(fl)
        src, metric = BWD_NORM_TC_SRC, BWD_METRIC
        tc = True
    elif bwd and w.normalize:
        # two fp32 forwards and the upstream-gradient kernel, the backward of the values,
        # the backward of the unit column and the gradient sums (all fp32, CUDA cores)
        params = hla.make_params(sets[0][0][0], sets[0][0][2], w.chunk, gamma, True, w.eps)
        ws_bytes = hla.hla_backward_workspace_size(params)
        names = ("norm_forwards_upstream", "norm_bwd_values", "norm_bwd_unit_sums")
        w1 = dataclasses.replace(w, dv=NORM_UNIT_WIDTH)
        fl = dict(zip(names, (alg_flops_per_token_head(w) + alg_flops_per_token_head(w1),
                              sum(bwd_flops_per_token_head(w).values()),
                              sum(bwd_flops_per_token_head(w1).values()))))
        src, metric = BWD_NORM_SRC, BWD_METRIC
        tc = False
    elif bwd:
        params = hla.make_params(sets[0][0][0], sets[0][0][2], w.chunk, gamma)
        ws_bytes = hla.hla_backward_workspace_size(params)
        tc = w.dtype == "bf16" and w.d == w.dv == w.chunk == 64  # local sums and gradients on the tensor cores
        names = ("bwd_local_tc_kernel" if tc else "bwd_local_kernel", "bwd_scan_tc_kernels" if tc else "bwd_scan_kernel",
                 "bwd_grad_tc_kernel" if tc else "bwd_grad_kernel")
        fl = dict(zip(names, bwd_flops_per_token_head(w).values()))
        src, metric = BWD_KERNEL_SRC, BWD_METRIC
    else:
        params = hla.make_params(sets[0][0][0], sets[0][0][2], w.chunk)
        ws_bytes = hla.hla_forward3_workspace_size(params)
        tc = w.dtype == "bf16" and w.d == w.dv == w.chunk == 64  # local sums and outputs on the tensor cores
        names = ("fwd3_local_tc_kernel" if tc else "fwd3_local_kernel",
                 "fwd3_scan_tc_kernels" if tc else "fwd3_scan_kernel",
                 "fwd3_out_tc_kernel" if tc else "fwd3_out_kernel")
        fl = dict(zip(names, fwd3_flops_per_token_head(w).values()))
        src, metric = FWD3_KERNEL_SRC, FWD3_METRIC
        st3 = hla.State3.empty(w.B * w.H, w.d, w.dv, device=dev)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def call(ins, outs, s, events=None):
        if bwd:
            hla.hla_backward_chunked_traced(params, *ins, *outs, ws, ws_bytes, s, events)
        else:
            hla.hla_forward3_chunked_traced(params, *ins, outs[0], None, st3, ws, ws_bytes, s, events)

    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            call(*sets[i % nsets], stream)
    hla.hla_sync_status(stream)
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for e4 in evs:  # create the events
        for e in e4:
            e.record(stream)
    stream.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(gpu_selector(local)) as clk, torch.cuda.stream(stream):
        ev0.record(stream)
        for i in range(K):
            call(*sets[i % nsets], stream, evs[i])
        ev1.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    barrier(dist)
    hla.hla_sync_status(stream)
    t_max = max_over_ranks(dist, ev0.elapsed_time(ev1))
    ms_per_step = t_max / K
    value = world * w.tokens * K / (t_max / 1e3)
    phase_ms = {nm: sum(e4[j].elapsed_time(e4[j + 1]) for e4 in evs) / K for j, nm in enumerate(names)}

    # ---- end to end: the inputs uploaded and the results read back every step;
    # step i+1's upload and step i-1's download overlap step i (two buffer sets)
    Ke = min(K, 100)
    outs_host = [[torch.empty(t.shape, dtype=tdt).pin_memory() for t in sets[0][1]] for _ in range(2)]
    s_up, s_down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {kk: [torch.cuda.Event() for _ in range(2)] for kk in ("up", "run", "down")}

    def e2e_steps(n):
        for i in range(n):
            b = i % 2
            ins, outs = sets[b]
            if i >= 2:
                s_up.wait_event(ev["run"][b])
            with torch.cuda.stream(s_up):
                for dst, n_ in zip(ins, in_names):
                    dst.copy_(host[n_], non_blocking=True)
            ev["up"][b].record(s_up)
            stream.wait_event(ev["up"][b])
            if i >= 2:
                stream.wait_event(ev["down"][b])
            call(ins, outs, stream)
            ev["run"][b].record(stream)
            s_down.wait_event(ev["run"][b])
            with torch.cuda.stream(s_down):
                for dst, src_ in zip(outs_host[b], outs):
                    dst.copy_(src_, non_blocking=True)
            ev["down"][b].record(s_down)
        stream.wait_stream(s_up)
        stream.wait_stream(s_down)

    te = time_e2e(e2e_steps, Ke, stream, s_up, s_down, dist)
    hla.hla_sync_status(stream)
    e2e = {"value": world * w.tokens * Ke / (te / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": int(sum(host[n].numel() * host[n].element_size() for n in host)),
           "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in outs_host[0])), "steps": Ke,
           "overlap": "upload of step i+1 and download of step i-1 on their own streams during step i",
           "replay": "CUDA graphs of up to 50 such steps (uploads, library calls, downloads and their "
                     "cross-stream order captured), replayed back to back"}

    # ---- roofline of the dominant kernel: fp32 FMA work on the CUDA cores, or bf16
    # MMAs for the tensor-core kernels
    peaks, peak_kind = load_peaks()
    alu_src = "derived: 152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz (fp32 FMA, CUDA cores)"
    tc_src = (f"{peak_kind} bf16 dense (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback bf16 dense")

    def bound_of(nm):
        return ("tensor", peaks["bf16_tflops"], tc_src) if "_tc_" in nm else ("alu", FP32_ALU_TFLOPS, alu_src)

    def source_of(nm):  # the file whose hash keys the committed DRAM traffic of this phase
        if nm.startswith("bwd_norm_tc_"):
            return BWD_NORM_TC_SRC
        if "_scan_tc_" in nm:
            return SCAN_TC_SRC
        if "_tc_" in nm:
            return BWD_TC_KERNEL_SRC if bwd else FWD3_TC_KERNEL_SRC
        return src

    top = max(phase_ms, key=phase_ms.get)
    flops_launch = fl[top] * w.token_heads
    ach = flops_launch / (phase_ms[top] / 1e3) / 1e12
    bnd, peak, psrc = bound_of(top)
    src_top = source_of(top)
    roofline = {"bound": bnd, "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                "peak_source": psrc, "traffic": traffic_for(top, w.name, src_top), "kernel": top,
                "alg_flops_per_launch": flops_launch,
                "phases": {nm: {"ms": phase_ms[nm], "alg_flops": fl[nm] * w.token_heads,
                                "tflops": fl[nm] * w.token_heads / (phase_ms[nm] / 1e3) / 1e12 if phase_ms[nm] else None,
                                "bound": bound_of(nm)[0], "traffic": traffic_for(nm, w.name, source_of(nm)),
                                "frac": (fl[nm] * w.token_heads / (phase_ms[nm] / 1e3) / 1e12) / bound_of(nm)[1]
                                if phase_ms[nm] else None}
                           for nm in names},
                "alg_bytes_per_step": set_bytes}
    cfg = config_dict(w, nsets, set_bytes, world)
    if bwd:
        cfg["variant"] = ("backward of the ratio-normalised masked forward" if w.normalize else
                          "backward of the masked forward") + (" with decay" if w.decay else "")
        cfg["inputs"] += f", dout N(0,1) seed {w.seed + 1000}"
    else:
        cfg["variant"] = "masked third order"
    line = {"metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if tc else "f32", "data": "synthetic",
            "config": cfg, "roofline": roofline, "e2e": e2e, "gpu_launches": launches_per_step(w) * K,
            "clocks": clk.summary(),
            "token_heads_per_s": world * w.token_heads * K / (t_max / 1e3)}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_backward(w, x, gout) if bwd else cpu_baseline_third(w, x)
    return line


# ----------------------------------------------------------------- decode bench
def bench_decode(args, dw: W.DecodeWorkload, rank, world, local, dist):
    import torch
    import causal_prefix_scan_gb300 as hla
    from causal_prefix_scan_gb300 import _build
    _build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    N, d, dv = dw.seqs * dw.H, dw.d, dw.dv
    third = dw.order == 3
    if third:  # a drawn third-order state (S^K symmetric)
        gs = torch.Generator(device=dev)
        gs.manual_seed(dw.seed)
        a_ = torch.randn((N, d, d), generator=gs, device=dev) * 0.05
        st = hla.State3((a_ + a_.transpose(1, 2)).contiguous(),
                        torch.randn((N, d, dv), generator=gs, device=dev) * 0.05,
                        torch.randn((N, d, dv), generator=gs, device=dev) * 0.05)
        del a_
    # prefill the state with the forward over a seeded prefix (drawn on the device)
    if not third:
        st = hla.State.empty(N, d, dv, device=dev)
        for b0, pw in W.decode_prefix_blocks(dw):
            px = W.make_inputs_device(pw, device=dev)
            sub = hla.State(*(a[b0 * dw.H:(b0 + pw.B) * dw.H] for a in st.astuple()))
            p = hla.make_params(px["q"], px["v"], dw.chunk)
            need = hla.hla_forward_workspace_size(p)
            ws = hla.new_workspace(need, dev)
            o = torch.empty_like(px["v"])
            hla.hla_forward_chunked(p, px["q"], px["k"], px["v"], o, None, sub, ws, need)
            del px, o, ws
    torch.cuda.synchronize()
    hla.hla_sync_status()
    steps = args.steps
    T = min(steps, 64)  # distinct token sets cycled through
    toks = W.decode_tokens_device(dw, T, device=dev)
    # the oracle's continuation starts from the exact fp32 state of a seeded sample of pairs
    cpu_sample = None
    if rank == 0 and not third and not args.no_cpu_baseline:
        idx = np.sort(np.random.default_rng(dw.seed + 500).choice(N, 64, replace=False))
        ti = torch.from_numpy(idx).to(dev)
        cpu_sample = (idx, [a.index_select(0, ti).double().cpu().numpy() for a in st.astuple()],
                      [tuple(t.index_select(0, ti).float().cpu().numpy() for t in ts) for ts in toks])
    o = torch.empty((N, dv), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(i, s):
        q, k, v = toks[i % T]
        if third:
            hla.hla_decode3_step(N, 1, d, dv, hla.HLA_BF16, 0, 0.0, None, st, q, k, v, o, s)
        else:
            hla.hla_decode_step(N, dw.H, 0, d, dv, hla.HLA_BF16, 0, 0.0, None, st, q, k, v, o, s)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i, stream)
    stream.synchronize()
    R = min(steps, 64)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=stream, capture_error_mode="thread_local"):
        for i in range(R):
            step(i, torch.cuda.current_stream())
    g_rem = None
    if steps % R:
        g_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_rem, stream=stream, capture_error_mode="thread_local"):
            for i in range(steps % R):
                step(i, torch.cuda.current_stream())
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(gpu_selector(local)) as clk, torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(steps // R):
            gr.replay()
        if g_rem is not None:
            g_rem.replay()
        ev1.record(stream)
        stream.synchronize()
    barrier(dist)
    hla.hla_sync_status(stream)
    t_max = max_over_ranks(dist, ev0.elapsed_time(ev1))
    ms = t_max / steps
    value = world * dw.seqs * steps / (t_max / 1e3)
    state_bytes = (d * d + 2 * d * dv + (0 if third else 2 * d)) * 4
    bytes_step = N * (2 * state_bytes + (2 * d + 2 * dv) * 2)
    peaks, peak_kind = load_peaks()
    ach = bytes_step / (ms / 1e3) / 1e9
    # e2e: q,k,v host->device and o device->host every step
    hq, hk, hv = (toks[0][i].cpu().pin_memory() for i in range(3))
    ho = torch.empty((N, dv), dtype=torch.bfloat16).pin_memory()
    q, k, v = (torch.empty_like(t) for t in toks[0])
    Ke = min(steps, 100)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(Ke):
            q.copy_(hq, non_blocking=True); k.copy_(hk, non_blocking=True); v.copy_(hv, non_blocking=True)
            if third:
                hla.hla_decode3_step(N, 1, d, dv, hla.HLA_BF16, 0, 0.0, None, st, q, k, v, o, stream)
            else:
                hla.hla_decode_step(N, dw.H, 0, d, dv, hla.HLA_BF16, 0, 0.0, None, st, q, k, v, o, stream)
            ho.copy_(o, non_blocking=True)
        e1.record(stream)
    stream.synchronize()
    te = max_over_ranks(dist, e0.elapsed_time(e1))
    line = {"metric": ("third-order " if third else "") + "HLA decode step tokens/s and % HBM roofline on 1 GB300",
            "value": value,
            "unit": "tokens/s", "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": dw.name, "seqs": dw.seqs, "H": dw.H, "d": d, "dv": dv, "prefix": dw.prefix,
                       "l2": f"state {N * state_bytes / 2**30:.2f} GiB >> L2",
                       "state": "drawn N(0, 0.05^2), S^K symmetric" if third else "prefilled by the forward"},
            "roofline": {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": ach / peaks["hbm_gbs"],
                         "traffic": traffic_for("decode3_kernel" if third else "decode_kernel", dw.name,
                                                FWD3_DISPATCH_SRC if third else DECODE_KERNEL_SRC),
                         "kernel": "decode3_kernel" if third else "decode_kernel", "alg_bytes_per_launch": bytes_step,
                         "peak_source": peak_kind},
            "e2e": {"value": world * dw.seqs * Ke / (te / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": 3 * N * d * 2, "d2h_bytes_per_step": N * dv * 2, "steps": Ke},
            "gpu_launches": steps, "clocks": clk.summary()}
    if cpu_sample is not None:
        line["cpu_baseline"] = cpu_baseline_decode(dw, *cpu_sample)
    return line


def oracle_decode_rate(dw: W.DecodeWorkload, state, tok_sets, steps: int, nthreads: int):
    """Continue the fp64 oracle's decode from `state` (the sampled pairs' fp32 state,
    as oracle.State) for `steps` steps with the workload's token sets; returns seconds."""
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    for i in range(steps):
        q, k, v = tok_sets[i % len(tok_sets)]
        oracle.decode_step(state, q, k, v, 1, nthreads=nthreads)
    return time.perf_counter() - t0


def cpu_baseline_decode(dw: W.DecodeWorkload, idx, state_arrays, tok_sets):
    """The oracle's decode step continued from the prefilled fp32 state of a seeded
    sample of (sequence, head) pairs for about 10 s; tokens/s counts sequence steps
    (H pair steps each), the unit of the GPU line."""
    import oracle
    cores = cpu_threads()
    used = min(cores, len(idx))
    st = oracle.State(*(np.array(a, dtype=np.float64) for a in state_arrays))
    secs = oracle_decode_rate(dw, st, tok_sets, 4, used)
    steps = int(max(4, min(dw.steps, 10.0 * 4 / max(secs, 1e-9))))
    st = oracle.State(*(np.array(a, dtype=np.float64) for a in state_arrays))
    secs = oracle_decode_rate(dw, st, tok_sets, steps, used)
    pair_steps = len(idx) * steps
    return {"value": pair_steps / dw.H / secs, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"fp64 decode step continued from the prefilled fp32 state of {len(idx)} of {dw.seqs * dw.H} "
                      f"(sequence, head) pairs for {steps} of {dw.steps} steps, threads over pairs; "
                      f"tokens = pair steps / H", "seconds": secs}


# ----------------------------------------------------------------- reference arm
def bench_reference(args, w, rank, world):
    """The oracle as it stands, on the host cores: each step one bounded sample of
    the workload (one batch row, all heads, a window of tokens)."""
    if isinstance(w, W.DecodeWorkload):
        if w.order == 3:
            return {"impl": "reference", "unavailable": "the oracle has no third-order decode step"}
        return bench_reference_decode(args, w, world)
    x = W.make_inputs(w)
    cores = min(cpu_threads(), w.H)
    if is_backward(w):
        return bench_reference_backward(args, w, x, cores, world)
    if is_third(w):
        return bench_reference_third(args, w, x, cores, world)
    secs, _ = oracle_rate(w, x, 1, min(w.n, 128), cores)
    budget = 90.0 / max(1, args.steps + args.warmup)
    n_s = int(max(16, min(w.n, 128 * budget / max(secs, 1e-9))))
    import oracle
    sl = lambda a, t0: np.ascontiguousarray(a[:1, :, t0:t0 + n_s], dtype=np.float64)
    g = None if x["gamma"] is None else np.asarray(x["gamma"], np.float64)
    offs = list(range(0, max(1, w.n - n_s + 1), max(1, n_s)))

    def one(i):
        t0 = offs[i % len(offs)]
        oracle.forward(sl(x["q"], t0), sl(x["k"], t0), sl(x["v"], t0), gamma=g, normalize=w.normalize,
                       eps=w.eps, nthreads=cores, unmasked=w.unmasked, asymmetric=w.asymmetric)

    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(i)
    dt = time.perf_counter() - t0
    value = n_s * args.steps / dt
    sample = f"fp64 serial recurrence on 1 batch row x {w.H} heads x {n_s}-token windows per step"
    return {"impl": "reference", "metric": metric_for(w), "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(w, 1, 0, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def bench_reference_decode(args, dw: W.DecodeWorkload, world):
    """The oracle's decode step on the host cores: 64 (sequence, head) pairs whose
    state the oracle prefills over a host-drawn 256-token prefix of the workload's
    recipe (untimed; the cost of a step does not depend on the state's values), then
    each step continues them for a window of steps sized so the run ends in about 90 s."""
    import oracle
    P = 64
    cores = min(cpu_threads(), P)
    pre = W.make_inputs(W.Workload("decode_ref_prefix", 1, P, 256, dw.d, dw.dv, 64, "bf16", "l2", seed=dw.seed))
    _, st = oracle.forward(pre["q"], pre["k"], pre["v"], nthreads=cores)
    toks = W.make_decode_tokens(1, P, dw.d, dw.dv, 16, seed=dw.seed)
    sets = [(toks["q"][i], toks["k"][i], toks["v"][i]) for i in range(16)]
    secs = oracle_decode_rate(dw, st.copy(), sets, 4, cores) / 4
    budget = 90.0 / max(1, args.steps + args.warmup)
    s_per = int(max(1, min(dw.steps, budget / max(secs, 1e-9))))
    for _ in range(args.warmup):
        oracle_decode_rate(dw, st, sets, s_per, cores)
    dt = sum(oracle_decode_rate(dw, st, sets, s_per, cores) for _ in range(args.steps))
    value = P * s_per * args.steps / dw.H / dt
    sample = (f"fp64 decode step on {P} of {dw.seqs * dw.H} (sequence, head) pairs x {s_per} steps per step, "
              f"from an oracle-prefilled 256-token prefix; tokens = pair steps / H")
    cfg = {"workload": dw.name, "seqs": dw.seqs, "H": dw.H, "d": dw.d, "dv": dw.dv, "prefix": dw.prefix,
           "sample": sample}
    return {"impl": "reference", "metric": "HLA decode step tokens/s and % HBM roofline on 1 GB300", "value": value,
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def bench_reference_third(args, w, x, cores, world):
    """The third-order oracle on the host cores: each step 1 batch row x H heads x a
    window of tokens (from a zero state)."""
    import oracle
    secs, _ = oracle3_rate(x, 1, min(w.n, 128), cores)
    budget = 90.0 / max(1, args.steps + args.warmup)
    n_s = int(max(16, min(w.n, 128 * budget / max(secs, 1e-9))))
    sl = lambda a, t0: np.ascontiguousarray(a[:1, :, t0:t0 + n_s], dtype=np.float64)
    offs = list(range(0, max(1, w.n - n_s + 1), max(1, n_s)))

    def one(i):
        t0 = offs[i % len(offs)]
        oracle.forward3(sl(x["q"], t0), sl(x["k"], t0), sl(x["v"], t0), nthreads=cores)

    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(i)
    dt = time.perf_counter() - t0
    value = n_s * args.steps / dt
    sample = f"fp64 serial third-order recurrence on 1 batch row x {w.H} heads x {n_s}-token windows per step"
    return {"impl": "reference", "metric": FWD3_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(w, 1, 0, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def bench_reference_backward(args, w, x, cores, world):
    """The oracle's gradient on the host cores: each step 1 batch row x H heads x a
    window of tokens (the gradient of a window from a zero state)."""
    import oracle
    gout = W.make_dout(w)
    secs, _ = oracle_bwd_rate(x, gout, 1, min(w.n, 128), cores, w)
    budget = 90.0 / max(1, args.steps + args.warmup)
    n_s = int(max(16, min(w.n, 128 * budget / max(secs, 1e-9))))
    sl = lambda a, t0: np.ascontiguousarray(a[:1, :, t0:t0 + n_s], dtype=np.float64)
    gam = None if x["gamma"] is None else np.asarray(x["gamma"], np.float64)
    offs = list(range(0, max(1, w.n - n_s + 1), max(1, n_s)))

    def one(i):
        t0 = offs[i % len(offs)]
        oracle.backward(sl(x["q"], t0), sl(x["k"], t0), sl(x["v"], t0), sl(gout, t0), gam, nthreads=cores,
                        **(dict(normalize=True, eps=w.eps) if w.normalize else {}))

    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(i)
    dt = time.perf_counter() - t0
    value = n_s * args.steps / dt
    sample = f"fp64 reverse-mode recurrence on 1 batch row x {w.H} heads x {n_s}-token windows per step"
    return {"impl": "reference", "metric": BWD_METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(w, 1, 0, world),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=W.FWD_BF16.name)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    rank, world, local = dist_env()
    w = workload_by_name(args.workload)
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(bench_reference(args, w, rank, world)), flush=True)
        return
    dist = dist_init(world)
    if isinstance(w, W.DecodeWorkload):
        line = bench_decode(args, w, rank, world, local, dist)
    elif is_backward(w) or is_third(w):
        line = bench_phased(args, w, rank, world, local, dist)
    else:
        line = bench_forward(args, w, rank, world, local, dist)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
