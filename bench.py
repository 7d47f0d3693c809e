#!/usr/bin/env python3
"""Benchmark of the fused attention forward on GB300.

``python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
[--workload NAME]`` prints ONE JSON line.

A step is one ``attn_fwd`` call over the whole workload (default: B=2, H=16,
Sq=Sk=8192, D=128, non-causal, bf16 N(0,1) inputs from seed 3).  ``value`` is
whole-job TFLOP/s (4*B*H*Sq*Sk*D per step, halved when causal) with inputs
resident in HBM; every step re-reads 192 MiB of Q/K/V (plus 64 MiB of O
written), more than the 129 MB L2, so no explicit flush is needed.  Smaller
workloads (``--workload``) get a 256 MiB L2 flush before every timed launch and
report the launch time alone.  The ``varlen_*`` workloads time
``attn_fwd_varlen`` on a packed batch of variable-length sequences, the
``paged_*`` ones ``attn_fwd_paged`` on the same batch with its keys and values
in a paged cache.

Under torchrun (N > 1) every rank runs the same workload on its own GPU (weak
scaling: the attention units shard with no exchange step); the barrier and the
max over ranks use torch.distributed, never the data path.

``--impl reference`` times the CPU oracle (fp64, materialised softmax) on the
host cores instead: each step is one 256-row query block of one head against
all keys, cycling over the workload's blocks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused attention fwd TFLOP/s (bf16) and % of GB300 dense BF16 tensor peak"
METRIC_BWD = "fused attention bwd TFLOP/s (bf16, 2.5x the forward FLOPs) and % of GB300 dense BF16 tensor peak"
FALLBACK_PEAK_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
# every source file of the translation unit that holds the forward kernel
# (attn_fwd.cu includes the PTX wrappers and the backward kernels)
KERNEL_SOURCES = ["exact_attention_86_gb300/csrc/attn_fwd.cu", "exact_attention_86_gb300/csrc/sm103_ptx.cuh",
                  "exact_attention_86_gb300/csrc/attn_bwd.cuh", "include/attn.h"]
TRAFFIC_FILE = "profiles/attn_fwd_kernel_s8192_d128_traffic.md"
L2_BYTES = 129 * 10**6


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source and this workload; else None."""
    path = os.path.join(ROOT, TRAFFIC_FILE)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    src = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    wl = re.search(r"workload:\s*(\S+)", text)
    val = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (src and wl and val) or src.group(1) != kernel_source_hash() or wl.group(1) != workload:
        return None
    return float(val.group(1))


def roofline_bound(flops: float, min_bytes: int, launch_ms: float, peak_tflops: float, hbm_gbs: float,
                   backward: bool = False) -> dict:
    """The launch against its ceiling: the tensor cores when the arithmetic
    intensity (FLOPs per algorithmic byte) is at or above the ridge of the two
    peaks, HBM below it (a query block against long keys, the small shapes).
    The backward reads and writes about twice the forward's bytes for 2.5 x
    its FLOPs and is taken as tensor-bound."""
    intensity = flops / min_bytes
    ridge = peak_tflops * 1e12 / (hbm_gbs * 1e9)
    if backward or intensity >= ridge:
        achieved = flops / (launch_ms * 1e-3) / 1e12
        out = {"bound": "tensor", "achieved": achieved, "peak": peak_tflops, "unit": "TFLOP/s"}
    else:
        achieved = min_bytes / (launch_ms * 1e-3) / 1e9
        out = {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s"}
    out["frac"] = achieved / out["peak"]
    out["intensity_flop_per_byte"] = intensity
    out["ridge_flop_per_byte"] = ridge
    return out


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((ts, parts))
        window = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05] or rows
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for _, p in window if num(p[1]) is not None]
        mx = [num(p[2]) for _, p in window if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, p in window:
            for name, val in zip(names, p[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(window),
                "power_w_max": max((num(p[3]) or 0.0) for _, p in window)}


def oracle_heads(w, q, k, v, kv):
    """The (q_head, k_head, v_head, kv_len) slices the CPU oracle walks: head 0
    of batch entry 0 for a padded workload; head 0 of every sequence for a
    packed variable-length one (``kv`` is then the offsets array)."""
    import numpy as np

    from exact_attention_86_gb300 import workloads

    f64 = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
    if isinstance(w, workloads.Fp8Workload):
        from oracle import decode_e4m3
        f64 = lambda t: decode_e4m3(t.numpy()) * w.descale  # noqa: E731
    if isinstance(w, workloads.VarlenWorkload):
        cu = [int(x) for x in kv]
        return [(f64(q[a:b, 0]), f64(k[a:b, 0]), f64(v[a:b, 0]), None)
                for a, b in zip(cu[:-1], cu[1:]) if b > a]
    return [(f64(q[0, 0]), f64(k[0, 0]), f64(v[0, 0]), None if kv is None else int(kv[0]))]


def cpu_oracle_steps(w, q, k, v, kv, n_steps: int, budget_s: float | None):
    """Runs the fp64 oracle on successive 256-row query blocks of the heads
    ``oracle_heads`` lists.  Returns (flops, seconds, blocks)."""
    from oracle import attention_rows

    blocks = [(h, r0) for h in oracle_heads(w, q, k, v, kv) for r0 in range(0, h[0].shape[0], 256)]
    flops = 0.0
    t0 = time.perf_counter()
    i = 0
    while True:
        (qh, kh, vh, kvb), r0 = blocks[i % len(blocks)]
        sq, sk = qh.shape[0], kh.shape[0]
        rows = list(range(r0, min(sq, r0 + 256)))
        attention_rows(qh, kh, vh, rows, w.scale, causal=w.causal, kv_len=kvb)
        keys = sk if kvb is None else min(max(kvb, 0), sk)
        for r in rows:
            n = min(keys, r + 1) if w.causal else keys
            flops += 4.0 * n * w.D
        i += 1
        el = time.perf_counter() - t0
        if n_steps is not None and i >= n_steps:
            break
        if budget_s is not None and el >= budget_s:
            break
    return flops, time.perf_counter() - t0, i


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        n = [d.get("num_threads") for d in info if d.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count() or 1


def max_over_ranks(values, device, world: int):
    """Element-wise maximum of a list of floats over all ranks (the job's time
    is its slowest rank's); a no-op for one rank.  torch.distributed carries
    only these timings, never attention data."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Weak scaling: every rank processes its own copy of the workload, so the
    job's rate is all ranks' units over the slowest rank's time (units/s)."""
    return units_per_rank * world / (ms * 1e-3)


def lookup(name):
    from exact_attention_86_gb300 import workloads
    tables = (workloads.WORKLOADS, workloads.VARLEN_WORKLOADS, workloads.PAGED_WORKLOADS, workloads.FP8_WORKLOADS)
    for table in tables:
        if name in table:
            return table[name]
    known = sorted(n for table in tables for n in table)
    raise SystemExit(f"unknown workload {name}; known: {known}")


def is_varlen(w) -> bool:
    """Packed variable-length workloads (paged ones included)."""
    from exact_attention_86_gb300 import workloads
    return isinstance(w, workloads.VarlenWorkload)


def is_paged(w) -> bool:
    from exact_attention_86_gb300 import workloads
    return isinstance(w, workloads.PagedWorkload)


def is_fp8(w) -> bool:
    from exact_attention_86_gb300 import workloads
    return isinstance(w, workloads.Fp8Workload)


def generate(w, draw: int):
    """(q, k, v, extra) with packed or padded keys: extra is kv_lens (padded)
    or the offsets (varlen; for a paged workload these are the same tokens
    its cache holds)."""
    from exact_attention_86_gb300 import workloads
    if is_varlen(w) or is_fp8(w):
        if draw != 0:
            raise SystemExit(f"workload {w.name} has a single draw")
    if is_varlen(w):
        return workloads.generate_varlen(w)
    if is_fp8(w):
        q8, k8, v8, _, kv = workloads.generate_fp8(w)
        return q8, k8, v8, kv
    return workloads.generate(w, draw)


class BwdJob:
    """The backward pass of a padded bf16 workload: the forward's O and LSE are
    computed once before timing; a step is one ``attn_bwd`` call (three
    kernels) for a fixed upstream gradient dO ~ N(0, 1) drawn after the
    workload's inputs."""

    def __init__(self, w, args, dev, attn, torch):
        from exact_attention_86_gb300 import workloads
        if is_varlen(w) or is_fp8(w) or args.splits > 0:
            raise SystemExit("--backward applies to padded bf16 workloads")
        self.stream = torch.cuda.current_stream(dev)
        sptr = self.stream.cuda_stream
        q, k, v, kv = workloads.generate(w, args.draw)
        g = torch.Generator().manual_seed(w.seed + 1000)
        dout = torch.randn(q.shape, generator=g).to(torch.bfloat16)
        qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), dout.to(dev)
        kvd = kv.to(dev) if kv is not None else None
        o, lse = attn.forward(qd, kd, vd, scale=w.scale, causal=w.causal, kv_lens=kvd)
        torch.cuda.synchronize(dev)
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        ws = torch.empty(max(attn.attn_bwd_workspace_size(w.B, w.H, w.Sq), 256), dtype=torch.uint8, device=dev)
        host = [q, k, v, o.cpu(), lse.cpu(), dout] + ([kv] if kv is not None else [])
        dev_t = [qd, kd, vd, o, lse, dod] + ([kvd] if kvd is not None else [])
        self.inputs = list(zip(host, dev_t))
        self.outputs = [dq, dk, dv]
        self.launches_per_step = 3
        kv_ptr = kvd.data_ptr() if kvd is not None else None

        def call():
            return attn.attn_bwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), dod.data_ptr(),
                                 lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.Sq, w.Sk,
                                 w.D, w.scale, int(w.causal), kv_ptr, ws.data_ptr(), ws.numel(), sptr)
        self._call = call
        self._attn = attn

    def step(self):
        st = self._call()
        if st != self._attn.ATTN_OK:
            raise self._attn.AttnError(st, "backward")


class Job:
    """Device buffers and the step of one workload.  ``inputs`` are (host,
    device) pairs the end-to-end step copies in; ``outputs`` the device
    tensors it copies back."""

    def __init__(self, w, args, dev, attn, torch):
        from exact_attention_86_gb300 import workloads
        self.stream = torch.cuda.current_stream(dev)
        sptr = self.stream.cuda_stream
        if args.splits > 0 and is_varlen(w):
            raise SystemExit("--splits applies to padded workloads only")
        if is_paged(w):
            q, kc, vc, cu, sk, table = workloads.generate_paged(w)
            host = [q, kc, vc, cu, sk, table]
        elif is_fp8(w):
            q, k8, _, vt8, kv = workloads.generate_fp8(w)
            host = [q, k8, vt8] + ([kv] if kv is not None else [])
        else:
            q, k, v, kv = generate(w, args.draw)
            host = [q, k, v] + ([kv] if kv is not None else [])
        dev_t = [t.to(dev) for t in host]
        self.inputs = list(zip(host, dev_t))
        o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        if is_varlen(w):
            lse = torch.empty(w.H, q.shape[0], dtype=torch.float32, device=dev)
        else:
            lse = torch.empty(w.B, w.H, w.Sq, dtype=torch.float32, device=dev)
        self.outputs = [o, lse]
        ptr = [t.data_ptr() for t in dev_t]
        total = q.shape[0]
        # packed and paged batches: dynamic scheduling through a persistent
        # counter (each launch leaves it zero); --static-schedule turns it off
        counter_ptr = None
        if is_varlen(w) and not args.static_schedule:
            self.counter = torch.zeros(2, dtype=torch.int32, device=dev)
            counter_ptr = self.counter.data_ptr()
        ws = None
        if args.splits > 0:
            ws_bytes = attn.attn_fwd_splitkv_workspace_size(w.B, w.H, w.Sq, w.D, args.splits)
            ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.launches_per_step = 2 if ws is not None else 1

        if is_paged(w):
            num_pages, page_size, max_pages = kc.shape[0], kc.shape[1], table.shape[1]

            def call():
                return attn.attn_fwd_paged(ptr[0], ptr[1], ptr[2], o.data_ptr(), lse.data_ptr(), ptr[3], ptr[4],
                                           ptr[5], w.batch, w.max_len, total, num_pages, page_size, max_pages, w.H,
                                           w.D, w.scale, int(w.causal), counter_ptr, sptr)
        elif is_fp8(w):
            kv_ptr = ptr[3] if len(ptr) > 3 else None

            def call():
                return attn.attn_fwd_fp8(ptr[0], ptr[1], ptr[2], o.data_ptr(), lse.data_ptr(), w.B, w.H, w.Sq, w.Sk,
                                         w.D, w.scale, int(w.causal), kv_ptr, w.descale, w.descale, w.descale, sptr)
        elif is_varlen(w):
            def call():
                return attn.attn_fwd_varlen(ptr[0], ptr[1], ptr[2], o.data_ptr(), lse.data_ptr(), ptr[3], ptr[3],
                                            w.batch, w.max_len, total, total, w.H, w.D, w.scale, int(w.causal),
                                            counter_ptr, sptr)
        elif ws is None:
            kv_ptr = ptr[3] if len(ptr) > 3 else None

            def call():
                return attn.attn_fwd(ptr[0], ptr[1], ptr[2], o.data_ptr(), lse.data_ptr(), w.B, w.H, w.Sq, w.Sk,
                                     w.D, w.scale, int(w.causal), kv_ptr, sptr)
        else:
            kv_ptr = ptr[3] if len(ptr) > 3 else None

            def call():
                return attn.attn_fwd_splitkv(ptr[0], ptr[1], ptr[2], o.data_ptr(), lse.data_ptr(), w.B, w.H, w.Sq,
                                             w.Sk, w.D, w.scale, int(w.causal), kv_ptr, args.splits, ws.data_ptr(),
                                             ws.numel(), sptr)
        self._call = call
        self._attn = attn

    def step(self):
        st = self._call()
        if st != self._attn.ATTN_OK:
            raise self._attn.AttnError(st, "forward")


def run_reference(args, w):
    """The CPU oracle as the reference arm."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    q, k, v, kv = generate(w, 0)
    cpu_oracle_steps(w, q, k, v, kv, n_steps=args.warmup, budget_s=None) if args.warmup > 0 else None
    flops, secs, blocks = cpu_oracle_steps(w, q, k, v, kv, n_steps=args.steps, budget_s=None)
    tflops = flops / secs / 1e12
    sample = (f"{blocks} steps; each one 256-row query block of head 0 of "
              f"{'a sequence' if is_varlen(w) else 'batch entry 0'} against all its keys, fp64 NumPy/BLAS")
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / max(blocks, 1) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "shape": w.label(), "oracle": "fp64 materialised softmax (CPU)"},
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None)
    ap.add_argument("--draw", type=int, default=0)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--static-schedule", action="store_true",
                    help="packed/paged workloads: deal the units round-robin instead of claiming them")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward pass (dQ, dK, dV) of the workload instead of the forward")
    ap.add_argument("--splits", type=int, default=0,
                    help="use the split-KV forward with this many key ranges (0: the plain forward; "
                         "-1: attn.suggest_num_splits for the device)")
    args = ap.parse_args()

    from exact_attention_86_gb300 import workloads
    w = lookup(args.workload or workloads.HEADLINE)
    varlen = is_varlen(w)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    if args.impl == "reference":
        return run_reference(args, w)

    import torch
    import torch.distributed as dist
    from exact_attention_86_gb300 import attn
    from exact_attention_86_gb300.build import build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    if args.splits < 0:
        if varlen:
            raise SystemExit("--splits applies to padded workloads only")
        args.splits = attn.suggest_num_splits(w.B, w.H, w.Sq, w.Sk,
                                              torch.cuda.get_device_properties(dev).multi_processor_count)

    if rank == 0:
        build()
    if world > 1:
        dist.barrier()
    attn.lib()

    job = (BwdJob if args.backward else Job)(w, args, dev, attn, torch)
    # FLOPs of a step: the forward's; the backward counts 2.5 times that (its
    # five products against the forward's two, the usual count)
    step_flops = w.flops * (2.5 if args.backward else 1.0)
    stream = job.stream
    sptr = stream.cuda_stream
    step = job.step

    # Workloads whose bytes fit in L2 get an L2 flush (a 256 MiB write) before
    # every timed launch; the launch events bracket the kernel alone.
    flush = None
    if w.min_bytes < 2 * L2_BYTES:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        step()
    st, site = attn.attn_check_device_status(sptr)
    if st != attn.ATTN_OK:
        raise attn.AttnError(st, f"warm-up (site {site})")

    # ---------------------------------------------------------- device-timed
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    for _ in range(max(args.warmup, 20)):
        step()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    barrier()
    wall0 = time.time()
    t_all0.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_all1.record(stream)
    barrier()
    wall1 = time.time()
    sampler.stop()
    st, site = attn.attn_check_device_status(sptr)
    if st != attn.ATTN_OK:
        raise attn.AttnError(st, f"timed region (site {site})")
    elapsed_ms = t_all0.elapsed_time(t_all1)
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    elapsed_ms, launch_ms = max_over_ranks([elapsed_ms, launch_ms], dev, world)
    # with an L2 flush between launches the step time is the launch alone
    ms_per_step = launch_ms if flush is not None else elapsed_ms / args.steps
    value = whole_job_rate(step_flops, world, ms_per_step) / 1e12
    clocks = sampler.summary(wall0, wall1)

    # ------------------------------------------------------------ end to end
    pinned = [(h.pin_memory(), d) for h, d in job.inputs]
    outs_h = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in job.outputs]

    def e2e_step():
        for h, d in pinned:
            d.copy_(h, non_blocking=True)
        step()
        for h, d in zip(outs_h, job.outputs):
            h.copy_(d, non_blocking=True)

    for _ in range(3):
        e2e_step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    (e2e_ms,) = max_over_ranks([e2e_ms], dev, world)
    h2d = sum(h.numel() * h.element_size() for h, _ in pinned)
    d2h = sum(t.numel() * t.element_size() for t in job.outputs)

    # -------------------------------------------------------------- roofline
    peaks = measured_peaks()
    if peaks and peaks.get("bf16_tflops"):
        peak = float(peaks["bf16_tflops"])
        peak_src = "measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)"
    else:
        peak = FALLBACK_PEAK_TFLOPS
        peak_src = "fallback (1.9 PFLOP/s bf16 burst)"
    if is_fp8(w):
        # the E4M3 contraction's own peak: the bf16 figure times the nominal
        # dense fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s)
        peak *= 2.0
        peak_src += " x 2 (nominal dense fp8 / bf16 ratio)"
    if peaks and peaks.get("hbm_gbs"):
        hbm = float(peaks["hbm_gbs"])
        hbm_src = "measured (MEASURED_PEAKS.json hbm_gbs, copy)"
    else:
        hbm = FALLBACK_HBM_GBS
        hbm_src = "fallback (6.8 TB/s copy)"
    roofline = roofline_bound(step_flops, w.min_bytes, launch_ms, peak, hbm, args.backward)
    roofline["peak_source"] = peak_src if roofline["bound"] == "tensor" else hbm_src
    roofline.update({"traffic": None if args.backward else recorded_traffic(w.name),
                     "kernel": "attn_bwd (delta, dq, dkdv kernels)" if args.backward else "attn_fwd_kernel",
                     "launch_ms": launch_ms, "algorithmic_flops_per_launch": step_flops,
                     "algorithmic_bytes_per_launch": w.min_bytes})

    # ----------------------------------------------------------- CPU oracle
    cpu = None
    if rank == 0 and not args.no_cpu_baseline and not args.backward:
        q, k, v, kv = generate(w, args.draw)
        flops, secs, blocks = cpu_oracle_steps(w, q, k, v, kv, n_steps=None, budget_s=args.cpu_budget_s)
        cpu = {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
               "sample": f"{blocks} query blocks of 256 rows of head 0 of "
                         f"{'the sequences' if varlen else 'batch entry 0'} against all their keys "
                         f"({secs:.1f} s of fp64 NumPy/BLAS)"}

    if rank == 0:
        line = {
            "metric": METRIC_BWD if args.backward else METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3" if is_fp8(w) else "bf16", "data": "synthetic",
            "config": {"workload": w.name, "shape": w.label(), "draw": args.draw,
                       "inputs": f"{'e4m3' if is_fp8(w) else 'bf16'} "
                                 f"N(0,{(w.std if args.draw == 0 else w.second_std) ** 2:g}) seed {w.seed}",
                       "l2": (f"flushed: a 256 MiB write before every timed launch (the workload moves "
                              f"{w.min_bytes / 2**20:.1f} MiB)") if flush is not None else
                             (f"no flush: each step moves {w.min_bytes / 2**20:.0f} MiB of Q/K/V/O/LSE, more "
                              f"than the 129 MB L2"),
                       "parallelism": f"weak: {world} replica(s) of the workload, one per GPU",
                       "splits": args.splits,
                       "schedule": ("static" if args.static_schedule or w.causal else "dynamic") if varlen
                                   else "static"},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": whole_job_rate(step_flops, world, e2e_ms) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "clocks": clocks,
            "gpu_launches": args.steps * job.launches_per_step,
            "pct_of_peak": 100.0 * value / world / peak,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
