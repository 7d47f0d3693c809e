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
# The sources each forward kernel's translation unit compiles from: a traffic
# record under profiles/ counts only while their hash is the one it names.
_CSRC = "exact_attention_86_gb300/csrc/"
KERNEL_SOURCES = {
    "attn_fwd_kernel": [_CSRC + n for n in ("attn_fwd.cu", "attn_common.cuh", "sm103_ptx.cuh", "attn_bwd.cuh",
                                            "attn_pair_host.h")] + ["include/attn.h"],
    "attn_fwd_pair_kernel": [_CSRC + n for n in ("attn_fwd_pair.cu", "attn_common.cuh", "sm103_ptx.cuh",
                                                 "attn_pair_host.h")],
}
L2_BYTES = 129 * 10**6


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary
    ``profiles/<kernel>_<workload>_traffic.md``, if it was taken on the current
    kernel source and this workload; else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}_traffic.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    src = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    wl = re.search(r"workload:\s*(\S+)", text)
    val = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (src and wl and val) or src.group(1) != kernel_source_hash(kernel) or wl.group(1) != workload:
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


def forward_kernel(w, splits: int, num_sms: int) -> str:
    """The kernel that does the forward's work for this workload, as the
    library chooses it: padded batches (bf16 or E4M3) without key ranges may
    run the two-query-tile kernel (attn_fwd_kernel_choice,
    attn_fwd_fp8_kernel_choice); packed and paged
    batches run it when a sequence may hold more than one query tile; split
    batches run the one-tile kernel."""
    from exact_attention_86_gb300 import attn
    if is_varlen(w):
        return "attn_fwd_pair_kernel" if w.max_len > 128 else "attn_fwd_kernel"
    choice = attn.attn_fwd_fp8_kernel_choice if is_fp8(w) else attn.attn_fwd_kernel_choice
    if splits == 0 and choice(w.B, w.H, w.Sq, w.Sk, w.D, int(w.causal), num_sms) == 1:
        return "attn_fwd_pair_kernel"
    return "attn_fwd_kernel"


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


class BufferSet:
    """One set of device buffers for a job: the inputs (device copies of the
    job's host tensors), the outputs, and the library call that reads and
    writes them on the compute stream."""

    def __init__(self, dev_inputs, outputs, call, keep=()):
        self.inputs = dev_inputs
        self.outputs = outputs
        self.call = call
        self.keep = list(keep)  # other device buffers the call uses (scheduling counter, workspace)


class _JobBase:
    """A workload's host inputs and one or more device buffer sets.  Set 0 is
    what the device-timed loop launches; the end-to-end loop alternates two
    sets so that one step's copies run under another step's kernel."""

    def add_set(self):
        self.sets.append(self._make_set())
        return self.sets[-1]

    def step(self, k: int = 0):
        st = self.sets[k].call()
        if st != self._attn.ATTN_OK:
            raise self._attn.AttnError(st, self._what)


class BwdJob(_JobBase):
    """The backward pass of a padded bf16 workload: the forward's O and LSE are
    computed once before timing; a step is one ``attn_bwd`` call (three
    kernels) for a fixed upstream gradient dO ~ N(0, 1) drawn after the
    workload's inputs."""

    def __init__(self, w, args, dev, attn, torch):
        from exact_attention_86_gb300 import workloads
        if is_varlen(w) or is_fp8(w) or args.splits > 0:
            raise SystemExit("--backward applies to padded bf16 workloads")
        self._attn, self._what, self.w, self.dev, self.torch = attn, "backward", w, dev, torch
        self.stream = torch.cuda.current_stream(dev)
        q, k, v, kv = workloads.generate(w, args.draw)
        g = torch.Generator().manual_seed(w.seed + 1000)
        dout = torch.randn(q.shape, generator=g).to(torch.bfloat16)
        kvd = kv.to(dev) if kv is not None else None
        o, lse = attn.forward(q.to(dev), k.to(dev), v.to(dev), scale=w.scale, causal=w.causal, kv_lens=kvd)
        torch.cuda.synchronize(dev)
        self.host = [q, k, v, o.cpu(), lse.cpu(), dout] + ([kv] if kv is not None else [])
        self.launches_per_step = 3
        self.sets = [self._make_set()]

    def _make_set(self):
        w, torch, attn = self.w, self.torch, self._attn
        d = [t.to(self.dev) for t in self.host]
        qd, kd, vd, o, lse, dod = d[:6]
        kv_ptr = d[6].data_ptr() if len(d) > 6 else None
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        ws = torch.empty(max(attn.attn_bwd_workspace_size(w.B, w.H, w.Sq), 256), dtype=torch.uint8, device=self.dev)
        sptr = self.stream.cuda_stream

        def call():
            return attn.attn_bwd(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), o.data_ptr(), dod.data_ptr(),
                                 lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), w.B, w.H, w.Sq, w.Sk,
                                 w.D, w.scale, int(w.causal), kv_ptr, ws.data_ptr(), ws.numel(), sptr)
        return BufferSet(d, [dq, dk, dv], call)


class Job(_JobBase):
    """The forward of one workload.  The host inputs are what the end-to-end
    step copies in; the outputs what it copies back."""

    def __init__(self, w, args, dev, attn, torch):
        self._attn, self._what, self.w, self.dev, self.torch, self.args = attn, "forward", w, dev, torch, args
        self.stream = torch.cuda.current_stream(dev)
        if args.splits > 0 and is_varlen(w):
            raise SystemExit("--splits applies to padded workloads only")
        if is_paged(w):
            q, kc, vc, cu, sk, table = workloads_mod().generate_paged(w)
            self.host = [q, kc, vc, cu, sk, table]
            self.paged_dims = (kc.shape[0], kc.shape[1], table.shape[1])
        elif is_fp8(w):
            q, k8, v8, vt8, kv = workloads_mod().generate_fp8(w)
            self.host = [q, k8, v8 if w.v_layout == "rows" else vt8] + ([kv] if kv is not None else [])
        else:
            q, k, v, kv = generate(w, args.draw)
            self.host = [q, k, v] + ([kv] if kv is not None else [])
        self.launches_per_step = 2 if args.splits > 0 else 1
        self.sets = [self._make_set()]

    def _make_set(self):
        w, torch, attn, args, dev = self.w, self.torch, self._attn, self.args, self.dev
        sptr = self.stream.cuda_stream
        dev_t = [t.to(dev) for t in self.host]
        q = self.host[0]
        o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        if is_varlen(w):
            lse = torch.empty(w.H, q.shape[0], dtype=torch.float32, device=dev)
        else:
            lse = torch.empty(w.B, w.H, w.Sq, dtype=torch.float32, device=dev)
        ptr = [t.data_ptr() for t in dev_t]
        total = q.shape[0]
        # packed and paged batches: dynamic scheduling through a persistent
        # counter (each launch leaves it zero); --static-schedule turns it off
        counter_ptr = None
        keep = []
        if is_varlen(w) and not args.static_schedule:
            counter = torch.zeros(2, dtype=torch.int32, device=dev)
            keep.append(counter)
            counter_ptr = counter.data_ptr()
        ws = None
        if args.splits > 0:
            ws_bytes = attn.attn_fwd_splitkv_workspace_size(w.B, w.H, w.Sq, w.D, args.splits)
            ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
            keep.append(ws)

        if is_paged(w):
            num_pages, page_size, max_pages = self.paged_dims

            def call():
                return attn.attn_fwd_paged(ptr[0], ptr[1], ptr[2], o.data_ptr(), lse.data_ptr(), ptr[3], ptr[4],
                                           ptr[5], w.batch, w.max_len, total, num_pages, page_size, max_pages, w.H,
                                           w.D, w.scale, int(w.causal), counter_ptr, sptr)
        elif is_fp8(w):
            kv_ptr = ptr[3] if len(self.host) > 3 else None

            layout = attn.ATTN_V_ROWS if w.v_layout == "rows" else attn.ATTN_V_TRANSPOSED

            def call():
                return attn.attn_fwd_fp8_ex(ptr[0], ptr[1], ptr[2], o.data_ptr(), lse.data_ptr(), w.B, w.H, w.Sq,
                                            w.Sk, w.D, w.scale, int(w.causal), kv_ptr, w.descale, w.descale,
                                            w.descale, layout, sptr)
        elif is_varlen(w):
            def call():
                return attn.attn_fwd_varlen(ptr[0], ptr[1], ptr[2], o.data_ptr(), lse.data_ptr(), ptr[3], ptr[3],
                                            w.batch, w.max_len, total, total, w.H, w.D, w.scale, int(w.causal),
                                            counter_ptr, sptr)
        elif ws is None:
            kv_ptr = ptr[3] if len(self.host) > 3 else None

            def call():
                return attn.attn_fwd(ptr[0], ptr[1], ptr[2], o.data_ptr(), lse.data_ptr(), w.B, w.H, w.Sq, w.Sk,
                                     w.D, w.scale, int(w.causal), kv_ptr, sptr)
        else:
            kv_ptr = ptr[3] if len(self.host) > 3 else None

            def call():
                return attn.attn_fwd_splitkv(ptr[0], ptr[1], ptr[2], o.data_ptr(), lse.data_ptr(), w.B, w.H, w.Sq,
                                             w.Sk, w.D, w.scale, int(w.causal), kv_ptr, args.splits, ws.data_ptr(),
                                             ws.numel(), sptr)
        return BufferSet(dev_t, [o, lse], call, keep)


def workloads_mod():
    from exact_attention_86_gb300 import workloads
    return workloads


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

    # ---------------------------------------------------------- launch floor
    # Small workloads: the same launch shape with no work (mode 0) and with
    # only the kernel's fixed set-up / tear-down (mode 1), each timed like the
    # workload (an L2 flush before every launch), so that the line separates
    # the floor from the work.
    floor = None
    if flush is not None and not args.backward and not is_varlen(w) and args.splits == 0:
        n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
        units = w.B * w.H * ((w.Sq + 127) // 128)
        grid = max(1, min(units, n_sms))
        floor = {"grid": grid}
        for mode, name in ((0, "empty_us"), (1, "setup_teardown_us")):
            n = min(args.steps, 200)
            fe = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
            for i in range(n + 3):
                flush.fill_(i & 0xFF)
                if i >= 3:
                    fe[i - 3][0].record(stream)
                st = attn.attn_selftest_launch_floor(grid, w.D, mode, sptr)
                if st != attn.ATTN_OK:
                    raise attn.AttnError(st, "launch floor")
                if i >= 3:
                    fe[i - 3][1].record(stream)
            torch.cuda.synchronize(dev)
            floor[name] = 1e3 * statistics.mean(a.elapsed_time(b) for a, b in fe)
        floor["workload_us"] = 1e3 * launch_ms

    # ------------------------------------------------------------ end to end
    # Every step copies its own inputs in from pinned host memory, runs the
    # library call and copies its own outputs back, all inside the timed
    # region.  Two device buffer sets alternate: the host-to-device copy of
    # step i+1 (copy-in stream) and the device-to-host copy of step i-1
    # (copy-out stream) run under the kernel of step i; events order each
    # copy after the last kernel that used its buffers.
    job.add_set()
    pinned_in = [t.pin_memory() for t in job.host]
    outs_h = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in job.sets[0].outputs] for _ in range(2)]
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)

    def new_event():
        return torch.cuda.Event()

    def e2e_run(n: int):
        computed = [None, None]    # kernel of the last step on set k done
        copied_out = [None, None]  # device-to-host copy of the last step on set k done
        start = new_event()
        start.record(stream)
        s_in.wait_event(start)
        s_out.wait_event(start)
        for i in range(n):
            kset = i % 2
            bs = job.sets[kset]
            with torch.cuda.stream(s_in):
                if computed[kset] is not None:
                    s_in.wait_event(computed[kset])
                for h, d in zip(pinned_in, bs.inputs):
                    d.copy_(h, non_blocking=True)
                copied_in = new_event()
                copied_in.record(s_in)
            stream.wait_event(copied_in)
            if copied_out[kset] is not None:
                stream.wait_event(copied_out[kset])
            job.step(kset)
            done = new_event()
            done.record(stream)
            computed[kset] = done
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                for h, d in zip(outs_h[kset], bs.outputs):
                    h.copy_(d, non_blocking=True)
                out_done = new_event()
                out_done.record(s_out)
                copied_out[kset] = out_done
        for e in copied_out:
            if e is not None:
                stream.wait_event(e)

    e2e_run(3)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.e2e_steps)
    e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    (e2e_ms,) = max_over_ranks([e2e_ms], dev, world)
    h2d = sum(h.numel() * h.element_size() for h in pinned_in)
    d2h = sum(t.numel() * t.element_size() for t in job.sets[0].outputs)

    # the box's pinned copy rates for these buffers, each direction alone
    def copy_ms(fn, reps=5):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        fn()
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / reps

    h2d_ms = copy_ms(lambda: [d.copy_(h, non_blocking=True) for h, d in zip(pinned_in, job.sets[0].inputs)])
    d2h_ms = copy_ms(lambda: [h.copy_(d, non_blocking=True) for h, d in zip(outs_h[0], job.sets[0].outputs)])
    e2e_bound_ms = max(h2d_ms, d2h_ms, ms_per_step)

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
    kernel = "attn_bwd (delta, dq, dkdv kernels)" if args.backward else forward_kernel(
        w, args.splits, torch.cuda.get_device_properties(dev).multi_processor_count)
    roofline.update({"traffic": None if args.backward else recorded_traffic(kernel, w.name),
                     "kernel": kernel,
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
                       "v_layout": (w.v_layout if is_fp8(w) else "rows"),
                       "schedule": ("static" if args.static_schedule or (w.causal and kernel == "attn_fwd_kernel")
                                    else "dynamic") if varlen else "static"},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": {"value": whole_job_rate(step_flops, world, e2e_ms) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "pipeline": "two device buffer sets; copy-in and copy-out streams overlap the next and "
                                "previous steps' copies with each kernel",
                    "h2d_gbs": h2d / (h2d_ms * 1e-3) / 1e9, "d2h_gbs": d2h / (d2h_ms * 1e-3) / 1e9,
                    "bound_ms_per_step": e2e_bound_ms,
                    "bound_value": whole_job_rate(step_flops, world, e2e_bound_ms) / 1e12},
            "clocks": clocks,
            "launch_floor": floor,
            "gpu_launches": args.steps * job.launches_per_step,
            "pct_of_peak": 100.0 * value / world / peak,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
