"""Benchmark of the MLA sparse prefill (kv_norm -> wkv_b -> sparse causal attention) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload headline] [--impl ours|reference]

One step = one mla_sparse_prefill call (selection bitsets, kv_norm + wkv_b GEMM, sparse attention)
over one batch of seeded synthetic inputs resident in HBM, with a preallocated workspace. Each
timed step is bracketed by CUDA events on the launching stream; a 256 MB buffer write between
steps (outside the event pair) flushes the 126 MB L2. Rank 0 prints one JSON line.

Metric: formula TFLOP/s = (2*B*T*H*512*256 + 2*H*sum_n*(192+128)) / time, sum_n being the number of
distinct causal selected keys summed over all queries (counted by the library's n_keys output).

--impl reference times the fp64 CPU oracle (the test oracle, as it stands) on the host cores, on a
bounded sample of the same workload per step.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA sparse prefill TFLOP/s & % bf16 tensor peak, T=4096 K=2048, 1×B300"
SPEC_BF16_TFLOPS = 2250.0


def formula_flops(B, T, H, sum_n):
    """(up-projection, attention) flops of the metric's formula."""
    up = 2.0 * B * T * H * 512 * 256
    attn = 2.0 * H * sum_n * (192 + 128)
    return up, attn


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), d.get("hbm_gbs"), "measured"
    return 1800.0, 1400.0, 6400.0, "fallback"


def _code_only(text: str) -> str:
    """C/C++/CUDA source with comments and whitespace removed (no source here has `//` or `/*`
    inside a string literal), so that editing a comment does not count as changing a kernel."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return "".join(text.split())


def kernel_sources_sha256() -> str:
    """sha256 over the code of libmla's kernel sources and header (the inputs of every kernel
    build), comments and whitespace excluded."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_latent_attention_norm_b300", "csrc")
    paths = [os.path.join(csrc, f) for f in sorted(os.listdir(csrc)) if f.endswith((".cu", ".cuh", ".h"))]
    for path in paths + [os.path.join(ROOT, "include", "mla.h")]:
        h.update(os.path.basename(path).encode())
        with open(path, encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()


def profiled_traffic(workload: str):
    """DRAM bytes (read + write) per launch of the attention kernel, from the committed ncu
    summary of the headline workload, or None when that capture predates the current sources."""
    if workload != "headline":
        return None
    path = os.path.join(ROOT, "profiles", "kernels_headline_full.md")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            if line.startswith("traffic: "):
                kv = dict(x.split("=", 1) for x in line.split()[1:] if "=" in x)
                if kv.get("kernel") == "sparse_attn_kernel" and kv.get("sources_sha256") == kernel_sources_sha256():
                    return int(kv["dram_bytes_per_launch"])
    return None


def dist_setup():
    """Under torchrun (WORLD_SIZE > 1) every rank runs an independent replica of the workload."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, None
    import torch
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
        backend = "nccl"
    else:
        backend = "gloo"
    dist.init_process_group(backend=backend)
    return rank, ws, dist


def max_over_ranks(x: float, dist) -> float:
    if dist is None:
        return x
    import torch
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"mla_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    @classmethod
    def parse(cls, lines):
        rows = []
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        seen = set()
        for *_, flags in rows:
            for n, f in zip(cls.REASONS, flags):
                if f.lower().startswith("active"):
                    seen.add(n)
        # "under load": samples drawing more than the median power of the run
        pw = statistics.median(r[2] for r in rows)
        loaded = [r[0] for r in rows if r[2] >= pw] or [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(seen), "samples": len(rows)}

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        with open(self.path) as f:
            return self.parse(f)


def cpu_baseline(inp, w, seconds_hint: float = 15.0):
    """The fp64 oracle, as it stands, on a bounded sample: all query rows of the first heads (at
    least one head per core: the oracle runs one thread per (batch, head)), doubling the head
    count until one run takes about `seconds_hint` / 2 or more."""
    import numpy as np
    import oracle
    cores = os.cpu_count() or 1
    heads, dt, nk = min(w.H, cores), 0.0, None
    while True:
        t0 = time.perf_counter()
        _, _, nk = oracle.prefill(inp, heads=(0, heads), threads=cores)
        dt = time.perf_counter() - t0
        if dt >= seconds_hint / 2 or heads >= w.H:
            break
        heads = min(w.H, heads * 2)
    sum_n = float(np.asarray(nk, dtype=np.int64).sum())
    up, attn = formula_flops(w.B, w.T, heads, sum_n)
    return {"value": (up + attn) / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{w.name}: heads 0..{heads - 1} of {w.H}, all {w.B * w.T} query rows, fp64 oracle, "
                      f"{dt:.1f} s"}


def run_reference(args, rank, world, dist, budget_s: float = 150.0):
    """The oracle timed on the host cores, same metric and workload. Each step is one bounded
    sample: the first (one per core) heads over all query rows, or, when K + W such steps would
    not fit in about `budget_s`, over the first R query rows of each batch (R sized from a timed
    first run)."""
    if rank != 0:
        return
    import numpy as np
    import mla_inputs as mi
    import oracle
    w = mi.WORKLOADS[args.workload]
    inp = mi.make_inputs(w)
    cores = os.cpu_count() or 1
    oracle.build()
    hs = min(w.H, cores)              # one head per core: the oracle runs one thread per (batch, head)
    t0 = time.perf_counter()
    oracle.prefill(inp, heads=(0, hs), threads=cores)
    t_full = time.perf_counter() - t0
    per_step = budget_s / (args.steps + args.warmup)
    R = w.T if t_full <= per_step else max(128, min(w.T, int(w.T * per_step / t_full)))
    rows = None if R == w.T else np.concatenate([b * w.T + np.arange(R) for b in range(w.B)]).astype(np.int64)
    times = []
    nk = None
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        _, _, nk = oracle.prefill(inp, rows=rows, heads=(0, hs), threads=cores)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    sum_n = float(np.asarray(nk, dtype=np.int64).sum())
    flops = 2.0 * w.B * R * hs * 512 * 256 + 2.0 * hs * sum_n * (192 + 128)   # positions up-projected + attention
    ms = 1e3 * sum(times) / len(times)
    value = flops / (ms / 1e3) / 1e12
    what = f"all {w.T} query rows" if rows is None else f"query rows 0..{R - 1}"
    sample = f"{w.name}: heads 0..{hs - 1} of {w.H}, {what} of each batch per step, fp64 oracle on {cores} threads"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(w.describe(), sample=sample),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def time_stage(fn, flush, stream, warmup, steps):
    """Mean CUDA-event time (ms) of fn() on `stream`, L2 flushed before every call.

    The calls are enqueued back to back (no host synchronisation between them), as in the timed
    steps: with a synchronisation after each call the device would idle between the flush and
    the next launch while the host prepares it, and that gap would land inside the event pair."""
    import torch
    n = warmup + steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs[warmup:])


def run_ours(args, rank, world, dist):
    import torch

    import mla_inputs as mi
    import sparse_latent_attention_norm_b300 as mla
    from sparse_latent_attention_norm_b300 import build as mla_build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    mla_build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    w = mi.WORKLOADS[args.workload]
    host = mi.make_inputs(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    B, T, H, K = w.B, w.T, w.H, w.K
    ws = mla.alloc_workspace(B, T, H, K, device=dev)
    out = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"], out=out, lse=lse,
                           workspace=ws, stream=stream)

    # selected-key count for the formula (outside any timed region)
    _, _, nk = mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"],
                                  workspace=ws, n_keys=True)
    sum_n = float(nk.to(torch.int64).sum().item())
    up_flops, attn_flops = formula_flops(B, T, H, sum_n)
    total_flops = up_flops + attn_flops
    mla.clear_status()

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    barrier(dist)
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = max_over_ranks(sum(step_ms) / len(step_ms), dist)
    status = mla.get_status()
    if status != 0:
        raise SystemExit(f"device status {mla.status_string(status)} after the timed region")
    if args.kernels_only:
        if rank == 0:
            print(json.dumps({"kernels_only": True, "workload": w.name, "ms_per_step": ms,
                              "tflops": world * total_flops / (ms / 1e3) / 1e12}), flush=True)
        return

    # each stage alone through the staged entry points, same stream, L2 flushed before each call
    n_stage = min(args.steps, 50)
    bits, _ = mla.canon_select(d["topk_idx"], T, n_keys=False)
    kv, klo = mla.kvnorm_wkvb(d["c_kv"], d["gamma"], d["wkv_b"])
    attn_avg = time_stage(lambda: mla.sparse_attention(d["q"], d["k_pe"], kv, klo, bits, stream=stream),
                          flush, stream, args.warmup, n_stage)
    gemm_avg = time_stage(lambda: mla.kvnorm_wkvb(d["c_kv"], d["gamma"], d["wkv_b"], stream=stream),
                          flush, stream, args.warmup, n_stage)
    canon_avg = time_stage(lambda: mla.canon_select(d["topk_idx"], T, n_keys=False, stream=stream),
                           flush, stream, args.warmup, n_stage)
    del kv, klo, bits

    # end to end from pinned host memory through the public API: every step copies its inputs
    # host->device and its results device->host; the pipeline overlaps step i's input copies with
    # step i-1's compute and step i-2's result copies (copy engines in both directions)
    pipe = mla.HostPrefillPipeline(B, T, H, K, device=dev)
    hin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    for _ in range(max(2, args.warmup)):
        pipe.result(pipe.submit(hin))
    e2e_steps = max(4, min(args.steps, 12))
    barrier(dist)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    handles = [pipe.submit(hin) for _ in range(e2e_steps)]
    for hnd in handles[-pipe.depth:]:
        pipe.result(hnd)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, dist)

    if rank != 0:
        return
    peak_burst, peak_sust, hbm, peak_kind = measured_peaks()
    achieved = attn_flops / (attn_avg / 1e3) / 1e12
    value = world * total_flops / (ms / 1e3) / 1e12
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": dict(w.describe(), l2="flushed between steps (256 MB write outside each step's event pair)",
                       parallelism="replicas" if world > 1 else "single GPU",
                       sum_selected_keys=int(sum_n)),
        "frac_of_spec_bf16": value / world / SPEC_BF16_TFLOPS,
        "frac_of_measured_bf16": value / world / peak_burst,
        "queries_heads_per_s": world * B * T * H / (ms / 1e3),
        "kernel_ms": {"sparse_attn": attn_avg, "kvnorm_wkvb": gemm_avg, "canon_select": canon_avg},
        "kvnorm_wkvb_tflops": up_flops / (gemm_avg / 1e3) / 1e12,
        "roofline": {"kernel": "sparse_attn_kernel", "bound": "tensor", "achieved": achieved, "peak": peak_burst,
                     "unit": "TFLOP/s", "frac": achieved / peak_burst, "traffic": profiled_traffic(w.name),
                     "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                     "peak_kind": f"{peak_kind} bf16 burst",
                     "algorithmic": "2*H*sum_n*(192+128) flops per launch"},
        "cpu_baseline": cpu_baseline(host, w),
        "e2e": {"value": world * total_flops / e2e_s / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": pipe.h2d_bytes(hin), "d2h_bytes_per_step": pipe.d2h_bytes(),
                "how": "HostPrefillPipeline: pinned host inputs -> device -> pinned host results each step, "
                       "steps overlapped on three streams"},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="headline")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--kernels-only", action="store_true",
                    help="time the prefill steps only (no stage timings, e2e or CPU baseline): for profilers")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank, world, dist = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, rank, world, dist)
        else:
            run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
