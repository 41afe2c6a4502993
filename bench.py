"""Benchmark of the MLA sparse prefill (kv_norm -> wkv_b -> sparse causal attention) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload headline] [--impl ours|reference]

One step = one mla_sparse_prefill call (selection bitsets, kv_norm + wkv_b GEMM, sparse attention)
over one batch of seeded synthetic inputs resident in HBM, with a preallocated workspace. Each
timed step is bracketed by CUDA events on the launching stream; a 256 MB buffer write between
steps (outside the event pair) flushes the 126 MB L2. Rank 0 prints one JSON line.

Besides the headline workload the line carries a sustained figure (the same step back to back
for a few seconds, against the measured sustained peak) and `per_config`: every other workload
(tiny, dense_causal, stress, long_context) timed the same way, each with its formula TFLOP/s,
queries*heads/s, fractions of peak, the attention stage alone, the hardware/formula MMA ratio and
the oracle on a bounded sample (single-threaded too on tiny and dense_causal).

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


def hardware_mma_flops(B, T, H):
    """(GEMM stage, attention stage) tensor-core work the kernels issue, in 16-bit-equivalent flops
    (an f8f6f4 UMMA of K=32 takes the time of a 16-bit one of K=16 and is counted as that):
      GEMM stage: per 128-row tile, head and half (k_nope or v), 32 UMMAs of 128x128x16;
      attention: per (batch, head, 128-query tile qt) qt + 1 key blocks of 24 UMMAs of 128x128x16
      (8 fp16 q_nope.k_hi, 4 bf16 q_pe.k_pe, 4 f8 residual, 8 fp16 P.V), over the whole block
      whether or not a key is selected."""
    umma = 2.0 * 128 * 128 * 16
    nqt = (T + 127) // 128
    gemm = B * nqt * H * 2 * 32 * umma
    attn = B * H * (nqt * (nqt + 1) // 2) * 24 * umma
    return gemm, attn


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


# the files the attention kernel's code comes from (its device code, the PTX helpers it calls and
# the header whose constants it reads)
ATTENTION_SOURCES = ("sparse_attn.cuh", "ptx.cuh")


def kernel_sources_sha256(files=None) -> str:
    """sha256 over the code of libmla's kernel sources (all of them, or the csrc files named in
    `files`) and its header, comments and whitespace excluded."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_latent_attention_norm_b300", "csrc")
    names = sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")) and (files is None or f in files))
    paths = [os.path.join(csrc, f) for f in names]
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
    path = os.path.join(ROOT, "profiles", "sparse_attn_headline.md")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        for line in f:
            if line.startswith("traffic: "):
                kv = dict(x.split("=", 1) for x in line.split()[1:] if "=" in x)
                if kv.get("kernel") == "sparse_attn_kernel" and \
                        kv.get("sources_sha256") == kernel_sources_sha256(ATTENTION_SOURCES):
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

    _count = 0

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        ClockSampler._count += 1   # one file per sampler: a later sampler must not overwrite it
        self.path = os.path.join("/tmp", f"mla_clocks_{os.getpid()}_{ClockSampler._count}.csv")
        self._summary = None

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
        if self._summary is None:
            if self.proc is None or not os.path.exists(self.path):
                self._summary = {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
            else:
                with open(self.path) as f:
                    self._summary = self.parse(f)
        return self._summary


def cpu_baseline(inp, w, seconds_hint: float = 15.0, threads: int = 0):
    """The fp64 oracle, as it stands, on a bounded sample: all query rows of the first heads (at
    least one head per thread: the oracle runs one thread per (batch, head)), doubling the head
    count until one run takes about `seconds_hint` / 2 or more. threads = 0: all host cores."""
    import numpy as np
    import oracle
    cores = threads if threads > 0 else (os.cpu_count() or 1)
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
            "queries_heads_per_s": w.B * w.T * heads / dt,
            "sample": f"{w.name}: heads 0..{heads - 1} of {w.H}, all {w.B * w.T} query rows, fp64 oracle, "
                      f"{dt:.1f} s on {cores} thread(s)"}


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


def make_device_inputs(w, dev, batch=None):
    """Seeded host inputs of workload `w` (optionally with its batch cut to `batch`) and their
    device copies."""
    import torch
    import mla_inputs as mi
    if batch is not None and batch != w.B:
        w = mi.custom(w.name + f"_b{batch}", batch, w.T, w.H, w.K, w.pattern, stress=w.stress, seed_id=w.seed_id,
                      recent=w.recent)
    host = mi.make_inputs(w)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    return w, host, d


def time_steps(step, flush, stream, warmup, steps):
    """Per-step CUDA-event times (ms) of `steps` calls of step() after `warmup` untimed ones, the
    L2 flushed (256 MB write) before each call outside its event pair."""
    import torch
    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


def measure_config(w, host, d, dev, flush, stream, warmup, steps, peak_burst, cpu_seconds, single_thread):
    """Formula TFLOP/s, queries*heads/s, fractions of peak, the attention stage alone and the
    hardware/formula MMA ratio of one workload, next to the oracle on a bounded sample."""
    import torch
    import sparse_latent_attention_norm_b300 as mla
    B, T, H, K = w.B, w.T, w.H, w.K
    ws = mla.alloc_workspace(B, T, H, K, device=dev)
    out = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    _, _, nk = mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"],
                                  workspace=ws, n_keys=True)
    sum_n = float(nk.to(torch.int64).sum().item())
    up, attn = formula_flops(B, T, H, sum_n)
    hw_gemm, hw_attn = hardware_mma_flops(B, T, H)

    def step():
        mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"], out=out, lse=lse,
                           workspace=ws, stream=stream)

    ms = statistics.mean(time_steps(step, flush, stream, warmup, steps))
    bits, _ = mla.canon_select(d["topk_idx"], T, n_keys=False)
    kv, klo = mla.kvnorm_wkvb(d["c_kv"], d["gamma"], d["wkv_b"])
    attn_ms = time_stage(lambda: mla.sparse_attention(d["q"], d["k_pe"], kv, klo, bits, stream=stream),
                         flush, stream, warmup, steps)
    status = mla.get_status()
    if status != 0:
        raise SystemExit(f"device status {mla.status_string(status)} after timing {w.name}")
    del kv, klo, bits, ws, out, lse
    res = {
        "B": B, "T": T, "H": H, "K": K, "sum_selected_keys": int(sum_n), "steps": steps,
        "ms_per_step": ms,
        "formula_tflops": (up + attn) / (ms / 1e3) / 1e12,
        "queries_heads_per_s": B * T * H / (ms / 1e3),
        "frac_of_measured_bf16": (up + attn) / (ms / 1e3) / 1e12 / peak_burst,
        "frac_of_spec_bf16": (up + attn) / (ms / 1e3) / 1e12 / SPEC_BF16_TFLOPS,
        "attn_ms": attn_ms,
        "attn_formula_tflops": attn / (attn_ms / 1e3) / 1e12,
        "attn_frac_of_measured_bf16": attn / (attn_ms / 1e3) / 1e12 / peak_burst,
        "hw_to_formula_mma": (hw_gemm + hw_attn) / (up + attn),
        "attn_hw_to_formula_mma": hw_attn / attn,
        "attn_hw_tflops": hw_attn / (attn_ms / 1e3) / 1e12,
        "cpu_baseline": cpu_baseline(host, w, seconds_hint=cpu_seconds),
    }
    if single_thread:
        res["cpu_baseline_1_thread"] = cpu_baseline(host, w, seconds_hint=cpu_seconds, threads=1)
    return res


def fp8_weight_of(wkv_b):
    """An FP8 block-scaled copy of a bf16 wkv_b for the benchmark's variant: per 128 x 128 block,
    scale = max|w| / 448 and e4m3 codes of w / scale (torch's float8 cast, outside any timed
    region; the scale rule is the one the library reads for the latent)."""
    import torch
    rows = wkv_b.shape[0]
    blocks = wkv_b.float().reshape(rows // 128, 128, 4, 128)
    amax = blocks.abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (blocks / scale[:, None, :, None]).to(torch.float8_e4m3fn)
    return q.reshape(rows, 512).view(torch.uint8).contiguous(), scale.contiguous()


def measure_variants(w, d, dev, flush, stream, steps, total_flops):
    """Headline step time with each option of mla_sparse_prefill_opt on, and all of them."""
    import torch
    import sparse_latent_attention_norm_b300 as mla
    B, T, H, K = w.B, w.T, w.H, w.K
    w8, scale = fp8_weight_of(d["wkv_b"])
    kv_cache = torch.empty((B, T, 512), dtype=torch.bfloat16, device=dev)
    pe_cache = torch.empty((B, T, 64), dtype=torch.bfloat16, device=dev)
    out = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    cases = {
        "fp8_wkv_b": dict(wkv_b=w8, wkv_b_scale=scale),
        "fp8_latent_and_kv_cache": dict(fp8_latent=True, kv_cache=kv_cache, pe_cache=pe_cache),
        "yarn_rope": dict(rope=True),
        "all": dict(wkv_b=w8, wkv_b_scale=scale, fp8_latent=True, rope=True, kv_cache=kv_cache, pe_cache=pe_cache),
    }
    res = {}
    for name, kw in cases.items():
        kw = dict(kw)
        wkv = kw.pop("wkv_b", d["wkv_b"])
        opt = mla.options(flags=(mla.FLAG_ROPE if kw.get("rope") else 0),
                          wkv_b_scale=kw.get("wkv_b_scale"))
        ws = mla.alloc_workspace(B, T, H, K, device=dev, opt=opt)

        def step():
            mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], wkv, d["topk_idx"], out=out, lse=lse,
                               workspace=ws, stream=stream, **kw)

        ms = statistics.mean(time_steps(step, flush, stream, 3, steps))
        res[name] = {"ms_per_step": ms, "formula_tflops": total_flops / (ms / 1e3) / 1e12, "steps": steps}
        del ws
    status = mla.get_status()
    if status != 0:
        raise SystemExit(f"device status {mla.status_string(status)} after the variants")
    return res


def run_ours(args, rank, world, dist):
    import torch

    import mla_inputs as mi
    import sparse_latent_attention_norm_b300 as mla
    from sparse_latent_attention_norm_b300 import build as mla_build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    mla_build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    w, host, d = make_device_inputs(mi.WORKLOADS[args.workload], dev, args.batch)
    B, T, H, K = w.B, w.T, w.H, w.K
    ws = mla.alloc_workspace(B, T, H, K, device=dev)
    out = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    # --options: the step with the model's own steps around the MHA excerpt (for profilers)
    opt_kw, wkv = {}, d["wkv_b"]
    if args.options:
        names = set(args.options.split(","))
        if "fp8_wkv_b" in names:
            w8, scale = fp8_weight_of(d["wkv_b"])
            opt_kw["wkv_b_scale"] = scale
            wkv = w8
        if "fp8_latent" in names:
            opt_kw["fp8_latent"] = True
            opt_kw["kv_cache"] = torch.empty((B, T, 512), dtype=torch.bfloat16, device=dev)
            opt_kw["pe_cache"] = torch.empty((B, T, 64), dtype=torch.bfloat16, device=dev)
        if "rope" in names:
            opt_kw["rope"] = True
        ws = mla.alloc_workspace(B, T, H, K, device=dev,
                                 opt=mla.options(flags=mla.FLAG_ROPE if opt_kw.get("rope") else 0,
                                                 wkv_b_scale=opt_kw.get("wkv_b_scale")))

    def step():
        mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], wkv, d["topk_idx"], out=out, lse=lse,
                           workspace=ws, stream=stream, **opt_kw)

    # selected-key count for the formula (outside any timed region)
    _, _, nk = mla.sparse_prefill(d["q"], d["c_kv"], d["k_pe"], d["gamma"], d["wkv_b"], d["topk_idx"],
                                  workspace=ws, n_keys=True)
    sum_n = float(nk.to(torch.int64).sum().item())
    up_flops, attn_flops = formula_flops(B, T, H, sum_n)
    total_flops = up_flops + attn_flops
    hw_gemm, hw_attn = hardware_mma_flops(B, T, H)
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
    main_clocks = clocks.summary()
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

    # sustained: the same step back to back for about `sustain_s` seconds (the part settles at its
    # power cap), against the measured sustained bf16 peak
    sustained = None
    if args.sustain_s > 0:
        n_sus = max(args.steps, int(args.sustain_s * 1e3 / max(ms, 1e-3)))
        with ClockSampler(torch.cuda.current_device()) as sus_clocks:
            sus_ms = statistics.mean(time_steps(step, flush, stream, 0, n_sus))
        sustained = {"steps": n_sus, "ms_per_step": sus_ms, "value": world * total_flops / (sus_ms / 1e3) / 1e12,
                     "unit": "TFLOP/s", "clocks": sus_clocks.summary()}

    # end to end from pinned host memory through the public API: every step copies its inputs
    # (the activations q, c_kv, k_pe and topk_idx; the weights gamma and wkv_b are uploaded once,
    # before the timed region, as a serving process holds them) host->device and its results
    # device->host; the pipeline overlaps step i's input copies with step i-1's compute and step
    # i-2's result copies (copy engines in both directions)
    pipe = mla.HostPrefillPipeline(B, T, H, K, device=dev)
    hin = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
    pipe.set_weights(hin["gamma"], hin["wkv_b"])
    e2e_h2d = pipe.h2d_bytes(hin)
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
    del pipe, hin

    if rank != 0:
        return
    peak_burst, peak_sust, hbm, peak_kind = measured_peaks()
    if sustained is not None:
        sustained.update(peak=peak_sust, frac=sustained["value"] / world / peak_sust,
                         peak_kind=f"{peak_kind} bf16 sustained")
    cpu = cpu_baseline(host, w)

    # the headline step with the model's own steps around the MHA excerpt switched on (FP8
    # block-scaled wkv_b, FP8 round trip of the latent with the KV-cache write, YaRN RoPE of q and
    # k_pe), each timed like the main step
    variants = {}
    if not args.no_per_config:
        variants = measure_variants(w, d, dev, flush, stream, args.config_steps, total_flops)

    # every other workload of the metric's family, one after the other on this GPU
    per_config = {}
    if not args.no_per_config:
        del ws, out, lse, d
        torch.cuda.empty_cache()
        for name in [n for n in mi.WORKLOADS if n != w.name]:
            wc, hc, dc = make_device_inputs(mi.WORKLOADS[name], dev)
            per_config[name] = measure_config(wc, hc, dc, dev, flush, stream, 3, args.config_steps, peak_burst,
                                              cpu_seconds=6.0, single_thread=name in ("tiny", "dense_causal"))
            del hc, dc
            torch.cuda.empty_cache()

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
        "hw_to_formula_mma": (hw_gemm + hw_attn) / total_flops,
        "attn_hw_to_formula_mma": hw_attn / attn_flops,
        "attn_hw_tflops": hw_attn / (attn_avg / 1e3) / 1e12,
        "roofline": {"kernel": "sparse_attn_kernel", "bound": "tensor", "achieved": achieved, "peak": peak_burst,
                     "unit": "TFLOP/s", "frac": achieved / peak_burst, "traffic": profiled_traffic(w.name),
                     "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
                     "peak_kind": f"{peak_kind} bf16 burst",
                     "algorithmic": "2*H*sum_n*(192+128) flops per launch"},
        "sustained": sustained,
        "cpu_baseline": cpu,
        "e2e": {"value": world * total_flops / e2e_s / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": e2e_h2d,
                "d2h_bytes_per_step": B * T * H * 128 * 2 + B * T * H * 4,
                "how": "HostPrefillPipeline: each step copies its activations (q, c_kv, k_pe, topk_idx) "
                       "from pinned host memory to the device and out / lse back to pinned host memory, "
                       "steps overlapped on three streams; the weights (gamma, wkv_b) are uploaded once "
                       "before the timed region"},
        "variants": variants,
        "per_config": per_config,
        "gpu_launches": 3 * args.steps,
        "clocks": main_clocks,
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
    ap.add_argument("--batch", type=int, default=None,
                    help="cut the workload's batch to this many sequences (smaller profiler captures)")
    ap.add_argument("--sustain-s", type=float, default=4.0,
                    help="seconds of back-to-back steps for the sustained figure (0: skip)")
    ap.add_argument("--config-steps", type=int, default=10, help="timed steps per other workload")
    ap.add_argument("--no-per-config", action="store_true", help="time the chosen workload only")
    ap.add_argument("--options", default="",
                    help="with --kernels-only: comma list of fp8_wkv_b, fp8_latent, rope to switch on (profilers)")
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
