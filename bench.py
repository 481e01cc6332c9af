"""Benchmark of the ring-attention forward on GB300.

One step = one cp_ring_attn_fwd call over the whole workload (every virtual
rank, every visible K/V tile) with Q/K/V already resident in HBM.  The
metric is effective causal TFLOP/s: 4 d FLOPs per visible (q, k) pair, summed
over (b, h), divided by the device time of the step.  Inputs are far larger
than L2 (3 GiB at the 128K workload), so no flush is needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--no-cpu-baseline]
For N > 1 it is launched by torch.distributed.run, one process per GPU; each
rank runs an independent replica of the workload (the single-GPU path has no
exchange step to shard), the step time is the max over ranks and the value is
the work of all ranks divided by that time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from context_ring_attention_fwd_gb300 import inputs  # noqa: E402

METRIC = "effective causal TFLOP/s of ring-attention fwd (1 GB300) and % of bf16 dense peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "bf16_causal_128k"
# DRAM bytes (read + write) per launch of the fused attention kernel, from one
# ncu capture of dram__bytes_read.sum + dram__bytes_write.sum limited to that
# kernel (-k regex:ring_attn_bf16 -c 1) on this bench command with the
# workload named.  Each figure holds only for the kernel source it was taken
# on: "sources" is the SHA-256 prefix of the forward kernel's source files
# (KERNEL_SOURCES), and a line whose sources differ reports traffic null.
KERNEL_SOURCES = ("context_ring_attention_fwd_gb300/csrc/attn_sm103.cu",
                  "context_ring_attention_fwd_gb300/csrc/attn_common.cuh",
                  "context_ring_attention_fwd_gb300/csrc/ptx.cuh")
BWD_KERNEL_SOURCES = ("context_ring_attention_fwd_gb300/csrc/attn_bwd_sm103.cu",
                      "context_ring_attention_fwd_gb300/csrc/attn_common.cuh",
                      "context_ring_attention_fwd_gb300/csrc/ptx.cuh")
NCU_TRAFFIC = {
    # 16.718 GB read + 1.084 GB written (ncu, ring_attn_bf16_kernel<128, 0, 0>, 1 pass)
    "bf16_causal_128k": {"bytes": 16.71847808e9 + 1.084292352e9, "sources": "a2bf8212ad5f2d98"},
    # the FP8 forward (--fp8; ring_attn_fp8_kernel<128>: 2.137 GB read + 1.063 GB
    # written) and the backward's dK/dV kernel (--bwd; ring_attn_bwd_kernel<128, 1>:
    # 5.995 GB read + 2.124 GB written), same capture form
    "fp8:bf16_causal_128k": {"bytes": 2.136846848e9 + 1.063047936e9,
                             "sources": "a2bf8212ad5f2d98"},
    "bwd:bf16_causal_128k": {"bytes": 5.995067904e9 + 2.123589376e9,
                             "sources": "22a468516fa74477", "files": BWD_KERNEL_SOURCES},
}
# tcgen05 dense bf16 -> fp32 rate per SM and clock: a 128x128x16 MMA
# (524,288 FLOPs) every 64 clocks.
TCGEN05_BF16_FLOP_PER_CLK_SM = 8192


# ------------------------------------------------------------------ helpers
def visible_pairs(S: int, causal: bool, docs) -> int:
    """Visible (q, k) pairs of one (b, h): S(S+1)/2 causal, S^2 full, and per
    document L(L+1)/2 or L^2 with packed documents."""
    spans = [S] if docs is None else [b - a for a, b in zip(docs[:-1], docs[1:])]
    return sum(L * (L + 1) // 2 if causal else L * L for L in spans)


def effective_flops(w, docs) -> int:
    return 4 * w.d * visible_pairs(w.S, w.causal, docs) * w.B * w.H


def kernel_sources_digest(files=KERNEL_SOURCES) -> str:
    """SHA-256 prefix over a kernel's source files (default: the forward's)."""
    import hashlib
    h = hashlib.sha256()
    for rel in files:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(name: str):
    """The recorded DRAM traffic of the kernel for this workload, or None when
    it was not recorded for the kernel source as it stands."""
    rec = NCU_TRAFFIC.get(name)
    if (not rec or rec["bytes"] is None
            or rec["sources"] != kernel_sources_digest(rec.get("files", KERNEL_SOURCES))):
        return None
    return rec["bytes"]


def computed_tile_ratio(S: int, n_shards: int, tile: int = 128) -> float:
    """Causal over full count of the (query tile, key tile) pairs the fused
    kernel computes, with tiles laid from each shard's first row."""
    L = S // n_shards
    T = -(-L // tile)
    first = np.array([i * L + a * tile for i in range(n_shards) for a in range(T)])
    last = np.minimum(first + tile, (first // L + 1) * L) - 1
    # key tile (k0, .) is computed for query tile (., q1) iff k0 <= q1
    causal = int(np.searchsorted(first, last, side="right").sum())
    return causal / (first.size ** 2)


def blas_threads():
    """Threads of the BLAS numpy calls into, or None when it cannot be asked."""
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:  # noqa: BLE001 - optional module, absent on some hosts
        pass
    import ctypes
    try:
        with open("/proc/self/maps") as f:
            libs = {ln.split()[-1] for ln in f if "blas" in ln.lower() and ".so" in ln}
    except OSError:
        return None
    for path in sorted(libs):
        try:
            h = ctypes.CDLL(path)
        except OSError:
            continue
        for sym in ("openblas_get_num_threads", "scipy_openblas_get_num_threads64_",
                    "openblas_get_num_threads64_"):
            fn = getattr(h, sym, None)
            if fn is not None:
                fn.restype = ctypes.c_int
                return int(fn())
    return None


def core_record():
    cpu = os.cpu_count() or 1
    try:
        aff = len(os.sched_getaffinity(0))
    except AttributeError:
        aff = cpu
    bt = blas_threads()
    # the matrix products run on the BLAS threads; the rest of numpy on one
    return {"cores": bt if bt else aff, "cpu_count": cpu, "affinity_cores": aff,
            "blas_threads": bt}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend)


def barrier(world: int, device=None):
    if world > 1:
        if device is not None and torch.distributed.get_backend() == "nccl":
            torch.distributed.barrier(device_ids=[device.index])
        else:
            torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a host scalar over all ranks (timing only, no data path)."""
    if world <= 1:
        return float(x)
    dev = device if (device is not None and torch.distributed.get_backend() == "nccl") else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), "measured"
    return 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power) if power else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def gpu_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        items = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(items) and items[local_rank].isdigit():
            return int(items[local_rank])
    return local_rank


# ------------------------------------------------------------ oracle timing
def oracle_sample(w, get_head, docs, budget_s: float, rows_per_head: int, seed: int = 0,
                  max_heads: int = 1 << 30):
    """Time the fp64 oracle on sampled query rows of the workload, one (b, h)
    head after another, until the budget is spent (at least one head).
    get_head(b, h) returns that head's q, k, v as [1, S, 1, d] fp32 numpy
    arrays (fetched outside the timed part).  Returns (effective FLOPs
    done, seconds, description)."""
    from oracle import ref  # the CPU baseline leg: the only bench use of the oracle

    flops = 0
    heads_done = 0
    dt = 0.0
    combos = [(b, h) for b in range(w.B) for h in range(w.H)]
    rng = np.random.default_rng(seed)
    rng.shuffle(combos)
    kk = np.asarray(docs) if docs is not None else None
    for b, h in combos[:max_heads]:
        rows = inputs.sample_rows(w.S, rows_per_head, seed=seed * 1000 + b * w.H + h)
        qh, kh, vh = get_head(b, h)
        t0 = time.perf_counter()
        ref.attention_rows(qh, kh, vh, 0, 0, rows, w.causal, docs)
        dt += time.perf_counter() - t0
        # visible keys of each sampled row
        if kk is None:
            cnt = (rows + 1) if w.causal else np.full(rows.shape, w.S)
        else:
            t = np.searchsorted(kk, rows, side="right") - 1
            cnt = (rows - kk[t] + 1) if w.causal else (kk[t + 1] - kk[t])
        flops += int(4 * w.d * int(np.sum(cnt)))
        heads_done += 1
        if dt >= budget_s:
            break
    what = ("all query rows" if rows_per_head >= w.S else f"{rows_per_head} seeded query rows")
    whole = " (the whole workload)" if rows_per_head >= w.S and heads_done == w.B * w.H else ""
    desc = (f"{what} x {heads_done} (b,h) heads of {w.name} ({w.describe()}){whole}, "
            f"fp64 numpy oracle")
    return flops, dt, desc


# ------------------------------------------------------------------- arms
def run_reference(args, w, rank, world):
    """The reference arm: the fp64 CPU oracle, on rank 0 only, each step a
    bounded sample of the workload."""
    if rank != 0:
        return None
    docs = (inputs.make_doc_offsets(w.S, w.seed + 1, w.doc_min, w.doc_max)
            if w.packed_docs else None)
    cache = {}

    def get_head(b, h):
        # one head's Q/K/V drawn on the CPU with a per-head seed: the same
        # shape and distribution as the workload, without drawing all heads
        key = (b, h)
        if key not in cache:
            qh, kh, vh = inputs.make_qkv(1, w.S, 1, w.d, w.seed * 1000 + b * w.H + h,
                                         w.torch_dtype, w.scale)
            cache.clear()
            cache[key] = tuple(t.float().numpy() for t in (qh, kh, vh))
        return cache[key]

    rows = max(8, min(256, int(2 ** 22 // max(1, w.S))))
    for s in range(args.warmup):
        oracle_sample(w, get_head, docs, budget_s=0.0, rows_per_head=rows, seed=s + 100,
                      max_heads=1)
    t_total, f_total = 0.0, 0
    desc = ""
    for s in range(args.steps):
        f, dt, desc = oracle_sample(w, get_head, docs, budget_s=0.0, rows_per_head=rows,
                                    seed=s + 1, max_heads=1)
        t_total += dt
        f_total += f
    value = f_total / t_total / 1e12
    ms = 1e3 * t_total / args.steps
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": _config(w, docs, world),
        "cpu_baseline": {"value": value, "unit": UNIT, **core_record(), "kind": "oracle",
                         "sample": "each step: " + desc,
                         # the whole workload at the sample's rate (extrapolated, not run)
                         "extrapolated_full_seconds": effective_flops(w, docs) / (value * 1e12)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    return line


def _config(w, docs, world):
    return {"workload": w.describe(), "name": w.name, "B": w.B, "S": w.S, "H": w.H, "d": w.d,
            "n_shards": w.n_shards, "causal": w.causal,
            "n_docs": None if docs is None else len(docs) - 1,
            "replicas": world, "l2_flush": "none: inputs (3*B*S*H*d*2 bytes) exceed the 129 MB L2"}


def run_ours(args, w, rank, world, local):
    import context_ring_attention_fwd_gb300 as pkg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pkg.lib()
    q, k, v = inputs.make_qkv(w.B, w.S, w.H, w.d, w.seed, w.torch_dtype, w.scale, device=str(dev))
    docs = (inputs.make_doc_offsets(w.S, w.seed + 1, w.doc_min, w.doc_max)
            if w.packed_docs else None)
    docs_t = pkg.doc_offsets_tensor(docs, dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    call = pkg.cp_ring_attn_fwd if w.dtype == "bf16" else pkg.cp_ring_attn_fwd_f32

    def step():
        call(q, k, v, out, lse, w.n_shards, w.causal, docs_t, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if pkg.cp_get_last_status(stream) != 0:
        raise RuntimeError("device error during warm-up")

    clocks = ClockSampler(gpu_index(local))
    clocks.start()
    time.sleep(0.3)
    launches0 = pkg.launch_counts()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world, dev)
    torch.cuda.synchronize(dev)
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    t_all0.record(stream)
    for s in range(args.steps):
        ev[s][0].record(stream)
        step()
        ev[s][1].record(stream)
    t_all1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world, dev)
    launches1 = pkg.launch_counts()
    clk = clocks.stop()
    if pkg.cp_get_last_status(stream) != 0:
        raise RuntimeError("device error during the timed region")
    total_ms = t_all0.elapsed_time(t_all1)
    per_launch_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(total_ms, world, dev)
    ms = total_ms / args.steps
    flops = effective_flops(w, docs)
    value = flops * world * args.steps / (total_ms * 1e-3) / 1e12
    gpu_launches = int(sum(launches1) - sum(launches0))

    # roofline of the dominant kernel (the fused attention kernel: one launch per step)
    avg_launch_ms = statistics.mean(per_launch_ms)
    achieved = flops / (avg_launch_ms * 1e-3) / 1e12
    peak_burst, peak_sust, peak_src = measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    tc_at_clock = (TCGEN05_BF16_FLOP_PER_CLK_SM * sms * clk["sm_mhz"] * 1e6 / 1e12
                   if clk.get("sm_mhz") else None)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak_burst, "unit": "TFLOP/s",
                "frac": achieved / peak_burst,
                "traffic": args.traffic if args.traffic is not None else ncu_traffic(w.name),
                "traffic_sources": kernel_sources_digest(),
                "algorithmic_bytes": 4 * w.B * w.S * w.H * w.d * w.elem_bytes
                + 4 * w.B * w.H * w.S,
                "peak_kind": f"{peak_src} bf16 dense burst (cuBLAS)",
                "frac_of_sustained": achieved / peak_sust if peak_sust else None,
                # the tensor pipe's own rate at the SM clock sampled in the timed region
                "tcgen05_peak_at_sampled_clock": tc_at_clock,
                "frac_of_tcgen05_at_sampled_clock": achieved / tc_at_clock if tc_at_clock
                else None}

    # the schedule's acceptance checks on this shape (untimed for the metric)
    gates = None
    if docs is None and not args.no_gates:
        gates = schedule_gates(pkg, w, q, k, v, out, lse, stream, dev)

    # end to end through the C ABI's host-buffer entry point (cp_ring_attn_fwd_host)
    e2e = None
    if args.e2e_steps > 0:
        hq = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
        hk = torch.empty_like(hq, pin_memory=True)
        hv = torch.empty_like(hq, pin_memory=True)
        hq.copy_(q)
        hk.copy_(k)
        hv.copy_(v)
        del q, k, v, out, lse
        torch.cuda.empty_cache()
        esz = hq.element_size()
        bufs = (torch.empty(pkg.cp_ring_attn_fwd_host_workspace_bytes(
                    w.B, w.S, w.H, w.d, w.n_shards, esz), dtype=torch.uint8, device=dev),
                torch.empty(hq.shape, dtype=hq.dtype, pin_memory=True),
                torch.empty((w.B, w.H, w.S), dtype=torch.float32, pin_memory=True))
        pkg.ring_attn_fwd_host(hq, hk, hv, w.n_shards, w.causal, docs, buffers=bufs)
        barrier(world, dev)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        marks = [t0]
        for _ in range(args.e2e_steps):
            pkg.ring_attn_fwd_host(hq, hk, hv, w.n_shards, w.causal, docs, buffers=bufs)
            marks.append(time.perf_counter())
        dt = marks[-1] - t0
        dt = max_over_ranks(dt, world, dev)
        elem = hq.numel() * hq.element_size()
        e2e = {"value": flops * world * args.e2e_steps / dt / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": 3 * elem,
               "d2h_bytes_per_step": elem + w.B * w.H * w.S * 4,
               "ms_per_step": 1e3 * dt / args.e2e_steps, "steps": args.e2e_steps,
               "ms_each": [1e3 * (b - a) for a, b in zip(marks[:-1], marks[1:])],
               "ms_median": 1e3 * statistics.median(
                   b - a for a, b in zip(marks[:-1], marks[1:])),
               "entry_point": "cp_ring_attn_fwd_host"}
        if docs is not None:
            e2e["doc_offsets"] = "resident on the device, as the C ABI takes them"
        host_inputs = (hq, hk, hv)
        del bufs
    else:
        host_inputs = tuple(t.cpu() for t in (q, k, v))

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        def get_head(b, h):
            return tuple(t[b:b + 1, :, h:h + 1].float().numpy() for t in host_inputs)

        rows = args.cpu_rows if args.cpu_rows is not None else (w.S if w.S <= 8192 else 512)
        # the whole oracle on every head when the rows are all of them
        budget = args.cpu_budget if rows < w.S else max(args.cpu_budget, 60.0)
        f, dt, desc = oracle_sample(w, get_head, docs, budget_s=budget, rows_per_head=rows)
        cpu = {"value": f / dt / 1e12, "unit": UNIT, **core_record(), "kind": "oracle",
               "sample": desc, "seconds": dt,
               # the whole workload at the sample's rate (extrapolated, not run)
               "extrapolated_full_seconds": effective_flops(w, docs) / (f / dt)}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": _config(w, docs, world),
        "frac_of_peak": value / world / peak_burst,
        # each timed launch between its own events: the median and the spread
        "ms_launch_median": statistics.median(per_launch_ms),
        "ms_launch_min_max": [min(per_launch_ms), max(per_launch_ms)],
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": gpu_launches,
        "clocks": clk, "gates": gates,
        "effective_flops_per_step": flops * world,
    }
    return line


def schedule_gates(pkg, w, q, k, v, out, lse, stream, dev, rounds: int = 3):
    """The schedule's acceptance checks on the workload's shape: the causal
    forward's time over the same shape without the causal mask (ideal: the
    computed-tile ratio; gate <= 0.53), and the causal time at N = 1, 2, 4, 8
    shards (equal work; gate: spread <= 3 %).  The five configurations are
    timed round-robin, one launch each per round after one warm-up launch
    each, with CUDA events on the launching stream, and each takes its median
    over the rounds, so the clock's drift under the power cap falls on every
    configuration alike instead of on the ones measured last."""
    configs = [(n, True) for n in (1, 2, 4, 8) if w.S % n == 0] + [(w.n_shards, False)]

    def launch(cfg):
        pkg.cp_ring_attn_fwd(q, k, v, out, lse, cfg[0], cfg[1], None, stream)

    for cfg in configs:
        launch(cfg)
    torch.cuda.synchronize(dev)
    times = {cfg: [] for cfg in configs}
    for _ in range(rounds):
        for cfg in configs:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch(cfg)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            times[cfg].append(e0.elapsed_time(e1))
    if pkg.cp_get_last_status(stream) != 0:
        raise RuntimeError("device error in the schedule checks")
    med = {cfg: statistics.median(t) for cfg, t in times.items()}
    by_n = {n: med[(n, True)] for n in (1, 2, 4, 8) if w.S % n == 0}
    t_full = med[(w.n_shards, False)]
    t_causal = med[(w.n_shards, True)] if (w.n_shards, True) in med else by_n[min(by_n)]
    ideal = computed_tile_ratio(w.S, w.n_shards)
    spread = (max(by_n.values()) - min(by_n.values())) / min(by_n.values())
    ratio = t_causal / t_full
    # the stated limit at the 128K shape; elsewhere the same margin over the
    # computed-tile ratio (shorter sequences carry more diagonal tiles)
    limit = 0.53 if (w.S, w.H, w.d, w.n_shards) == (131072, 32, 128, 4) else ideal + 0.03
    return {"ms_causal": t_causal, "ms_full": t_full, "causal_over_full": ratio,
            "computed_tile_ratio": ideal, "causal_over_full_limit": limit,
            "causal_over_full_ok": ratio <= limit,
            "ms_causal_by_n_shards": {str(n): t for n, t in by_n.items()},
            "n_shards_spread": spread, "n_shards_spread_ok": spread <= 0.03,
            "rounds": rounds, "timing": "round-robin over the configurations, median per one"}


def run_ring_emulation(args, w, local):
    """Time the ring with explicit per-rank buffers: transfers overlapped on
    a copy stream, transfers in order on the compute stream, and the fused
    kernel, on the same inputs.  One JSON line (impl "ring_emulated")."""
    import context_ring_attention_fwd_gb300 as pkg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    q, k, v = inputs.make_qkv(w.B, w.S, w.H, w.d, w.seed, w.torch_dtype, w.scale, device=str(dev))
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
    ws = torch.empty(pkg.cp_ring_emulated_workspace_bytes(w.B, w.S, w.H, w.d, w.n_shards),
                     dtype=torch.uint8, device=dev)
    cs = torch.cuda.Stream(device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / args.steps

    recv = []
    ms_ov = timed(lambda: recv.append(pkg.cp_ring_attn_fwd_emulated(
        q, k, v, out, lse, w.n_shards, w.causal, ws, stream, cs)))
    ms_ser = timed(lambda: pkg.cp_ring_attn_fwd_emulated(
        q, k, v, out, lse, w.n_shards, w.causal, ws, stream, None))
    ms_fused = timed(lambda: pkg.cp_ring_attn_fwd(q, k, v, out, lse, w.n_shards, w.causal, None,
                                                  stream))
    if pkg.cp_get_last_status(stream) != 0:
        raise RuntimeError("device error in the ring emulation")
    flops = effective_flops(w, None)
    moved = int(sum(recv[-1]))
    return {
        "metric": METRIC, "impl": "ring_emulated", "unit": UNIT,
        "value": flops / (ms_ov * 1e-3) / 1e12, "ms_per_step": ms_ov,
        "ms_transfers_in_order": ms_ser, "ms_fused_kernel": ms_fused,
        "transfer_time_hidden_ms": ms_ser - ms_ov,
        "bytes_received_per_step": moved, "bytes_received_per_rank": recv[-1],
        "steps": args.steps, "warmup": args.warmup, "n_gpus": 1, "dtype": w.dtype,
        "data": "synthetic", "config": _config(w, None, 1),
    }


def run_ulysses(args, w, local):
    """Time the all-to-all (Ulysses) form against the fused ring kernel on the
    same inputs.  The time of the form's head-group attention launch alone
    is taken on head-split copies of the inputs; the rest of the step is the
    permutations (HBM-bound, reported against the measured copy peak) and
    the LSE copies.  One JSON line."""
    import context_ring_attention_fwd_gb300 as pkg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    q, k, v = inputs.make_qkv(w.B, w.S, w.H, w.d, w.seed, w.torch_dtype, w.scale, device=str(dev))
    docs = (inputs.make_doc_offsets(w.S, w.seed + 1, w.doc_min, w.doc_max)
            if w.packed_docs else None)
    dd = pkg.doc_offsets_tensor(docs, dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
    ws = torch.empty(pkg.cp_ulysses_workspace_bytes(w.B, w.S, w.H, w.d, w.n_shards),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / args.steps

    moved = []
    ms_u = timed(lambda: moved.append(pkg.cp_ulysses_attn_fwd(q, k, v, out, lse, w.n_shards,
                                                              w.causal, dd, ws, stream)))
    ms_f = timed(lambda: pkg.cp_ring_attn_fwd(q, k, v, out, lse, w.n_shards, w.causal, dd, stream))
    # The attention part alone: the launch the Ulysses form makes over its
    # head groups (batch N * B, H / N heads), on head-split copies made here
    # (outside the timing).
    N, Hg = w.n_shards, w.H // w.n_shards
    split = [t.view(w.B, w.S, N, Hg, w.d).permute(2, 0, 1, 3, 4).contiguous()
             .view(N * w.B, w.S, Hg, w.d) for t in (q, k, v)]
    o_g = torch.empty_like(split[0])
    l_g = torch.empty((N * w.B, Hg, w.S), dtype=torch.float32, device=dev)

    def heads_only():
        pkg.cp_ring_attn_fwd(split[0], split[1], split[2], o_g, l_g, 1, w.causal, dd, stream)
    ms_a = timed(heads_only)
    if pkg.cp_get_last_status(stream) != 0:
        raise RuntimeError("device error in the Ulysses form")
    flops = effective_flops(w, docs)
    tensor_bytes = q.numel() * q.element_size()
    perm_bytes = 8 * tensor_bytes  # Q, K, V in and O out, each read once and written once
    hbm, _, _ = measured_peaks_hbm()
    return {
        "metric": METRIC, "impl": "ulysses_all_to_all", "unit": UNIT,
        "value": flops / (ms_u * 1e-3) / 1e12, "ms_per_step": ms_u, "ms_fused_ring": ms_f,
        "ms_head_group_attention": ms_a,
        "a2a_bytes_counted": moved[-1], "permutation_bytes_in_hbm": perm_bytes,
        # the form's time beyond its attention launch: a difference of two
        # totals, so it carries their noise (no bandwidth is derived from it)
        "ms_permutations_and_lse": ms_u - ms_a,
        "hbm_peak_GBps": hbm,
        "steps": args.steps, "warmup": args.warmup, "n_gpus": 1, "dtype": w.dtype,
        "data": "synthetic", "config": _config(w, docs, 1),
    }


def run_fp8(args, w, local):
    """Time the FP8 (E4M3) form on the workload's inputs stored as FP8: the
    quantisation of Q, K, V and the FP8 forward, each with CUDA events, and
    the bf16 forward on the same bf16 inputs beside them.  The roofline of
    the FP8 forward is taken against the FP8 dense peak: the measured bf16
    burst figure times the nominal FP8 / bf16 ratio (4.5 / 2.25 PFLOP/s).
    One JSON line."""
    import context_ring_attention_fwd_gb300 as pkg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    q, k, v = inputs.make_qkv(w.B, w.S, w.H, w.d, w.seed, w.torch_dtype, w.scale, device=str(dev))
    docs = (inputs.make_doc_offsets(w.S, w.seed + 1, w.doc_min, w.doc_max)
            if w.packed_docs else None)
    dd = pkg.doc_offsets_tensor(docs, dev)
    stream = torch.cuda.current_stream(dev)
    fp8 = pkg.fp8_quantize_qkv(q, k, v, stream)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / args.steps

    clocks = ClockSampler(gpu_index(local))
    clocks.start()
    time.sleep(0.3)
    ms_8 = timed(lambda: pkg.cp_ring_attn_fwd_fp8(*fp8, out, lse, w.n_shards, w.causal, dd,
                                                  stream))
    clk = clocks.stop()
    ms_q = timed(lambda: pkg.fp8_quantize_qkv(q, k, v, stream))
    ms_b = timed(lambda: pkg.cp_ring_attn_fwd(q, k, v, out, lse, w.n_shards, w.causal, dd,
                                              stream))
    if pkg.cp_get_last_status(stream) != 0:
        raise RuntimeError("device error in the FP8 form")
    flops = effective_flops(w, docs)
    achieved = flops / (ms_8 * 1e-3) / 1e12
    peak_burst, peak_sust, peak_src = measured_peaks()
    g8 = pkg.cp_ring_traffic(w.B, w.S, w.H, w.d, 1, w.n_shards, w.causal)
    g16 = pkg.cp_ring_traffic(w.B, w.S, w.H, w.d, 2, w.n_shards, w.causal)
    return {
        "metric": METRIC, "impl": "fp8_e4m3", "unit": UNIT, "value": achieved,
        "ms_per_step": ms_8, "ms_quantize_qkv": ms_q, "ms_bf16_fused": ms_b,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": 2 * peak_burst,
                     "unit": "TFLOP/s", "frac": achieved / (2 * peak_burst),
                     "traffic": ncu_traffic("fp8:" + w.name),
                     "traffic_sources": kernel_sources_digest(),
                     # Q, K, V read once as E4M3; O (bf16) and LSE written once
                     "algorithmic_bytes": 3 * w.B * w.S * w.H * w.d + 2 * w.B * w.S * w.H * w.d
                     + 4 * w.B * w.H * w.S,
                     "peak_kind": f"{peak_src} bf16 dense burst (cuBLAS) x 2 (nominal FP8/bf16)"},
        "ring_send_plus_recv_bytes_fp8": int(sum(g8)),
        "ring_send_plus_recv_bytes_bf16": int(sum(g16)),
        "clocks": clk, "steps": args.steps, "warmup": args.warmup, "n_gpus": 1,
        "dtype": "e4m3 (fp32 accumulate)", "data": "synthetic", "config": _config(w, docs, 1),
    }


def run_bwd(args, w, local):
    """Time the backward (cp_ring_attn_bwd: the row sums D, the dK/dV kernel
    and the dQ kernel) on the workload, after one forward for its out and
    lse.  Algorithmic work: 10 d FLOPs per visible pair (dP, dV, dK, dQ and
    the recomputed S, 2 d each); the two kernels execute 14 d (S and dP are
    formed in both).  Roofline against the bf16 dense peak.  One JSON line."""
    import context_ring_attention_fwd_gb300 as pkg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    q, k, v = inputs.make_qkv(w.B, w.S, w.H, w.d, w.seed, w.torch_dtype, w.scale, device=str(dev))
    dout = inputs.make_qkv(w.B, w.S, w.H, w.d, w.seed + 50, w.torch_dtype, device=str(dev))[0]
    docs = (inputs.make_doc_offsets(w.S, w.seed + 1, w.doc_min, w.doc_max)
            if w.packed_docs else None)
    dd = pkg.doc_offsets_tensor(docs, dev)
    stream = torch.cuda.current_stream(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
    pkg.cp_ring_attn_fwd(q, k, v, out, lse, w.n_shards, w.causal, dd, stream)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    ws = torch.empty(pkg.cp_ring_attn_bwd_workspace_bytes(w.B, w.S, w.H, w.d, w.n_shards),
                     dtype=torch.uint8, device=dev)

    def step():
        pkg.cp_ring_attn_bwd(q, k, v, out, lse, dout, dq, dk, dv, w.n_shards, w.causal, dd, ws,
                             stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(gpu_index(local))
    clocks.start()
    time.sleep(0.3)
    launches0 = pkg.launch_counts()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    launches1 = pkg.launch_counts()
    clk = clocks.stop()
    if pkg.cp_get_last_status(stream) != 0:
        raise RuntimeError("device error in the backward")
    ms = e0.elapsed_time(e1) / args.steps
    fwd_flops = effective_flops(w, docs)        # 4 d per visible pair
    flops = fwd_flops * 10 // 4
    achieved = flops / (ms * 1e-3) / 1e12
    peak_burst, peak_sust, peak_src = measured_peaks()
    return {
        "metric": "effective TFLOP/s of the ring-attention backward (1 GB300)", "impl": "bwd",
        "unit": UNIT, "value": achieved, "ms_per_step": ms, "higher_is_better": True,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_burst,
                     "unit": "TFLOP/s", "frac": achieved / peak_burst,
                     # DRAM bytes of one launch of the dominant kernel (dK/dV)
                     "traffic": ncu_traffic("bwd:" + w.name),
                     "traffic_kernel": "ring_attn_bwd_kernel<128, 1> (dK, dV)",
                     "traffic_sources": kernel_sources_digest(BWD_KERNEL_SOURCES),
                     "peak_kind": f"{peak_src} bf16 dense burst (cuBLAS)",
                     "executed_tflops": achieved * 14 / 10},
        "gpu_launches": int(sum(launches1) - sum(launches0)),
        "clocks": clk, "steps": args.steps, "warmup": args.warmup, "n_gpus": 1,
        "dtype": w.dtype, "data": "synthetic", "config": _config(w, docs, 1),
    }


def run_skip_check(args, w, local):
    """The schedule's acceptance checks on the workload's shape: the time of
    the causal forward over the time of the same shape without the causal
    mask (the computed-tile ratio is the ideal), and the causal time at
    N = 1, 2, 4, 8 shards (equal work, so equal time).  One JSON line."""
    import context_ring_attention_fwd_gb300 as pkg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    q, k, v = inputs.make_qkv(w.B, w.S, w.H, w.d, w.seed, w.torch_dtype, w.scale, device=str(dev))
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def timed(n_shards, causal):
        for _ in range(args.warmup):
            pkg.cp_ring_attn_fwd(q, k, v, out, lse, n_shards, causal, None, stream)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            pkg.cp_ring_attn_fwd(q, k, v, out, lse, n_shards, causal, None, stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / args.steps

    t_causal = timed(w.n_shards, True)
    t_full = timed(w.n_shards, False)
    by_n = {n: timed(n, True) for n in (1, 2, 4, 8) if w.S % n == 0}
    if pkg.cp_get_last_status(stream) != 0:
        raise RuntimeError("device error in the schedule check")
    L = w.S // w.n_shards
    T = -(-L // 128)
    n_tiles = w.n_shards * T
    causal_tiles = sum(min(n_tiles, (qt // T) * T + qt % T + 1) for qt in range(n_tiles))
    ideal = causal_tiles / (n_tiles * n_tiles)
    spread = (max(by_n.values()) - min(by_n.values())) / min(by_n.values())
    return {
        "metric": "schedule checks of the fused forward", "impl": "skip_check",
        "ms_causal": t_causal, "ms_full": t_full, "causal_over_full": t_causal / t_full,
        "computed_tile_ratio": ideal, "ms_causal_by_n_shards": by_n,
        "n_shards_spread": spread, "steps": args.steps, "warmup": args.warmup,
        "n_gpus": 1, "dtype": w.dtype, "data": "synthetic", "config": _config(w, None, 1),
    }


def run_hbm_kernels(args, w, local):
    """Time the bandwidth-bound kernels at the workload's shape, each against
    the measured HBM copy peak: the online merge and the finalize over one
    rank's fp32 state [B, S/N, H, d] (cp_lse_merge, cp_lse_finalize) and the
    FP8 quantiser of one bf16 tensor (cp_fp8_quantize, plain and transposed);
    the all-to-all permutation of the Ulysses form is reported by --ulysses.
    Algorithmic bytes per unit: merge 12 d + 24 per (b, row, h) (O, m, l of
    both operands read, the running state written); finalize 4 d + 8 read and
    2 d + 4 written (bf16 out); quantiser 2 B read for the amax, then 2 B read
    and 1 B written per element.  One JSON line."""
    import context_ring_attention_fwd_gb300 as pkg

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    B, H, d, N = w.B, w.H, w.d, w.n_shards
    L = w.S // N
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    o_acc = torch.randn((B, L, H, d), generator=g, device=dev)
    o_p = torch.randn((B, L, H, d), generator=g, device=dev)
    m_acc = torch.randn((B, H, L), generator=g, device=dev)
    m_p = torch.randn((B, H, L), generator=g, device=dev)
    l_acc = torch.rand((B, H, L), generator=g, device=dev) + 1.0
    l_p = torch.rand((B, H, L), generator=g, device=dev) + 1.0
    out = torch.empty((B, L, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    x = torch.randn((w.B, w.S, w.H, w.d), generator=g, device=dev).to(torch.bfloat16)
    x8 = torch.empty((w.B, w.S, w.H, w.d), dtype=torch.uint8, device=dev)
    x8t = torch.empty((w.B, w.H, w.d, w.S), dtype=torch.uint8, device=dev)
    desc = torch.empty((w.B, w.H), dtype=torch.float32, device=dev)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        times = []
        for _ in range(args.steps):
            flush.zero_()   # 512 MB written: the L2 (129 MB) holds nothing of the inputs
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            times.append(e0.elapsed_time(e1))
        return statistics.median(times)

    rows = B * L * H
    elems = w.B * w.S * w.H * w.d
    hbm, _, hbm_src = measured_peaks_hbm()
    kernels = []

    def add(name, ms, nbytes, unit_desc):
        gbs = nbytes / (ms * 1e-3) / 1e9
        kernels.append({"kernel": name, "ms": ms, "bytes": int(nbytes), "GB/s": gbs,
                        "frac_of_hbm": gbs / hbm, "units": unit_desc})

    add("lse_merge_kernel (cp_lse_merge)",
        timed(lambda: pkg.cp_lse_merge(o_acc, m_acc, l_acc, o_p, m_p, l_p, stream)),
        rows * (12 * d + 24), f"{rows} (b,row,h) x (12 d + 24) B")
    add("lse_finalize_kernel (cp_lse_finalize, bf16 out)",
        timed(lambda: pkg.cp_lse_finalize(o_acc, m_acc, l_acc, out, lse, stream)),
        rows * (6 * d + 12), f"{rows} (b,row,h) x (6 d + 12) B")
    add("fp8 quantiser (cp_fp8_quantize, [B,S,H,d])",
        timed(lambda: pkg.cp_fp8_quantize(x, x8, desc, False, stream)),
        elems * 5, f"{elems} elements x 5 B")
    add("fp8 quantiser (cp_fp8_quantize, transposed [B,H,d,S])",
        timed(lambda: pkg.cp_fp8_quantize(x, x8t, desc, True, stream)),
        elems * 5, f"{elems} elements x 5 B")
    if pkg.cp_get_last_status(stream) != 0:
        raise RuntimeError("device error in the bandwidth-bound kernels")
    return {"metric": "achieved GB/s of the bandwidth-bound kernels (1 GB300)",
            "impl": "hbm_kernels", "unit": "GB/s", "hbm_peak_GBps": hbm,
            "hbm_peak_kind": f"{hbm_src} copy bandwidth", "kernels": kernels,
            "l2_flush": "512 MB written between timed launches",
            "steps": args.steps, "warmup": args.warmup, "n_gpus": 1, "data": "synthetic",
            "config": _config(w, None, 1)}


def measured_peaks_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f).get("hbm_gbs"), None, "measured"
    return 6800.0, None, "fallback"


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(inputs.BY_NAME))
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--cpu-rows", type=int, default=None,
                    help="query rows per head for the oracle timing (default: every row up "
                         "to S = 8192, where the whole oracle fits the budget; 512 above)")
    ap.add_argument("--no-gates", action="store_true",
                    help="leave the schedule checks out of the default line")
    ap.add_argument("--hbm-kernels", action="store_true",
                    help="time the bandwidth-bound kernels (merge, finalize, FP8 quantiser, "
                         "all-to-all permutation) against the measured HBM peak instead")
    ap.add_argument("--ring-emulation", action="store_true",
                    help="time the ring with explicit per-rank buffers instead")
    ap.add_argument("--ulysses", action="store_true",
                    help="time the all-to-all (Ulysses) form instead")
    ap.add_argument("--fp8", action="store_true",
                    help="time the FP8 (E4M3) form instead")
    ap.add_argument("--bwd", action="store_true", help="time the backward instead")
    ap.add_argument("--skip-check", action="store_true",
                    help="causal / full time ratio and shard-count invariance instead")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the attention kernel from an ncu capture")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    w = inputs.BY_NAME[args.workload]
    if (args.ring_emulation or args.ulysses or args.fp8 or args.bwd or args.skip_check
            or args.hbm_kernels):
        line = (run_ring_emulation(args, w, local) if args.ring_emulation
                else run_ulysses(args, w, local) if args.ulysses
                else run_fp8(args, w, local) if args.fp8
                else run_hbm_kernels(args, w, local) if args.hbm_kernels
                else run_bwd(args, w, local) if args.bwd else run_skip_check(args, w, local))
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    if args.impl == "reference":
        dist_init(world, "gloo")
        line = run_reference(args, w, rank, world)
    else:
        dist_init(world, "nccl" if torch.cuda.is_available() else "gloo")
        line = run_ours(args, w, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
