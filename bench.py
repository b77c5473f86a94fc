"""Benchmark: chunked-prefill attention over a paged KV cache on one GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload mixed_serving|mixed_serving_fp8|nonpow2|swa64|swa1024|mm|mixed|
                                mixed_fp8|mixed_window|mixed_cached|chunked|decode|decode_split|
                                decode_fp8|decode_fp8_inkernel|mixed_fp8_inkernel]
                    [--no-cpu-baseline] [--sweep windows|pages|splits|groups]

A step is one pass of the whole hot path over one batch: for every run (shape) of the
workload, stage 1 (live key-tile bounds and work list) and the attention kernel, through the
C ABI. The default workload is the mixed-serving sweep: one seeded batch of 32 sequences
(context U[4096, 32768], query U[512, 4096], 32 q / 4 kv heads, D 128, causal) run at each page
size 128, 512, 544, 1040, 1056 and 2048, without a window and with window_left 4096 (12 runs,
bf16 KV; ``mixed_serving_fp8`` runs the same sweep over an fp8 e4m3 cache). Values are seeded
N(0,1) (synthetic data). L2 (129 MB) is flushed between timed steps by writing 512 MiB; the
flush is outside the timed region. The CPU-baseline leg times the oracle on sampled rows and
compares those rows with the last timed step's output (``parity`` in the line).

Prints one JSON line (rank 0). ``value`` is TFLOP/s over live (query, key) pairs:
4 * D * Hq per pair, pairs counted by the library's own interval arithmetic.
Under torchrun each rank runs its own seeded batch (weak scaling, no data-path collective);
the step time is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill attn TFLOP/s (live pairs) & % GB300 bf16 TC peak; tokens/s at 1 GPU"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------------------
def make_workload(name: str, seed: int):
    from paged_kv_prefix_gb300 import workloads as wl
    if name in ("mixed_serving", "mixed_serving_fp8"):
        kv = "fp8_e4m3" if name.endswith("fp8") else "bf16"
        return ("mixed serving sweep: 32 seqs, ctx U[4096,32768], q U[512,4096], 32 q / 4 kv "
                "heads, D 128, causal; one run per page size in {128,512,544,1040,1056,2048} x "
                f"window_left in {{0,4096}} (12 runs, one seeded batch), {kv} KV cache"
                + (" (one per-tensor fp32 scale each for K and V)" if kv != "bf16" else ""),
                [wl.mixed(p, w, kv_dtype=kv, seed=seed) for w in (False, True)
                 for p in wl.MIXED_PAGE_SIZES])
    if name == "nonpow2":
        return ("non-power-of-2 pages: 8 seqs, ctx U[0,8192], q U[1,2048], causal; "
                "(Hq,G,D,P) = (64,1,128,544), (8,4,256,1040), (8,4,256,1056)",
                [wl.nonpow2(i, seed=seed) for i in range(3)])
    if name == "swa64":
        return ("sliding window 64/64 non-causal, 1 seq x 16384, 8 heads, D 64, page 16",
                [wl.swa_noncausal(seed=seed)])
    if name == "swa1024":
        return ("sliding window 1024 causal, 1 seq x 32768, 8 heads, D 64, page 16",
                [wl.swa_causal(seed=seed)])
    if name == "mm":
        return ("clamped multimodal: 4 seqs x 16384, 16 q / 8 kv heads, D 256, page 16, causal, "
                "window 1024, 60 ranges x 256 tokens", [wl.clamped_mm(seed=seed)])
    if name == "mixed":
        return ("mixed serving: 32 seqs, ctx U[4096,32768], q U[512,4096], 32 q / 4 kv heads, "
                "D 128, causal, page 544, no window, bf16 KV", [wl.mixed(544, False, seed=seed)])
    if name in ("mixed_fp8", "mixed_fp8_inkernel"):
        return ("mixed serving, fp8 e4m3 KV cache (one per-tensor scale each for K and V): 32 seqs, "
                "ctx U[4096,32768], q U[512,4096], 32 q / 4 kv heads, D 128, causal, page 544"
                + ("; e4m3 rows widened in the attention kernel" if name.endswith("inkernel")
                   else ""),
                [wl.mixed(544, False, kv_dtype="fp8_e4m3", seed=seed)])
    if name in ("decode_fp8", "decode_fp8_inkernel"):
        return ("decode over an fp8 e4m3 cache: 32 seqs, ctx U[8192,32768], 1 new token each, "
                "32 q / 8 kv heads, D 128, page 544, causal; "
                + ("e4m3 rows widened in the attention kernel" if name.endswith("inkernel")
                   else "live cache tiles dequantised into workspace first"),
                [wl.decode(seed=seed, kv_dtype="fp8_e4m3")])
    if name in ("decode", "decode_split"):
        return (f"decode: 32 seqs, ctx U[8192,32768], 1 new token each, 32 q / 8 kv heads, D 128, "
                f"page 544, causal"
                + (", split-KV in the library's tuned segments (32 key tiles)"
                   if name == "decode_split" else ""),
                [wl.decode(seed=seed)])
    if name == "chunked":
        return ("chunked-local attention: 4 seqs x 32768 new tokens, 32 q / 8 kv heads, D 128, "
                "page 544, causal, chunk 8192, lookback 0", [wl.chunked_local(seed=seed)])
    if name == "mixed_cached":
        return ("mixed serving, new tokens appended to the paged cache then attended from it "
                "(ppa_append_kv + cache-sourced attention): 32 seqs, ctx U[4096,32768], "
                "q U[512,4096], 32 q / 4 kv heads, D 128, causal, page 544, bf16 KV",
                [wl.mixed(544, False, seed=seed)])
    if name == "mixed_window":
        return ("mixed serving with window_left 4096: 32 seqs, ctx U[4096,32768], q U[512,4096], "
                "32 q / 4 kv heads, D 128, causal, page 2048, bf16 KV",
                [wl.mixed(2048, True, seed=seed)])
    raise SystemExit(f"unknown workload {name}")


# ---------------------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------------------
def _prepass(dc) -> bool:
    """An fp8 cache dequantised into workspace before the attention kernel (the default)."""
    from paged_kv_prefix_gb300 import binding
    return (dc.dims.kv_dtype == binding.PPA_KV_FP8_E4M3
            and not (dc.dims.flags & binding.PPA_FLAG_FP8_INKERNEL))


def _kv_in_cache(dc) -> bool:
    """The step appends the new tokens to the cache and attends from it."""
    from paged_kv_prefix_gb300 import binding
    return bool(dc.dims.flags & binding.PPA_FLAG_KV_IN_CACHE)


def _launches_per_step(dc) -> int:
    """Kernels of this library per step: the plan and the attention kernel, plus the fp8
    live-tile marking, staging-slot and dequantisation kernels, plus the KV append, plus the
    split-KV merge."""
    return (2 + (3 if _prepass(dc) else 0) + (1 if _kv_in_cache(dc) else 0)
            + (1 if dc.dims.kv_split_tiles != 0 else 0))


def workload_flags(name: str) -> int:
    from paged_kv_prefix_gb300 import binding
    if name == "mixed_cached":
        return binding.PPA_FLAG_KV_IN_CACHE
    return binding.PPA_FLAG_FP8_INKERNEL if name.endswith("_inkernel") else 0


def cache_token_bound(case, flags: int) -> int:
    """ppa_dims.max_cache_tokens as a serving engine would pass it for an fp8 cache: the cached
    positions of the batch (context, plus the new tokens when they are appended first)."""
    from paged_kv_prefix_gb300 import binding
    if case.kv_dtype == "bf16":
        return 0
    return int(case.context_lens.sum()) + (case.total_q if flags & binding.PPA_FLAG_KV_IN_CACHE
                                           else 0)


def append_bytes(case) -> float:
    """The KV append's algorithmic bytes: every new token's K and V row read (bf16) and
    written (bf16 or one byte per fp8 code)."""
    per = 2 + (1 if case.kv_dtype == "fp8_e4m3" else 2)
    return 2.0 * case.total_q * case.num_kv_heads * case.head_dim * per


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_prefix_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per attention launch from a committed ncu capture, if it still matches."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(workload)
    if not ent or ent.get("kernel_source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


def algorithmic_flops(binding, dc, case, stream) -> float:
    """4 * D * Hq per live (query, key) pair: QK^T and PV, 2*D each, per query head."""
    import torch
    cnt = torch.zeros(1, dtype=torch.int64, device=dc.q.device)
    binding.ppa_live_pairs(dc.dims, dc.cu_query_lens, dc.context_lens, dc.mm_ranges, cnt, stream)
    return 4.0 * case.head_dim * case.num_q_heads * float(cnt.item())


def algorithmic_bytes(binding, dc, case, stream) -> float:
    """Bytes one pass must move at least once: Q and O, k_new and v_new, every live cached
    token's K and V row once per KV head, the block-table entries read and the ranges."""
    import torch
    cnt = torch.zeros(1, dtype=torch.int64, device=dc.q.device)
    binding.ppa_live_kv_tokens(dc.dims, dc.cu_query_lens, dc.context_lens, dc.mm_ranges, cnt,
                               stream)
    D, Hq, Hkv = case.head_dim, case.num_q_heads, case.num_kv_heads
    kv_bytes = 1 if case.kv_dtype == "fp8_e4m3" else 2
    ctx = case.context_lens.numpy().astype(np.int64)
    table = int(((ctx + case.page_size - 1) // case.page_size).sum()) * 4
    ranges = 0 if case.mm_ranges is None else case.mm_ranges.numel() * 4
    return (case.total_q * (2 * Hq * D + 2 * Hkv * D) * 2
            + float(cnt.item()) * 2 * Hkv * D * kv_bytes + table + ranges)


def roofline(flops: float, nbytes: float, seconds: float, peaks: dict, peak_src: str) -> dict:
    """The bound of one launch: tensor cores when its intensity is above the ridge of the
    measured peaks, HBM below it."""
    tflops_peak = float(peaks["bf16_tflops"])
    gbs_peak = float(peaks["hbm_gbs"])
    ridge = tflops_peak * 1e12 / (gbs_peak * 1e9)
    intensity = flops / max(nbytes, 1.0)
    if intensity >= ridge:
        a = flops / seconds / 1e12
        return {"bound": "tensor", "achieved": a, "peak": tflops_peak, "unit": "TFLOP/s",
                "frac": a / tflops_peak, "intensity_flop_per_byte": intensity,
                "peak_source": f"{peak_src} bf16 dense (burst)"}
    a = nbytes / seconds / 1e9
    return {"bound": "hbm", "achieved": a, "peak": gbs_peak, "unit": "GB/s", "frac": a / gbs_peak,
            "intensity_flop_per_byte": intensity, "peak_source": f"{peak_src} HBM copy"}


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
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
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "t0", 0.0), getattr(self, "t1", float("inf"))
        inside = [ln for ts, ln in self.lines if t0 <= ts <= t1 + 0.05]
        if not inside and self.lines:  # timed region shorter than the sampling period
            mid = 0.5 * (t0 + min(t1, self.lines[-1][0]))
            inside = [min(self.lines, key=lambda x: abs(x[0] - mid))[1]]
        for line in inside:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        return dist, rank, world, local
    return None, rank, world, local


def max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------------------
# CPU oracle baseline (the only place bench.py runs oracle/)
# ---------------------------------------------------------------------------------------
def oracle_sample(cases, budget_s: float, rng_seed: int = 0):
    """Times the oracle on evenly spaced query tokens of each case until ~budget_s of CPU
    work. Returns (live-pair FLOPs computed, seconds, description, rows): ``rows`` lists, per
    case, (sequence, query tokens, the oracle's output rows) of the last sample taken."""
    from oracle import ref
    flops, secs, tokens = 0.0, 0.0, 0
    per_case = budget_s / len(cases)
    rows = []
    for case in cases:
        inp = case.numpy_inputs()
        cu = inp["cu_query_lens"]
        B = case.num_seqs
        b = int(np.argmax([(cu[i + 1] - cu[i]) * (inp["context_lens"][i] + cu[i + 1] - cu[i])
                           for i in range(B)]))
        c = int(inp["context_lens"][b])
        n = int(cu[b + 1] - cu[b])
        kv = (ref.gather_kv(inp, b, "k"), ref.gather_kv(inp, b, "v"))
        spent, count = 0.0, 2
        last = None
        while spent < per_case and count <= n:
            toks = np.linspace(0, n - 1, num=min(count, n)).astype(np.int64)
            t0 = time.perf_counter()
            out = ref.attention_rows(inp, b, toks, kv=kv)
            dt = time.perf_counter() - t0
            last = (b, toks, out)
            pairs = int(ref.allowed_mask(c + toks, c + n, case.causal, case.window_left,
                                         case.window_right, None if inp["mm_ranges"] is None
                                         else inp["mm_ranges"][b], case.clamp_mm,
                                         case.chunk_size, case.chunk_lookback).sum())
            flops += 4.0 * case.head_dim * case.num_q_heads * pairs
            secs += dt
            tokens += len(toks)
            spent += dt
            count *= 2
        rows.append(last)
    return (flops, secs,
            f"{tokens} query tokens (all heads) of the heaviest sequence of each shape", rows)


def sampled_parity(cases, dcs, rows) -> dict:
    """The oracle rows the CPU baseline computed, against the same rows of the timed run's
    output: max abs error and the number of elements outside |err| <= 2e-2 + 2e-2 |want|."""
    worst, bad, n_el = 0.0, 0, 0
    for case, dc, r in zip(cases, dcs, rows):
        if r is None:
            continue
        b, toks, want = r
        q0 = int(case.cu_query_lens[b])
        got = dc.out[q0 + toks].float().cpu().numpy()
        err = np.abs(got - want)
        worst = max(worst, float(err.max()))
        bad += int((err > 2e-2 + 2e-2 * np.abs(want)).sum())
        n_el += err.size
    return {"parity_max_abs": worst, "elements_outside_2e-2": bad, "elements_checked": n_el}


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------------------
def run_reference(args):
    dist, rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    desc, cases = make_workload(args.workload, seed=0)
    per_step = args.ref_step_seconds
    for _ in range(args.warmup):
        oracle_sample(cases, per_step / 4)
    total_f, total_s, sample = 0.0, 0.0, ""
    for _ in range(args.steps):
        f, s, sample, _ = oracle_sample(cases, per_step)
        total_f += f
        total_s += s
    tflops = total_f / total_s / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": desc},
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------
def run_ours(args):
    import torch
    from paged_kv_prefix_gb300 import binding

    dist, rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    binding.lib()
    desc, cases = make_workload(args.workload, seed=rank)
    if args.split is not None:
        desc += f"; kv_split_tiles {args.split}"
    if args.runs:  # a subset of the workload's runs (e.g. one launch for a profiler)
        keep = [int(x) for x in args.runs.split(",")]
        cases = [cases[i] for i in keep]
        desc += f"; runs {keep} only: " + ", ".join(c.name for c in cases)
    flags = workload_flags(args.workload)
    dcs = [binding.DeviceCase(c, device=dev, flags_extra=flags,
                              kv_split_tiles=(args.split if args.split is not None
                                              else -1 if args.workload == "decode_split" else 0),
                              max_cache_tokens=cache_token_bound(c, flags))
           for c in cases]
    stream = torch.cuda.current_stream(dev)

    # live pairs and FLOPs, live cache tokens and algorithmic bytes, from the library's own
    # interval arithmetic
    flops, nbytes, tokens = [], [], 0
    for dc, case in zip(dcs, cases):
        flops.append(algorithmic_flops(binding, dc, case, stream))
        nbytes.append(algorithmic_bytes(binding, dc, case, stream))
        tokens += case.total_q
    step_flops = sum(flops)

    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def step(ev_list):
        for i, dc in enumerate(dcs):
            ev_list[i][0].record(stream)
            if _kv_in_cache(dc):
                dc.append(stream)
            ev_list[i][3].record(stream)
            dc.plan(stream)
            ev_list[i][1].record(stream)
            dc.attend(stream)
            ev_list[i][2].record(stream)

    # per shape: step start, after the plan, after the attention, after the append
    mk = lambda: [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in dcs]
    # clocks: the sampler runs from before the warm-up; samples inside the timed region count
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    for _ in range(args.warmup):
        flush.zero_()
        step(mk())
    torch.cuda.synchronize()
    for dc in dcs:
        st = dc.read_status(stream)
        if st != 0:
            raise SystemExit(f"device status {st}: {binding.status_string(st)}")

    events = [mk() for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark(True)
    t_wall = time.perf_counter()
    for k in range(args.steps):
        flush.zero_()
        step(events[k])
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    if dist is not None:
        dist.barrier()
    if sampler:
        sampler.mark(False)
    clocks = sampler.stop() if sampler else None

    step_ms = [sum(ev[i][0].elapsed_time(ev[i][2]) for i in range(len(dcs))) for ev in events]
    attend_ms = np.array([[ev[i][1].elapsed_time(ev[i][2]) for i in range(len(dcs))]
                          for ev in events])  # [steps, shapes]
    plan_ms = np.array([[ev[i][3].elapsed_time(ev[i][1]) for i in range(len(dcs))]
                        for ev in events])
    app_ms = np.array([[ev[i][0].elapsed_time(ev[i][3]) for i in range(len(dcs))]
                       for ev in events])
    total_ms = max_over_ranks(dist, float(sum(step_ms)), dev)
    all_flops = sum_over_ranks(dist, step_flops * args.steps, dev)
    all_tokens = sum_over_ranks(dist, float(tokens * args.steps), dev)
    for dc in dcs:
        st = dc.read_status(stream)
        if st != 0:
            raise SystemExit(f"device status {st}: {binding.status_string(st)}")

    # ---- e2e: host buffers in, host result out, through the same public API ----
    e2e = run_e2e(args, cases, dcs, step_flops, stream, dev)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    value = all_flops / (total_ms * 1e-3) / 1e12
    # dominant kernel: the attention launch with the largest total time
    shape_tot = attend_ms.sum(axis=0)
    dom = int(np.argmax(shape_tot))
    dom_avg_s = float(attend_ms[:, dom].mean()) * 1e-3
    peak = float(peaks["bf16_tflops"])
    roof = roofline(flops[dom], nbytes[dom], dom_avg_s, peaks, peak_src)
    roof["traffic"] = recorded_traffic(args.workload)
    roof["kernel"] = (f"{'fp8 dequant + ' if _prepass(dcs[dom]) else ''}"
                      f"{'attn_pair_kernel' if cases[dom].head_dim == 256 else 'attn_ws_kernel'}"
                      f"{' + split merge' if dcs[dom].dims.kv_split_tiles != 0 else ''} "
                      f"({cases[dom].name})")
    shapes = []
    for i, case in enumerate(cases):
        a = float(attend_ms[:, i].mean())
        shapes.append({"shape": case.name, "attend_ms": round(a, 4),
                       "plan_ms": round(float(plan_ms[:, i].mean()), 4),
                       "tflops": round(flops[i] / (a * 1e-3) / 1e12, 2),
                       "gbs": round(nbytes[i] / (a * 1e-3) / 1e9, 1),
                       "live_tflop": round(flops[i] / 1e12, 4),
                       "algorithmic_mb": round(nbytes[i] / 1e6, 2)})
        if _kv_in_cache(dcs[i]):  # the append kernel against the HBM roofline
            am = float(app_ms[:, i].mean())
            gbs = append_bytes(case) / (am * 1e-3) / 1e9
            shapes[-1]["append"] = {"kernel": "append_kv_kernel", "ms": round(am, 4),
                                    "algorithmic_mb": round(append_bytes(case) / 1e6, 2),
                                    "gbs": round(gbs, 1), "peak": float(peaks["hbm_gbs"]),
                                    "frac": round(gbs / float(peaks["hbm_gbs"]), 4)}
    cpu = None
    check = None
    if not args.no_cpu_baseline and world == 1:
        f, s, sample, rows = oracle_sample(cases, args.cpu_seconds)
        cpu = {"value": f / s / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": sample + f" ({s:.1f} s)"}
        # the rows the oracle just computed, against the output of the last timed step
        check = sampled_parity(cases, dcs, rows)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": desc, "l2": "flushed between timed steps (512 MiB write)",
                   "seed_per_rank": "rank"},
        "pct_bf16_peak": 100.0 * value / peak,
        "tokens_per_s": all_tokens / (total_ms * 1e-3),
        "roofline": roof,
        "shapes": shapes,
        "e2e": e2e,
        "gpu_launches": sum(_launches_per_step(dc) for dc in dcs) * args.steps,
        "clocks": clocks,
        "wall_s_timed_region": t_wall,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
        line["parity"] = check
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_e2e(args, cases, dcs, step_flops, stream, dev):
    """Same metric with host inputs: per step, pinned-host -> device copies of every input,
    the C-ABI call, and a device -> host copy of the output, all inside the timed region."""
    import torch
    from paged_kv_prefix_gb300 import binding

    names = ["q", "k_new", "v_new", "k_cache", "v_cache", "block_table", "cu_query_lens",
             "context_lens"]
    host = []
    h2d = d2h = 0
    pinned = {}  # one pinned copy per host tensor (runs of a sweep share their value tensors)

    def pin(t):
        if id(t) not in pinned:
            pinned[id(t)] = t.pin_memory()
        return pinned[id(t)]

    for case, dc in zip(cases, dcs):
        hs = {n: pin(getattr(case, n)) for n in names}
        if case.mm_ranges is not None:
            hs["mm_ranges"] = case.mm_ranges.pin_memory()
        hs["k_scale"] = torch.tensor([case.k_scale], dtype=torch.float32).pin_memory()
        hs["v_scale"] = torch.tensor([case.v_scale], dtype=torch.float32).pin_memory()
        hs["out"] = torch.empty_like(case.q).pin_memory()
        h2d += sum(v.numel() * v.element_size() for k, v in hs.items() if k != "out")
        d2h += hs["out"].numel() * hs["out"].element_size()
        host.append(hs)

    def one():
        for hs, dc in zip(host, dcs):
            for n in names:
                getattr(dc, n).copy_(hs[n], non_blocking=True)
            if dc.mm_ranges is not None:
                dc.mm_ranges.copy_(hs["mm_ranges"], non_blocking=True)
            dc.k_scale.copy_(hs["k_scale"], non_blocking=True)
            dc.v_scale.copy_(hs["v_scale"], non_blocking=True)
            if _kv_in_cache(dc):
                dc.append(stream)
            dc.run(stream)
            hs["out"].copy_(dc.out, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        one()
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, 5))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": step_flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": ms}


def run_window_sweep(args):
    """Causal sliding-window prefill over a grid of sequence lengths and windows: time should
    follow the live pairs (~ L * W), not L^2. One JSON line per point."""
    import torch
    from paged_kv_prefix_gb300 import binding
    from paged_kv_prefix_gb300 import workloads as wl
    torch.cuda.set_device(0)
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for seq_len in (16384, 32768, 65536):
        for window in (512, 1024, 2048):
            case = wl.swa_causal(seed=0, seq_len=seq_len, window=window)
            dc = binding.DeviceCase(case)
            flops = algorithmic_flops(binding, dc, case, stream)
            nbytes = algorithmic_bytes(binding, dc, case, stream)
            dc.plan(stream)
            ms = []
            for k in range(args.warmup + args.steps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                dc.attend(stream)
                e1.record(stream)
                torch.cuda.synchronize()
                if k >= args.warmup:
                    ms.append(e0.elapsed_time(e1))
            st = dc.read_status(stream)
            t = float(np.median(ms)) * 1e-3
            print(json.dumps({"sweep": "sliding_window_causal", "seq_len": seq_len, "window": window,
                              "attend_ms": t * 1e3, "live_pairs_per_head": flops / (4 * 64 * 8),
                              "tflops": flops / t / 1e12, "gbs": nbytes / t / 1e9,
                              "ns_per_mpair": t * 1e9 / (flops / (4 * 64 * 8) / 1e6),
                              "roofline": roofline(flops, nbytes, t, peaks, peak_src),
                              "status": st}), flush=True)
            del dc


def run_page_sweep(args):
    """One ragged batch (8 sequences, context U[0, 8192], 1-2048 new tokens, causal) at every
    page size the pages name and each head shape: with key tiles that straddle pages, the
    throughput should not depend on the page size. One JSON line per point."""
    import torch
    from paged_kv_prefix_gb300 import binding
    from paged_kv_prefix_gb300 import workloads as wl
    torch.cuda.set_device(0)
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(0)
    ctx = rng.integers(0, 8193, size=8)
    qlen = rng.integers(1, 2049, size=8)
    for hq, hkv, d in ((64, 64, 128), (32, 8, 128), (8, 2, 256), (16, 16, 64)):
        for page in (16, 128, 512, 544, 1040, 1056, 2048):
            case = wl.build_case(f"pages_h{hq}_g{hq // hkv}_d{d}_p{page}", ctx, qlen, hq, hkv, d,
                                 page, causal=True, seed=0)
            dc = binding.DeviceCase(case)
            flops = algorithmic_flops(binding, dc, case, stream)
            nbytes = algorithmic_bytes(binding, dc, case, stream)
            dc.plan(stream)
            ms = []
            for k in range(args.warmup + args.steps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                dc.attend(stream)
                e1.record(stream)
                torch.cuda.synchronize()
                if k >= args.warmup:
                    ms.append(e0.elapsed_time(e1))
            st = dc.read_status(stream)
            t = float(np.median(ms)) * 1e-3
            print(json.dumps({"sweep": "page_size", "num_q_heads": hq, "group": hq // hkv,
                              "head_dim": d, "page_size": page, "attend_ms": t * 1e3,
                              "tflops": flops / t / 1e12, "gbs": nbytes / t / 1e9,
                              "roofline": roofline(flops, nbytes, t, peaks, peak_src),
                              "status": st}), flush=True)
            del dc


def run_group_sweep(args):
    """One ragged causal batch (8 sequences, context U[0, 8192], 1-2048 new tokens, page 544)
    for every head dimension and GQA group size (8 KV heads, 8 * G query heads): how the tile
    shape (a query tile holds 128 / G tokens of G heads) and the head dimension move the
    tensor throughput. One JSON line per point."""
    import torch
    from paged_kv_prefix_gb300 import binding
    from paged_kv_prefix_gb300 import workloads as wl
    torch.cuda.set_device(0)
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(0)
    ctx = rng.integers(0, 8193, size=8)
    qlen = rng.integers(1, 2049, size=8)
    for d in (64, 128, 256):
        for g in (1, 2, 4, 8):
            case = wl.build_case(f"groups_d{d}_g{g}", ctx, qlen, 8 * g, 8, d, 544, causal=True,
                                 seed=0)
            dc = binding.DeviceCase(case)
            flops = algorithmic_flops(binding, dc, case, stream)
            dc.plan(stream)
            ms = []
            for k in range(args.warmup + args.steps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                dc.attend(stream)
                e1.record(stream)
                torch.cuda.synchronize()
                if k >= args.warmup:
                    ms.append(e0.elapsed_time(e1))
            st = dc.read_status(stream)
            t = float(np.median(ms)) * 1e-3
            print(json.dumps({"sweep": "head_dim_and_group", "head_dim": d, "group": g,
                              "num_q_heads": 8 * g, "attend_ms": t * 1e3,
                              "tflops": flops / t / 1e12,
                              "frac_bf16": flops / t / 1e12 / float(peaks["bf16_tflops"]),
                              "status": st}), flush=True)
            del dc


def run_split_sweep(args):
    """Decode and verification batches (1 or 4 new tokens per sequence over 8K-32K contexts)
    at several split-KV segment lengths (kv_split_tiles, 0 = unsplit): the time per launch
    (plan, attention and merge) and the achieved HBM bandwidth. One JSON line per point."""
    import torch
    from paged_kv_prefix_gb300 import binding
    from paged_kv_prefix_gb300 import workloads as wl
    torch.cuda.set_device(0)
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    for num_seqs in (8, 32):
        for new_tokens in (1, 4):
            case = wl.decode(seed=0, num_seqs=num_seqs, new_tokens=new_tokens)
            for split in (0, 4, 8, 16, 32, 64, -1):
                dc = binding.DeviceCase(case, kv_split_tiles=split)
                nbytes = algorithmic_bytes(binding, dc, case, stream)
                ms = []
                for k in range(args.warmup + args.steps):
                    flush.zero_()
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    dc.run(stream)
                    e1.record(stream)
                    torch.cuda.synchronize()
                    if k >= args.warmup:
                        ms.append(e0.elapsed_time(e1))
                st = dc.read_status(stream)
                t = float(np.median(ms)) * 1e-3
                print(json.dumps({"sweep": "kv_split_tiles", "num_seqs": num_seqs,
                                  "new_tokens": new_tokens, "kv_split_tiles": split,
                                  "ms": t * 1e3, "gbs": nbytes / t / 1e9,
                                  "frac_hbm": nbytes / t / 1e9 / float(peaks["hbm_gbs"]),
                                  "workspace_mb": dc.workspace.numel() / 1e6, "status": st}),
                      flush=True)
                del dc


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mixed_serving")
    ap.add_argument("--split", type=int, default=None,
                    help="kv_split_tiles for every run (-1: the library's tuned length)")
    ap.add_argument("--runs", default="",
                    help="comma-separated indices: run only these runs (shapes) of the workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-step-seconds", type=float, default=6.0)
    ap.add_argument("--sweep", choices=["windows", "pages", "splits", "groups"], default=None,
                    help="print one line per point of a window / length sweep instead")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.sweep == "windows":
        run_window_sweep(args)
    elif args.sweep == "pages":
        run_page_sweep(args)
    elif args.sweep == "splits":
        run_split_sweep(args)
    elif args.sweep == "groups":
        run_group_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
