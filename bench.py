#!/usr/bin/env python3
"""Benchmark of the paged decode attention layer-step on GB300.

One step = one decode layer-step of the whole batch: reshape_and_cache of the
new token of every sequence, then decode attention through the block tables
(split kernel + log-sum-exp merge, or the single pass).  Inputs are seeded
synthetic workloads resident in HBM; L2 is flushed before
every step (a 256 MiB write, then a 256 MiB read) and only the step's own
kernels sit between its CUDA events.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config llama8b]
    python bench.py --impl reference ...   # the CPU reference on host cores

Prints one JSON line (rank 0).  Metric: KV GB/s of the layer-step, with
bytes = K/V of every context token read + q read + output written.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_226_gb300 import build as pa_build  # noqa: E402
from paged_kv_cache_226_gb300 import inputs as pin  # noqa: E402
from paged_kv_cache_226_gb300 import lib  # noqa: E402

METRIC = "paged decode attention KV GB/s and % of GB300 HBM peak; µs per layer-step"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
FP8_K_SCALE, FP8_V_SCALE = 1.0 / 64, 1.0 / 48
_CSRC = os.path.join(ROOT, "paged_kv_cache_226_gb300", "csrc")
_TILE_SOURCES = ["decode_tile.cuh", "pa_device.cuh", "pa_internal.h"]
# the sources each timed kernel is compiled from: a committed DRAM-traffic
# figure counts only while these are unchanged
KERNEL_SOURCES = {
    "paged_decode": ["decode_kernel.cuh"] + _TILE_SOURCES,
    "paged_decode_split": ["decode_kernel.cuh"] + _TILE_SOURCES,
    "paged_decode_step": ["decode_kernel.cuh"] + _TILE_SOURCES,
    "balanced_step": ["balanced.cu"] + _TILE_SOURCES,
    "paged_prefill": ["prefill.cu", "prefill_tc.cu", "tc_device.cuh", "prefill_internal.h"] + _TILE_SOURCES,
}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    return int(os.environ.get("RANK", "0")), ws, int(os.environ.get("LOCAL_RANK", "0"))


def rank_seed(config: str, rank: int) -> int:
    """Each rank draws its own batch of the same shape (weak scaling)."""
    return pin.CONFIGS[config][0] + 1000 * rank


def max_over_ranks(value: float, device=None) -> float:
    """MAX of a per-rank scalar over the process group (identity without one)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank_step: int, world: int, ms_per_step: float) -> float:
    """All ranks' bytes per step over the slowest rank's step time."""
    return bytes_per_rank_step * world / (ms_per_step * 1e-3) / 1e9


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(_CSRC, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(config: str, kernel: str, partition=None):
    """DRAM bytes per launch from a committed ncu summary
    (profiles/<kernel>_<config>.json), if it was taken on the kernel's current
    sources and, for a partitioned launch, at the same partition size; else
    None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{config}.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        p = json.load(f)
    if p.get("source_sha256_16") != source_hash(kernel):
        return None
    if partition is not None and p.get("partition_tokens") != partition:
        return None
    return p.get("dram_bytes_per_launch")


def step_bytes(w: pin.Workload, mode: str, partition: int, cache_elem_bytes: int = 2):
    """Algorithmic bytes: the layer-step and each kernel of it."""
    e = 2
    B, hq, hkv, d = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim
    kv = w.kv_bytes_logical() * cache_elem_bytes // 2
    q = B * hq * d * e
    out = B * hq * d * e
    new_tok = w.num_tokens * hkv * d * e * 2           # read k, v
    write_tok = int((w.slot_mapping >= 0).sum()) * hkv * d * cache_elem_bytes * 2
    parts = sum(-(-int(L) // partition) for L in w.context_lens)
    split_w = parts * hq * (d + 2) * 4                  # tmp_out + max_logits + exp_sums
    kernels = {"reshape_and_cache": new_tok + write_tok + w.num_tokens * 8}
    if mode in ("fused", "balanced"):
        name = "paged_decode_step" if mode == "fused" else "balanced_step"
        kernels = {name: kv + q + out + new_tok + write_tok + w.num_tokens * 8}
    elif mode == "split":
        kernels["paged_decode_split"] = kv + q + split_w
        kernels["lse_reduce"] = split_w + out
    else:
        kernels["paged_decode"] = kv + q + out
    return {"layer_step": kv + q + out, "kernels": kernels, "partitions": parts, "kv": kv}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.f = None

    def __enter__(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
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
        return False

    def summary(self, t0: float = None, t1: float = None):
        """Median SM clock and the throttle reasons seen between wall times
        t0 and t1 (time.time()); all samples when not given."""
        if self.proc is None or self.f is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        import datetime
        self.f.flush()
        self.f.seek(0)
        rows = [r.strip().split(", ") for r in self.f.read().splitlines() if r.strip()]
        os.unlink(self.f.name)
        sm, smax, reasons, n_all = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk, cmax = float(r[2]), float(r[3])
            except ValueError:
                continue
            n_all += 1
            if t0 is not None and not (t0 - 0.03 <= ts <= t1 + 0.03):
                continue
            sm.append(clk)
            smax.append(cmax)
            for n, v in zip(names, r[6:10]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm), "samples_total": n_all}


class L2Flush:
    """Evicts the 129 MB L2 between steps: writes one 256 MiB buffer, then
    reads another, so that the step starts with L2 holding only clean lines
    of the second buffer (no write-back of dirty flush data is left for the
    step's own kernels to pay for)."""

    def __init__(self, dev):
        n = L2_FLUSH_BYTES // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.ones(n, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self, value: float):
        self.w.fill_(value)
        torch.sum(self.r, dim=(0,), out=self.sink)


def run_step(plan, evs=None, stream=None):
    """One layer-step through the prepared C-ABI calls, with an event before,
    between and after its kernels when ``evs`` is given."""
    if evs:
        evs[0].record(stream)
    plan.reshape_and_cache()
    if evs:
        evs[1].record(stream)
    plan.decode()
    if evs:
        evs[2].record(stream)
    plan.reduce()
    if evs:
        evs[3].record(stream)


def cpu_baseline(w: pin.Workload, budget_s: float = 12.0):
    """The CPU reference as it stands, timed on the host cores over whole
    passes of the workload (at least one, up to ~budget_s)."""
    import oracle
    qb, kc, vc = pin.bits(w.q), pin.bits(w.k_cache), pin.bits(w.v_cache)
    kn, vn = pin.bits(w.k_new), pin.bits(w.v_new)
    bytes_per = w.kv_bytes_logical() + w.qo_bytes()
    passes, t0 = 0, time.perf_counter()
    while True:
        kc2, vc2, _ = oracle.reshape_and_cache(kn, vn, w.slot_mapping, kc, vc, w.block_size)
        oracle.paged_decode(qb, kc2, vc2, w.block_tables, w.context_lens, w.scale, w.dtype)
        passes += 1
        el = time.perf_counter() - t0
        if el >= budget_s or el / passes * (passes + 1) > 2.5 * budget_s:
            break
    cores = oracle.max_threads()
    # one pass on a single thread beside it
    oracle.set_threads(1)
    try:
        t1 = time.perf_counter()
        kc2, vc2, _ = oracle.reshape_and_cache(kn, vn, w.slot_mapping, kc, vc, w.block_size)
        oracle.paged_decode(qb, kc2, vc2, w.block_tables, w.context_lens, w.scale, w.dtype)
        el1 = time.perf_counter() - t1
    finally:
        oracle.set_threads(cores)
    return {"value": passes * bytes_per / el / 1e9, "unit": "GB/s", "cores": cores,
            "kind": "oracle", "value_1thread": bytes_per / el1 / 1e9,
            "sample": f"{passes} full pass(es) of the {w.name} workload (reshape_and_cache + fp64 "
                      f"paged decode of all {w.num_seqs} sequences), {el:.1f} s; one more pass "
                      f"on 1 thread, {el1:.1f} s"}


def make_workload(args, rank: int) -> pin.Workload:
    """The named workload, with --params (JSON) overriding its parameters."""
    if not args.params:
        return pin.build_workload(args.config, seed=rank_seed(args.config, rank))
    seed, params = pin.CONFIGS[args.config]
    params = dict(params, **json.loads(args.params))
    w = pin.build_workload(args.config, seed=seed + 1000 * rank, params=params)
    w.name = args.config
    return w


def bench_reference(args):
    """CPU reference on the host cores; each step one full pass of the workload
    (or of its first sequences when a pass would take longer than ~3 s)."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    w = pin.build_workload(args.config)
    qb, kc, vc = pin.bits(w.q), pin.bits(w.k_cache), pin.bits(w.v_cache)
    kn, vn = pin.bits(w.k_new), pin.bits(w.v_new)
    # size the per-step sample: whole sequences, about 3 s of work at most
    t0 = time.perf_counter()
    oracle.paged_decode(qb[:1], kc, vc, w.block_tables[:1], w.context_lens[:1], w.scale, w.dtype)
    per_tok = (time.perf_counter() - t0) / max(1, int(w.context_lens[0]))
    n = w.num_seqs
    while n > 1 and per_tok * int(w.context_lens[:n].sum()) / max(1, oracle.max_threads()) > 3.0:
        n = max(1, n // 2)
    sl = slice(0, n)

    def step():
        kc2, vc2, _ = oracle.reshape_and_cache(kn[sl], vn[sl], w.slot_mapping[sl], kc, vc,
                                               w.block_size)
        oracle.paged_decode(qb[sl], kc2, vc2, w.block_tables[sl], w.context_lens[sl], w.scale,
                            w.dtype)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    e = 2
    bytes_step = int(w.context_lens[sl].astype(np.int64).sum()) * w.num_kv_heads * \
        w.head_dim * e * 2 + 2 * n * w.num_q_heads * w.head_dim * e
    value = bytes_step * args.steps / el / 1e9
    sample = (f"first {n} of {w.num_seqs} sequences of the {w.name} workload per step "
              f"(reshape_and_cache + fp64 paged decode)")
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": f"{w.name}: {pin.DESCRIPTIONS[w.name]}",
                       "l2": "n/a (host)", "mode": "cpu oracle"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s",
                             "cores": oracle.max_threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def decode_setup(w: pin.Workload, dev, mode: str, partition: int, kv_dtype: str, fp8_seed: int):
    """Device inputs and the marshalled layer-step (lib.StepPlan) of a
    workload; with kv_dtype "fp8" the pools are replaced by E4M3 codes."""
    max_len = int(w.context_lens.max())
    kc, vc, scales = w.k_cache, w.v_cache, {}
    if kv_dtype == "fp8":
        if mode not in ("fused", "balanced"):
            raise SystemExit("--kv-dtype fp8 runs the fused steps")
        if w.k_cache.is_cuda:
            gen = torch.Generator(device=dev)
            gen.manual_seed(fp8_seed)
            kc = pin.fp8_codes_device(gen, tuple(w.k_cache.shape), FP8_K_SCALE, dev)
            vc = pin.fp8_codes_device(gen, tuple(w.v_cache.shape), FP8_V_SCALE, dev)
        else:
            rng = np.random.default_rng(fp8_seed)
            kc = pin.fp8_codes(rng, tuple(w.k_cache.shape), FP8_K_SCALE)
            vc = pin.fp8_codes(rng, tuple(w.v_cache.shape), FP8_V_SCALE)
        scales = dict(k_scale=FP8_K_SCALE, v_scale=FP8_V_SCALE)
    d = {k: v.to(dev) for k, v in dict(
        q=w.q, k_new=w.k_new, v_new=w.v_new, k_cache=kc, v_cache=vc,
        block_tables=torch.from_numpy(w.block_tables),
        context_lens=torch.from_numpy(w.context_lens),
        slot_mapping=torch.from_numpy(w.slot_mapping)).items()}
    plan = lib.StepPlan(d["q"], d["k_new"], d["v_new"], d["slot_mapping"], d["k_cache"],
                        d["v_cache"], d["block_tables"], d["context_lens"], w.scale, max_len,
                        mode=mode, partition_size=partition, **scales)
    nb = step_bytes(w, mode, partition, 1 if kv_dtype == "fp8" else 2)
    return d, plan, nb


def time_steps(plan, flush, dev, stream, steps: int, warmup: int, gpu_index: int, world: int):
    """Warm-up, then the timed region.  Phase 1 (the K timed steps): events
    only at step boundaries, so consecutive kernels of a step overlap their
    launch latency (programmatic dependent launch).  Phase 2 (kernel
    attribution, min(K, 1000) more steps): events between the kernels as
    well, which serialises them, to time each kernel for the roofline.
    Returns per-step and per-kernel milliseconds and the clocks seen."""
    for _ in range(warmup):
        flush(1.0)
        run_step(plan)
    torch.cuda.synchronize(dev)
    assert lib.read_device_errors(dev) == 0
    n_attr = min(steps, 1000)
    step_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n_attr)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(gpu_index) as clk:
        time.sleep(0.4)
        t_epoch0 = time.time()
        t_wall = time.perf_counter()
        # Hold the GPU briefly so the host queues the steps ahead of it: the
        # events then see only GPU time, not Python launch overhead.
        torch.cuda._sleep(int(2e7))
        for i in range(steps):
            flush(float(i))
            step_ev[i][0].record(stream)
            run_step(plan)
            step_ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
        torch.cuda._sleep(int(2e7))
        for i in range(n_attr):
            flush(float(i))
            run_step(plan, evs[i], stream)
        torch.cuda.synchronize(dev)
        t_epoch1 = time.time()
        time.sleep(0.1)
    if world > 1:
        dist.barrier()
    step_ms = [e[0].elapsed_time(e[1]) for e in step_ev]
    return {"step_ms": step_ms,
            "k1_ms": [e[0].elapsed_time(e[1]) for e in evs],
            "k2_ms": [e[1].elapsed_time(e[2]) for e in evs],
            "k3_ms": [e[2].elapsed_time(e[3]) for e in evs],
            "serial_ms": sum(e[0].elapsed_time(e[3]) for e in evs) / n_attr,
            "n_attr": n_attr, "t_wall": t_wall, "clocks": clk.summary(t_epoch0, t_epoch1)}


DOMINANT = {"split": "paged_decode_split", "single": "paged_decode",
            "fused": "paged_decode_step", "balanced": "balanced_step"}
LAUNCHES_PER_STEP = {"split": 3, "single": 2, "fused": 1, "balanced": 2}


def decode_summary(w: pin.Workload, mode: str, partition: int, kv_dtype: str, nb: dict,
                   tm: dict, dev, world: int, hbm: float, peak_src: str, traffic_key: str):
    """Step time statistics, per-kernel times and the dominant kernel's
    roofline of one timed decode workload."""
    ms = max_over_ranks(sum(tm["step_ms"]) / len(tm["step_ms"]), dev)
    ms_median = max_over_ranks(float(np.median(tm["step_ms"])), dev)
    ms_p99 = max_over_ranks(float(np.percentile(tm["step_ms"], 99)), dev)
    dom = DOMINANT[mode]
    dom_ms = sum(tm["k2_ms"]) / len(tm["k2_ms"])
    dom_bytes = nb["kernels"][dom]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    kern = {dom: round(1e3 * dom_ms, 2)}
    if mode not in ("fused", "balanced"):
        kern["reshape_and_cache"] = round(1e3 * sum(tm["k1_ms"]) / len(tm["k1_ms"]), 2)
    if mode == "split":
        kern["lse_reduce"] = round(1e3 * sum(tm["k3_ms"]) / len(tm["k3_ms"]), 2)
    kern["note"] = (f"event-bracketed, serialised, over {tm['n_attr']} more steps; the same "
                    f"step serialised takes {1e3 * tm['serial_ms']:.2f} us")
    value = whole_job_gbs(nb["layer_step"], world, ms)
    return {
        "value": round(value, 3), "unit": "GB/s", "ms_per_step": round(ms, 5),
        "us_per_layer_step": round(ms * 1e3, 2),
        "us_per_layer_step_median": round(ms_median * 1e3, 2),
        "us_per_layer_step_p99": round(ms_p99 * 1e3, 2),
        "hbm_frac_of_measured" if peak_src == "measured" else "hbm_frac_of_fallback":
            round(value / world / hbm, 4),
        "mode": mode, "partition_tokens": partition if mode != "single" else None,
        "kv_dtype": w.dtype if kv_dtype != "fp8" else "e4m3",
        "kv_bytes": nb["kv"],
        "kv_bytes_unique": int(w.kv_bytes_unique() * (1 if kv_dtype != "fp8" else 0.5)),
        "bytes_per_step": nb["layer_step"],
        "kernels_us": kern,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 2),
                     "peak": hbm, "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "traffic": profiled_traffic(
                         traffic_key, dom,
                         partition if dom in ("paged_decode_step", "paged_decode_split") else None)},
        "clocks": tm["clocks"],
        "gpu_launches": LAUNCHES_PER_STEP[mode] * len(tm["step_ms"]),
    }


# Further workloads timed in the same run (N = 1) and reported under
# "configs": name -> (workload, mode, partition tokens (0: chosen from the
# batch shape), cache type).
SUB_CONFIGS = {
    "llama8b_split512": ("llama8b", "split", 512, "auto"),
    "llama8b_fp8": ("llama8b", "fused", 0, "fp8"),
    "prefix": ("prefix", "fused", 0, "auto"),
    "prefix_balanced": ("prefix", "balanced", 0, "auto"),
    "llama70b": ("llama70b", "fused", 0, "auto"),
    "long16": ("long16", "fused", 0, "auto"),
    "long16_split512": ("long16", "split", 512, "auto"),
    "long32": ("long32", "fused", 0, "auto"),
    "long32_split512": ("long32", "split", 512, "auto"),
    "prefill8b": ("prefill8b", "prefill", 0, "auto"),
}


def bench_sub_configs(names, args, dev, stream, flush, hbm, peak_src):
    """Each named workload built with its pools drawn on the device, timed
    like the headline (same steps, warm-up and L2 flush), then freed."""
    out = {}
    for name in names:
        cfg, mode, partition, kv_dtype = SUB_CONFIGS[name]
        t0 = time.perf_counter()
        if mode == "prefill":
            res = time_prefill(cfg, dev, args.steps, args.warmup, 0, flush, stream)
            res.pop("metric", None)
            out[name] = res
        else:
            w = pin.build_workload(cfg, seed=rank_seed(cfg, 0), pool_device=dev)
            max_len = int(w.context_lens.max())
            p = partition or lib.choose_partition(w.num_seqs, w.num_kv_heads, max_len,
                                                  w.block_size, dev, w.context_lens)
            d, plan, nb = decode_setup(w, dev, mode, p, kv_dtype, rank_seed(cfg, 0) + 7)
            tm = time_steps(plan, flush, dev, stream, args.steps, args.warmup, dev.index or 0, 1)
            res = decode_summary(w, mode, p, kv_dtype, nb, tm, dev, 1, hbm, peak_src,
                                 cfg + ("_fp8" if kv_dtype == "fp8" else ""))
            res["workload"] = f"{cfg}: {pin.DESCRIPTIONS[cfg]}"
            res["device_errors"] = lib.read_device_errors(dev)
            out[name] = res
            del d, plan, w
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        out[name]["build_and_time_s"] = round(time.perf_counter() - t0, 2)
    return out


def bench_ours(args):
    rank, world, local_rank = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pa_build.build()
    lib.load()

    w = make_workload(args, rank)
    max_len = int(w.context_lens.max())
    mode = args.mode if args.mode != "auto" else "fused"
    partition = args.partition or lib.choose_partition(w.num_seqs, w.num_kv_heads, max_len,
                                                       w.block_size, dev, w.context_lens)
    d, plan, nb = decode_setup(w, dev, mode, partition, args.kv_dtype,
                               rank_seed(args.config, rank) + 7)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    tm = time_steps(plan, flush, dev, stream, args.steps, args.warmup, local_rank, world)
    errs = lib.read_device_errors(dev)

    # End to end through the public API, with the step's inputs in pinned host
    # memory and its output read back there every step, inside the events
    # (the L2 flush before each step is outside them; the host synchronises
    # after every step).  Headline form: the fused step reads q, the new K/V,
    # slots, tables and lengths straight from the pinned host buffers and
    # stores its output into pinned host memory (unified addressing over the
    # host link; no copy launch).  Also timed: the staged form, one packed
    # upload kernel, the step on device buffers, one read-back kernel.
    e2e = None
    if not args.no_e2e:
        names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
        src = {k: (torch.from_numpy(getattr(w, k)) if isinstance(getattr(w, k), np.ndarray)
                   else getattr(w, k)) for k in names}
        stage = lib.InputStaging({k: (tuple(t.shape), t.dtype) for k, t in src.items()}, dev)
        for k, t in src.items():
            stage.h[k].copy_(t)
        scales = dict(k_scale=FP8_K_SCALE, v_scale=FP8_V_SCALE) if args.kv_dtype == "fp8" else {}
        h2d = stage.nbytes
        n_e2e = min(args.steps, 200)

        def e2e_time(plan):
            e_ms = []
            for it in range(args.warmup + n_e2e):
                flush(0.5)
                ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                ea.record(stream)
                plan.replay()
                eb.record(stream)
                stream.synchronize()
                if it >= args.warmup:
                    e_ms.append(ea.elapsed_time(eb))
            return max_over_ranks(sum(e_ms) / len(e_ms), dev)

        forms = {}
        if mode == "fused":
            out_h = torch.empty(tuple(src["q"].shape), dtype=src["q"].dtype).pin_memory()
            plan_zc = lib.StepPlan(stage.h["q"], stage.h["k_new"], stage.h["v_new"],
                                   stage.h["slot_mapping"], d["k_cache"], d["v_cache"],
                                   stage.h["block_tables"], stage.h["context_lens"], w.scale,
                                   max_len, out=out_h, mode=mode, partition_size=partition,
                                   **scales)
            plan_zc.capture_graph()
            forms["zero_copy"] = (e2e_time(plan_zc), out_h.numel() * out_h.element_size(),
                                  "none: the fused step reads its inputs from the pinned host "
                                  "buffers and stores its output into pinned host memory",
                                  "one CUDA graph per step (the layer-step)")
            del plan_zc
        plan_e2e = lib.StepPlan(stage.d["q"], stage.d["k_new"], stage.d["v_new"],
                                stage.d["slot_mapping"], d["k_cache"], d["v_cache"],
                                stage.d["block_tables"], stage.d["context_lens"], w.scale,
                                max_len, mode=mode, partition_size=partition, **scales)
        out_s = torch.empty(plan_e2e.out.shape, dtype=plan_e2e.out.dtype).pin_memory()
        plan_e2e.capture_graph(before=stage.upload,
                               after=lambda: lib.copy_async(out_s, plan_e2e.out))
        forms["staged"] = (e2e_time(plan_e2e), out_s.numel() * out_s.element_size(),
                           "1 host-to-device (inputs packed), 1 device-to-host (out), each a "
                           "short kernel on pinned host memory (pa_copy_async)",
                           "one CUDA graph per step (upload, layer-step, read-back)")
        del plan_e2e, stage
        head = "zero_copy" if "zero_copy" in forms else "staged"
        e2e_ms, d2h, copies, launch = forms[head]
        e2e = {"value": round(whole_job_gbs(nb["layer_step"], world, e2e_ms), 3),
               "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_ms, 5), "steps": n_e2e, "form": head,
               "copies_per_step": copies, "launch": launch}
        for name, (ms, _, copies, launch) in forms.items():
            if name != head:
                e2e[name] = {"value": round(whole_job_gbs(nb["layer_step"], world, ms), 3),
                             "ms_per_step": round(ms, 5), "copies_per_step": copies,
                             "launch": launch}

    hbm, peak_src = peaks()
    summ = decode_summary(w, mode, partition, args.kv_dtype, nb, tm, dev, world, hbm, peak_src,
                          args.config + ("_fp8" if args.kv_dtype == "fp8" else ""))
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)
    configs = None
    if world == 1 and args.configs != "none":
        names = list(SUB_CONFIGS) if args.configs == "all" else \
            [n for n in args.configs.split(",") if n]
        del d, plan
        torch.cuda.empty_cache()
        configs = bench_sub_configs(names, args, dev, stream, flush, hbm, peak_src)
    frac_key = "hbm_frac_of_measured" if peak_src == "measured" else "hbm_frac_of_fallback"
    line = {
        "metric": METRIC, "value": summ["value"], "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": summ["ms_per_step"],
        "us_per_layer_step": summ["us_per_layer_step"],
        "us_per_layer_step_median": summ["us_per_layer_step_median"],
        "us_per_layer_step_p99": summ["us_per_layer_step_p99"],
        frac_key: summ[frac_key],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype if args.kv_dtype != "fp8" else f"{w.dtype} (q, out), e4m3 (K/V cache)",
        "data": "synthetic (seeded N(0,1) q/K/V, seeded block placement)",
        "config": {"workload": f"{w.name}: {pin.DESCRIPTIONS[w.name]}"
                               + (f" with {args.params}" if args.params else ""), "mode": mode,
                   "partition_tokens": summ["partition_tokens"],
                   "l2": "flushed before every step (256 MiB write, then 256 MiB read of another "
                         "buffer; outside the step's events)",
                   "kv_bytes": summ["kv_bytes"], "kv_bytes_unique": summ["kv_bytes_unique"],
                   "bytes_per_step": summ["bytes_per_step"], "seqs_per_gpu": w.num_seqs},
        "kernels_us": summ["kernels_us"],
        "roofline": summ["roofline"],
        "clocks": summ["clocks"],
        "gpu_launches": summ["gpu_launches"],
        "device_errors": errs,
        "wall_s_timed": round(tm["t_wall"], 4),
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    if configs is not None:
        line["configs"] = configs
        line["configs_note"] = (
            "further workloads timed in the same run, each with its pools drawn on the device "
            "by a seeded generator; same steps, warm-up and L2 flush as the headline; not in "
            "value, gpu_launches or wall_s_timed")
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def bench_copy(args):
    """Whole-block copies (pa_copy_blocks): copy-on-write inside the device
    pool and swap-out to pinned host memory, over the workload's pool."""
    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pa_build.build()
    lib.load()
    w = make_workload(args, rank)
    rng = np.random.default_rng(5)
    nb = w.num_blocks
    n_pairs = min(4096, nb // 2)
    perm = rng.permutation(nb)
    cow = torch.from_numpy(np.stack([perm[:n_pairs], perm[n_pairs:2 * n_pairs]], 1)).to(dev)
    kc, vc = w.k_cache.to(dev), w.v_cache.to(dev)
    hk = torch.empty((n_pairs,) + tuple(kc.shape[1:]), dtype=kc.dtype).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    swap = torch.from_numpy(np.stack([perm[:n_pairs], np.arange(n_pairs)], 1)).to(dev)
    block_bytes = kc[0].numel() * kc.element_size() * 2          # K and V
    res = {}
    for name, (src, dst, mp) in {"copy_on_write": ((kc, vc), (kc, vc), cow),
                                 "swap_out": ((kc, vc), (hk, hv), swap),
                                 "swap_in": ((hk, hv), (kc, vc),
                                             torch.flip(swap, [1]).contiguous())}.items():
        for _ in range(args.warmup):
            lib.copy_blocks(*src, *dst, mp)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            lib.copy_blocks(*src, *dst, mp)
        e1.record()
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / args.steps
        # bytes moved: read + write of every copied block
        res[name] = {"us": round(ms * 1e3, 2),
                     "GBps_rw": round(2 * n_pairs * block_bytes / (ms * 1e-3) / 1e9, 1)}
    hbm, peak_src = peaks()
    line = {"metric": "block copy GB/s (read + write), copy-on-write and swap",
            "value": res["copy_on_write"]["GBps_rw"], "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": f"{w.name} pool, {n_pairs} block pairs of "
                                   f"{block_bytes} bytes (K + V)"},
            "roofline": {"bound": "hbm", "achieved": res["copy_on_write"]["GBps_rw"],
                         "peak": hbm, "unit": "GB/s",
                         "frac": round(res["copy_on_write"]["GBps_rw"] / hbm, 4)},
            "ops": res}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def prefill_flops(w) -> int:
    """Algorithmic FLOPs of one chunked-prefill call: new token at position p
    of a head attends p + 1 keys, 2 D FLOPs for its score and 2 D for its
    share of P V each."""
    lens = w.context_lens.astype(np.int64)
    chunks = np.diff(w.query_start).astype(np.int64)
    attended = 0
    for L, C in zip(lens, chunks):
        first = L - C + 1                       # keys seen by the first new token
        attended += C * first + C * (C - 1) // 2
    return int(4 * w.head_dim * w.num_q_heads * attended)


def time_prefill(name: str, dev, steps: int, warmup: int, rank: int, flush, stream,
                 world: int = 1):
    """Chunked-prefill attention (pa_prefill) over the paged cache, every new
    token of every sequence attending causally through its block table:
    timed with CUDA events around each call, L2 flushed before each call."""
    w = pin.build_prefill_workload(name, seed=pin.PREFILL_CONFIGS[name][0] + 1000 * rank)
    d = {k: v.to(dev) if isinstance(v, torch.Tensor) else torch.from_numpy(v).to(dev)
         for k, v in dict(q=w.q, kn=w.k_new, vn=w.v_new, kc=w.k_cache, vc=w.v_cache,
                          bt=w.block_tables, cl=w.context_lens, qs=w.query_start,
                          sm=w.slot_mapping).items()}
    lib.reshape_and_cache(d["kn"], d["vn"], d["sm"], d["kc"], d["vc"])
    max_q = int(np.diff(w.query_start).max())
    out = torch.empty_like(d["q"])
    shp = lib.make_shape(w.num_seqs, d["q"].shape[1], d["kc"], d["bt"].shape[1])
    ws_bytes = lib.prefill_workspace_size(shp, max_q)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    launches_per_call = 2 if ws_bytes else 1          # the ordering plan, then attention

    def call():
        lib.prefill(d["q"], d["kc"], d["vc"], d["bt"], d["cl"], d["qs"], w.scale, max_q, out,
                    workspace=ws)

    for _ in range(warmup):
        flush(1.0)
        call()
    torch.cuda.synchronize(dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    import torch.distributed as dist
    sync_ranks = dist.is_available() and dist.is_initialized()
    with ClockSampler(dev.index or 0) as clocks:
        time.sleep(0.2)
        if sync_ranks:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t_start = time.time()
        for i in range(steps):
            flush(float(i))
            evs[i][0].record(stream)
            call()
            evs[i][1].record(stream)
        torch.cuda.synchronize(dev)
        t_end = time.time()
        if sync_ranks:
            dist.barrier()
        time.sleep(0.2)
    clk = clocks.summary(t_start, t_end)
    times = [a.elapsed_time(b) for a, b in evs]
    ms = max_over_ranks(sum(times) / steps, dev)
    flops = prefill_flops(w)
    tflops = flops * world / (ms * 1e-3) / 1e12
    with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
        peak = float(json.load(f)["bf16_tflops"])
    kv_tokens = int(w.context_lens.sum())
    kv_bytes = kv_tokens * w.num_kv_heads * w.head_dim * 2 * 2
    return {"metric": "chunked-prefill attention TFLOP/s over the paged cache",
            "value": round(tflops, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 5),
            "us_per_call_median": round(1e3 * float(np.median(times)), 2),
            "us_per_call_p99": round(1e3 * float(np.percentile(times, 99)), 2),
            "dtype": w.dtype,
            "workload": f"{w.name}: {pin.PREFILL_DESCRIPTIONS[w.name]}",
            "new_tokens": int(w.query_start[-1]), "kv_tokens": kv_tokens,
            "kv_bytes": kv_bytes, "flops_per_call": flops,
            "roofline": {"bound": "tensor", "kernel": "paged_prefill",
                         "achieved": round(tflops / world, 2),
                         "peak": peak, "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops, "
                                                      "burst; tcgen05 kernel, kernel='auto')",
                         "unit": "TFLOP/s", "frac": round(tflops / world / peak, 4),
                         "traffic": profiled_traffic(name, "paged_prefill")},
            "clocks": clk, "gpu_launches": steps * launches_per_call,
            "device_errors": lib.read_device_errors(dev)}


def bench_prefill(args):
    """The chunked-prefill bench line (--op prefill)."""
    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pa_build.build()
    lib.load()
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    r = time_prefill(args.prefill_config, dev, args.steps, args.warmup, rank, flush, stream,
                     world)
    line = {"metric": r["metric"], "value": r["value"], "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": r["dtype"], "data": "synthetic (seeded N(0,1) q/K/V, seeded block placement)",
            "config": {"workload": r["workload"], "new_tokens": r["new_tokens"],
                       "kv_tokens": r["kv_tokens"], "kv_bytes": r["kv_bytes"],
                       "flops_per_call": r["flops_per_call"],
                       "l2": "flushed before every call (outside its events)"},
            "roofline": r["roofline"], "clocks": r["clocks"],
            "gpu_launches": r["gpu_launches"], "device_errors": r["device_errors"]}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--op", choices=["step", "copy", "prefill"], default="step",
                    help="what to time: the decode layer-step, whole-block copies, or "
                         "chunked-prefill attention")
    ap.add_argument("--prefill-config", default="prefill8b", choices=sorted(pin.PREFILL_CONFIGS))
    ap.add_argument("--config", default="llama8b", choices=sorted(pin.CONFIGS))
    ap.add_argument("--mode", default="auto", choices=["auto", "single", "split", "fused",
                                                       "balanced"])
    ap.add_argument("--partition", type=int, default=0,
                    help="tokens per partition (0: chosen from the batch shape)")
    ap.add_argument("--params", default="", help="JSON overrides of the workload parameters")
    ap.add_argument("--kv-dtype", default="auto", choices=["auto", "fp8"],
                    help="cache element type: the workload's fp16/bf16, or E4M3 codes")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--configs", default="all",
                    help="further workloads timed after the headline at N = 1 and reported "
                         "under \"configs\": all, none, or a comma list of " +
                         ", ".join(SUB_CONFIGS))
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)        # at least 3 untimed warm-up steps
    if args.impl == "reference":
        return bench_reference(args)
    if args.op == "copy":
        return bench_copy(args)
    if args.op == "prefill":
        return bench_prefill(args)
    return bench_ours(args)


if __name__ == "__main__":
    sys.exit(main())
