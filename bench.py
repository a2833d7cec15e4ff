"""Benchmark of the look-ahead sparse decode layer-step (OasisKV) on GB300.

Workload (default): one Qwen3-8B-shaped layer, 128 requests x 16384 tokens
(1024 blocks of 16), 32 query / 8 KV heads, head dim 128, K = 128 resident
blocks per (request, KV head), fetch cap 0.05 (6 admissions per head per
step); 5 % planted hot blocks per head, queries aligned with the hot
direction, draft query 0.95-correlated with the next step's query.  The full
KV store (8 GiB bf16) sits in pinned host memory; HBM holds the resident pool
(1 GiB + spares), the min/max summaries (512 MiB) and the tables.

One step = one layer-step of the whole hot path through the C ABI
(oasis_step): look-ahead attention on the main stream; summary scan + top-K,
capped eviction and the host->HBM gather on the side stream.

Output: one JSON line (rank 0).  `--impl reference` times the CPU oracle on
the same workload instead (bounded samples of (request, KV head) pairs).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_kv_block_gb300 import workload  # noqa: E402

METRIC = "look-ahead decode layer-steps/s at 16K ctx×128 req; % of HBM & host-link roofline"
UNIT = "layer-steps/s"
UNIT_BYTES = 8192          # keys + values of one 16-token block of one KV head (bf16)
SUMM_BYTES = 512           # min + max rows of one block of one KV head (bf16)


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return ws, rank, local


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), power=float(f[3]),
                                 hw=f[5], hwt=f[6], swt=f[7], swp=f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        reasons = set()
        for r in rows:
            if r["hw"].lower().startswith("active"):
                reasons.add("hw_slowdown")
            if r["hwt"].lower().startswith("active"):
                reasons.add("hw_thermal_slowdown")
            if r["swt"].lower().startswith("active"):
                reasons.add("sw_thermal_slowdown")
            if r["swp"].lower().startswith("active"):
                reasons.add("sw_power_cap")
        loaded = [r for r in rows if r["power"] > 200.0] or rows
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "samples_under_load": len(loaded)}


def build_layer(shape, seed, dev, side_groups=0, schedule=3, num_drafts=1):
    """Allocate and fill one layer (untimed setup); returns (engine, q, qd, lens, host)."""
    from sparse_kv_block_gb300.oasis import Oasis, make_config
    lens = workload.ctx_lens(shape)
    host = torch.empty((shape.R, shape.Hkv, shape.NBmax, 2, 16, 128), dtype=torch.bfloat16,
                       pin_memory=True)
    gen = dev if dev.type == "cuda" else "cpu"
    workload.host_kv(shape, seed, 0, lens, device=gen, out=host)
    cfg = make_config(shape.R, shape.NBmax, shape.Hq, shape.Hkv, shape.K, shape.fetch_ratio,
                      device=dev.index or 0, side_groups=side_groups, schedule=schedule,
                      num_drafts=num_drafts)
    eng = Oasis(cfg, host_kv=[host])
    eng.set_context(lens)
    eng.oasis_build_summaries(0, 0)
    return eng, lens, host


class _DeviceView:
    """__cuda_array_interface__ of a pinned host tensor at its device address."""

    def __init__(self, t: torch.Tensor, dev_ptr: int):
        self.__cuda_array_interface__ = {"shape": (t.numel(),), "typestr": "<i2",
                                         "data": (dev_ptr, False), "version": 2,
                                         "strides": None}


def pinned_device_alias(t: torch.Tensor, dev) -> torch.Tensor:
    """A CUDA tensor over a pinned host bf16 tensor's memory (its device
    mapping), so torch kernels read and write it over the host link."""
    from sparse_kv_block_gb300.oasis import lib
    import ctypes
    fn = lib().cudaHostGetDevicePointer
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p, ctypes.c_uint]
    p = ctypes.c_void_p()
    if fn(ctypes.byref(p), ctypes.c_void_p(t.data_ptr()), 0) != 0 or not p.value:
        raise RuntimeError("store is not mapped page-locked memory")
    with torch.cuda.device(dev):
        flat = torch.as_tensor(_DeviceView(t, p.value), device=dev)
    return flat.view(torch.bfloat16).view(t.shape)


def pretouch_host(host: torch.Tensor, dev) -> None:
    """Read the whole pinned host store once through its device mapping (a
    sequential GPU read, untimed), as a store in long use would have been:
    the gather's random 8 KiB reads run several times slower while the
    store's pages are still cold on the device side (measured: a first timed
    pass of 1192 against 2416 layer-steps/s in the next pass of one process;
    under a profiler that replays each launch cold, 12x slower)."""
    alias = pinned_device_alias(host, dev)
    flat = alias.view(-1)
    step = 1 << 28
    acc = torch.zeros((), dtype=torch.float32, device=dev)
    for i in range(0, flat.numel(), step):
        acc += flat[i:i + step].float().sum()
    torch.cuda.synchronize(dev)


def warm_start(eng, shape, q0, dev):
    """Resident set = the summary-ranked top-K of the first query (warm cache)."""
    topk = torch.empty((shape.R, shape.Hkv, shape.K), dtype=torch.int32, device=dev)
    eng.oasis_score_topk(0, 0, q0, topk)
    torch.cuda.synchronize(dev)
    eng.res_ids[0][0].copy_(topk)
    eng.oasis_load_resident(0, 0)
    eng.oasis_sync()


def oracle_rate(shape, host, lens, q, qd, budget_s: float, threads: int = 1):
    """Time the CPU oracle on whole (request, all KV heads) samples, on
    `threads` host threads at once (each steps its own requests; the oracle's
    C functions release the interpreter lock).

    Returns (layer-steps/s extrapolated to the whole batch = the sum of the
    threads' pair-step rates over the batch's pairs, pairs timed, busy
    seconds summed over threads, sample description)."""
    import concurrent.futures
    import oracle
    hb = workload.bf16_bits(host)
    res0 = workload.initial_resident(shape, 0, 0, lens)
    qb_all = workload.bf16_bits(q[0].cpu().contiguous())
    qdb_all = workload.bf16_bits(qd[0].cpu().contiguous())
    oracle.build()

    def worker(k):
        t_pairs, t_sec, r = 0, 0.0, k % shape.R
        while t_sec < budget_s:
            sub = np.ascontiguousarray(hb[r:r + 1])
            sl = np.ascontiguousarray(lens[r:r + 1])
            summ = oracle.summary_build(sub, sl)
            orc = oracle.LayerOracle(sub, summ, sl, res0[r:r + 1], shape.K, shape.C,
                                     [(0, h) for h in range(shape.Hkv)])
            qb = np.ascontiguousarray(qb_all[r:r + 1])
            qdb = np.ascontiguousarray(qdb_all[r:r + 1])
            t0 = time.perf_counter()
            orc.step(qb, qdb, 0)
            t_sec += time.perf_counter() - t0
            t_pairs += shape.Hkv
            r = (r + threads) % shape.R
        return t_pairs, t_sec

    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
        res = list(ex.map(worker, range(threads)))
    pairs_per_s = sum(p / s for p, s in res)
    t_pairs = sum(p for p, _ in res)
    t_sec = sum(s for _, s in res)
    rate = pairs_per_s / (shape.R * shape.Hkv)
    desc = (f"oracle_step (attention + summary score + top-K + capped eviction, fp64) on "
            f"{t_pairs} (request, KV head) pair-steps of the {shape.name} layer, "
            f"{budget_s:.0f} s on each of {threads} host thread(s) (rates summed), "
            f"extrapolated to {shape.R * shape.Hkv} pairs")
    return rate, t_pairs, t_sec, desc


def run_reference(args, ws, rank):
    """The reference arm: the CPU oracle as it stands (fp64, sequential per
    (request, KV head) pair) on this machine's host cores, on the same workload,
    metric and config as the CUDA arm.  Every step is a whole layer-step:
    all of the layer's pairs, split over one host thread per core (the
    oracle's C functions release the interpreter lock), timed from the first
    pair's start to the last pair's end.  Nothing is extrapolated."""
    if rank != 0:
        return
    import concurrent.futures
    import oracle
    shape = get_shape(args)
    cuda = torch.cuda.is_available()
    lens = workload.ctx_lens(shape)
    host = torch.empty((shape.R, shape.Hkv, shape.NBmax, 2, 16, 128), dtype=torch.bfloat16,
                       pin_memory=cuda)
    gen = torch.device("cuda", 0) if cuda else "cpu"
    workload.host_kv(shape, args.seed, 0, lens, device=gen, out=host)
    nq = min(args.queries, 8)
    q, qd = workload.queries(shape, args.seed, 0, nq, device=gen)
    qb = [np.ascontiguousarray(workload.bf16_bits(q[i].cpu().contiguous())) for i in range(nq)]
    qdb = [np.ascontiguousarray(workload.bf16_bits(qd[i].cpu().contiguous())) for i in range(nq)]
    hb = workload.bf16_bits(host)
    summ = oracle.summary_build(hb, lens)
    res0 = workload.initial_resident(shape, args.seed, 0, lens)
    cores = os.cpu_count() or 1
    pairs = [(r, h) for r in range(shape.R) for h in range(shape.Hkv)]
    parts = [pairs[k::cores] for k in range(cores)]
    orcs = [oracle.LayerOracle(hb, summ, lens, res0, shape.K, shape.C, p) for p in parts if p]
    state = {"t": 0}

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(orcs)) as ex:
        def one_step():
            t = state["t"]
            t0 = time.perf_counter()
            list(ex.map(lambda o: o.step(qb[t % nq], qdb[t % nq], t), orcs))
            state["t"] += 1
            return time.perf_counter() - t0

        for _ in range(args.warmup):
            one_step()
        secs = [one_step() for _ in range(args.steps)]
    total = sum(secs)
    value = args.steps / total
    sample = (f"whole layer-steps: oracle_step (attention + summary score + top-K + capped "
              f"eviction, fp64) on all {len(pairs)} (request, KV head) pairs of the "
              f"{shape.name} layer per step, split over {len(orcs)} host threads; "
              f"{args.steps} steps timed in {total:.1f} s")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * total / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(shape, ws), "tokens_per_s": round(value * shape.R, 3),
            "step_ms_spread": spread([1000.0 * x for x in secs]),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": len(orcs), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


L2_BYTES = 129 * 10 ** 6   # GB300 L2


def l2_note(shape) -> str:
    """Whether one layer-step's resident units + summaries exceed L2 (the
    timing rule's alternative to flushing it between steps)."""
    nbytes = shape.R * shape.Hkv * (shape.K * UNIT_BYTES + shape.NBmax * SUMM_BYTES)
    rel = "larger" if nbytes > L2_BYTES else "smaller"
    size = f"{nbytes / 2 ** 30:.2f} GiB" if nbytes >= 2 ** 28 else f"{nbytes / 2 ** 20:.1f} MiB"
    return f"inputs {rel} than L2: {size} of pool + summaries read per layer-step"


def config_dict(shape, ws) -> dict:
    """The `config` of both arms' lines: what was run, no results."""
    return {"workload": workload_desc(shape), "parallelism": f"replicas{ws}",
            "l2": l2_note(shape)}


def get_shape(args):
    import dataclasses
    shape = workload.SHAPES[args.workload]
    if args.requests:
        shape = dataclasses.replace(shape, R=args.requests, name=f"{shape.name}_r{args.requests}")
    return shape


def workload_desc(shape) -> str:
    return (f"{shape.name}: {shape.layers} layer(s) x {shape.R} requests x {shape.ctx} tokens, "
            f"{shape.Hq} q / {shape.Hkv} KV heads, d=128, B=16, K={shape.K}, "
            f"fetch cap {shape.fetch_ratio} (C={shape.C}), hot {shape.hot_frac:.0%} blocks")


def h2d_bandwidth(dev) -> float:
    """Pinned host -> device copy bandwidth (GB/s), 256 MiB, best of 5."""
    n = 256 << 20
    h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    h.fill_(1)
    d = torch.empty(n, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(dev)
    best = 1e9
    for _ in range(6):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            d.copy_(h, non_blocking=True)
            e1.record(s)
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1))
    return n / (best * 1e-3) / 1e9


# Nominal HBM3e bandwidth of one GB300, for a second fraction beside the
# measured copy peak.
HBM_SPEC_GBS = 7900.0

# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum, one ncu
# capture) by workload and reported kernel, with the SHA-256 (first 16 hex
# digits) of the kernel's source file when the counters were taken: a
# kernel whose source has changed since reports traffic null.  Captured on a
# reduced case and scaled by (request, KV head) pairs where marked.
PROFILED_TRAFFIC = {
    "qwen3_8b_16k": {
        "attention": (1083310592, "f53ce477022af819"),
        "summary_scan": (547601920, "41a81604dd3ab5ff"),
        "topk_select": (4326400, "41a81604dd3ab5ff"),
        "prefetch": (653312, "06148c34713b870d"),
    },
}


def source_digest(name: str) -> str:
    import hashlib
    path = os.path.join(ROOT, "sparse_kv_block_gb300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


KERNEL_SOURCES = {"attention": "attn.cu", "summary_scan": "score_topk.cu",
                  "topk_select": "score_topk.cu", "prefetch": "admit_gather.cu"}


def profiled_traffic(workload_name: str, kernel: str):
    entry = PROFILED_TRAFFIC.get(workload_name, {}).get(kernel)
    if entry is None:
        return None
    nbytes, digest = entry
    return nbytes if source_digest(KERNEL_SOURCES[kernel]) == digest else None


def traffic_fields(workload_name: str, kernel: str) -> dict:
    """`traffic` (DRAM bytes per launch from the recorded capture, or None)
    and where it comes from: never from this run."""
    t = profiled_traffic(workload_name, kernel)
    if t is None:
        src = "none: no ncu capture of this kernel's current source for this workload"
    else:
        src = ("ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, recorded "
               f"capture of {KERNEL_SOURCES[kernel]} sha256 "
               f"{PROFILED_TRAFFIC[workload_name][kernel][1]} (not measured in this run)")
    return {"traffic": t, "traffic_source": src}


def kernel_rooflines(shape, ms_sum, counts, off_sum, steps, link_bytes, h2d_gbs, peaks):
    """Per-kernel rooflines of one timed pass: summed CUDA-event durations of
    each kind's launches per step (several request groups per step for the
    side work), against the algorithmic bytes of one step.  Returns
    (per-kernel dict, name of the longest kernel)."""
    from sparse_kv_block_gb300.oasis import PROFILE_KINDS
    show = {"score_topk": "summary_scan"}
    names = [show.get(n, n) for n in PROFILE_KINDS]
    avg_ms = {n: (ms_sum[i] / steps if counts[i] else None) for i, n in enumerate(names)}
    avg_start = {n: (off_sum[i] / counts[i] if counts[i] else None) for i, n in enumerate(names)}
    launches = {n: counts[i] / steps for i, n in enumerate(names)}
    R, Hq, Hkv, K, NB = shape.R, shape.Hq, shape.Hkv, shape.K, shape.NBmax
    qo_bytes = 4 * R * Hq * 128 * 2
    attn_bytes = R * Hkv * K * UNIT_BYTES + qo_bytes
    # The scan reads every summary row and the draft queries and writes one
    # fp32 score per block.
    scan_bytes = R * Hkv * NB * SUMM_BYTES + R * Hq * 128 * 2 + R * Hkv * NB * 4
    hbm_src = ("measured hbm_gbs (MEASURED_PEAKS.json)" if peaks["source"] == "measured"
               else "fallback 6.8 TB/s")
    per_kernel = {}
    for n, b, bound, peak in [("attention", attn_bytes, "hbm", peaks["hbm_gbs"]),
                              ("summary_scan", scan_bytes, "hbm", peaks["hbm_gbs"]),
                              ("prefetch", link_bytes, "host-link", h2d_gbs)]:
        if avg_ms[n]:
            a = b / (avg_ms[n] * 1e-3) / 1e9
            k = {"bound": bound, "achieved": round(a, 1), "peak": round(peak, 1),
                 "unit": "GB/s", "frac": round(a / peak, 4),
                 "bytes_per_step": int(b), "ms_per_step": round(avg_ms[n], 5),
                 "launches_per_step": launches[n], "avg_start_ms": round(avg_start[n], 5),
                 "peak_source": (hbm_src if bound == "hbm" else
                                 "pinned cudaMemcpyAsync H2D, 256 MiB, measured in this run"),
                 **traffic_fields(shape.name, n)}
            if bound == "hbm":
                k["frac_of_spec"] = round(a / HBM_SPEC_GBS, 4)
                k["spec_gbs"] = HBM_SPEC_GBS
            per_kernel[n] = k
    if avg_ms["topk_select"]:
        per_kernel["topk_select"] = {
            "bound": "latency", "ms_per_step": round(avg_ms["topk_select"], 5),
            "launches_per_step": launches["topk_select"],
            "avg_start_ms": round(avg_start["topk_select"], 5),
            "note": "head-wise top-K of the scan's fp32 scores and the fused capped "
                    "eviction; overlaps the attention",
            **traffic_fields(shape.name, "topk_select")}
    timed = [n for n in ("attention", "summary_scan", "prefetch") if avg_ms[n]]
    dominant = max(timed, key=lambda n: avg_ms[n])
    return per_kernel, dominant


def whole_step_rates(per_kernel, link_bytes, steps_per_s, peaks, h2d_gbs) -> dict:
    """HBM and host-link rates of the whole step at `steps_per_s` (one GPU),
    and their fractions of the measured peaks."""
    hbm = per_kernel["attention"]["bytes_per_step"] + per_kernel["summary_scan"]["bytes_per_step"]
    hbm_gbs = hbm * steps_per_s / 1e9
    link_gbs = link_bytes * steps_per_s / 1e9
    return {"hbm_bytes_per_step": int(hbm), "hbm_gbs": round(hbm_gbs, 1),
            "hbm_frac": round(hbm_gbs / peaks["hbm_gbs"], 4),
            "link_bytes_per_step": int(link_bytes), "link_gbs": round(link_gbs, 1),
            "link_frac": round(link_gbs / h2d_gbs, 4)}


def spread(per_step_ms) -> dict:
    """min / median / max of per-step times (ms)."""
    v = sorted(per_step_ms)
    return {"min": round(v[0], 4), "median": round(v[len(v) // 2], 4), "max": round(v[-1], 4),
            "steps": len(v)}


def run_oasis(args, ws, rank, local):
    from sparse_kv_block_gb300.oasis import PROFILE_KINDS, lib
    lib()  # fail loudly if the CUDA library is missing
    if not torch.cuda.is_available():
        raise RuntimeError("the CUDA path needs a GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    # The clock sampler starts now, seconds before the timed region, so that
    # its start-up is over by then.
    clocks = ClockSampler(local)
    clocks.start()
    shape = get_shape(args)
    nq = args.queries
    eng, lens, host = build_layer(shape, args.seed + rank, dev, args.side_groups, args.schedule)
    q, qd = workload.queries(shape, args.seed + rank, 0, nq, device=dev)
    warm_start(eng, shape, q[0], dev)
    if not args.no_host_pretouch:
        pretouch_host(host, dev)
    odt = torch.bfloat16
    out = torch.empty((shape.R, shape.Hq, 128), dtype=odt, device=dev)
    outd = torch.empty_like(out)
    main = torch.cuda.Stream(dev)
    h2d_gbs = h2d_bandwidth(dev)

    step = 0

    def one_step():
        nonlocal step
        eng.oasis_step(0, step, q[step % nq], qd[step % nq], out, outd, main)
        step += 1

    # No idle gap between the warm-up steps and the timed region.
    with torch.cuda.stream(main):
        for _ in range(args.warmup):
            one_step()
    eng.oasis_sync()

    # ---------------- timed region: K layer-steps, inputs resident in HBM

    def timed_pass(profiled: bool):
        """K steps between CUDA events on the main stream (barrier + sync on
        both sides); with `profiled`, the library also brackets every kernel
        with CUDA events on its own stream."""
        eng.oasis_profile_enable(profiled)
        barrier(ws)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(main)
        for _ in range(args.steps):
            one_step()
        eng.oasis_join(0, main)
        e1.record(main)
        torch.cuda.synchronize(dev)
        barrier(ws)
        return e0.elapsed_time(e1)

    # Pass 1 gives `value`; pass 2 repeats it with per-kernel events (which
    # cost some time themselves) for the kernel rooflines.
    ms = timed_pass(False)
    ms_prof = timed_pass(True)
    ms_sum, counts, off_sum = eng.oasis_profile_read(len(PROFILE_KINDS))
    eng.oasis_profile_enable(False)
    clk = clocks.stop()
    eng.oasis_sync()
    ms_max = max_over_ranks(ms, ws)
    value = ws * args.steps / (ms_max * 1e-3)

    # ---------------- admitted traffic (a few extra steps, read back)
    n_adm = []
    for _ in range(8):
        lists = eng.step_lists(0, step)
        with torch.cuda.stream(main):
            one_step()
        eng.oasis_join(0, main)
        torch.cuda.synchronize(dev)
        n_adm.append(int(lists["n_admit"].sum().item()))
    adm_units = sum(n_adm) / len(n_adm)
    link_bytes = adm_units * UNIT_BYTES

    # ---------------- end to end: host buffers through oasis_step_host
    # Inputs: the step's queries in pinned host memory (a ring of 8 distinct
    # steps, filled before timing); each step copies its own inputs to the
    # device.  Outputs: two pinned sets, the host reading step i - 2's result
    # once that step has ended while steps i - 1 and i are in flight; every
    # copy is inside the timed region.
    def pinned():
        return torch.empty((shape.R, shape.Hq, 128), dtype=torch.bfloat16, pin_memory=True)
    n_in = min(nq, 8)
    qh = [pinned() for _ in range(n_in)]
    qdh = [pinned() for _ in range(n_in)]
    for j in range(n_in):
        qh[j].copy_(q[j].cpu())
        qdh[j].copy_(qd[j].cpu())
    oh, odh = [pinned(), pinned()], [pinned(), pinned()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    e2e_steps = args.steps

    def e2e_pass(async_outputs: bool) -> float:
        """Wall seconds for e2e_steps host-buffer steps.  async_outputs: the
        outputs come back on the library's output stream
        (oasis_step_host_async + oasis_wait_outputs); else on `main`
        (oasis_step_host + an event per step)."""
        nonlocal step
        checksum = 0.0
        barrier(ws)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        first = step
        for i in range(e2e_steps):
            b = i & 1
            if i >= 2:                              # step i - 2 finished: read its result
                if async_outputs:
                    if not eng.oasis_wait_outputs(0, step - 2, 60000.0):
                        raise RuntimeError("outputs not back within 60 s")
                else:
                    done[b].synchronize()
                checksum += float(oh[b][0, 0, 0])
            if async_outputs:
                eng.oasis_step_host_async(0, step, qh[i % n_in], qdh[i % n_in], oh[b], odh[b],
                                          main)
            else:
                eng.oasis_step_host(0, step, qh[i % n_in], qdh[i % n_in], oh[b], odh[b], main)
                done[b].record(main)
            step += 1
        for j in range(max(e2e_steps - 2, 0), e2e_steps):
            if async_outputs:
                eng.oasis_wait_outputs(0, first + j, 60000.0)
            else:
                done[j & 1].synchronize()
            checksum += float(oh[j & 1][0, 0, 0])
        eng.oasis_join(0, main)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - t0
        barrier(ws)
        return wall

    e2e_sync_s = max_over_ranks(e2e_pass(False), ws)
    e2e_s = max_over_ranks(e2e_pass(True), ws)
    e2e_value = ws * e2e_steps / e2e_s
    e2e_sync_value = ws * e2e_steps / e2e_sync_s
    eng.oasis_sync()

    # ---------------- roofline of the dominant kernel
    peaks = measured_peaks()
    per_kernel, dominant = kernel_rooflines(shape, ms_sum, counts, off_sum, args.steps,
                                            link_bytes, h2d_gbs, peaks)
    R, Hq = shape.R, shape.Hq
    # The dominant kernel is the longest per step; the attention (the largest
    # HBM reader) is also reported on its own below.
    dk = per_kernel.get(dominant, per_kernel["attention"])
    roofline = {"bound": dk["bound"], "kernel": dominant,
                "achieved": dk["achieved"], "peak": dk["peak"], "unit": "GB/s",
                "frac": dk["frac"], "traffic": dk.get("traffic"),
                "traffic_source": dk.get("traffic_source"), "peak_source": dk["peak_source"]}

    line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": config_dict(shape, ws), "tokens_per_s": round(value * shape.R, 1),
            "roofline": roofline, "roofline_hbm": per_kernel.get("attention"),
            "kernels": per_kernel,
            # one GPU's whole step against the two peaks it shares: every
            # HBM byte of its kernels (attention + scan) and every link byte,
            # at the per-GPU step rate
            "whole_step": whole_step_rates(per_kernel, link_bytes, value / ws, peaks, h2d_gbs),
            "host_link": {"h2d_memcpy_gbs": round(h2d_gbs, 1),
                          "admitted_units_per_step": adm_units,
                          "bytes_per_step": int(link_bytes)},
            "e2e": {"value": round(e2e_value, 2), "unit": UNIT,
                    "h2d_bytes_per_step": 2 * R * Hq * 128 * 2,
                    "d2h_bytes_per_step": 2 * R * Hq * 128 * 2,
                    "note": "oasis_step_host_async: each step copies its q/q_draft from "
                            "pinned host memory (a ring of 8 steps' inputs) and its "
                            "attention outputs back; the host reads every result once "
                            "oasis_wait_outputs says it is back, two steps in flight",
                    "stream_ordered_value": round(e2e_sync_value, 2),
                    "stream_ordered_note": "the same loop through oasis_step_host (outputs "
                                           "copied back on the step's stream)"},
            "gpu_launches": int(sum(counts)), "clocks": clk,
            "profiled_pass_ms_per_step": round(ms_prof / args.steps, 5)}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        # The oracle on every host core (its (request, KV head) pairs are
        # independent), and on one core for reference.
        ncores = os.cpu_count() or 1
        rate, pairs, sec, desc = oracle_rate(shape, host, lens, q.cpu(), qd.cpu(),
                                             budget_s=args.cpu_budget / 2, threads=ncores)
        rate1, _, _, desc1 = oracle_rate(shape, host, lens, q.cpu(), qd.cpu(),
                                         budget_s=args.cpu_budget / 2, threads=1)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": ncores, "kind": "oracle",
                                "sample": desc, "single_thread_value": rate1,
                                "single_thread_sample": desc1}
    if rank == 0:
        print(json.dumps(line), flush=True)
    eng.close()


def run_oasis_layers(args, ws, rank, local):
    """Multi-layer decode loop: every step runs oasis_step for each layer in
    order on one main stream; each layer's side work overlaps the next
    layers.  Host stores are shared by layers l and l + M when the host
    cannot pin one per layer (M = --host-stores); every layer keeps its own
    summaries, resident pool and tables, and its queries point at its
    store's hot blocks.  With hot-block drift (the 36-layer workload), the
    hot blocks move between steps, untimed: the pipeline is drained, the
    host stores rewritten, and each layer's summaries and resident copies of
    the moved blocks refreshed (oasis_refresh_blocks); each step is then
    timed on its own and the steps' times are summed."""
    from sparse_kv_block_gb300.oasis import PROFILE_KINDS, Oasis, lib, make_config
    lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    shape = get_shape(args)
    L, nq = shape.layers, min(args.queries, 16)
    M = max(1, min(L, args.host_stores))
    lens = workload.ctx_lens(shape)
    stores = []
    for m in range(M):
        h = torch.empty((shape.R, shape.Hkv, shape.NBmax, 2, 16, 128), dtype=torch.bfloat16,
                        pin_memory=True)
        workload.host_kv(shape, args.seed + rank, m, lens, device=dev, out=h)
        stores.append(h)
    cfg = make_config(shape.R, shape.NBmax, shape.Hq, shape.Hkv, shape.K, shape.fetch_ratio,
                      layers=L, device=local, side_groups=args.side_groups,
                      schedule=args.schedule)
    eng = Oasis(cfg, host_kv=[stores[l % M] for l in range(L)])
    eng.set_context(lens)
    if not args.no_host_pretouch:
        for h in stores:
            pretouch_host(h, dev)
    qs, qds = [], []
    for l in range(L):
        q, qd = workload.queries(shape, args.seed + rank, l, nq, device=dev,
                                 direction_layer=l % M)
        qs.append(q)
        qds.append(qd)
        eng.oasis_build_summaries(l, 0)
        topk = torch.empty((shape.R, shape.Hkv, shape.K), dtype=torch.int32, device=dev)
        eng.oasis_score_topk(l, 0, q[0], topk)
        torch.cuda.synchronize(dev)
        eng.res_ids[l][0].copy_(topk)
        eng.oasis_load_resident(l, 0)
    eng.oasis_sync()
    outs = [torch.empty((shape.R, shape.Hq, 128), dtype=torch.bfloat16, device=dev)
            for _ in range(2)]
    main = torch.cuda.Stream(dev)
    h2d_gbs = h2d_bandwidth(dev)
    step = 0

    grow = shape.grow_steps > 0
    if grow and args.steps + args.warmup > shape.grow_steps:
        raise SystemExit(f"{shape.name}: steps + warmup must be <= {shape.grow_steps}")
    if grow:   # a few distinct new tokens, cycled (drawn untimed)
        toks = [workload.new_tokens(shape, args.seed + rank, 0, i, device=dev) for i in range(4)]

    drift = shape.hot_move_prob > 0 and not args.no_hot_drift
    if drift:
        hots = [workload.hot_blocks(shape, args.seed + rank, m, lens) for m in range(M)]
        max_ids = 2 * max(len(x) for row in hots[0] for x in row)
        ids_h = torch.full((shape.R, shape.Hkv, max_ids), -1, dtype=torch.int32)
        nid_h = torch.zeros((shape.R, shape.Hkv), dtype=torch.int32)
        ids_d = [torch.empty((shape.R, shape.Hkv, max_ids), dtype=torch.int32, device=dev)
                 for _ in range(M)]
        nid_d = [torch.empty((shape.R, shape.Hkv), dtype=torch.int32, device=dev)
                 for _ in range(M)]
    moved = [0]

    if drift:
        # The moved blocks are rewritten by GPU kernels through the stores'
        # device mappings: CPU stores would leave the lines dirty in the host
        # caches, and the next steps' gathers of those blocks (they are the
        # new hot blocks, soon admitted) then run at about half speed
        # (measured: 2082 against 3127 layer-steps/s without rewriting).
        views = [pinned_device_alias(st, dev) for st in stores]

    def drift_between_steps():
        """Untimed: drain, move hot blocks in every host store, refresh."""
        for l in range(L):
            eng.oasis_join(l, main)
        main.synchronize()
        for m in range(M):
            mv = workload.move_hot_blocks(shape, args.seed + rank, m, step, hots[m], lens)
            with torch.cuda.stream(main):
                workload.apply_hot_moves(shape, args.seed + rank, m, views[m], mv, lens)
            moved[0] += len(mv)
            ids_h.fill_(-1)
            nid_h.zero_()
            for (r, h, old, new) in mv:
                n = int(nid_h[r, h])
                ids_h[r, h, n] = old
                ids_h[r, h, n + 1] = new
                nid_h[r, h] = n + 2
            ids_d[m].copy_(ids_h)
            nid_d[m].copy_(nid_h)
        for l in range(L):
            eng.oasis_refresh_blocks(l, step, ids_d[l % M], nid_d[l % M], main)
        main.synchronize()

    def one_step():
        nonlocal step
        for l in range(L):
            eng.oasis_step(l, step, qs[l][step % nq], qds[l][step % nq], outs[0], outs[1], main)
        if grow:
            # the decoded token of every request joins each layer's host
            # store, tail summary and resident copy; then the context grows
            k_new, v_new = toks[step % len(toks)]
            for l in range(L):
                eng.oasis_append_token(l, step, k_new, v_new, main)
            eng.oasis_advance_context(step, 1, main)
        step += 1

    # The clock sampler starts before the warm-up: no idle gap between the
    # warm-up steps and the timed region.
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    for _ in range(args.warmup):
        one_step()
        if drift:
            drift_between_steps()
    for l in range(L):
        eng.oasis_join(l, main)
    torch.cuda.synchronize(dev)
    eng.oasis_sync()
    moved[0] = 0
    eng.oasis_profile_enable(True)
    barrier(ws)
    torch.cuda.synchronize(dev)
    step_spread = None
    if drift:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for i in range(args.steps):
            ev[i][0].record(main)
            one_step()
            for l in range(L):
                eng.oasis_join(l, main)
            ev[i][1].record(main)
            drift_between_steps()
        torch.cuda.synchronize(dev)
        per_step = sorted(a.elapsed_time(b) for a, b in ev)
        ms = sum(per_step)
        step_spread = spread(per_step)
    else:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        e0.record(main)
        for i in range(args.steps):
            one_step()
            marks[i].record(main)   # after the step's last attention (steps overlap)
        for l in range(L):
            eng.oasis_join(l, main)
        e1.record(main)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1)
        gaps = [e0.elapsed_time(marks[0])] + [marks[i - 1].elapsed_time(marks[i])
                                               for i in range(1, args.steps)]
        step_spread = spread(gaps)
    barrier(ws)
    ms_sum, counts, off_sum = eng.oasis_profile_read(len(PROFILE_KINDS))
    eng.oasis_profile_enable(False)
    clk = clocks.stop()
    eng.oasis_sync()
    ms_max = max_over_ranks(ms, ws)
    value = ws * args.steps * L / (ms_max * 1e-3)
    adm = 0
    for l in range(L):
        adm += int(eng.step_lists(l, step - 1)["n_admit"].sum().item())
    link_bytes = adm / L * UNIT_BYTES
    peaks = measured_peaks()
    R, Hq, Hkv, K, NB = shape.R, shape.Hq, shape.Hkv, shape.K, shape.NBmax
    names = [{"score_topk": "summary_scan"}.get(n, n) for n in PROFILE_KINDS]
    per = {}
    for i, n in enumerate(names):
        if counts[i]:
            per[n] = {"ms_per_layer_step": round(ms_sum[i] / (args.steps * L), 5),
                      "launches_per_layer_step": counts[i] / (args.steps * L)}
    attn_bytes = R * Hkv * K * UNIT_BYTES + 4 * R * Hq * 128 * 2
    scan_bytes = R * Hkv * NB * SUMM_BYTES
    if counts[1]:
        sb = scan_bytes + R * Hq * 128 * 2 + R * Hkv * NB * 4
        s_gbs = sb / (ms_sum[1] / counts[1] * 1e-3) / 1e9
        per["summary_scan"].update({"achieved_gbs": round(s_gbs, 1),
                                    "frac": round(s_gbs / peaks["hbm_gbs"], 4)})
    a_ms = ms_sum[0] / counts[0]
    line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_desc(shape), "host_stores": M,
                       "note": f"layers l and l+{M} share one pinned host store"
                               + ("; one token appended per request per step (timed)"
                                  if grow else "")
                               + (f"; hot blocks moved between steps (untimed, "
                                  f"{moved[0] / args.steps:.0f} moves per step over "
                                  f"{M} stores), each step timed alone" if drift else ""),
                       "tokens_per_s": round(value * R / L, 1),
                       "l2": l2_note(shape)},
            "roofline": {"bound": "hbm", "kernel": "attention",
                         "achieved": round(attn_bytes / (a_ms * 1e-3) / 1e9, 1),
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(attn_bytes / (a_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                         **traffic_fields(shape.name, "attention")},
            "hbm_bytes_per_layer_step": attn_bytes + scan_bytes,
            "hbm_achieved_gbs_whole_step": round((attn_bytes + scan_bytes) * value / 1e9, 1),
            "host_link": {"h2d_memcpy_gbs": round(h2d_gbs, 1),
                          "bytes_per_layer_step": int(link_bytes),
                          "achieved_gbs_whole_step": round(link_bytes * value / 1e9, 1)},
            "kernels": per, "gpu_launches": int(sum(counts)), "clocks": clk}
    if step_spread is not None:
        line["step_ms_spread"] = step_spread
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        # Every layer-step does the same work, so the oracle is timed on layer
        # 0's store and first step (a bounded sample), on every host core.
        ncores = os.cpu_count() or 1
        rate, pairs, sec, desc = oracle_rate(shape, stores[0], lens, qs[0].cpu(), qds[0].cpu(),
                                             budget_s=args.cpu_budget / 2, threads=ncores)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": ncores, "kind": "oracle",
                                "sample": desc + " (layer 0, first step)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    eng.close()


def run_kernels_alone(args, ws, rank, local):
    """Each stage of the step timed alone (CUDA events on its stream, after
    warm-up) on the single-layer workload, through the stage-level C ABI
    calls; reports achieved GB/s against the HBM / host-link peaks."""
    from sparse_kv_block_gb300.oasis import PROFILE_KINDS, lib
    lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    shape = get_shape(args)
    eng, lens, host = build_layer(shape, args.seed, dev)
    q, qd = workload.queries(shape, args.seed, 0, 4, device=dev)
    warm_start(eng, shape, q[0], dev)
    R, Hq, Hkv, K, C, NB = shape.R, shape.Hq, shape.Hkv, shape.K, shape.C, shape.NBmax
    out = torch.empty((R, Hq, 128), dtype=torch.bfloat16, device=dev)
    outd = torch.empty_like(out)
    topk = torch.empty((R, Hkv, K), dtype=torch.int32, device=dev)
    sc = torch.empty((R, Hkv, K), dtype=torch.float32, device=dev)
    aid = torch.empty((R, Hkv, max(C, 1)), dtype=torch.int32, device=dev)
    asl, evi = torch.empty_like(aid), torch.empty_like(aid)
    nad = torch.empty((R, Hkv), dtype=torch.int32, device=dev)
    st = torch.cuda.Stream(dev)
    n = max(5, min(args.steps, 50))

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(n):
            fn()
        e1.record(st)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / n

    res = {}
    res["attention_ms"] = timed(lambda: eng.oasis_lookahead_attn(0, 0, q[1], qd[1], out, outd, st))
    res["score_topk_ms"] = timed(lambda: eng.oasis_score_topk(0, 0, qd[1], topk, sc, st))
    # The same call with per-kernel events: the scan and the ranking apart.
    eng.oasis_profile_enable(True)
    for _ in range(n):
        eng.oasis_score_topk(0, 0, qd[1], topk, sc, st)
    kms, kcnt, _ = eng.oasis_profile_read(len(PROFILE_KINDS))
    eng.oasis_profile_enable(False)
    res["scan_ms"] = kms[1] / max(1, kcnt[1])
    res["select_ms"] = kms[6] / max(1, kcnt[6]) if kcnt[6] else None
    eng.oasis_score_topk(0, 0, qd[1], topk, sc, st)
    torch.cuda.synchronize(dev)
    res["admit_evict_ms"] = timed(lambda: eng.oasis_admit_evict(0, 0, topk, aid, asl, evi, nad, st))
    eng.oasis_admit_evict(0, 0, topk, aid, asl, evi, nad, st)
    torch.cuda.synchronize(dev)
    units = int(nad.sum())
    res["prefetch_ms"] = timed(lambda: eng.oasis_prefetch(0, 0, aid, asl, nad, st))
    # Dense anchor: the whole KV of the context in HBM, attention over all of it.
    kv_dense = host.to(dev)
    res["dense_ms"] = timed(lambda: eng.oasis_dense_attn(kv_dense, 0, q[1], qd[1], out, outd, st))
    del kv_dense
    eng.oasis_sync()
    peaks = measured_peaks()
    h2d = h2d_bandwidth(dev)
    dense_b = R * Hkv * NB * UNIT_BYTES + 4 * R * Hq * 128 * 2
    attn_b = R * Hkv * K * UNIT_BYTES + 4 * R * Hq * 128 * 2
    scan_b = R * Hkv * NB * SUMM_BYTES + R * Hq * 128 * 2
    scan_only_b = scan_b + R * Hkv * NB * 4
    gb = lambda b, ms: b / (ms * 1e-3) / 1e9
    line = {"mode": "kernels-alone", "workload": workload_desc(shape), "iters": n,
            "attention": {"ms": round(res["attention_ms"], 5), "bytes": attn_b,
                          "GBs": round(gb(attn_b, res["attention_ms"]), 1),
                          "frac_hbm": round(gb(attn_b, res["attention_ms"]) / peaks["hbm_gbs"], 4)},
            "score_topk": {"ms": round(res["score_topk_ms"], 5), "bytes": scan_b,
                           "GBs": round(gb(scan_b, res["score_topk_ms"]), 1),
                           "frac_hbm": round(gb(scan_b, res["score_topk_ms"]) / peaks["hbm_gbs"], 4),
                           "note": "oasis_score_topk as a whole (scan, then ranking)"},
            "summary_scan": {"ms": round(res["scan_ms"], 5), "bytes": scan_only_b,
                             "GBs": round(gb(scan_only_b, res["scan_ms"]), 1),
                             "frac_hbm": round(gb(scan_only_b, res["scan_ms"]) / peaks["hbm_gbs"], 4),
                             "frac_of_spec": round(gb(scan_only_b, res["scan_ms"]) / HBM_SPEC_GBS, 4)},
            "topk_select": {"ms": None if res["select_ms"] is None else round(res["select_ms"], 5)},
            "admit_evict": {"ms": round(res["admit_evict_ms"], 5)},
            "prefetch": {"ms": round(res["prefetch_ms"], 5), "units": units,
                         "GBs": round(gb(units * UNIT_BYTES, res["prefetch_ms"]), 1),
                         "frac_h2d_memcpy": round(gb(units * UNIT_BYTES, res["prefetch_ms"]) / h2d, 4)},
            "dense_attention": {"ms": round(res["dense_ms"], 5), "bytes": dense_b,
                                "GBs": round(gb(dense_b, res["dense_ms"]), 1),
                                "frac_hbm": round(gb(dense_b, res["dense_ms"]) / peaks["hbm_gbs"], 4),
                                "layer_steps_per_s": round(1e3 / res["dense_ms"], 1)},
            "hbm_peak_gbs": peaks["hbm_gbs"], "h2d_memcpy_gbs": round(h2d, 1)}
    if rank == 0:
        print(json.dumps(line), flush=True)
    eng.close()


def run_miss_stall(args, ws, rank, local):
    """The "stall" outcome of a look-ahead miss against the look-ahead step
    ("drop"), both through the C ABI on the same workload.

    Stall (oasis_step_stall): each step ranks every block with its own normal
    query, fetches every block of that top-K the look-ahead did not bring
    (uncapped, on the critical path), attends, then runs the look-ahead side
    work.  Drop (oasis_step): the attention reads what the look-ahead
    brought.  Reports each mode's rate, the kernels of the stall step, and
    the demand units per step (the top-K blocks the look-ahead missed)."""
    from sparse_kv_block_gb300.oasis import PROFILE_KINDS, lib
    lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    shape = get_shape(args)
    R, Hq, Hkv, K = shape.R, shape.Hq, shape.Hkv, shape.K
    nq = min(args.queries, 16)
    results = {}
    clocks = ClockSampler(local)
    clocks.start()
    for mode in ("stall", "lookahead"):
        eng, lens, host = build_layer(shape, args.seed, dev, args.side_groups, args.schedule)
        q, qd = workload.queries(shape, args.seed, 0, nq, device=dev)
        warm_start(eng, shape, q[0], dev)
        if not args.no_host_pretouch:
            pretouch_host(host, dev)
        out = torch.empty((R, Hq, 128), dtype=torch.bfloat16, device=dev)
        outd = torch.empty_like(out)
        st = torch.cuda.Stream(dev)
        fn = eng.oasis_step_stall if mode == "stall" else eng.oasis_step
        step = 0

        def one():
            nonlocal step
            t = step % nq
            fn(0, step, q[t], qd[t], out, outd, st)
            step += 1

        def timed(profiled):
            eng.oasis_profile_enable(profiled)
            eng.oasis_join(0, st)
            torch.cuda.synchronize(dev)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(st)
            for _ in range(args.steps):
                one()
            eng.oasis_join(0, st)
            e1.record(st)
            torch.cuda.synchronize(dev)
            return e0.elapsed_time(e1) / args.steps

        for _ in range(args.warmup):
            one()
        ms = timed(False)
        timed(True)
        ms_sum, counts, _ = eng.oasis_profile_read(len(PROFILE_KINDS))
        eng.oasis_profile_enable(False)
        res = {"ms_per_step": round(ms, 4), "layer_steps_per_s": round(1e3 / ms, 1),
               "kernel_ms_per_step": {PROFILE_KINDS[i]: round(ms_sum[i] / args.steps, 4)
                                      for i in range(len(PROFILE_KINDS)) if counts[i]}}
        if mode == "stall":
            demand = []
            for _ in range(8):
                with torch.cuda.stream(st):
                    one()
                eng.oasis_join(0, st)
                torch.cuda.synchronize(dev)
                demand.append(int(eng.stall_lists(0, step - 1)["n_admit"].sum().item()))
            res["demand_units_per_step"] = sum(demand) / len(demand)
            res["demand_share_of_topk"] = round(sum(demand) / len(demand) / (R * Hkv * K), 4)
        eng.oasis_sync()
        results[mode] = res
        eng.close()
        del eng, host
        torch.cuda.empty_cache()
    clk = clocks.stop()
    if rank == 0:
        print(json.dumps({"mode": "miss-stall vs look-ahead", "workload": workload_desc(shape),
                          "steps": args.steps, "warmup": args.warmup, "clocks": clk,
                          **results}), flush=True)


def run_drafts(args, ws, rank, local):
    """Several draft queries per step (an option of the three-stream
    pipeline): the look-ahead step with D = 1, 2, 3 drafts on the same
    workload, each draft attending over the one resident set and the drafts'
    summary bounds summed for the ranking.  Reports the step rate and the
    attention kernel alone (same resident bytes, 1 + D query kinds)."""
    from sparse_kv_block_gb300.oasis import PROFILE_KINDS, lib
    lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    shape = get_shape(args)
    R, Hq, Hkv, K = shape.R, shape.Hq, shape.Hkv, shape.K
    nq = min(args.queries, 16)
    peak = measured_peaks().get("hbm_gbs")
    results = {}
    # Two rounds over D, the second one reported: the first engine of a
    # process ran ~10 % slower than later ones, whatever its D.
    for D in (1, 2, 3, 1, 2, 3):
        eng, lens, host = build_layer(shape, args.seed, dev, args.side_groups, args.schedule,
                                      num_drafts=D)
        q, qd = workload.draft_queries(shape, args.seed, 0, nq, D, device=dev)
        warm_start(eng, shape, qd[0], dev)
        if not args.no_host_pretouch:
            pretouch_host(host, dev)
        out = torch.empty((R, Hq, 128), dtype=torch.bfloat16, device=dev)
        outd = torch.empty((D, R, Hq, 128), dtype=torch.bfloat16, device=dev)
        st = torch.cuda.Stream(dev)
        for i in range(args.warmup):
            eng.oasis_step(0, i, q[i % nq], qd[i % nq], out, outd, st)
        eng.oasis_join(0, st)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for i in range(args.warmup, args.warmup + args.steps):
            eng.oasis_step(0, i, q[i % nq], qd[i % nq], out, outd, st)
        eng.oasis_join(0, st)
        e1.record(st)
        torch.cuda.synchronize(dev)
        eng.oasis_sync()
        ms = e0.elapsed_time(e1) / args.steps
        last = args.warmup + args.steps - 1
        admitted = float(eng.step_lists(0, last)["n_admit"].float().mean())
        # a profiled pass (per-kernel durations and start offsets in the step)
        n_prof = min(args.steps, 200)
        eng.oasis_profile_enable(True)
        for i in range(last + 1, last + 1 + n_prof):
            eng.oasis_step(0, i, q[i % nq], qd[i % nq], out, outd, st)
        eng.oasis_join(0, st)
        torch.cuda.synchronize(dev)
        ms_sum, counts, off_sum = eng.oasis_profile_read(len(PROFILE_KINDS))
        eng.oasis_profile_enable(False)
        names = [{"score_topk": "summary_scan"}.get(n, n) for n in PROFILE_KINDS]
        kern = {n: {"ms": round(ms_sum[k] / max(counts[k], 1), 4),
                    "start_ms": round(off_sum[k] / max(counts[k], 1), 4)}
                for k, n in enumerate(names) if counts[k]}
        # attention alone on the resident set the loops left behind
        nxt = last + 1 + n_prof
        n_attn = 50
        for _ in range(3):
            eng.oasis_lookahead_attn(0, nxt, q[0], qd[0], out, outd, st)
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record(st)
        for _ in range(n_attn):
            eng.oasis_lookahead_attn(0, nxt, q[0], qd[0], out, outd, st)
        a1.record(st)
        torch.cuda.synchronize(dev)
        eng.oasis_sync()
        ams = a0.elapsed_time(a1) / n_attn
        # resident units + q and the D draft planes read + 1 + D outputs written
        nbytes = R * Hkv * K * 8192 + 2 * (1 + D) * R * Hq * 128 * 2
        gbs = nbytes / (ams * 1e-3) / 1e9
        results[f"drafts_{D}"] = {
            "ms_per_step": round(ms, 4), "layer_steps_per_s": round(1e3 / ms, 1),
            "admitted_per_head": round(admitted, 3), "profiled_kernels": kern,
            "attention_alone_us": round(ams * 1e3, 1), "attention_gbs": round(gbs, 1),
            "attention_frac_of_measured_hbm": round(gbs / peak, 4) if peak else None}
        eng.close()
        del eng, host
        torch.cuda.empty_cache()
    if rank == 0:
        print(json.dumps({"mode": "draft queries per step", "workload": workload_desc(shape),
                          "steps": args.steps, "l2": "attention reads 1 GiB of units per launch",
                          **results}), flush=True)


def run_remote(args, ws, rank, local):
    """Remote tier (emulated prefill-decode disaggregation with remote partial
    fetch) on the single-layer shape: the full cache stays in the remote
    store; the decode side holds a local host tier that a block enters the
    first time it is needed (warm start, then admissions), moved by host
    threads at an emulated network rate.  Every step uses a fresh query, so
    the admitted blocks are not replayed.  Reports layer-steps/s, remote
    traffic per step, and the decode-side host memory held at the end against
    the full cache, next to the same steps without a remote tier."""
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    shape = get_shape(args)
    R, Hq, Hkv, K = shape.R, shape.Hq, shape.Hkv, shape.K
    n = args.steps + args.warmup
    q, qd = workload.queries(shape, args.seed, 0, n, device=dev)
    lens = workload.ctx_lens(shape)
    nb = np.array([-(-int(x) // 16) for x in lens], dtype=np.int64)
    full_units = int(nb.sum()) * Hkv
    results = {}
    for mode in ["local"] + [f"remote_{g:g}GBps" for g in args.remote_gbps]:
        eng, lens, host = build_layer(shape, args.seed, dev, args.side_groups, args.schedule)
        rt = None
        if mode != "local":
            gbps = float(mode[len("remote_"):-len("GBps")])
            rt = eng.oasis_remote_attach(0, shape.NBmax, gbps, args.remote_threads)
        warm_start(eng, shape, q[0], dev)
        out = torch.empty((R, Hq, 128), dtype=torch.bfloat16, device=dev)
        outd = torch.empty_like(out)
        st = torch.cuda.Stream(dev)
        for t in range(args.warmup):
            eng.oasis_step(0, t, q[t], qd[t], out, outd, st)
        eng.oasis_join(0, st)
        torch.cuda.synchronize(dev)
        s0 = eng.oasis_remote_stats(0) if rt is not None else None
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for t in range(args.warmup, n):
            eng.oasis_step(0, t, q[t], qd[t], out, outd, st)
        eng.oasis_join(0, st)
        e1.record(st)
        torch.cuda.synchronize(dev)
        eng.oasis_sync()
        ms = e0.elapsed_time(e1) / args.steps
        r = {"ms_per_step": round(ms, 4), "layer_steps_per_s": round(1e3 / ms, 1)}
        if rt is not None:
            s1 = eng.oasis_remote_stats(0)
            du = s1["units"] - s0["units"]
            held = int(rt["local_count"].sum().item())
            r.update({
                "remote_units_per_step": round(du / args.steps, 1),
                "remote_GB_per_step": round(du * 8192 / args.steps / 1e9, 4),
                "transfer_ms_per_step": round((s1["seconds"] - s0["seconds"]) * 1e3 / args.steps, 4),
                "transfer_GBps": round(du * 8192 / max(s1["seconds"] - s0["seconds"], 1e-9) / 1e9, 1),
                "decode_host_units_held": held,
                "full_cache_units": full_units,
                "decode_host_fraction": round(held / full_units, 4),
                "admission_fraction": round(R * Hkv * K / full_units, 4),
                "bad_entries": s1["bad_entries"]})
        results[mode] = r
        eng.close()
        del eng, host
        torch.cuda.empty_cache()
    if rank == 0:
        print(json.dumps({"mode": "remote tier", "workload": workload_desc(shape),
                          "steps": args.steps, "warmup": args.warmup,
                          "remote_threads": args.remote_threads, **results}), flush=True)


def run_cap_sweep(args, ws, rank, local):
    """Fetch-cap sweep on the single-layer shape: for each cap, layer-steps/s,
    host-to-device bytes per step, and the top-K agreement between the draft
    query's selection at step t and the next step's true query: ranked by the
    summary score through oasis_score_topk, and (on the first 4 requests)
    against the exact blocks of the next query, scored by
    max over tokens of sum over the group's query heads of q . k."""
    import dataclasses
    from sparse_kv_block_gb300.oasis import Oasis, lib, make_config
    lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    base = get_shape(args)
    lens = workload.ctx_lens(base)
    host = torch.empty((base.R, base.Hkv, base.NBmax, 2, 16, 128), dtype=torch.bfloat16,
                       pin_memory=True)
    workload.host_kv(base, args.seed, 0, lens, device=dev, out=host)
    if not args.no_host_pretouch:
        pretouch_host(host, dev)
    nq = args.queries
    q, qd = workload.queries(base, args.seed, 0, nq + 1, device=dev)
    main = torch.cuda.Stream(dev)
    ns = min(4, base.R)
    keys_s = host[:ns, :, :, 0].to(dev).float()             # [ns][Hkv][NB][B][d]
    tok = torch.arange(base.NBmax * base.B, device=dev).view(base.NBmax, base.B)
    valid_s = tok[None] < torch.as_tensor(lens[:ns], device=dev).view(ns, 1, 1)

    def exact_topk(qn):
        """Exact next-step top-K ids of the sampled pairs, [ns][Hkv][K]."""
        qg = qn[:ns].float().view(ns, base.Hkv, base.G, base.d).sum(2)
        sc = torch.einsum("rhbtd,rhd->rhbt", keys_s, qg)
        sc = sc.masked_fill(~valid_s[:, None], float("-inf")).amax(-1)
        return sc.topk(min(base.K, base.NBmax), dim=-1).indices

    results = []
    clocks = ClockSampler(local)
    clocks.start()
    for cap in (0.01, 0.05, 0.25, 1.0):
        shape = dataclasses.replace(base, fetch_ratio=cap)
        cfg = make_config(shape.R, shape.NBmax, shape.Hq, shape.Hkv, shape.K, cap,
                          device=local, side_groups=args.side_groups, schedule=args.schedule)
        eng = Oasis(cfg, host_kv=[host])
        eng.set_context(lens)
        eng.oasis_build_summaries(0, 0)
        warm_start(eng, shape, q[0], dev)
        out = torch.empty((shape.R, shape.Hq, 128), dtype=torch.bfloat16, device=dev)
        outd = torch.empty_like(out)
        true_topk = torch.empty((shape.R, shape.Hkv, shape.K), dtype=torch.int32, device=dev)
        P, NB, K = shape.R * shape.Hkv, shape.NBmax, shape.K
        agree, agree_x, agree_s, adm = [], [], [], []
        step = 0
        for _ in range(args.warmup):
            eng.oasis_step(0, step, q[step % nq], qd[step % nq], out, outd, main)
            step += 1
        eng.oasis_join(0, main)
        torch.cuda.synchronize(dev)
        for _ in range(8):      # agreement and admissions, read back per step
            t = step % nq
            eng.oasis_step(0, step, q[t], qd[t], out, outd, main)
            eng.oasis_join(0, main)
            eng.oasis_score_topk(0, step, q[t + 1], true_topk, None, main)
            lists = eng.step_lists(0, step)
            torch.cuda.synchronize(dev)
            a = torch.zeros((P, NB + 1), device=dev)
            b = torch.zeros((P, NB + 1), device=dev)
            a.scatter_(1, lists["topk_ids"].view(P, K).long() + 1, 1.0)
            b.scatter_(1, true_topk.view(P, K).long() + 1, 1.0)
            agree.append(float(((a * b)[:, 1:].sum(1) / K).mean()))
            ex = exact_topk(q[t + 1])
            ax = torch.zeros((ns * shape.Hkv, NB + 1), device=dev)
            bx = torch.zeros((ns * shape.Hkv, NB + 1), device=dev)
            ax.scatter_(1, lists["topk_ids"][:ns].reshape(-1, K).long() + 1, 1.0)
            bx.scatter_(1, ex.reshape(-1, K) + 1, 1.0)
            agree_x.append(float(((ax * bx)[:, 1:].sum(1) / K).mean()))
            cx = torch.zeros((ns * shape.Hkv, NB + 1), device=dev)
            cx.scatter_(1, true_topk[:ns].reshape(-1, K).long() + 1, 1.0)
            agree_s.append(float(((cx * bx)[:, 1:].sum(1) / K).mean()))
            adm.append(int(lists["n_admit"].sum()))
            step += 1
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        e0.record(main)
        for i in range(args.steps):
            eng.oasis_step(0, step, q[step % nq], qd[step % nq], out, outd, main)
            marks[i].record(main)
            step += 1
        eng.oasis_join(0, main)
        e1.record(main)
        torch.cuda.synchronize(dev)
        eng.oasis_sync()
        ms = e0.elapsed_time(e1) / args.steps
        gaps = [e0.elapsed_time(marks[0])] + [marks[i - 1].elapsed_time(marks[i])
                                               for i in range(1, args.steps)]
        results.append({"fetch_ratio": cap, "C": shape.C,
                        "layer_steps_per_s": round(1e3 / ms, 1),
                        "ms_per_step": round(ms, 4),
                        "step_ms_spread": spread(gaps),
                        "h2d_GB_per_layer_step": round(sum(adm) / len(adm) * UNIT_BYTES / 1e9, 5),
                        "admitted_units_per_step": sum(adm) / len(adm),
                        "topk_agreement_draft_vs_next": round(sum(agree) / len(agree), 5),
                        "topk_agreement_draft_vs_next_exact":
                            round(sum(agree_x) / len(agree_x), 5),
                        "topk_agreement_summary_vs_exact_same_query":
                            round(sum(agree_s) / len(agree_s), 5)})
        eng.close()
        del eng
        torch.cuda.empty_cache()
    clk = clocks.stop()
    if rank == 0:
        print(json.dumps({"mode": "cap-sweep", "metric": METRIC, "unit": UNIT,
                          "cap_sweep": results, "workload": workload_desc(base),
                          "steps": args.steps, "warmup": args.warmup, "clocks": clk,
                          "data": "synthetic"}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="oasis", choices=["oasis", "reference"])
    ap.add_argument("--workload", default="qwen3_8b_16k",
                    choices=["qwen3_8b_16k", "tiny", "qwen3_8b_36l", "llama31_8b_32k"])
    ap.add_argument("--miss-stall", action="store_true",
                    help="fetch on the critical path (stall) against the look-ahead step")
    ap.add_argument("--kernels-alone", action="store_true",
                    help="time each stage alone on the single-layer workload")
    ap.add_argument("--cap-sweep", action="store_true",
                    help="fetch-cap sweep (0.01, 0.05, 0.25, 1.0) on the single-layer shape")
    ap.add_argument("--host-stores", type=int, default=12,
                    help="distinct pinned host stores of a multi-layer workload")
    ap.add_argument("--no-hot-drift", action="store_true",
                    help="36-layer workload: keep the hot blocks in place (one timed region)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--queries", type=int, default=64, help="distinct query steps, cycled")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-host-pretouch", action="store_true",
                    help="skip the one untimed read of every host store through its device "
                         "mapping before timing")
    ap.add_argument("--side-groups", type=int, default=0,
                    help="request groups of the side work (0 = library default)")
    ap.add_argument("--schedule", type=int, default=3,
                    help="0 scan first, 1 concurrent, 2 the pages' three background streams, "
                         "3 auto (scan first on device buffers, concurrent on host buffers), "
                         "4 early scan (the scan of step t beside the attention of step t-1)")
    ap.add_argument("--drafts", action="store_true",
                    help="step rate and attention time with 1, 2 and 3 draft queries per step")
    ap.add_argument("--remote", action="store_true",
                    help="remote tier (emulated disaggregated partial fetch) on the single-layer shape")
    ap.add_argument("--remote-gbps", type=float, nargs="+", default=[0.0, 50.0, 25.0],
                    help="emulated network rates for --remote (0 = unthrottled host copy)")
    ap.add_argument("--remote-threads", type=int, default=16)
    ap.add_argument("--requests", type=int, default=0,
                    help="override the request count (small cases for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    elif args.cap_sweep:
        run_cap_sweep(args, ws, rank, local)
    elif args.kernels_alone:
        run_kernels_alone(args, ws, rank, local)
    elif args.miss_stall:
        run_miss_stall(args, ws, rank, local)
    elif args.remote:
        run_remote(args, ws, rank, local)
    elif args.drafts:
        run_drafts(args, ws, rank, local)
    elif workload.SHAPES[args.workload].layers > 1:
        run_oasis_layers(args, ws, rank, local)
    else:
        run_oasis(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
