#!/usr/bin/env python3
"""Benchmark of the Kamera KV-reuse hot path on GB300.

One step = one kamera_reuse_batched call over the whole batch (every layer,
K and V): gather the canonical chunks, re-rotate the keys by delta, add the
rank-m patch, scatter into the paged pool.  Default workload (the largest
single-GPU one): long-video reorder + recall on a GQA 8B-shaped backbone
(32 layers, 8 KV heads x 128, base 5e5): 128 permuted chunks x 1296 tokens
with rank-64 orbit patches plus 32 recalled chunks with fresh rank-64
patches, page 64, shuffled block table -- 57.4 GB moved per call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints one JSON line.  ``value`` = reused tokens/s with inputs resident in
HBM (device time, CUDA events on the launching stream, max over ranks);
``e2e`` = the same metric with the step's inputs copied host->device from
pinned memory and the call's status read back inside the timed region.  The
headline inputs are far larger than L2, so no flush is needed between steps.
With one GPU the line also carries ``configs``: the device-timed figures of
the other four workloads (tiny MHA, GQA video, MLA, sliding window), each
timed in the same process (those smaller than 4x L2 with an L2 flush
between launches).  ``--impl reference`` times the fp64 CPU oracle on a
bounded sample.  ``--workload gqa_video_compressed`` times
kamera_reuse_compressed on the GQA video batch read from a compressed
canonical store (int8 K, 3-bit V).
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
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from synth import workloads as W  # noqa: E402

METRIC = "reused KV tokens/sec (rotate + rank-m patch), achieved HBM GB/s vs roofline"
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal bandwidth (the "~8 TB/s" figure); the roofline uses the measured copy
UNIT = "tokens/s"
# the device sources of each profiled kernel: a committed capture counts only while they are unchanged
KERNEL_SOURCES = ["position_invariant_kv_kamera_gb300/csrc/kamera_kernel.cuh",
                  "position_invariant_kv_kamera_gb300/csrc/ptx.cuh"]
FACTOR_SOURCES = ["position_invariant_kv_kamera_gb300/csrc/kamera_factor.cuh"]
ORBIT_SOURCES = ["position_invariant_kv_kamera_gb300/csrc/kamera_orbit.cuh"]
DESCRIPTIONS = {
    "gqa_video": "GQA Qwen2.5-VL-7B-shaped: 28 layers, 4 KV heads x 128, base 1e6, 16 chunks x 1024 tokens, "
                 "1% outlier channels x8, rank-32 patch per layer per K/V, delta in [-32768, 32768], "
                 "page 64, shuffled block table",
    "tiny_mha": "MHA 1 layer, 4 heads x 64, one 256-token chunk, rank 8, delta 1000, contiguous output",
    "mla_lite": "MLA DeepSeek-V2-Lite-shaped: 27 layers, c_KV 512 + k_rope 64, 8 chunks x 2048, rank 16, page 64",
    "sliding_window": "sliding-window survival, GQA 8B-shaped (32 layers, 8 KV heads x 128, base 5e5): 56 of 64 "
                      "resident 1024-token chunks re-rotated in place by -8192, no patch, page 64",
    "long_video": "long-video reorder + recall, GQA 8B-shaped: 128 permuted chunks x 1296 with rank-64 orbit "
                  "patches + 32 recalled chunks with fresh rank-64 patches, page 64",
    "gqa_video_compressed": "the gqa_video batch reused from a compressed canonical store (PolyKV scheme: int8 K "
                            "with one scale per (chunk, layer), 3-bit Walsh-Hadamard/Lloyd-Max V with one norm per "
                            "head row), decoded on gather; store encoded on the GPU before timing",
}
COMPRESSED = {"gqa_video_compressed": "gqa_video"}


def kernel_hash(sources: list[str] = KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for f in sources:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def profile_traffic(workload: str, kernel: str = "reuse_kernel", sources: list[str] = KERNEL_SOURCES) -> float | None:
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    h = re.search(r"kernel_sources_sha256_16:\s*([0-9a-f]+)", txt)
    if not h or h.group(1) != kernel_hash(sources):
        return None
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if m:
        return float(m.group(1))
    # a reduced capture of a workload too large to profile: scaled by the units processed
    m = re.search(r"dram_bytes_per_launch_reduced:\s*([0-9.eE+]+)", txt)
    f = re.search(r"traffic_scale_to_full:\s*([0-9.eE+]+)", txt)
    return float(m.group(1)) * float(f.group(1)) if m and f else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.out = out
        else:
            self.out = ""

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(value: float, torch, device) -> float:
    """Max over ranks (timing only; the data path has no collective)."""
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


SCALED = {  # reduced chunk counts, for profiler captures that must stay small
    "gqa_video": lambda n: W.gqa_video(n_chunks=n),
    "mla_lite": lambda n: W.mla_lite(n_chunks=n),
    "sliding_window": lambda n: W.sliding_window(n_resident=n + max(1, n // 8), n_evict=max(1, n // 8)),
    "long_video": lambda n: W.long_video(n_reorder=n - n // 4, n_recall=n // 4),
}


def rank_workload(name: str, rank: int, world: int, chunks: int = 0) -> W.Workload:
    """Weak scaling: every rank reuses its own batch of the same shape (its own
    seed); there is no data exchange between ranks.  chunks > 0 selects a
    reduced batch of that many chunks (profiling captures only)."""
    name = COMPRESSED.get(name, name)
    base = SCALED[name](chunks) if chunks and name in SCALED else W.WORKLOADS[name]()
    return base.replace(seed=base.seed + 1000 * rank) if world > 1 else base


def aggregate(tokens_per_rank: int, world: int, max_elapsed_s: float, steps: int) -> float:
    """Whole-job throughput: the units all ranks processed / the slowest rank's time."""
    return tokens_per_rank * world * steps / max_elapsed_s


# ---- CPU oracle timing (cpu_baseline and the reference arm) -----------------------------------

FULL_T = {"gqa_video": 1024, "mla_lite": 2048, "long_video": 1296, "sliding_window": 1024, "tiny_mha": 256}


def oracle_sample_workload(name: str, n_items: int, n_tokens: int | None = None) -> W.Workload:
    """A bounded sample of the workload with the same shapes (layers, row
    width, rank, page size): its first n_items chunks, optionally truncated
    to n_tokens tokens each."""
    if name == "gqa_video":
        return W.gqa_video(n_chunks=n_items, T=n_tokens or 1024)
    if name == "mla_lite":
        return W.mla_lite(n_chunks=n_items, T=n_tokens or 2048)
    if name == "long_video":
        return W.long_video(n_reorder=n_items, n_recall=0, T=n_tokens or 1296)
    if name == "sliding_window":
        T = 1024 if not n_tokens else max(64, n_tokens // 64 * 64)  # whole pages: the relocation is in place
        return W.sliding_window(n_resident=n_items + 1, n_evict=1, T=T)
    return W.WORKLOADS[name]()


def oracle_call(wl: W.Workload, compressed: bool = False):
    """The oracle over wl as a ready-to-run closure: every input (the bf16 or
    the compressed store, patches, pools) is generated here, once."""
    import oracle

    m = oracle.model(wl.family, wl.num_layers, wl.num_kv_heads, wl.head_dim, wl.rope_dim, wl.latent_dim,
                     wl.pairing, wl.patch_frame)
    th = oracle.theta(wl.rope_base, wl.rope_dim)
    kw = {}
    if wl.rank and wl.mode != "relocate_in_place":
        kw.update(patch=wl.host_patch(), patch_off=wl.patch_off, patch_len=np.array(wl.patch_lens, np.int32),
                  rank=wl.rank)
    pk_in = wl.host_pool(0)
    pv_in = wl.host_pool(1) if wl.n_ch == 2 else None
    if compressed:
        cs = oracle.compress_store(m, wl.host_store(), wl.store_off, np.array(wl.chunk_lens, np.int32))
        return lambda: oracle.reuse_compressed(m, th, cs, items=wl.items, block_table=wl.block_table,
                                               num_pages=wl.num_pages, page_size=wl.page_size, pool_k_in=pk_in,
                                               pool_v_in=pv_in, **kw)
    if wl.mode == "reuse":
        kw.update(store=wl.host_store(), store_off=wl.store_off, store_len=np.array(wl.chunk_lens, np.int32))
    mode = {"reuse": oracle.MODE_REUSE, "relocate_in_place": oracle.MODE_RELOCATE_IN_PLACE,
            "apply_patch": oracle.MODE_PATCH_IN_PLACE}[wl.mode]
    return lambda: oracle.reuse(m, th, mode, items=wl.items, block_table=wl.block_table, num_pages=wl.num_pages,
                                page_size=wl.page_size, pool_k_in=pk_in, pool_v_in=pv_in, **kw)


def timed(fn) -> float:
    t0 = time.perf_counter()
    fn()
    return time.perf_counter() - t0


def host_cores() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_parallel(call, workers: int) -> float:
    """Wall seconds of `workers` concurrent runs of the same oracle closure.
    The oracle is C behind ctypes, which releases the GIL for the call, so
    threads run on separate cores; inputs are shared read-only, every run
    writes its own output images."""
    from concurrent.futures import ThreadPoolExecutor

    with ThreadPoolExecutor(max_workers=workers) as ex:
        t0 = time.perf_counter()
        list(ex.map(lambda _: call(), range(workers)))
        return time.perf_counter() - t0


def oracle_sample(name: str, seconds: float) -> tuple[W.Workload, bool]:
    """One chunk of the workload, truncated so that one single-threaded oracle
    call over it takes about `seconds` (sized from a warm probe: a cold first
    call overstates the cost per token)."""
    comp = name in COMPRESSED
    base = COMPRESSED.get(name, name)
    full_T = FULL_T.get(base)
    if not full_T:  # patch formation / orbit mean have their own baselines
        raise ValueError(name)
    probe = oracle_sample_workload(base, 1, 64)
    call = oracle_call(probe, compressed=comp)
    call()
    per_tok = timed(call) / max(probe.tokens, 1)
    n_tok = max(64, min(full_T, int(seconds / max(per_tok, 1e-9))))
    return oracle_sample_workload(base, 1, n_tok if n_tok < full_T else None), comp


def cpu_baseline(name: str, budget_s: float = 10.0) -> dict:
    """The oracle as it stands (plain fp64 C, unchanged) on a bounded sample of
    the workload: one chunk, all layers and channels, truncated to about
    budget_s of single-core work; timed once on one core and once as one
    independent run per host core at the same time."""
    wl, comp = oracle_sample(name, budget_s)
    call = oracle_call(wl, compressed=comp)
    dt1 = timed(call)
    cores = host_cores()
    dtn = run_parallel(call, cores)
    what = "decoding the compressed store" if comp else "bf16 store"
    return {"value": cores * wl.tokens / dtn, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"one chunk truncated to {wl.tokens} tokens, all {wl.num_layers} layers and channels "
                      f"({what}); {cores} concurrent single-threaded runs of the fp64 C oracle, one per host core, "
                      f"in {dtn:.1f} s",
            "single_core": {"value": wl.tokens / dt1, "unit": UNIT, "cores": 1, "seconds": dt1}}


def run_reference(args) -> None:
    """The reference arm: the fp64 oracle (the method's plain definition; the
    pages publish no code to install) timed on the host cores.  Each step runs
    one single-threaded oracle call per host core concurrently, each over the
    same token sample of one chunk (all layers and channels), sized so that
    warm-up plus timed steps take about two minutes."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    name = args.workload
    if name not in FULL_T and COMPRESSED.get(name) not in FULL_T:
        print(json.dumps({"impl": "reference", "unavailable": f"no CPU reference for workload {name}"}), flush=True)
        return
    cores = host_cores()
    budget = 120.0 / (args.steps + args.warmup)
    wl, comp = oracle_sample(name, budget)
    call = oracle_call(wl, compressed=comp)  # inputs generated once, outside the timing
    for _ in range(args.warmup):
        run_parallel(call, cores)
    total = 0.0
    for _ in range(args.steps):
        total += run_parallel(call, cores)
    toks = cores * wl.tokens * args.steps
    value = toks / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": f"{name}: {DESCRIPTIONS.get(name, '')}",
                       "sample_per_step": f"{cores} concurrent oracle runs over {wl.tokens} tokens of one chunk, "
                                          f"all {wl.num_layers} layers"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"each step: {cores} x {wl.tokens} tokens x {wl.num_layers} layers"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---- GPU arm ----------------------------------------------------------------------------------

L2_BYTES = 129 * 10**6  # GB300 L2


def make_call(name: str, wl: W.Workload, torch, device, stream):
    """(device inputs, one_call(inputs, stream)) for a workload; the compressed
    variant encodes its store on the GPU first (write-once, off the timed path)."""
    import position_invariant_kv_kamera_gb300 as pk
    from tests import harness as H

    if name in COMPRESSED:
        t = H.device_inputs(wl, torch, device)
        cstore, ct = H.empty_compressed(wl, torch, device)
        pk.kamera_compress_chunks(H.model_for(wl), pk.chunk_store(t["store"], t["store_off"], t["store_len"]),
                                  cstore, t["err"].data_ptr(), stream.cuda_stream)
        torch.cuda.synchronize(device)
        for n in ("store", "store_off", "store_len"):
            del t[n]
        t.update(ct)

        def one_call(d, s):
            cs = pk.compressed_store(d["k_codes"], d["k_scale"], d["v_codes"], d["v_norm"], d["row_offset"],
                                     d["len"])
            return H.call_compressed(wl, d, cs, stream=s)
    else:
        t = H.device_inputs(wl, torch, device)

        def one_call(d, s):
            return H.call(wl, d, stream=s)
    torch.cuda.synchronize(device)
    return t, one_call


def device_time(one_call, t, torch, device, stream, steps: int, warmup: int, flush: bool) -> dict:
    """Device time of `steps` launches on the launching stream after `warmup`
    untimed ones.  Inputs larger than L2: the launches run back to back
    between two events.  Otherwise (flush=True) every launch is bracketed by
    its own events, with a write of twice the L2 size between launches so
    that each starts with a cold L2; the flush writes are outside the timed
    intervals."""
    for _ in range(warmup):
        one_call(t, stream)
    torch.cuda.synchronize(device)
    if int(t["err"].item()) != 0:
        raise RuntimeError(f"device error flag {int(t['err'].item())}")
    if not flush:
        b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b.record(stream)
        for _ in range(steps):
            one_call(t, stream)
        e.record(stream)
        torch.cuda.synchronize(device)
        total = b.elapsed_time(e) / 1e3
    else:
        scrub = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=device)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        with torch.cuda.stream(stream):
            for b, e in ev:
                scrub.fill_(1.0)
                b.record(stream)
                one_call(t, stream)
                e.record(stream)
        torch.cuda.synchronize(device)
        total = sum(b.elapsed_time(e) for b, e in ev) / 1e3
        del scrub
    if int(t["err"].item()) != 0:
        raise RuntimeError(f"device error flag {int(t['err'].item())}")
    return {"elapsed": total, "per_launch": total / steps, "steps": steps}


CONFIG_ORDER = ["tiny_mha", "gqa_video", "mla_lite", "sliding_window"]


def time_configs(names, torch, device, stream, steps: int, warmup: int, peak_gbs: float) -> dict:
    """Device-timed figures of other workloads in this process (one at a time,
    freeing each before the next)."""
    out = {}
    for name in names:
        wl = W.WORKLOADS[name]()
        t, one_call = make_call(name, wl, torch, device, stream)
        nbytes = wl.algorithmic_bytes()
        flush = nbytes < 4 * L2_BYTES
        n = max(steps, 100) if flush else steps
        r = device_time(one_call, t, torch, device, stream, n, warmup, flush)
        gbs = nbytes / r["per_launch"] / 1e9
        out[name] = {"description": DESCRIPTIONS[name], "ms_per_call": 1e3 * r["per_launch"],
                     "tokens_per_s": wl.tokens / r["per_launch"], "algorithmic_bytes": nbytes, "gbs": gbs,
                     "frac_of_measured_peak": gbs / peak_gbs, "frac_of_nominal": gbs / NOMINAL_HBM_GBS,
                     "launches": n, "l2": "flushed before every launch" if flush else "inputs larger than L2",
                     "traffic": profile_traffic(name)}
        del t
        torch.cuda.empty_cache()
    return out


def run_gpu(args) -> None:
    import torch

    import position_invariant_kv_kamera_gb300 as pk

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pk.load()

    wl = rank_workload(args.workload, rank, world, args.chunks)
    comp = args.workload in COMPRESSED
    stream = torch.cuda.current_stream(device)
    t, one_call = make_call(args.workload, wl, torch, device, stream)
    alg_bytes = wl.compressed_bytes() if comp else wl.algorithmic_bytes()
    flush = alg_bytes < 4 * L2_BYTES

    for _ in range(args.warmup):
        one_call(t, stream)
    torch.cuda.synchronize(device)
    if int(t["err"].item()) != 0:
        raise RuntimeError(f"device error flag {int(t['err'].item())}")

    # timed region: K launches on the launching stream, bracketed by a barrier and a synchronize
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    with ClockSampler(local) as clocks:
        time.sleep(0.25)  # let the sampler start before the timed region
        r = device_time(one_call, t, torch, device, stream, args.steps, 0, flush)
    if world > 1:
        torch.distributed.barrier()
    elapsed = r["elapsed"]
    max_elapsed = reduce_max(elapsed, torch, device)
    value = aggregate(wl.tokens, world, max_elapsed, args.steps)

    # end to end: the step's inputs from pinned host memory, the status read back
    e2e = run_e2e(wl, t, torch, device, stream, min(args.steps, args.e2e_steps), one_call)
    e2e_value = reduce_max_time_value(e2e, wl.tokens, world, torch, device)
    del t
    torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    peaks = measured_peaks()
    configs = None
    if world == 1 and args.configs and not args.chunks:
        names = [n for n in CONFIG_ORDER if n != args.workload]
        configs = time_configs(names, torch, device, stream, args.steps, args.warmup, peaks["hbm_gbs"])
    avg_launch_s = r["per_launch"]
    achieved = alg_bytes / avg_launch_s / 1e9
    traffic = profile_traffic(args.workload)
    cpu = cpu_baseline(args.workload) if world == 1 or rank == 0 else None
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * max_elapsed / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8/3-bit codes in, fp32 math, bf16 out" if comp else "bf16",
        "data": "synthetic",
        "config": {"workload": f"{args.workload}: {DESCRIPTIONS.get(args.workload, '')}"
                               + (f" [reduced to {args.chunks} chunks]" if args.chunks else ""),
                   "tokens_per_step": wl.tokens, "algorithmic_bytes_per_step": alg_bytes,
                   "patch_flops_per_step": wl.patch_flops(),
                   "l2": "L2 flushed before every launch" if flush else "inputs larger than L2 (no flush needed)",
                   "parallelism": f"replicas x{world} (independent batches, no collective)"},
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "peak_source": peaks["source"] + " (burst copy)",
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "kernel": "kamera::reuse_kernel", "launch_ms_mean": 1e3 * avg_launch_s},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": e2e["h2d"],
                "d2h_bytes_per_step": e2e["d2h"], "steps": e2e["steps"]},
        "gpu_launches": args.steps,
        "clocks": clocks.summary(),
    }
    if configs is not None:
        line["configs"] = configs
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_e2e(wl, t, torch, device, stream, steps: int, one_call) -> dict:
    """Host-buffer variant through the same public call: every step uploads
    its inputs (canonical chunks, patches, items, block table) from pinned
    host memory, runs the call, and reads back the call's status word (the
    device error flag).  The rebuilt pool stays in HBM, where attention reads
    it -- the analogue of a training step reading back its loss.  Two device
    buffer sets and separate upload / compute / download streams let step
    i+1's upload overlap step i."""
    names = [n for n in ("store", "store_off", "store_len", "k_codes", "k_scale", "v_codes", "v_norm", "row_offset",
                         "len", "patch", "patch_off", "patch_len", "items", "block_table", "section_delta") if n in t]
    # pinned host copies, allocated pinned (no pageable intermediate: the long-video inputs are 30 GB)
    host_in = {n: torch.empty(t[n].shape, dtype=t[n].dtype, pin_memory=True).copy_(t[n]) for n in names}
    host_err = [torch.empty(1, dtype=torch.int32, pin_memory=True) for _ in range(2)]
    sets = [t, {**{n: torch.empty_like(t[n]) for n in names}, "pool_k": t["pool_k"], "pool_v": t.get("pool_v"),
                "err": torch.zeros_like(t["err"])}]
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = 4
    s_up, s_down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    comp_done = [torch.cuda.Event() for _ in range(2)]
    down_done = [torch.cuda.Event() for _ in range(2)]
    for e in comp_done + down_done:
        e.record(stream)

    def step(i):
        b = i & 1
        d = sets[b]
        with torch.cuda.stream(s_up):
            s_up.wait_event(comp_done[b])   # the call of step i-2 no longer reads these inputs
            for n in names:
                d[n].copy_(host_in[n], non_blocking=True)
        up = torch.cuda.Event()
        up.record(s_up)
        stream.wait_event(up)
        stream.wait_event(down_done[b])     # step i-2's status has been read back
        one_call(d, stream)
        comp_done[b].record(stream)
        with torch.cuda.stream(s_down):
            s_down.wait_event(comp_done[b])
            host_err[b].copy_(d["err"], non_blocking=True)
        down_done[b].record(s_down)

    step(0)
    step(1)
    torch.cuda.synchronize(device)
    begin, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    begin.record(s_up)
    stream.wait_event(begin)
    s_down.wait_event(begin)
    for i in range(steps):
        step(i)
    end_c = torch.cuda.Event()
    end_c.record(stream)
    s_down.wait_event(end_c)
    end.record(s_down)
    torch.cuda.synchronize(device)
    if any(int(x.item()) for x in host_err):
        raise RuntimeError("device error flag set in the end-to-end leg")
    return {"elapsed": begin.elapsed_time(end) / 1e3, "steps": steps, "h2d": h2d, "d2h": d2h}


def reduce_max_time_value(e2e: dict, tokens: int, world: int, torch, device) -> float:
    mx = reduce_max(e2e["elapsed"], torch, device)
    return aggregate(tokens, world, mx, e2e["steps"])


# ---- patch formation (rank-m factors of a deficit) -----------------------------------------------

FACTOR_SHAPE = dict(n_slabs=16 * 28 * 2, T=1024, D=512, rank=32, oversample=16, power_iters=2, true_rank=40)


def factor_flops(T: int, D: int, k: int, m: int, q: int) -> int:
    """Algorithmic flops of one slab: the GEMMs (Delta Omega, 2q subspace
    products, Q^T Delta, B B^T, the two output products) and one QR of each
    of the 2q+1 panels (2 k^2 n for an n x k panel; a reorthogonalisation
    pass is overhead and not counted)."""
    gemm = 2 * T * D * k * (2 + 2 * q) + 2 * D * k * k + 2 * (T + D) * k * m
    orth = 2 * k * k * (T + q * (T + D))
    return gemm + orth


def factor_bytes(n: int, T: int, D: int, m: int, q: int) -> int:
    """HBM bytes the method moves: every product with Delta reads the fp32
    slab once (2 q + 2 products), and U_m, V_m are written once in bf16."""
    return n * ((2 * q + 2) * T * D * 4 + (T + D) * m * 2)


def run_factor(args) -> None:
    import torch

    import position_invariant_kv_kamera_gb300 as pk
    from synth import gen

    torch.cuda.set_device(0)
    fs = FACTOR_SHAPE
    n, T, D, m, p, q, r = (fs[k] for k in ("n_slabs", "T", "D", "rank", "oversample", "power_iters", "true_rank"))
    # seeded deficits of rank r (factors from the counter generator, product formed on the device)
    st = gen.stream_id(0x4B414D45, gen.STREAM_DEFICIT)
    A = torch.from_numpy(gen.normal_f32(st, np.arange(n * T * r, dtype=np.uint64)).reshape(n, T, r)).cuda()
    B = torch.from_numpy(gen.normal_f32(st, np.uint64(1 << 40) + np.arange(n * D * r, dtype=np.uint64))
                         .reshape(n, D, r)).cuda()
    spec = torch.linspace(10, 1, r, device="cuda")
    delta = torch.bmm(A * spec, B.transpose(1, 2)).contiguous() / float(np.sqrt(T * D))
    del A, B
    om = torch.from_numpy(gen.gaussian_test_matrix(0x4B414D45, D, m + p)).cuda()
    desc = pk.factor_desc(delta, n, T, D, m, p, q, om)
    nbytes = pk.kamera_factor_workspace_size(desc)
    ws = torch.empty(nbytes // 4 + 64, dtype=torch.float32, device="cuda")
    out = torch.empty(n * (T + D) * m, dtype=torch.int16, device="cuda")
    stream = torch.cuda.current_stream()

    def call():
        pk.kamera_factor_patches(desc, out.data_ptr(), out.data_ptr() + 2 * T * m, (T + D) * m, ws.data_ptr(),
                                 nbytes, stream.cuda_stream)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 20))
    b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clocks:
        time.sleep(0.25)
        b.record(stream)
        for _ in range(steps):
            call()
        e.record(stream)
        torch.cuda.synchronize()
    sec = b.elapsed_time(e) / 1e3 / steps
    flops = n * factor_flops(T, D, m + p, m, q)
    peaks = measured_peaks()
    # the products with Delta run in TF32 on the tensor cores: the measured bf16
    # burst peak scaled by the nominal dense tf32 : bf16 ratio (1.1 : 2.25 PFLOP/s)
    tf32_peak = peaks["bf16_tflops"] * 1.1 / 2.25
    # the method reads Delta once per product: 2 q + 2 passes (Y, q x (Z, Y), B),
    # plus the bf16 factors written once
    nbytes = factor_bytes(n, T, D, m, q)
    # CPU: the oracle's exact Jacobi SVD of one slab
    import oracle
    A1 = delta[0].double().cpu().numpy()
    t0 = time.perf_counter()
    oracle.jacobi_svd(A1)
    cpu_s = time.perf_counter() - t0
    line = {"metric": "patch formation: rank-m factors of conditioning deficits (slabs/s)", "value": n / sec,
            "unit": "slabs/s", "n_gpus": 1, "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{n} slabs of {T}x{D} (16 patches x 28 layers x K/V of the GQA video shape), "
                                   f"rank {m}, oversample {p}, {q} subspace iterations, deficit rank {r}"},
            "roofline": {"bound": "hbm", "achieved": nbytes / sec / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": nbytes / sec / 1e9 / peaks["hbm_gbs"],
                         "traffic": profile_traffic("patch_formation", "factor_kernel", FACTOR_SOURCES),
                         "peak_source": peaks["source"] + " (burst copy)",
                         "bytes": f"{2 * q + 2} reads of the fp32 deficits + the bf16 factors written"},
            "tensor": {"achieved": flops / sec / 1e12, "peak": tf32_peak, "unit": "TFLOP/s",
                       "frac": flops / sec / 1e12 / tf32_peak,
                       "peak_source": f"{peaks['source']} bf16 burst {peaks['bf16_tflops']:.1f} TFLOP/s x nominal "
                                      "tf32:bf16 1.1:2.25"},
            "cpu_baseline": {"value": 1.0 / cpu_s, "unit": "slabs/s", "cores": 1, "kind": "oracle",
                             "sample": f"one {T}x{D} slab, exact one-sided Jacobi SVD ({cpu_s:.1f} s)"},
            "gpu_launches": steps, "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)


def orbit_traffic(slabs: int) -> float | None:
    """DRAM bytes per launch of the orbit mean over `slabs` slabs: the committed
    capture (scaled to 896 slabs) scaled by the slabs processed."""
    t = profile_traffic("orbit_mean", "orbit_mean_kernel", ORBIT_SOURCES)
    return t * slabs / 896 if t is not None else None


def run_orbit(args) -> None:
    """Orbit deficit: the mean over 4 sampled orderings of the headline batch's
    deficits (896 slabs of 1024 x 512 fp32 per ordering).  HBM-bound."""
    import torch

    import position_invariant_kv_kamera_gb300 as pk

    torch.cuda.set_device(0)
    slabs = 56 * args.chunks if args.chunks else 896  # 28 layers x K/V per chunk; --chunks for small captures
    n_ord, per = 4, slabs * 1024 * 512
    g = torch.Generator(device="cuda").manual_seed(0x4B414D45)
    d = torch.randn((n_ord, per), generator=g, device="cuda", dtype=torch.float32)
    out = torch.empty(per, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def call():
        pk.kamera_orbit_mean(d.data_ptr(), n_ord, per, per, out.data_ptr(), stream.cuda_stream)

    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 50))
    b, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(0) as clocks:
        time.sleep(0.25)
        b.record(stream)
        for _ in range(steps):
            call()
        e.record(stream)
        torch.cuda.synchronize()
    sec = b.elapsed_time(e) / 1e3 / steps
    nbytes = (n_ord + 1) * per * 4
    peaks = measured_peaks()
    x = d[:, : 1 << 24].double().cpu().numpy()
    import oracle
    t0 = time.perf_counter()
    oracle.orbit_mean(x.astype(np.float32))
    cpu_s = time.perf_counter() - t0
    line = {"metric": "orbit deficit: mean over sampled orderings (slabs/s)", "value": slabs / sec, "unit": "slabs/s",
            "n_gpus": 1, "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 * sec, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{n_ord} orderings x {slabs} slabs of 1024x512 fp32 deficits"},
            "roofline": {"bound": "hbm", "achieved": nbytes / sec / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": nbytes / sec / 1e9 / peaks["hbm_gbs"],
                         "traffic": orbit_traffic(slabs),
                         "frac_of_nominal": nbytes / sec / 1e9 / NOMINAL_HBM_GBS,
                         "peak_source": peaks["source"] + " (burst copy)"},
            "cpu_baseline": {"value": (1 << 24) / (1024 * 512) / cpu_s, "unit": "slabs/s", "cores": 1,
                             "kind": "oracle", "sample": f"2^24 elements x {n_ord} orderings ({cpu_s:.2f} s)"},
            "gpu_launches": steps, "clocks": clocks.summary()}
    print(json.dumps(line), flush=True)


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="long_video",
                    choices=sorted(W.WORKLOADS) + sorted(COMPRESSED) + ["patch_formation", "orbit_mean"])
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="time only the selected workload (no configs object)")
    ap.add_argument("--chunks", type=int, default=0,
                    help="reduced batch of this many chunks (profiler captures); 0 = the full workload")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "patch_formation":
        run_factor(args)
    elif args.workload == "orbit_mean":
        run_orbit(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
