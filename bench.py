"""Benchmark of the batched ragged exact top-k on GB300.

One step = one call of the library on one batch of seeded synthetic scores
already resident in HBM (all rows, the whole hot path: sampling, streaming
filter, exact cutoff, emission). Default workload: B=1024 rows of width
262144, lengths uniform in [0.8w, w], k=512, paged output (page_size 64); the
B=1024 x 131072, k=2048 ragged workload is measured too and reported under
"also". Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

``--impl reference`` times the CPU oracle (the reference arm) on
a bounded sample of the same workload instead.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs/call and scores-read GB/s (% of HBM peak) at B=1024, 80–100% ragged, k=512/2048"
UNIT = "µs/call"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20  # GB300
# The pages' own B300 (GB300 GPU) warm latencies for the same B=1024 ragged
# workloads (vLLM PR 56346, 执行摘要), context only.
PAGE_LATENCY_US = {3: 207.06, 4: 301.72}
WORKLOADS = {"w262144_k512_paged": 4, "w131072_k2048_ragged": 3,
             # prefill shapes (short-row kernel), for profiling runs with --quick
             "w8192_k512_prefill": 6, "w16384_k2048_prefill": 7}


# The files that make up each kernel's device code and launch shape. DRAM
# counters are reported as a kernel's traffic only while the code-only hash of
# these files equals the one recorded beside the counters.
_LAUNCH_FILES = ("ptx.cuh", "topk_kernel.cuh", "topk_launch.cuh", "topk_abi.cu")
KERNEL_SOURCES = {
    "topk_rows_kernel": _LAUNCH_FILES + tuple(f"topk_k{k}_{o}.cu" for k in (512, 1024, 2048)
                                              for o in ("ragged", "paged")),
    "topk_short_kernel": _LAUNCH_FILES + ("topk_short.cuh",) + tuple(f"topk_short_k{k}.cu"
                                                                   for k in (512, 1024, 2048)),
    "topk_short_bf16_kernel": _LAUNCH_FILES + ("topk_short.cuh", "topk_short_bf16.cuh")
    + tuple(f"topk_short_k{k}.cu" for k in (512, 1024, 2048)),
    "amax8_kernel": ("ptx.cuh", "topk_kernel.cuh", "topk_blocks.cu"),
    "sort_blocks_kernel": ("ptx.cuh", "topk_kernel.cuh", "topk_blocks.cu"),
}


def _code_only(text: str) -> str:
    """The source without // comments and blank lines: the hash follows the
    code, so an edited comment does not mark the counters stale."""
    lines = []
    for line in text.splitlines():
        code = line.split("//", 1)[0].rstrip()
        if code.strip():
            lines.append(code)
    return "\n".join(lines)


def kernel_source_hash(kernel: str = "topk_rows_kernel", csrc: str = "") -> str:
    csrc = csrc or os.path.join(ROOT, "sparse_attention_indexer_fp32_gb300", "csrc")
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            doc = json.load(f)
    except (OSError, ValueError):
        return None
    entry = doc.get("workloads", {}).get(workload)
    if not entry or entry.get("kernel") not in KERNEL_SOURCES:
        return None
    if entry.get("kernel_source_hash") != kernel_source_hash(entry["kernel"]):
        return None
    return entry.get("dram_bytes_per_launch")


def workload_config(spec) -> dict:
    """The `config` object of a bench line for a workload (both arms print it)."""
    return {"workload": spec.name, "B": spec.B, "stride": spec.stride, "k": spec.k,
            "lengths": "uniform integer in [ceil(0.8*stride), stride]",
            "paged": bool(spec.page_size), "page_size": spec.page_size or None,
            "scores": "f32", "keys": "u32 order-preserving keys of the f32 scores (exact ranking)",
            "scores_bytes": int(spec.B) * int(spec.stride) * 4,
            "l2": "inputs larger than L2 (no flush needed)"}


def algorithmic_bytes(lengths: np.ndarray, stride: int, B: int, k: int) -> int:
    n = np.clip(lengths.astype(np.int64), 0, stride)
    return int(n.sum() * 4 + B * k * 4)


def hbm_roofline(algo: int, us: float, traffic=None) -> dict:
    """The roofline object of a launch that moves `algo` algorithmic bytes in
    `us` microseconds, against the measured HBM peak."""
    peak, peak_kind = measured_peak()
    achieved = algo / (us * 1e-6) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_kind": f"{peak_kind} hbm_gbs (burst copy)",
            "traffic": traffic, "algorithmic_bytes_per_launch": int(algo)}


# ----------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.path is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        power = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------ distributed


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, local, world


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (every rank gets it)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------- GPU arm


def time_device(fn, steps: int, warmup: int, world: int):
    import torch

    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        fn()
    end.record()
    torch.cuda.synchronize()
    barrier(world)
    return start.elapsed_time(end)  # ms for all steps


def bench_workload(config: int, steps: int, warmup: int, world: int, local: int, with_e2e: bool,
                   e2e_steps: int, clocks: bool, rows=None):
    import torch

    import sparse_attention_indexer_fp32_gb300 as tk
    from synth import CONFIGS, make_workload

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = make_workload(config, B=rows)
    s = torch.from_numpy(w.scores).to(dev)
    l = torch.from_numpy(w.lengths).to(dev)
    pt = None if w.page_table is None else torch.from_numpy(w.page_table).to(dev)
    out = torch.empty((w.B, w.k), dtype=torch.int32, device=dev)
    if pt is None:
        fn = lambda: tk.topk_ragged(s, l, w.k, out=out)  # noqa: E731
    else:
        fn = lambda: tk.topk_paged(s, l, w.k, pt, w.page_size, out=out)  # noqa: E731

    sampler = ClockSampler(torch.cuda.current_device()) if clocks else None
    if sampler:
        sampler.__enter__()
    ms_total = time_device(fn, steps, warmup, world)
    if sampler:
        sampler.__exit__()
    ms_total = max_over_ranks(ms_total, world, dev)
    us_per_call = 1000.0 * ms_total / steps

    algo = algorithmic_bytes(w.lengths, w.stride, w.B, w.k)
    peak, peak_kind = measured_peak()
    achieved = algo / (us_per_call * 1e-6) / 1e9
    res = {
        "workload": w.name,
        "us_per_call": us_per_call,
        "rows_per_s": w.B / (us_per_call * 1e-6),
        "scores_read_gbs": (algo - w.B * w.k * 4) / (us_per_call * 1e-6) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": f"{peak_kind} hbm_gbs (burst copy)",
                     "traffic": profiled_traffic(w.name),
                     "algorithmic_bytes_per_launch": algo},
        "config": dict(workload_config(CONFIGS[config]), B=w.B, scores_bytes=int(w.scores.nbytes)),
        "gpu_launches": steps,
        "sampler": sampler.summary() if sampler else None,
    }
    if with_e2e:
        res["e2e"] = bench_e2e(w, dev, e2e_steps, world)
    del s, l, pt, out
    torch.cuda.empty_cache()
    return res


def bench_prefill(config: int, local: int, steps: int, warmup: int, world: int, bf16: bool = False):
    """Prefill-shaped batch (many rows of at most 16384 scores): the
    short-row kernel, FP32 scores or the same scores rounded to BF16."""
    import torch

    import sparse_attention_indexer_fp32_gb300 as tk
    from synth import make_workload, to_bf16_bits

    dev = torch.device("cuda", local)
    w = make_workload(config)
    if bf16:
        s = torch.from_numpy(to_bf16_bits(w.scores).view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        s = torch.from_numpy(w.scores).to(dev)
    l = torch.from_numpy(w.lengths).to(dev)
    out = torch.empty((w.B, w.k), dtype=torch.int32, device=dev)
    if bf16:
        fn = lambda: tk.topk_select_bf16(s, l, w.k, out=out)  # noqa: E731
    else:
        fn = lambda: tk.topk_ragged(s, l, w.k, out=out)  # noqa: E731
    ms = max_over_ranks(time_device(fn, steps, warmup, world), world, dev)
    us = 1000.0 * ms / steps
    n = np.clip(w.lengths.astype(np.int64), 0, w.stride)
    algo = int(n.sum() * (2 if bf16 else 4) + w.B * w.k * 4)
    peak, peak_kind = measured_peak()
    achieved = algo / (us * 1e-6) / 1e9
    del s, l, out
    torch.cuda.empty_cache()
    return {"workload": w.name + ("_bf16" if bf16 else ""), "kind": "prefill", "us_per_call": us,
            "rows_per_s": w.B / (us * 1e-6), "steps": steps,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": f"{peak_kind} hbm_gbs (burst copy)",
                         "traffic": profiled_traffic(w.name + ("_bf16" if bf16 else "")),
                         "algorithmic_bytes_per_launch": algo},
            "config": {"workload": w.name, "B": w.B, "stride": w.stride, "k": w.k,
                       "dtype": "bf16" if bf16 else "f32",
                       "lengths": "uniform integer in [ceil(0.8*stride), stride]",
                       "l2": "inputs larger than L2 (no flush needed)"}}


def two_level_rooflines(res: dict, nb: np.ndarray, keys_stride: int, B: int, k_blocks: int,
                        workload: str) -> None:
    """Adds the roofline of each two-level stage to `res` (stage -> {"us_per_call"}),
    from the rows' block counts `nb`."""
    res["sort_candidate_blocks"]["note"] = ("the kernel alone (the table is sorted in place; repeated "
                                            "calls redo the same counting sort); algorithmic bytes: "
                                            "ids read and written, one page-table entry read and one "
                                            "pool slot written per id")
    # keys: the scores read (the newest block is +inf, not read) and the keys written
    algo_keys = int((nb - 1).clip(min=0).sum() * 32 + nb.sum() * 4)
    res["amax8_varlen"]["roofline"] = hbm_roofline(
        algo_keys, res["amax8_varlen"]["us_per_call"],
        profiled_traffic("amax8_varlen_" + workload.split("_k")[0]))
    # top-k over the keys: the keys read and the block ids written
    shape = workload.split("_k")[0]
    algo_sel = algorithmic_bytes(nb, keys_stride, B, k_blocks)
    res["topk_over_keys"]["roofline"] = hbm_roofline(
        algo_sel, res["topk_over_keys"]["us_per_call"], profiled_traffic("topk_over_keys_" + shape))
    algo_table = 4 * B * k_blocks * 4
    res["sort_candidate_blocks"]["roofline"] = hbm_roofline(
        algo_table, res["sort_candidate_blocks"]["us_per_call"],
        profiled_traffic("sort_candidate_blocks_" + shape))


def bench_two_level(local: int, steps: int, warmup: int, world: int):
    """The two-level indexer's chain on the paged workload's rows: block-max
    keys (one pass over the scores), top-k over the keys (k = 512 blocks), the
    sorted block table with pool slots (64-token pages). Each stage timed on
    its own, and the keys stage against the HBM roofline."""
    import torch

    import sparse_attention_indexer_fp32_gb300 as tk
    from synth import make_workload

    dev = torch.device("cuda", local)
    w = make_workload(4)
    k_blocks, page_size = 512, 64
    s = torch.from_numpy(w.scores).to(dev)
    l = torch.from_numpy(w.lengths).to(dev)
    n = np.clip(w.lengths.astype(np.int64), 0, w.stride)
    nb = -(-n // 8)
    blen = torch.from_numpy(nb.astype(np.int32)).to(dev)
    pt = torch.from_numpy(np.ascontiguousarray(w.page_table)).to(dev)
    keys = torch.empty((w.B, -(-w.stride // 8)), dtype=torch.float32, device=dev)
    sel = torch.empty((w.B, k_blocks), dtype=torch.int32, device=dev)
    table = torch.empty_like(sel)
    pages = torch.empty_like(sel)
    stages = {
        "amax8_varlen": lambda: tk.amax8_varlen(s, l, k_blocks, out=keys),
        "topk_over_keys": lambda: tk.topk_ragged(keys, blen, k_blocks, out=sel),
        # in place: after the first call the table is already ascending, and a
        # repeated call redoes the same counting sort (its cost does not depend
        # on the order of the ids)
        "sort_candidate_blocks": lambda: tk.sort_candidate_blocks(table, l, w.stride, pt, page_size,
                                                                  out_pages=pages),
    }
    res = {}
    for name, fn in stages.items():
        if name == "sort_candidate_blocks":  # the selection, once, outside the timed region
            stages["topk_over_keys"]()
            table.copy_(sel)
        ms = max_over_ranks(time_device(fn, steps, warmup, world), world, dev)
        res[name] = {"us_per_call": 1000.0 * ms / steps}
    two_level_rooflines(res, nb, int(keys.shape[1]), w.B, k_blocks, w.name)
    del s, l, blen, pt, keys, sel, table, pages
    torch.cuda.empty_cache()
    return {"workload": w.name, "kind": "two_level", "k_blocks": k_blocks, "page_size": page_size,
            "steps": steps, "stages": res}


def bench_latency(config: int, local: int, steps: int = 200, cold_steps: int = 50):
    """Per-call latency of a small decode batch: eager calls through the
    Python API, and replays of one call captured in a CUDA graph (the
    launch path a decode loop uses; lengths may change between replays)."""
    import torch

    import sparse_attention_indexer_fp32_gb300 as tk
    from synth import make_workload

    dev = torch.device("cuda", local)
    w = make_workload(config)
    s = torch.from_numpy(w.scores).to(dev)
    l = torch.from_numpy(w.lengths).to(dev)
    out = torch.empty((w.B, w.k), dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for _ in range(10):
            tk.topk_ragged(s, l, w.k, out=out)
        stream.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            tk.topk_ragged(s, l, w.k, out=out)
        b.record()
        b.synchronize()
        eager = 1000.0 * a.elapsed_time(b) / steps
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            tk.topk_ragged(s, l, w.k, out=out)
        for _ in range(10):
            graph.replay()
        stream.synchronize()
        a.record()
        for _ in range(steps):
            graph.replay()
        b.record()
        b.synchronize()
        replay = 1000.0 * a.elapsed_time(b) / steps

        # Cold L2: before every call a buffer twice the L2's size is written
        # (outside the timed events), so the call finds none of its inputs there.
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)
        cold = {}
        for mode, fn in (("eager", lambda: tk.topk_ragged(s, l, w.k, out=out)),
                         ("graph_replay", graph.replay)):
            times = []
            for i in range(cold_steps):
                flush.fill_(i)
                a.record()
                fn()
                b.record()
                b.synchronize()
                times.append(1000.0 * a.elapsed_time(b))
            cold[mode] = statistics.median(times)
        del flush
    return {"workload": w.name, "kind": "latency", "eager_us_per_call": eager,
            "graph_replay_us_per_call": replay, "steps": steps,
            "cold_l2_eager_us_per_call": cold["eager"],
            "cold_l2_graph_replay_us_per_call": cold["graph_replay"], "cold_steps": cold_steps,
            "note": "warm: back-to-back calls on one stream; cold: median of single calls, each "
                    "after writing a buffer of twice the L2 size; the graph holds one captured call"}


E2E_CHUNKS = 8
E2E_WINDOWS = 3


def bench_e2e(w, dev, steps: int, world: int):
    """Same work through the public API with host buffers: every step copies the
    inputs from pinned host memory to the device and reads the result back.
    The batch goes in E2E_CHUNKS row chunks: while the copy engine brings in
    chunk c + 1, a second stream selects chunk c, so that only the last
    chunk's selection is not hidden behind the host-to-device copy (the
    CPU-GPU link bounds this leg: about 211 GB/s on GB300 for the copy engine
    and for kernel loads from mapped pinned memory alike)."""
    import torch

    import sparse_attention_indexer_fp32_gb300 as tk

    hs = torch.from_numpy(w.scores).pin_memory()
    hl = torch.from_numpy(w.lengths).pin_memory()
    hpt = None if w.page_table is None else torch.from_numpy(w.page_table).pin_memory()
    hout = torch.empty((w.B, w.k), dtype=torch.int32).pin_memory()
    ds = torch.empty_like(hs, device=dev)
    dl = torch.empty_like(hl, device=dev)
    dpt = None if hpt is None else torch.empty_like(hpt, device=dev)
    dout = torch.empty((w.B, w.k), dtype=torch.int32, device=dev)
    nchunks = max(1, min(E2E_CHUNKS, w.B))
    bounds = [w.B * c // nchunks for c in range(nchunks + 1)]
    comp = torch.cuda.Stream(device=dev)
    landed = [torch.cuda.Event() for _ in range(nchunks)]
    done = torch.cuda.Event()

    def step():
        cur = torch.cuda.current_stream(dev)
        for c in range(nchunks):
            r0, r1 = bounds[c], bounds[c + 1]
            if r0 == r1:
                continue
            dl[r0:r1].copy_(hl[r0:r1], non_blocking=True)
            if dpt is not None:
                dpt[r0:r1].copy_(hpt[r0:r1], non_blocking=True)
            ds[r0:r1].copy_(hs[r0:r1], non_blocking=True)
            landed[c].record(cur)
            comp.wait_event(landed[c])
            with torch.cuda.stream(comp):
                if dpt is None:
                    tk.topk_ragged(ds[r0:r1], dl[r0:r1], w.k, out=dout[r0:r1])
                else:
                    tk.topk_paged(ds[r0:r1], dl[r0:r1], w.k, dpt[r0:r1], w.page_size, out=dout[r0:r1])
        done.record(comp)
        cur.wait_event(done)  # the next step's copies and the read-back follow every chunk's selection
        hout.copy_(dout, non_blocking=True)

    # Three timed windows of `steps` steps each, after 5 warm-up steps: the
    # host-to-device link's rate varies from window to window on a shared
    # host (one window in several runs ~45 % slower, copies alone included),
    # so the line reports the median window and lists all three.
    windows = []
    for i in range(E2E_WINDOWS):
        ms = max_over_ranks(time_device(step, steps, 5 if i == 0 else 0, world), world, dev)
        windows.append(1000.0 * ms / steps)
    h2d = hs.nbytes + hl.nbytes + (0 if hpt is None else hpt.nbytes)
    return {"value": sorted(windows)[len(windows) // 2], "unit": UNIT, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(hout.nbytes), "steps": steps, "row_chunks": nchunks,
            "windows_us": [round(v, 1) for v in windows]}


def cpu_baseline(config: int, budget_s: float = 12.0, min_rows: int = 8):
    """The CPU oracle as it stands (single thread) on a bounded sample of rows
    of the same workload, scaled to the whole batch."""
    import oracle
    from synth import CONFIGS, make_rows

    spec = CONFIGS[config]
    orc = oracle.load()
    rng = np.random.default_rng(0)
    order = rng.permutation(spec.B)
    done, elapsed = 0, 0.0
    while done < spec.B and (elapsed < budget_s or done < min_rows):
        rows = order[done: done + 8]
        wk = make_rows(config, rows)
        t0 = time.perf_counter()
        if wk.page_table is None:
            orc.topk_ragged(wk.scores, wk.lengths, wk.k)
        else:
            orc.topk_paged(wk.scores, wk.lengths, wk.k, wk.page_table, wk.page_size)
        elapsed += time.perf_counter() - t0
        done += len(rows)
    us = 1e6 * elapsed / done * spec.B
    return {"value": us, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{done} random rows of {spec.B} (single-threaded full sort per row), "
                      f"{elapsed:.1f} s, scaled to the whole batch"}


def _oracle_chunk(config: int, rows):
    """One worker of the parallel CPU baseline: the oracle on these rows
    (drawn before the clock starts); returns (rows, seconds)."""
    import oracle
    from synth import make_rows

    orc = oracle.load(rebuild_if_stale=False)
    wk = make_rows(config, rows)
    t0 = time.perf_counter()
    if wk.page_table is None:
        orc.topk_ragged(wk.scores, wk.lengths, wk.k)
    else:
        orc.topk_paged(wk.scores, wk.lengths, wk.k, wk.page_table, wk.page_size)
    return len(rows), time.perf_counter() - t0


def cpu_baseline_parallel(config: int, rows_per_core: int = 8):
    """The same oracle over all host cores: one process per core (spawned, so
    no CUDA state is inherited), each on its own rows; the whole batch's time
    is scaled from the slowest worker."""
    import multiprocessing as mp

    import oracle
    from synth import CONFIGS

    oracle.load()  # compiled once, before the workers start
    spec = CONFIGS[config]
    cores = os.cpu_count() or 1
    order = np.random.default_rng(1).permutation(spec.B)
    chunks = [order[i * rows_per_core: (i + 1) * rows_per_core].tolist() for i in range(cores)]
    chunks = [c for c in chunks if c]
    with mp.get_context("spawn").Pool(len(chunks)) as pool:
        res = pool.starmap(_oracle_chunk, [(config, c) for c in chunks])
    rows = sum(r for r, _ in res)
    slowest = max(t for _, t in res)
    us = 1e6 * slowest / rows_per_core * spec.B / len(chunks)
    return {"value": us, "unit": UNIT, "cores": len(chunks), "kind": "oracle",
            "sample": f"{rows} random rows, {rows_per_core} per process on {len(chunks)} "
                      f"processes (single-threaded full sort per row); the batch's time "
                      f"scaled from the slowest process ({slowest:.2f} s)"}


# ------------------------------------------------------------- dispatch sweep

SWEEP_WIDTHS = (4096, 8192, 16384, 32768, 65536, 131072, 196608, 262144)
SWEEP_BATCHES = (1, 4, 8, 16, 32, 48, 64, 96, 128, 192, 256, 1024, 2048)
SWEEP_KS = (512, 1024, 2048)
SWEEP_MAX_ELEMS = 2048 * 262144  # 2 GiB of scores at most


def _sweep_split_rows(B: int, sm_count: int) -> int:
    """The split-row count of the automatic policy without its width gate."""
    slots = 2 * sm_count
    r = B % slots if B >= slots else B
    return min(r, slots - r)


def sweep_paths(width: int, B: int, sm_count: int):
    """(name, options) of every path worth timing on rows of this width."""
    paths = [("auto", {})]
    if width <= 16384:
        paths += [("short", dict(short_rows=1)), ("short_regs", dict(short_rows=1, sample_mode=1))]
    for G in (1, 2, 4, 8, 16):
        if width // G < 4096:  # a CTA would stream less than one stage
            continue
        for sm in (1, 2):
            paths.append((f"G{G}_{'sampled' if sm == 2 else 'full'}",
                          dict(short_rows=-1, cluster_size=G, sample_mode=sm)))
    m = _sweep_split_rows(B, sm_count)
    if width >= 32768 and 0 < m <= 1024:
        paths.append((f"G1_split{m}", dict(short_rows=-1, cluster_size=1, split_rows=m)))
    if width >= 32768 and B <= 512 and B != m:
        paths.append(("G1_split_all", dict(short_rows=-1, cluster_size=1, split_rows=B)))
    return paths


SWEEP_REPS = 20


def _graph_time_us(fn, stream, start, end) -> float:
    """Device time per call of `fn`: SWEEP_REPS calls captured in one CUDA
    graph (so that the host's launch cost is not timed), replayed once to warm
    up, then twice under CUDA events."""
    import torch

    with torch.cuda.stream(stream):
        for _ in range(3):
            fn()
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(SWEEP_REPS):
                fn()
        graph.replay()
        start.record()
        graph.replay()
        graph.replay()
        end.record()
        end.synchronize()
    us = 1000.0 * start.elapsed_time(end) / (2 * SWEEP_REPS)
    del graph
    return us


def run_sweep(args):
    """Times every path of the library on N(0,1) rows over batch x width x k,
    with full and 80-100 % ragged lengths; writes the measurements (JSON) and
    a summary table (markdown) under the output folder."""
    import torch

    import sparse_attention_indexer_fp32_gb300 as tk

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    gen = torch.Generator(device=dev)
    gen.manual_seed(0x5EED0100)
    big = torch.randn(SWEEP_MAX_ELEMS, generator=gen, device=dev, dtype=torch.float32)
    ws = torch.zeros(tk.workspace_bytes(2048, 1024), dtype=torch.uint8, device=dev)
    cnt = torch.zeros(tk.NUM_COUNTERS, dtype=torch.int32, device=dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream = torch.cuda.Stream(dev)
    results = []
    t0 = time.time()
    for width in SWEEP_WIDTHS:
        for B in SWEEP_BATCHES:
            if B * width > SWEEP_MAX_ELEMS:
                continue
            scores = big[: B * width].view(B, width)
            for lmode in ("full", "ragged"):
                if lmode == "full":
                    lengths = torch.full((B,), width, dtype=torch.int32, device=dev)
                else:
                    lengths = torch.randint(-(-width * 4 // 5), width + 1, (B,), generator=gen,
                                            device=dev, dtype=torch.int32)
                n = int(lengths.clamp(0, width).sum().item())
                for k in SWEEP_KS:
                    out = torch.empty((B, k), dtype=torch.int32, device=dev)
                    rec = {"width": width, "B": B, "lengths": lmode, "k": k, "paths": {}}
                    for name, opts in sweep_paths(width, B, sms):
                        o = dict(opts)
                        if name == "auto" or "split_rows" in o:
                            o["workspace"] = ws  # the automatic policy with a workspace
                        fn = lambda o=o: tk.topk_select_ex(scores, lengths, k, out=out, **o)  # noqa: E731
                        rec["paths"][name] = _graph_time_us(fn, stream, start, end)
                    # what the automatic policy did, from the device counters
                    cnt.zero_()
                    tk.topk_select_ex(scores, lengths, k, out=out, counters=cnt,
                                      workspace=ws if width > 16384 else None)
                    c = cnt.cpu().tolist()
                    rec["auto_counters"] = {"short": c[tk.Counter.SHORT_ROWS],
                                            "cluster": c[tk.Counter.CLUSTER_ROWS],
                                            "split": c[tk.Counter.SPLIT_ROWS],
                                            "sampled": c[tk.Counter.SAMPLED]}
                    rec["algorithmic_bytes"] = n * 4 + B * k * 4
                    results.append(rec)
    clusters = {f"k{k}_G{g}": tk.max_active_clusters(k, False, g) for k in SWEEP_KS
                for g in (2, 4, 8, 16)}
    doc = {"sm_count": sms, "gpu": torch.cuda.get_device_name(dev), "seconds": time.time() - t0,
           "max_active_clusters": clusters,
           "reps": SWEEP_REPS, "warmup": 3, "command": "python bench.py --sweep --sweep-out DIR",
           "results": results}
    os.makedirs(args.sweep_out, exist_ok=True)
    with open(os.path.join(args.sweep_out, "dispatch_sweep.json"), "w") as f:
        json.dump(doc, f)
    with open(os.path.join(args.sweep_out, "dispatch_sweep.md"), "w") as f:
        f.write(sweep_markdown(doc))
    print(json.dumps({"sweep": len(results), "seconds": doc["seconds"]}), flush=True)


def sweep_markdown(doc: dict) -> str:
    """Summary tables of a sweep: per shape the automatic path against the
    best forced one, and the comparisons each dispatch gate rests on."""
    peak, _ = measured_peak()
    res = doc["results"]
    lines = [f"# Dispatch sweep: every path of the library over batch x width x k",
             "",
             f"GPU: {doc['gpu']} ({doc['sm_count']} SMs). Command: `{doc['command']}`. N(0,1) rows "
             f"(seeded torch generator on the device), lengths full or uniform in [0.8w, w]; each "
             f"path: {doc['warmup']} warm-up calls, then {doc['reps']} calls captured in one CUDA "
             f"graph, replayed once untimed and twice under CUDA events (device time, no host "
             f"launch cost; small shapes stay in L2). Times in us per call. `frac` = algorithmic "
             f"bytes / time / {peak:.0f} GB/s.",
             "",
             "Clusters resident at once (the CUDA driver's answer, ragged kernel): " +
             ", ".join(f"{n} {v}" for n, v in doc.get("max_active_clusters", {}).items()) + ".",
             ""]
    lines += ["## Automatic policy against the best forced path (ragged lengths)", "",
              "| k | width | B | auto us | frac | best path | best us | auto/best |",
              "|---|---|---|---|---|---|---|---|"]
    for r in res:
        if r["lengths"] != "ragged":
            continue
        p = r["paths"]
        best = min((v, n) for n, v in p.items() if n != "auto")
        frac = r["algorithmic_bytes"] / (p["auto"] * 1e-6) / 1e9 / peak
        lines.append(f"| {r['k']} | {r['width']} | {r['B']} | {p['auto']:.1f} | {frac:.2f} | "
                     f"{best[1]} | {best[0]:.1f} | {p['auto'] / best[0]:.2f} |")
    lines += ["", "## Gate: short-row kernel against the streaming kernel (width <= 16384)", "",
              "| k | width | B | lengths | short us | short_regs us | best streaming | us |",
              "|---|---|---|---|---|---|---|---|"]
    for r in res:
        if r["width"] > 16384:
            continue
        p = r["paths"]
        st = min((v, n) for n, v in p.items() if n.startswith("G"))
        lines.append(f"| {r['k']} | {r['width']} | {r['B']} | {r['lengths']} | {p['short']:.1f} | "
                     f"{p['short_regs']:.1f} | {st[1]} | {st[0]:.1f} |")
    lines += ["", "## Gate: sampled cutoff against the full stream (one CTA per row, ragged)", "",
              "| k | width | B | full us | sampled us | sampled/full |", "|---|---|---|---|---|---|"]
    for r in res:
        if r["lengths"] != "ragged" or "G1_full" not in r["paths"]:
            continue
        p = r["paths"]
        lines.append(f"| {r['k']} | {r['width']} | {r['B']} | {p['G1_full']:.1f} | "
                     f"{p['G1_sampled']:.1f} | {p['G1_sampled'] / p['G1_full']:.2f} |")
    lines += ["", "## Gate: split rows of the last wave (one CTA per row, sampled, ragged)", "",
              "| k | width | B | unsplit us | split path | split us | split/unsplit |",
              "|---|---|---|---|---|---|---|"]
    for r in res:
        if r["lengths"] != "ragged":
            continue
        p = r["paths"]
        for n, v in p.items():
            if n.startswith("G1_split") and "G1_sampled" in p:
                lines.append(f"| {r['k']} | {r['width']} | {r['B']} | {p['G1_sampled']:.1f} | {n} | "
                             f"{v:.1f} | {v / p['G1_sampled']:.2f} |")
    lines += ["", "## Gate: cluster size (sampled, ragged): time per G", "",
              "| k | width | B | G1 | G2 | G4 | G8 | G16 | best |", "|---|---|---|---|---|---|---|---|---|"]
    for r in res:
        if r["lengths"] != "ragged" or r["width"] <= 16384:
            continue
        p = r["paths"]
        cells = [p.get(f"G{g}_sampled") for g in (1, 2, 4, 8, 16)]
        vals = [(v, g) for v, g in zip(cells, (1, 2, 4, 8, 16)) if v is not None]
        best = min(vals)[1]
        lines.append(f"| {r['k']} | {r['width']} | {r['B']} | " +
                     " | ".join("-" if v is None else f"{v:.1f}" for v in cells) + f" | G{best} |")
    return "\n".join(lines) + "\n"


def run_gpu_arm(args):
    rank, local, world = dist_setup(args.gpus)
    primary = WORKLOADS[args.workload]
    secondary = 3 if primary == 4 else 4
    if args.bf16:  # profiling runs of the BF16 short-row kernel
        res = bench_prefill(primary, local, args.steps, args.warmup, world, bf16=True)
        if rank == 0:
            print(json.dumps({"quick": True, "workload": res["workload"], "B": res["config"]["B"],
                              "us_per_call": res["us_per_call"], "roofline": res["roofline"]}), flush=True)
        return
    res = bench_workload(primary, args.steps, args.warmup, world, local, with_e2e=not args.quick,
                         e2e_steps=args.e2e_steps, clocks=not args.quick, rows=args.rows)
    also = latency = prefill = two_level = None
    if not args.quick:
        also = bench_workload(secondary, max(args.steps // 2, 1), args.warmup, world, local,
                              with_e2e=False, e2e_steps=0, clocks=False, rows=args.rows)
        # every rank runs these (their timing takes the maximum over ranks)
        latency = bench_latency(1, local)
        two_level = bench_two_level(local, 200, args.warmup, world)
        prefill = [bench_prefill(6, local, 200, args.warmup, world),
                   bench_prefill(7, local, 200, args.warmup, world),
                   bench_prefill(6, local, 200, args.warmup, world, bf16=True)]
    if rank != 0:
        return
    if args.quick:  # profiling runs: timing of the primary workload only
        print(json.dumps({"quick": True, "workload": res["workload"], "B": res["config"]["B"],
                          "us_per_call": res["us_per_call"], "roofline": res["roofline"]}),
              flush=True)
        return
    clocks = res.pop("sampler")
    also.pop("sampler")
    also_line = {"workload": also["workload"], "us_per_call": also["us_per_call"],
                 "rows_per_s": also["rows_per_s"], "scores_read_gbs": also["scores_read_gbs"],
                 "roofline": also["roofline"], "config": also["config"],
                 "steps": max(args.steps // 2, 1), "page_b300_us": PAGE_LATENCY_US.get(secondary)}
    line = {
        "metric": METRIC,
        "value": res["us_per_call"],
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": res["us_per_call"] / 1000.0,
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded Philox rows shaped like the decode-step indexer workload)",
        "config": dict(res["config"], parallelism=f"replicas x{world}"),
        "rows_per_s": res["rows_per_s"] * world,
        "scores_read_gbs": res["scores_read_gbs"],
        "roofline": res["roofline"],
        "clocks": clocks,
        "e2e": res["e2e"],
        "gpu_launches": res["gpu_launches"],
        "latency": latency,
        "prefill": prefill,
        "two_level": two_level,
        "page_b300_us": PAGE_LATENCY_US.get(primary),
        "kernel_source_hash": {k: kernel_source_hash(k) for k in KERNEL_SOURCES},
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(primary)
        line["cpu_baseline_all_cores"] = cpu_baseline_parallel(primary)
    # The other metric workload, then a compact summary of every line: last,
    # so that a reader keeping only the end of the line still has them.
    line["also"] = [also_line]
    line["summary"] = summary_of(line)
    print(json.dumps(line), flush=True)


def summary_of(line: dict) -> list:
    """One short entry per timed workload: time per call, roofline fraction
    of the measured peak, DRAM traffic per launch (null when not captured on
    the current kernel source)."""
    def entry(name, us, roof):
        return {"w": name, "us": round(us, 2), "frac": round(roof["frac"], 3),
                "traffic": roof.get("traffic"), "algo": roof["algorithmic_bytes_per_launch"]}

    out = [entry(line["config"]["workload"], line["value"], line["roofline"])]
    out += [entry(a["workload"], a["us_per_call"], a["roofline"]) for a in line.get("also") or []]
    out += [entry(p["workload"], p["us_per_call"], p["roofline"]) for p in line.get("prefill") or []]
    tl = line.get("two_level")
    if tl:
        out += [entry(f"{name}_{tl['workload']}", st["us_per_call"], st["roofline"])
                for name, st in tl["stages"].items()]
    lat = line.get("latency")
    if lat:
        out.append({"w": lat["workload"], "eager_us": round(lat["eager_us_per_call"], 2),
                    "graph_us": round(lat["graph_replay_us_per_call"], 2),
                    "cold_eager_us": round(lat["cold_l2_eager_us_per_call"], 2),
                    "cold_graph_us": round(lat["cold_l2_graph_replay_us_per_call"], 2)})
    return out


def run_reference_arm(args):
    """The oracle, as it stands, on the host cores: each step is a bounded
    sample of rows of the same workload; the value is scaled to the batch."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from synth import CONFIGS, make_rows

    config = WORKLOADS[args.workload]
    spec = CONFIGS[config]
    orc = oracle.load()
    rows_per_step = 1
    rng = np.random.default_rng(1)
    order = rng.permutation(spec.B)
    # steps cycle through pre-drawn rows so that drawing is not timed
    pool = make_rows(config, order[: min(spec.B, 16)])

    def step(i):
        j = i % pool.B
        sl = slice(j, j + rows_per_step)
        if pool.page_table is None:
            orc.topk_ragged(pool.scores[sl], pool.lengths[sl], pool.k)
        else:
            orc.topk_paged(pool.scores[sl], pool.lengths[sl], pool.k, pool.page_table[sl],
                           pool.page_size)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    elapsed = time.perf_counter() - t0
    us = 1e6 * elapsed / (args.steps * rows_per_step) * spec.B
    line = {
        "impl": "reference",
        "metric": METRIC, "value": us, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1000.0 * elapsed / args.steps,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded Philox rows shaped like the decode-step indexer workload)",
        "config": dict(workload_config(spec), parallelism="replicas x1"),
        "cpu_baseline": {"value": us, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{args.steps} steps of {rows_per_step} row each, cycling over "
                                   f"{pool.B} random rows; scaled to the {spec.B}-row batch "
                                   "(the host oracle, one thread: no GPU and no replicas)"},
        "e2e": {"value": us, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="w262144_k512_paged")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rows", type=int, default=None,
                    help="use only the first ROWS rows of the workload (profiling runs)")
    ap.add_argument("--quick", action="store_true",
                    help="primary workload only, no e2e / clocks / CPU baseline (profiling runs)")
    ap.add_argument("--bf16", action="store_true",
                    help="with --quick and a prefill workload: its scores rounded to BF16, through "
                         "topk_select_bf16 (profiling runs)")
    ap.add_argument("--sweep", action="store_true",
                    help="time every path over batch x width x k instead (dispatch sweep)")
    ap.add_argument("--sweep-out", default="sweep_out",
                    help="folder for the sweep's JSON and markdown summary")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.bf16 and not (args.quick and WORKLOADS[args.workload] in (6, 7)):
        ap.error("--bf16 needs --quick and a prefill workload")
    if args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference_arm(args)
    else:
        run_gpu_arm(args)


if __name__ == "__main__":
    main()
