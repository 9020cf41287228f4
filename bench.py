#!/usr/bin/env python3
"""Benchmark of one DSA layer-step on GB300: µs per step, HBM GB/s, roofline.

Workload (default): decode, batch 64, every causal length 32768, page 64,
indexer 64 heads x 128 bf16, top-k 2048, 64 query / 8 KV heads, head dim 128,
bf16 K/V, softmax scale 1/sqrt(128).  One step = lightning indexer -> top-k
-> sparse attention (8 splits) -> merge, replayed as one CUDA graph with the
inputs resident in HBM.  Algorithmic bytes per step: index keys up to each
length (64 x 32768 x 256 B) + selected K/V (64 x 2048 x 8 heads x 128 x 2 B
x 2) = 1 GiB.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl dsa|reference]

Prints one JSON line.  Under torchrun (N > 1) every rank runs an independent
replica on its own GPU (the step does not shard; no collective on the data
path) and rank 0 prints the aggregate.  --impl reference times the CPU
oracle (fp64 numpy, one thread) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

if "--cpu-baseline-worker" in sys.argv or ("--impl" in sys.argv and "reference" in sys.argv):
    # the oracle is timed on one host thread: pin BLAS before numpy loads
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        os.environ[_v] = "1"

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per DSA layer-step and HBM GB/s (% of roofline), batch 64, 32k ctx, top-k 2048"
DEFAULT_WORKLOAD = 2
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 256 << 20  # > 129 MB L2
KERNEL_SOURCE = {"indexer": "indexer_tc.cu", "sparse_attn": "attn.cu"}  # file holding each timed kernel


def max_over_ranks(x: float, world: int) -> float:
    """The largest of every rank's value (the job's wall time is its slowest
    rank's); a plain value when there is one rank.  Uses the process group's
    backend device (CUDA tensors for NCCL, CPU tensors for gloo)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job(ms_max: float, rows_per_rank: int, world: int) -> dict:
    """Whole-job figures of N replicas that each run one full step at once:
    µs per layer-step as the job delivers them (the slowest rank's time over
    N) and rows per second over all ranks."""
    return {"us_per_step": ms_max * 1e3 / world, "rows_per_s": rows_per_rank * world / (ms_max * 1e-3)}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["dsa", "reference"], default="dsa")
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD)
    ap.add_argument("--splits", type=int, default=None, help="override the top-k split count")
    ap.add_argument("--kv-layout", choices=["interleaved", "separate"], default="interleaved",
                    help="K/V cache layout: one [pages, P, 2, Hkv, D] cache (default) or two [pages, P, Hkv, D]")
    ap.add_argument("--score-buffer-bytes", type=int, default=0,
                    help="score-buffer budget: the indexer and top-k run in row windows that fit it (0: one window)")
    ap.add_argument("--batch", type=int, default=None,
                    help="fewer decode requests (profiling captures only; the bench line uses the full batch)")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--flush", action="store_true",
                    help="also write a 256 MiB buffer between timed steps (outside the timed events); "
                         "not needed when a step streams far more than L2")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill-groups", action="store_true",
                    help="every row takes the per-row attention (DSA_FLAG_NO_PREFILL_GROUPS)")
    ap.add_argument("--other-workloads", default="3,4",
                    help="workloads also timed after the headline (comma list, '' for none); "
                         "their numbers go to the line's 'workloads' object")
    ap.add_argument("--cpu-baseline-worker", default=None, help=argparse.SUPPRESS)
    return ap.parse_args()


# ----------------------------------------------------------------------------
# workload description and algorithmic bytes
# ----------------------------------------------------------------------------
def score_windows_note(cfg) -> str:
    from sparse_attention_decode_paged_gb300 import dsa
    wr, nw = dsa.dsa_score_windows(cfg)
    return (f"score buffer budget {cfg.score_buffer_bytes} B: indexer and top-k over {nw} row windows of "
            f"{wr} rows ({wr * cfg.score_width * 4 / 2**20:.1f} MiB of scores)")


def describe(wl, cfg, step_bytes, flush=False) -> dict:
    kd = "fp8 e4m3 + fp32 per-token scale" if wl.idx_key_dtype else "bf16"
    return {
        "workload": f"{wl.name}: {wl.kind} step, {wl.max_rows} row slots, indexer {wl.idx_heads}x{wl.idx_dim} {kd}, "
                    f"page {wl.page_size}, top-k {wl.topk}, {wl.num_q_heads}q/{wl.num_kv_heads}kv heads, "
                    f"head dim {wl.head_dim} bf16",
        "batch": int(wl.max_reqs), "score_width": int(wl.score_width), "topk": int(wl.topk),
        "page_size": int(wl.page_size), "num_splits": int(cfg.num_splits),
        "kv_layout": ("interleaved: one cache [pages, P, 2, Hkv, D], a token's K row then its V row"
                      if cfg.flags & 2 else "separate K and V caches [pages, P, Hkv, D]"),
        **({"score_windows": score_windows_note(cfg)} if cfg.score_buffer_bytes else {}),
        "l2": f"inputs larger than L2: each step streams {step_bytes / 2**20:.0f} MiB of index keys and K/V "
              f"({step_bytes / 129e6:.1f}x the 129 MB L2)"
              + ("; plus a 256 MiB L2 flush between steps" if flush else ""),
        "timing": ("one CUDA-graph replay of dsa_step per step between CUDA events, the L2 flush outside them"
                   if flush else
                   "K CUDA-graph replays of dsa_step back to back between two CUDA events on the replay "
                   "stream, divided by K")
                  + "; the per-kernel table comes from a second loop over the same four launches with event "
                    "nodes between them",
    }


def algorithmic_bytes(wl, rows) -> dict:
    key_b = wl.idx_dim * (1 if wl.idx_key_dtype else 2) + (4 if wl.idx_key_dtype else 0)
    idx = 0
    for b in range(rows["num_blocks"]):
        f, n = int(rows["block_first"][b]), int(rows["block_nrows"][b])
        idx += int(max(rows["row_len"][f:f + n])) * key_b
    kv = sum(min(wl.topk, int(L)) for L in rows["row_len"][:rows["num_rows"]]) * wl.num_kv_heads * wl.head_dim * 2 * 2
    return {"indexer": idx, "sparse_attn": kv, "step": idx + kv}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def traffic_record(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it still
    describes the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    rec = d.get(kernel)
    if not rec or rec.get("source") != KERNEL_SOURCE.get(kernel):
        return None
    from sparse_attention_decode_paged_gb300 import build as B
    src = os.path.join(B.CSRC, rec["source"])
    import hashlib
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()
    if h != rec.get("source_sha256"):
        return None
    return rec["dram_bytes_per_launch"]


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.t_on = self.t_off = None
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["--id=GPU-" + uuid] if uuid else []
        except Exception:
            sel = []
        self.cmd = ["nvidia-smi"] + sel + ["--query-gpu=" + self.FIELDS,
                                           "--format=csv,noheader,nounits", "-lms", "100"]

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, on: bool):
        if on:
            self.t_on = time.time()
        else:
            self.t_off = time.time()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)
        rows = []
        for t, line in self.samples:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                rows.append((t, float(parts[2]), float(parts[3]), parts[5:]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t_on and self.t_off and self.t_on <= r[0] <= self.t_off + 0.1]
        window = "timed"
        if not inside:
            inside, window = rows, "timed+warmup"
        if not inside:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names, r[3][1:5]):
                if v.strip().lower() in ("active", "1", "yes"):
                    reasons.add(n)
        return {"sm_mhz": float(statistics.median(r[1] for r in inside)),
                "sm_max_mhz": float(max(r[2] for r in inside)),
                "reasons": sorted(reasons), "samples": len(inside), "window": window}


# ----------------------------------------------------------------------------
# CPU oracle on a bounded sample (cpu_baseline and the reference arm)
#
# Both arms measure the oracle through measure_cpu_oracle, with the same
# sample, pass counts and statistic.  A sample is a few rows of the step
# spread over its length mix; each pass runs the oracle's whole step (rows,
# indexer, top-k, attention) over them, either in one process held to one
# thread or in one process per core, each with one thread and its share of
# the rows.  A pass's time scales to the step by the step's total keys over
# the sample's (the indexer's work is linear in the row length).
# ----------------------------------------------------------------------------
_BLAS_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def host_cpu() -> dict:
    """The host the oracle runs on: logical CPUs, the ones this process may
    use, and the CPU model (lscpu, else /proc/cpuinfo)."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
    try:
        usable = len(os.sched_getaffinity(0))
    except AttributeError:
        usable = os.cpu_count() or 1
    return {"cpu_count": os.cpu_count(), "usable_cpus": usable, "cpu_model": model,
            "machine": platform.machine()}


def sample_rows(row_len, num_rows: int, nrows: int) -> list:
    """nrows rows spread over the step's length mix: the non-pad rows sorted
    by length, one taken from the middle of each of nrows equal slices."""
    order = sorted((r for r in range(num_rows) if row_len[r] > 0), key=lambda r: (int(row_len[r]), r))
    n = len(order)
    if n == 0:
        return []
    m = min(nrows, n)
    return sorted(order[(2 * j + 1) * n // (2 * m)] for j in range(m))


def cpu_sample(inp, rows, picks):
    """The picked rows as a problem of their own: each becomes a one-token
    request whose cache length is the row's length, with its request's page
    table row (cut at the row's length) and its own q_idx, w and q rows; the
    pages those rows reach are compacted into a small pool.  The oracle's
    work on it is its work on those rows in the full step."""
    import dataclasses
    wl = inp["workload"]
    picks = np.asarray(picks, np.int64)
    lens = rows["row_len"][picks].astype(np.int32)
    pt = np.asarray(inp["page_table"])[rows["row_req"][picks]]
    npg = (lens + wl.page_size - 1) // wl.page_size
    pt = np.where(np.arange(pt.shape[1])[None, :] < npg[:, None], pt, -1)
    used = np.unique(pt[pt >= 0])
    remap = np.full(inp["num_pages"], -1, np.int32)
    remap[used] = np.arange(used.size, dtype=np.int32)
    sub_pt = np.where(pt >= 0, remap[np.maximum(pt, 0)], -1).astype(np.int32)
    sub_wl = dataclasses.replace(wl, max_rows=len(picks), max_reqs=len(picks), block_rows=1)
    arrays = dict(cache_len=lens, new_tokens=np.ones(len(picks), np.int32), page_table=sub_pt,
                  q_idx=inp["q_idx"][picks], w=inp["w"][picks], idx_cache=inp["idx_cache"][used],
                  q=inp["q"][picks], k_cache=inp["k_cache"][used], v_cache=inp["v_cache"][used])
    if inp["idx_scale"] is not None:
        arrays["idx_scale"] = inp["idx_scale"][used]
    return sub_wl, arrays


def _oracle_problem(meta, arrays, idx):
    """Rows idx of a saved sample as an oracle input (the caches shared)."""
    import dataclasses
    from sparse_attention_decode_paged_gb300 import workloads as W
    wl = dataclasses.replace(W.workload(meta["workload"]), max_rows=len(idx), max_reqs=len(idx), block_rows=1)
    inp = {k: (v if k in ("idx_cache", "idx_scale", "k_cache", "v_cache") else np.ascontiguousarray(v[idx]))
           for k, v in arrays.items()}
    inp["workload"] = wl
    inp.setdefault("idx_scale", None)
    inp["num_pages"] = int(arrays["idx_cache"].shape[0])
    return inp


def _load_sample(path):
    with open(os.path.join(path, "meta.json")) as f:
        meta = json.load(f)
    arrays = {k: np.load(os.path.join(path, k + ".npy"), mmap_mode="r") for k in meta["arrays"]}
    return meta, arrays


def _oracle_proc(path, idx, passes, barrier, q):
    """One process of an all-cores pass: its rows, one thread, in step with
    the others at every pass."""
    from oracle import dsa_oracle as O
    meta, arrays = _load_sample(path)
    inp = _oracle_problem(meta, arrays, np.asarray(idx))
    times = []
    for _ in range(passes):
        barrier.wait()
        t0 = time.perf_counter()
        O.step(inp)
        times.append(time.perf_counter() - t0)
    q.put(times)


def cpu_oracle_worker(path: str):
    """Runs in a child process whose BLAS / OpenMP pools hold one thread;
    prints the seconds of each pass (warm-up passes included)."""
    meta, arrays = _load_sample(path)
    procs, passes = meta["procs"], meta["passes"]
    n = int(arrays["cache_len"].shape[0])
    if procs <= 1:
        from oracle import dsa_oracle as O
        inp = _oracle_problem(meta, arrays, np.arange(n))
        times = []
        for _ in range(passes):
            t0 = time.perf_counter()
            O.step(inp)
            times.append(time.perf_counter() - t0)
    else:
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        barrier, q = ctx.Barrier(procs), ctx.Queue()
        # rows dealt out longest first so every process gets a like share
        order = sorted(range(n), key=lambda r: -int(arrays["cache_len"][r]))
        groups = [order[p::procs] for p in range(procs)]
        ps = [ctx.Process(target=_oracle_proc, args=(path, g, passes, barrier, q)) for g in groups if g]
        for p in ps:
            p.start()
        per = [q.get(timeout=900) for _ in ps]
        for p in ps:
            p.join(timeout=60)
        times = [max(t[i] for t in per) for i in range(passes)]  # a pass ends with its slowest process
    print(json.dumps({"times": times}))


def measure_cpu_oracle(inp, rows, wl_index: int, procs: int, nrows: int, passes: int, warmup: int) -> dict:
    """Seconds per step of the CPU oracle: `warmup` + `passes` passes over a
    sample of nrows rows in `procs` one-thread processes (child processes, so
    nothing in this process competes with them); the fastest timed pass (the
    host is shared, and the median of the passes moved by up to ~20% between
    runs; the fastest pass is the least disturbed), scaled by the step's keys
    over the sample's."""
    picks = sample_rows(rows["row_len"], rows["num_rows"], nrows)
    sub_wl, arrays = cpu_sample(inp, rows, picks)
    keys_all = int(np.sum(rows["row_len"][:rows["num_rows"]]))
    keys_sample = int(np.sum(arrays["cache_len"]))
    procs = max(1, min(procs, len(picks)))
    with tempfile.TemporaryDirectory() as td:
        for k, v in arrays.items():
            np.save(os.path.join(td, k + ".npy"), np.ascontiguousarray(v))
        with open(os.path.join(td, "meta.json"), "w") as f:
            json.dump({"workload": wl_index, "procs": procs, "passes": warmup + passes,
                       "arrays": sorted(arrays)}, f)
        env = dict(os.environ)
        for v in _BLAS_VARS:
            env[v] = "1"
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-worker", td],
                           capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(r.stderr.strip()[-300:])
    times = json.loads(r.stdout.strip().splitlines()[-1])["times"][warmup:]
    scale = keys_all / keys_sample
    return {"s_per_step": min(times) * scale, "times": times, "procs": procs, "rows": picks,
            "scale": scale, "keys_all": keys_all, "keys_sample": keys_sample}


def cpu_baseline_record(m1: dict, mall: dict | None, num_rows: int, host: dict) -> dict:
    """The cpu_baseline object: the all-cores figure when there is one (the
    oracle on the host's cores), with the one-thread figure beside it."""
    def desc(m):
        return (f"{len(m['rows'])} of {num_rows} rows per pass (rows {m['rows']}, spread over the length mix), "
                f"{m['procs']} one-thread process(es), the fastest of {len(m['times'])} timed passes, scaled to the "
                f"step by its keys over the sample's ({m['keys_all']}/{m['keys_sample']} = {m['scale']:.3g}); "
                f"fp64 numpy oracle, whole step (indexer, top-k, attention)")
    main = mall if mall is not None else m1
    rec = {"value": main["s_per_step"] * 1e6, "unit": "us", "cores": main["procs"], "threads": main["procs"],
           "kind": "oracle", "sample": desc(main), **host,
           "one_thread": {"value": m1["s_per_step"] * 1e6, "unit": "us", "threads": 1, "sample": desc(m1)}}
    return rec


CPU_ONE_THREAD_ROWS = 2  # rows per one-thread pass
CPU_PASSES, CPU_WARMUP = 6, 1


def run_cpu_baseline(inp, rows, wl_index: int, host: dict) -> dict:
    m1 = measure_cpu_oracle(inp, rows, wl_index, 1, CPU_ONE_THREAD_ROWS, CPU_PASSES, CPU_WARMUP)
    procs = host["usable_cpus"]
    mall = None
    if procs > 1:
        mall = measure_cpu_oracle(inp, rows, wl_index, procs, procs, CPU_PASSES, CPU_WARMUP)
    return cpu_baseline_record(m1, mall, rows["num_rows"], host)


# ----------------------------------------------------------------------------
# the reference arm: the CPU oracle, timed on the host
# ----------------------------------------------------------------------------
def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from sparse_attention_decode_paged_gb300 import workloads as W
    inp = W.generate(args.workload)
    wl = inp["workload"]
    from oracle import dsa_oracle as O
    rows = O.build_rows(inp["cache_len"], inp["new_tokens"], wl.max_rows, wl.block_rows)
    host = host_cpu()
    t0 = time.perf_counter()
    # one step = one all-cores pass over a sample of the step (one row per
    # process), scaled to the step; the one-thread figure beside it
    procs = host["usable_cpus"]
    mall = measure_cpu_oracle(inp, rows, args.workload, procs, procs, max(args.steps, 1), max(args.warmup, 0))
    m1 = measure_cpu_oracle(inp, rows, args.workload, 1, CPU_ONE_THREAD_ROWS, CPU_PASSES, CPU_WARMUP)
    wall = time.perf_counter() - t0
    cpu = cpu_baseline_record(m1, mall if procs > 1 else None, rows["num_rows"], host)
    us = cpu["value"]
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": "us", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.name} (CPU oracle on a bounded sample)", "batch": int(wl.max_reqs),
                   "score_width": int(wl.score_width), "topk": int(wl.topk)},
        "cpu_baseline": cpu,
        "e2e": {"value": us, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "timing_note": ("ms_per_step is a sampled pass scaled to the whole step (see cpu_baseline.sample); "
                        "the run's wall time covers the sampled passes only"),
        "wall_s": wall,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# the CUDA path
# ----------------------------------------------------------------------------
def run_dsa(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)

    from sparse_attention_decode_paged_gb300 import build as B
    B.build()
    from sparse_attention_decode_paged_gb300 import dsa
    from sparse_attention_decode_paged_gb300 import workloads as W
    from sparse_attention_decode_paged_gb300.harness import DeviceStep

    t_gen = time.time()
    wl0 = W.workload(args.workload)
    if args.batch:
        import dataclasses
        wl0 = dataclasses.replace(wl0, max_rows=args.batch, max_reqs=args.batch)
    inp = W.generate(wl0)
    wl = inp["workload"]
    override = {"num_splits": args.splits} if args.splits else {}
    # the per-kernel calls below mirror dsa_step, which hands the indexer's
    # key histogram to the top-k
    override["flags"] = dsa.DSA_FLAG_TOPK_HISTOGRAM
    if args.kv_layout == "interleaved":  # a token's K and V rows adjacent: one copy per selected token
        override["flags"] |= dsa.DSA_FLAG_KV_INTERLEAVED
    if args.no_prefill_groups:
        override["flags"] |= dsa.DSA_FLAG_NO_PREFILL_GROUPS
    if args.score_buffer_bytes:
        override["score_buffer_bytes"] = args.score_buffer_bytes
    dev = DeviceStep(inp, **override)
    cfg, t, v = dev.cfg, dev.t, dev.views
    gen_s = time.time() - t_gen
    nbytes = algorithmic_bytes(wl, dev.rows)
    # the CPU oracle first, while this process and the GPU are idle (the
    # children it runs in then share the host with nothing of ours)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            cpu = run_cpu_baseline(inp, dev.rows, args.workload, host_cpu())
        except Exception as exc:  # report, do not fail the GPU measurement
            cpu = {"error": repr(exc)[:300]}

    stream = torch.cuda.Stream()
    # the launches dsa_step makes: indexer and top-k once per score window
    # (one window without a budget), then the attention and the merge
    wr, nw = dsa.dsa_score_windows(cfg)
    launches = []
    for lo in range(0, cfg.max_rows, wr):
        win = None if nw == 1 else (lo, min(lo + wr, cfg.max_rows))
        launches.append(("indexer", lambda s, win=win: dsa.dsa_indexer_scores(
            cfg, t["q_idx"], t["w"], t["idx_cache"], t["idx_scale"], t["page_table"], t["row_req"],
            t["row_len"], t["block_first"], t["block_nrows"], v["scores"], dev.workspace, s, window=win)))
        launches.append(("topk", lambda s, win=win: dsa.dsa_topk(
            cfg, v["scores"], t["row_len"], v["topk_idx"], dev.workspace, s, window=win)))
    launches.append(("sparse_attn", lambda s: dsa.dsa_sparse_attn(
        cfg, t["q"], t["k_cache"], t["v_cache"], t["page_table"], t["row_req"], t["row_len"], v["topk_idx"],
        v["part_m"], v["part_l"], v["part_acc"], dev.workspace, s)))
    launches.append(("merge", lambda s: dsa.dsa_merge(
        cfg, v["part_m"], v["part_l"], v["part_acc"], t["out"], t["lse"], s)))
    names = ["indexer", "topk", "sparse_attn", "merge"]
    nev = len(launches) + 1
    try:
        ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(nev)]
        events_in_graph = True
    except TypeError:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(nev)]
        events_in_graph = False

    def kernels(s, record):
        # dsa_step's launches, with event nodes between them
        if record:
            ev[0].record(s)
        for i, (_, fn) in enumerate(launches):
            fn(s)
            if record:
                ev[i + 1].record(s)

    def add_kernel_times(per_kernel):
        # each kernel's time summed over its launches (one per window)
        for n in names:
            per_kernel[names.index(n)].append(
                sum(ev[i].elapsed_time(ev[i + 1]) for i, (m, _) in enumerate(launches) if m == n))

    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        kernels(stream, record=True)  # eager warm-up (also sets kernel attributes)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        kernels(torch.cuda.current_stream(), record=events_in_graph)
    torch.cuda.synchronize()
    # the headline graph: the one dsa_step call a user makes (its launches keep
    # their programmatic-dependency edges, which event nodes would cut)
    step_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(step_graph, stream=stream):
        dsa.dsa_step(cfg, dev.args, dev.workspace, torch.cuda.current_stream())
    torch.cuda.synchronize()
    status = dsa.dsa_read_device_status(dev.workspace)
    flush = torch.empty(FLUSH_BYTES if args.flush else 16, dtype=torch.uint8, device="cuda")
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    sampler = ClockSampler(local)
    sampler.start()
    with torch.cuda.stream(stream):
        for k in range(max(args.warmup, 3)):
            if args.flush:
                flush.fill_(k & 0xFF)
            step_graph.replay()
            graph.replay()
        stream.synchronize()
        status = dsa.dsa_read_device_status(dev.workspace, stream)
        if status:  # a device-side check fired: report it instead of timing a broken step
            sampler.stop()
            print(json.dumps({"metric": METRIC, "error": f"device status 0x{status:x} after warm-up"}), flush=True)
            sys.exit(1)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        sampler.mark(True)
        t_wall = time.perf_counter()
        per_step, per_kernel, per_inst = [], [[] for _ in range(4)], []
        # the headline: K dsa_step graph replays back to back, as a decode
        # loop issues them (each replay's launch overlaps the previous step)
        step_ev[0].record(stream)
        for k in range(args.steps):
            if args.flush:
                flush.fill_(k & 0xFF)
            step_graph.replay()
        step_ev[1].record(stream)
        stream.synchronize()
        ms_back_to_back = step_ev[0].elapsed_time(step_ev[1]) / args.steps  # flushes included when --flush
        wall_s = time.perf_counter() - t_wall
        for k in range(args.steps if args.flush else min(args.steps, 200)):  # one replay at a time
            if args.flush:
                flush.fill_(k & 0xFF)
            step_ev[0].record(stream)
            step_graph.replay()
            step_ev[1].record(stream)
            stream.synchronize()
            per_step.append(step_ev[0].elapsed_time(step_ev[1]))
        torch.cuda.synchronize()
        if events_in_graph:  # the per-kernel breakdown: same launches, event nodes between them
            for k in range(args.steps):
                if args.flush:
                    flush.fill_(k & 0xFF)
                step_ev[0].record(stream)
                graph.replay()
                step_ev[1].record(stream)
                stream.synchronize()
                per_inst.append(step_ev[0].elapsed_time(step_ev[1]))
                add_kernel_times(per_kernel)
        torch.cuda.synchronize()
        sampler.mark(False)
        if world > 1:
            dist.barrier()
    clocks = sampler.stop()

    if not events_in_graph:  # torch without graph event nodes: time the kernels eagerly instead
        with torch.cuda.stream(stream):
            for k in range(max(20, args.steps // 10)):
                if args.flush:
                    flush.fill_(k & 0xFF)
                kernels(stream, record=True)
                stream.synchronize()
                add_kernel_times(per_kernel)

    # with --flush the flush writes sit between the replays, so the step is
    # timed one replay at a time (events around the replay only)
    ms_step = statistics.mean(per_step) if args.flush else ms_back_to_back
    ms_max = max_over_ranks(ms_step, world)

    k_ms = {n: statistics.mean(x) for n, x in zip(names, per_kernel)}
    per_row_kv = None
    if wl.kind == "mixed":
        # rows of one request (a prefill chunk) share their gathers: the
        # attention's HBM floor is the distinct K/V rows, per request the
        # union of its rows' selections; the per-row gathers beyond it are
        # reported beside it (served by L2)
        per_row_kv = nbytes["sparse_attn"]
        union = union_kv_bytes(wl, dev.rows, v["topk_idx"].cpu().numpy())
        nbytes = {"indexer": nbytes["indexer"], "sparse_attn": union, "step": nbytes["indexer"] + union}
    dominant = max(("indexer", "sparse_attn"), key=lambda n: k_ms[n])
    peak, peak_kind = measured_peaks()
    ach = nbytes[dominant] / (k_ms[dominant] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": dominant, "achieved": ach, "peak": peak, "unit": "GB/s",
                "frac": ach / peak, "traffic": traffic_record(dominant),
                "algorithmic_bytes": nbytes[dominant], "peak_source": f"{peak_kind} copy bandwidth",
                "timing": ("graph event nodes, second timed loop" if events_in_graph
                           else "eager launches, events")}
    step_gbs = nbytes["step"] / (ms_max * 1e-3) / 1e9
    kernel_table = {n: {"us": k_ms[n] * 1e3} for n in names}
    for n in ("indexer", "sparse_attn"):
        kernel_table[n]["algorithmic_bytes"] = nbytes[n]
        kernel_table[n]["gbs"] = nbytes[n] / (k_ms[n] * 1e-3) / 1e9
        kernel_table[n]["frac_of_peak"] = kernel_table[n]["gbs"] / peak
    if per_row_kv is not None:
        roofline["bytes_note"] = ("algorithmic bytes: the distinct K/V rows the step selects (per request, the union "
                                  "of its rows' selections) and the index keys; per-row gathers in the kernel table")
        kernel_table["sparse_attn"]["per_row_gather_bytes"] = per_row_kv
        kernel_table["sparse_attn"]["per_row_gather_gbs"] = per_row_kv / (k_ms["sparse_attn"] * 1e-3) / 1e9

    # ---- end to end through the public API, host buffers
    e2e = run_e2e(args, dsa, dev, inp, stream, flush) if args.e2e_steps > 0 else None
    try:
        probe = run_read_probe(dev, nbytes["indexer"], stream)
    except Exception as exc:  # a measurement aid; report, do not fail the run
        probe = {"error": repr(exc)[:200]}
    kv_probe = None
    if args.kv_layout == "interleaved" and per_row_kv is None:
        try:
            kv_probe = run_read_probe_kv(dev, stream)
        except Exception as exc:
            kv_probe = {"error": repr(exc)[:200]}
        probe = dict(probe, kv_rows=kv_probe)
    if "us" in probe:
        kernel_table["indexer"]["frac_of_read_probe"] = (nbytes["indexer"] / (k_ms["indexer"] * 1e-3) / 1e9) / probe["gbs"]
        # the attention against the same read of its own 4 KiB K/V rows when
        # measured, else against the page read
        ref = kv_probe if kv_probe is not None and "gbs" in kv_probe else probe
        kernel_table["sparse_attn"]["frac_of_read_probe"] = (
            (nbytes["sparse_attn"] / (k_ms["sparse_attn"] * 1e-3) / 1e9) / ref["gbs"])

    others = {}
    wanted = [int(x) for x in args.other_workloads.split(",") if x.strip()] if args.other_workloads else []
    wanted = [i for i in wanted if i != args.workload]
    if wanted and not args.batch and args.score_buffer_bytes == 0 and not args.splits:
        del graph, step_graph
        for i in wanted:
            try:
                others[str(i)] = run_other_workload(i, args, stream, peak)
            except Exception as exc:  # report, do not fail the headline measurement
                others[str(i)] = {"error": repr(exc)[:300]}

    job = whole_job(ms_max, dev.rows["num_rows"], world)  # replicas run concurrently
    us = job["us_per_step"]
    line = {
        "metric": METRIC, "value": us, "unit": "us", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": describe(wl, cfg, nbytes["step"], args.flush),
        "rows_per_s": job["rows_per_s"],
        "hbm_gbs_step": step_gbs, "step_roofline_frac": step_gbs / peak,
        "roofline": roofline, "kernels": kernel_table, "read_probe": probe, "cpu_baseline": cpu, "e2e": e2e,
        "clocks": clocks, "gpu_launches": (2 * nw + 2) * args.steps, "device_status": status,
        "workloads": others or None,
        "isolated_step_us": {"median": statistics.median(per_step) * 1e3, "min": min(per_step) * 1e3,
                             "note": "one replay per synchronize, graph launch latency included"},
        "wall_s": wall_s, "setup_s": gen_s,
        "instrumented_step_us": statistics.mean(per_inst) * 1e3 if per_inst else None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def union_kv_bytes(wl, rows, topk_idx) -> int:
    """Bytes of the distinct K/V rows the step selects: per request, the
    union of its rows' selected positions (what an HBM floor counts when the
    rows of one request share their gathers, e.g. a prefill chunk's)."""
    per_tok = wl.num_kv_heads * wl.head_dim * 2 * 2
    total = 0
    req = rows["row_req"][:rows["num_rows"]]
    for b in np.unique(req):
        sel = topk_idx[:rows["num_rows"]][req == b]
        total += np.unique(sel[sel >= 0]).size * per_tok
    return int(total)


def run_other_workload(i: int, args, stream, peak: float) -> dict:
    """One more workload's dsa_step graph, timed like the headline: K replays
    back to back between CUDA events (inputs larger than L2), and also one
    replay at a time after a 256 MiB L2 flush (median); the roofline against
    the step's algorithmic bytes, and for steps whose rows share requests
    (prefill) also against the distinct K/V rows the step gathers."""
    import torch
    from sparse_attention_decode_paged_gb300 import dsa
    from sparse_attention_decode_paged_gb300 import workloads as W
    from sparse_attention_decode_paged_gb300.harness import DeviceStep
    inp = W.generate(i)
    wl = inp["workload"]
    flags = dsa.DSA_FLAG_TOPK_HISTOGRAM
    if args.kv_layout == "interleaved":
        flags |= dsa.DSA_FLAG_KV_INTERLEAVED
    dev = DeviceStep(inp, flags=flags)
    cfg = dev.cfg
    nbytes = algorithmic_bytes(wl, dev.rows)
    g = dev.capture(stream)
    status = dsa.dsa_read_device_status(dev.workspace, stream)
    union = union_kv_bytes(wl, dev.rows, dev.views["topk_idx"].cpu().numpy())
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    steps = max(1, min(args.steps, 200))
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            g.replay()
        stream.synchronize()
        ev[0].record(stream)
        for _ in range(steps):
            g.replay()
        ev[1].record(stream)
        stream.synchronize()
        us = ev[0].elapsed_time(ev[1]) / steps * 1e3
        cold = []
        for k in range(min(steps, 50)):
            flush.fill_(k & 0xFF)
            ev[0].record(stream)
            g.replay()
            ev[1].record(stream)
            stream.synchronize()
            cold.append(ev[0].elapsed_time(ev[1]) * 1e3)
    status = status or dsa.dsa_read_device_status(dev.workspace, stream)
    rec = {"name": wl.name, "us": us, "us_cold_l2": statistics.median(cold), "steps": steps,
           "rows": int(dev.rows["num_rows"]), "row_slots": int(cfg.max_rows), "num_splits": int(cfg.num_splits),
           "algorithmic_bytes": nbytes["step"], "indexer_bytes": nbytes["indexer"],
           "kv_gather_bytes": nbytes["sparse_attn"],
           "gbs": nbytes["step"] / (us * 1e-6) / 1e9, "frac": nbytes["step"] / (us * 1e-6) / 1e9 / peak,
           "device_status": status,
           "timing": "dsa_step graph: back-to-back replays between CUDA events (us); one replay per "
                     "synchronize after a 256 MiB L2 flush, median (us_cold_l2)"}
    if union != nbytes["sparse_attn"]:
        # rows of one request share their gathers: the roofline counts the
        # distinct K/V rows (per request, the union of its rows' selections);
        # the per-row gather rate is reported beside it (served by L2)
        hbm = nbytes["indexer"] + union
        rec.update({"algorithmic_bytes": hbm, "kv_gather_bytes": union,
                    "gbs": hbm / (us * 1e-6) / 1e9, "frac": hbm / (us * 1e-6) / 1e9 / peak,
                    "bytes_note": "index keys + the distinct K/V rows the step selects (per request, the union of "
                                  "its rows' selections); the per-row gathers beyond it are served by L2",
                    "per_row_gather_bytes": nbytes["sparse_attn"],
                    "per_row_gbs": (nbytes["indexer"] + nbytes["sparse_attn"]) / (us * 1e-6) / 1e9})
    del dev, g
    torch.cuda.empty_cache()
    return rec


def _probe_reads(base_ptr, order, page_bytes, stream, reps=25):
    """Median µs of CUDA-event-timed launches of the plain read probe over
    `order` (device int32 chunk indices) chunks of `page_bytes` from base."""
    import ctypes
    import torch
    from sparse_attention_decode_paged_gb300 import build as B
    lib = ctypes.CDLL(B.PROBE_LIB)
    lib.dsa_probe_read_pages.restype = ctypes.c_int
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sink = torch.empty(16 * sms * 256 // 32, dtype=torch.int32, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    times = []
    for _ in range(reps):
        ev[0].record(stream)
        rc = lib.dsa_probe_read_pages(ctypes.c_void_p(base_ptr), ctypes.c_void_p(order.data_ptr()), int(order.numel()),
                                      page_bytes, ctypes.c_void_p(sink.data_ptr()), 16, 256,
                                      ctypes.c_void_p(stream.cuda_stream))
        ev[1].record(stream)
        stream.synchronize()
        if rc != 0:
            raise RuntimeError(f"cuda error {rc}")
        times.append(ev[0].elapsed_time(ev[1]))
    return statistics.median(times[5:]) * 1e3


def run_read_probe_kv(dev, stream):
    """The same plain read over the K/V rows the step's attention gathers: one
    4 KiB interleaved K/V row per selected token (the step's own selection),
    row after row in selection order."""
    import torch
    wl = dev.inp["workload"]
    nr = int(dev.rows["num_rows"])
    idx = dev.views["topk_idx"][:nr]
    req = dev.t["row_req"][:nr].long()
    P = wl.page_size
    pos = idx.clamp(min=0).long()
    tok = dev.t["page_table"].long()[req[:, None], pos // P] * P + pos % P
    order = tok[idx >= 0].to(torch.int32).contiguous()
    row_bytes = 2 * wl.num_kv_heads * wl.head_dim * 2
    t_us = _probe_reads(dev.t["k_cache"].data_ptr(), order, row_bytes, stream)
    nbytes = int(order.numel()) * row_bytes
    return {"bytes": nbytes, "us": t_us, "gbs": nbytes / (t_us * 1e-6) / 1e9,
            "what": "plain read of the attention's selected K/V rows (4 KiB each, interleaved cache) in selection "
                    "order, 16-byte loads, 16x256 threads per SM, median of CUDA-event-timed launches"}


def run_read_probe(dev, nbytes_idx, stream, reps=25):
    """A plain read of the pages the step's indexer streams (page-table order,
    16-byte loads, 16 x 256 threads per SM, no shared memory): the read-only
    stream rate this GPU reaches on those bytes, timed like the kernels (CUDA
    events around one launch, median)."""
    import ctypes
    import torch
    from sparse_attention_decode_paged_gb300 import build as B
    lib = ctypes.CDLL(B.PROBE_LIB)
    lib.dsa_probe_read_pages.restype = ctypes.c_int
    wl = dev.inp["workload"]
    page_bytes = wl.page_size * wl.idx_dim * (1 if wl.idx_key_dtype else 2)
    pt = dev.t["page_table"].flatten()
    pt = pt[pt >= 0]
    npages = int(min(pt.numel(), max(1, nbytes_idx // page_bytes)))
    order = pt[:npages].to(torch.int32).contiguous()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sink = torch.empty(16 * sms * 256 // 32, dtype=torch.int32, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    times = []
    for _ in range(reps):
        ev[0].record(stream)
        rc = lib.dsa_probe_read_pages(ctypes.c_void_p(dev.t["idx_cache"].data_ptr()), ctypes.c_void_p(order.data_ptr()),
                                      npages, page_bytes, ctypes.c_void_p(sink.data_ptr()), 16, 256,
                                      ctypes.c_void_p(stream.cuda_stream))
        ev[1].record(stream)
        stream.synchronize()
        if rc != 0:
            return {"error": f"cuda error {rc}"}
        times.append(ev[0].elapsed_time(ev[1]))
    t_us = statistics.median(times[5:]) * 1e3
    nbytes = npages * page_bytes
    return {"bytes": nbytes, "us": t_us, "gbs": nbytes / (t_us * 1e-6) / 1e9,
            "what": "plain read of the indexer's key pages in page-table order, 16-byte loads, "
                    "16x256 threads per SM, median of CUDA-event-timed launches"}


def run_e2e(args, dsa, dev, inp, stream, flush):
    """µs per step through the public API with host buffers: per step the rows
    are built on the host (dsa_build_rows, straight into the pinned staging
    copy of the device input arena), then one CUDA graph copies that arena
    (row maps, page table, q_idx, w, q) host -> device in one copy, runs
    dsa_step and copies the output arena (out, lse) back in one copy (the way
    a serving loop replays a captured step), and the host waits for it.  The
    same sequence issued eagerly is reported too."""
    import torch
    from sparse_attention_decode_paged_gb300.harness import DEVICE_ROW_KEYS
    cfg, R = dev.cfg, dev.cfg.max_rows
    h_in = dev.inputs.cpu().pin_memory()  # this step's inputs, staged on the host
    h_out = torch.empty_like(dev.outputs, device="cpu").pin_memory()
    # host views of the staged row maps (same offsets as the device arena)
    staged = {k: h_in[dev.t[k].data_ptr() - dev.inputs.data_ptr():][:4 * R].view(torch.int32)
              for k in DEVICE_ROW_KEYS}
    staged["row_pos"] = torch.empty(R, dtype=torch.int32)  # not needed on the device
    h2d, d2h = dev.inputs.numel(), dev.outputs.numel()
    cache_len = np.ascontiguousarray(inp["cache_len"], dtype=np.int32)
    new_tokens = np.ascontiguousarray(inp["new_tokens"], dtype=np.int32)

    def host_rows():
        dsa.dsa_build_rows(cfg, cache_len, new_tokens, out=staged)

    def device_part(s):
        dev.inputs.copy_(h_in, non_blocking=True)
        dsa.dsa_step(cfg, dev.args, dev.workspace, s)
        h_out.copy_(dev.outputs, non_blocking=True)

    with torch.cuda.stream(stream):
        host_rows()
        device_part(stream)  # warm-up
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            device_part(torch.cuda.current_stream())
        stream.synchronize()
        times, eager, host_t, dev_t = [], [], [], []
        ge = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        for k in range(args.e2e_steps + 3):
            if args.flush:
                flush.fill_(k & 0xFF)
            stream.synchronize()
            t0 = time.perf_counter()
            host_rows()
            t1 = time.perf_counter()
            ge[0].record(stream)
            graph.replay()
            ge[1].record(stream)
            stream.synchronize()
            if k >= 3:
                times.append(time.perf_counter() - t0)
                host_t.append(t1 - t0)
                dev_t.append(ge[0].elapsed_time(ge[1]) * 1e-3)
        # where the device time goes: the same three operations issued
        # eagerly with events between them
        pe = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        parts = {"h2d": [], "step": [], "d2h": []}
        for k in range(min(args.e2e_steps, 20) + 3):
            stream.synchronize()
            pe[0].record(stream)
            dev.inputs.copy_(h_in, non_blocking=True)
            pe[1].record(stream)
            dsa.dsa_step(cfg, dev.args, dev.workspace, stream)
            pe[2].record(stream)
            h_out.copy_(dev.outputs, non_blocking=True)
            pe[3].record(stream)
            stream.synchronize()
            if k >= 3:
                for i, n in enumerate(("h2d", "step", "d2h")):
                    parts[n].append(pe[i].elapsed_time(pe[i + 1]) * 1e3)
        for k in range(args.e2e_steps + 3):
            if args.flush:
                flush.fill_(k & 0xFF)
            stream.synchronize()
            t0 = time.perf_counter()
            host_rows()
            device_part(stream)
            stream.synchronize()
            if k >= 3:
                eager.append(time.perf_counter() - t0)
    wall, host_us, dev_us = statistics.median(times) * 1e6, statistics.median(host_t) * 1e6, statistics.median(dev_t) * 1e6
    return {"value": wall, "unit": "us", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": len(times),
            "eager_us": statistics.median(eager) * 1e6,
            "split_us": {"host_rows": host_us, "graph_on_device": dev_us,
                         "launch_and_wait": wall - host_us - dev_us,
                         "h2d_eager": statistics.median(parts["h2d"]), "step_eager": statistics.median(parts["step"]),
                         "d2h_eager": statistics.median(parts["d2h"]),
                         "note": "medians: host_rows = dsa_build_rows into pinned staging (host clock); "
                                 "graph_on_device = CUDA events around the graph replay (H2D + step + D2H); "
                                 "launch_and_wait = the rest of the wall time (graph launch, host wait); the "
                                 "*_eager parts time the three operations one by one"},
            "path": "dsa_build_rows into the pinned input staging + one CUDA-graph replay of (one H2D copy of "
                    "the input arena, dsa_step, one D2H copy of the output arena) + host wait, wall clock "
                    "median; eager_us: the same calls issued eagerly"}


def main():
    args = parse_args()
    if args.cpu_baseline_worker:
        cpu_oracle_worker(args.cpu_baseline_worker)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_dsa(args)


if __name__ == "__main__":
    main()
