"""Benchmark of the low-bit dual-path MLA decode hot path on one GB300 (one JSON line).

A step is one decode step of one layer: the fused writer appends one token to every sequence
of the layer's cache, then decode attention reads the whole cache (packed pages + BF16
protected tokens) for every head. Steps rotate over several layer caches whose total size is
several times the L2 cache, so every step streams its cache from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

--impl reference times the fp64 CPU oracle (the reference arm of this build) on the host.
Under torchrun (N > 1) every rank runs an independent replica over its own sequences (the path
shards by sequence with no exchange); the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "decode attn µs/layer and packed-cache HBM GB/s (fraction of 8 TB/s) on 1 GB300"
DEFAULT_WORKLOAD = "v2lite_c4r4_b32_h16_t8k"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--layers", type=int, default=0, help="layer caches rotated (0 = enough for 3x L2)")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra-workloads", default="auto",
                    help="other workloads measured in the same run ('auto': the target configurations when the "
                         "default workload runs; 'none'; or a comma-separated list)")
    ap.add_argument("--sweep", action="store_true",
                    help="latency sweep: C4R4 decode against the BF16 paged comparator over 1K..1M tokens")
    ap.add_argument("--sweep-batches", default="1,8,32")
    ap.add_argument("--sweep-heads", type=int, default=16)
    ap.add_argument("--sweep-max-tokens", type=int, default=1 << 20)
    ap.add_argument("--multi", action="store_true",
                    help="multi-token decode: q_len new tokens per sequence in one call")
    ap.add_argument("--proj", action="store_true",
                    help="projections either side of attention: query absorption and W_UV up-projection")
    ap.add_argument("--record-traffic", metavar="NCU_CSV",
                    help="write profiles/traffic_<workload>.json from an ncu --csv log of dram__bytes_read.sum and "
                         "dram__bytes_write.sum (no GPU needed)")
    ap.add_argument("--traffic-kernel", default=None, help="kernel-name regex for --record-traffic")
    ap.add_argument("--traffic-command", default="", help="the ncu command that wrote the log (recorded)")
    ap.add_argument("--transform", action="store_true",
                    help="per-layer cost of the latent transform A_c: standalone kernel vs fused in the writer")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_sequences(batch: int, rank: int, world: int) -> range:
    """Global sequence ids owned by a rank of a replicas-only job: every rank serves its own
    batch of sequences (weak scaling), rank r the ids [r*batch, (r+1)*batch)."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    return range(rank * batch, (rank + 1) * batch)


def replica_workload(w: workloads.Workload, rank: int) -> workloads.Workload:
    """The workload a rank serves: its own sequences, drawn from a seed of its own (rank 0
    serves exactly the single-GPU workload)."""
    return dataclasses.replace(w, seed=w.seed + 1000 * rank) if rank else w


def max_over_ranks(value: float, device=None) -> float:
    """Replicas only: the job's time is the slowest rank's (all ranks hold identical work)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ algorithmic work per step

def decode_bytes(w: workloads.Workload, seq_lens, heads) -> int:
    """Bytes the method must move per decode call: packed copies of unprotected tokens
    (codes + per-token group metadata + per-page k_R metadata), BF16 rows of protected tokens,
    the queries and the outputs."""
    P, S, W = w.page_size, w.n_sink, w.n_recent
    per_tok = 64 * w.bits_c + 32 + 16  # latent codes + k_R codes + latent metadata
    total = 0
    for T in seq_lens:
        T = int(T)
        prot = min(T, S) + max(0, T - max(T - W, min(T, S)))
        packed = T - prot
        pages = math.ceil(max(T - W, 0) / P) if packed else 0
        total += packed * per_tok + pages * 256 + prot * 576 * 2
    B = len(seq_lens)
    total += B * heads * 576 * 2 + B * heads * (512 + 1) * 4
    return total


def decode_flops(seq_lens, heads) -> int:
    return int(sum(int(T) for T in seq_lens)) * heads * 2 * (576 + 512)


def peaks():
    """(HBM GB/s, dense 16-bit tensor TFLOP/s burst, which): the measured copy bandwidth and
    bf16 GEMM rate of this GPU pool (FP16 and BF16 share the dense tensor rate)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def dominant_kernel_regex(w: workloads.Workload) -> str:
    """Name pattern of the kernel that carries the decode's packed-page stream."""
    return r"decode_tc_kernel" if w.heads % 64 == 0 else r"decode_kernel"


# the sources each decode kernel is compiled from: a kernel's recorded DRAM traffic holds while
# these are unchanged
KERNEL_SOURCES = {"decode_kernel": ("decode.cu", "kernels.cuh", "ptx.cuh"),
                  "decode_tc_kernel": ("decode_tc.cu", "kernels.cuh", "ptx.cuh")}


def source_sha(kernel_regex: str) -> str:
    """Hash of the sources of the kernel that kernel_regex names."""
    files = KERNEL_SOURCES["decode_tc_kernel" if "decode_tc" in kernel_regex else "decode_kernel"]
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_mla_kv_qcache_gb300", "csrc")
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def traffic_path(workload: str) -> str:
    return os.path.join(ROOT, "profiles", f"traffic_{workload}.json")


def profiled_traffic(workload: str):
    """DRAM bytes (read + write) per launch of the dominant decode kernel, from the record that
    ``--record-traffic`` wrote out of an ncu CSV, if it was taken on the current kernel sources
    (else None)."""
    path = traffic_path(workload)
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    if rec.get("source_sha") != source_sha(rec.get("kernel_regex", "")):
        return None
    return float(rec["dram_bytes_per_launch"])


_BYTE_UNITS = {"byte": 1.0, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9, "tbyte": 1e12,
               "b": 1.0, "kb": 1e3, "mb": 1e6, "gb": 1e9, "kib": 1024.0, "mib": 1024.0 ** 2, "gib": 1024.0 ** 3}


def ncu_dram_bytes(csv_path: str, kernel_regex: str):
    """Per-launch dram__bytes_read.sum + dram__bytes_write.sum of the launches whose kernel name
    matches kernel_regex, from an ncu ``--csv`` metrics log (one row per launch and metric)."""
    import csv
    rows = []
    with open(csv_path, newline="") as f:
        lines = [ln for ln in f if ln.startswith('"')]  # ncu's own log lines are not CSV rows
    reader = csv.DictReader(lines)
    per = {}
    for r in reader:
        name, metric = r.get("Kernel Name", ""), r.get("Metric Name", "")
        if metric not in ("dram__bytes_read.sum", "dram__bytes_write.sum") or not re.search(kernel_regex, name):
            continue
        unit = r.get("Metric Unit", "byte").strip().lower()
        val = float(r["Metric Value"].replace(",", "")) * _BYTE_UNITS[unit]
        d = per.setdefault(r["ID"], {"kernel": name})
        d[metric] = val
    for launch_id, d in per.items():
        if "dram__bytes_read.sum" in d and "dram__bytes_write.sum" in d:
            rows.append((launch_id, d["kernel"], d["dram__bytes_read.sum"], d["dram__bytes_write.sum"]))
    if not rows:
        raise RuntimeError(f"no launch of a kernel matching {kernel_regex!r} with both DRAM metrics in {csv_path}")
    return rows


def record_traffic(csv_path: str, workload: str, kernel_regex: str, command: str) -> dict:
    rows = ncu_dram_bytes(csv_path, kernel_regex)
    per_launch = [rd + wr for _, _, rd, wr in rows]
    rec = {"workload": workload, "kernel_regex": kernel_regex, "kernels": sorted({k for _, k, _, _ in rows}),
           "launches": len(rows), "dram_bytes_read_per_launch": statistics.mean(r for _, _, r, _ in rows),
           "dram_bytes_write_per_launch": statistics.mean(w for _, _, _, w in rows),
           "dram_bytes_per_launch": statistics.mean(per_launch), "source_sha": source_sha(kernel_regex), "command": command}
    with open(traffic_path(workload), "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    return rec


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle (baseline / reference arm)

def oracle_step(w: workloads.Workload):
    """Build the oracle's cache for the whole workload (every sequence, prefilled by the oracle
    writer) and return a closure that runs one full layer step on it: the oracle writes one new
    token to every sequence, then decodes every sequence and head. Nothing is sampled or scaled:
    the closure's time is the time of one step of the workload."""
    import oracle
    inp = workloads.make_inputs(w, extra_pages=1)
    B = w.batch
    cfg = oracle.make_config(**w.config_kwargs())
    pool = np.zeros((inp.n_pages, oracle.page_bytes(cfg)), np.uint8)
    sink = np.zeros((B, cfg.n_sink, 576), np.uint16)
    ring = np.zeros((B, cfg.n_recent, 576), np.uint16)
    oracle.write(cfg, inp.c, inp.kr, inp.cu, np.zeros(B, np.int32), int(inp.seq_lens.max()), inp.page_table, pool,
                 sink, ring)
    rng = np.random.default_rng(123)
    state = {"lens": inp.seq_lens.astype(np.int32).copy()}
    max_tokens = inp.page_table.shape[1] * w.page_size

    def step():
        c1, k1 = workloads.draw_tokens(rng, B, w.latent_dist, inp.outliers, w.outlier_scale)
        if int(state["lens"].max()) + 1 > max_tokens:  # keep within the page table: restart from the prefill
            state["lens"] = inp.seq_lens.astype(np.int32).copy()
        t0 = time.perf_counter()
        oracle.write(cfg, c1, k1, np.arange(B + 1, dtype=np.int32), state["lens"], 1, inp.page_table, pool, sink,
                     ring)
        state["lens"] = state["lens"] + 1
        oracle.decode(cfg, inp.q_lat, inp.q_rope, inp.page_table, state["lens"], pool, sink, ring, w.softmax_scale)
        return time.perf_counter() - t0

    return step


def cpu_cores() -> int:
    return os.cpu_count() or 1


def oracle_threads_summary(step, all_threads: int, steps_all: int, steps_1: int):
    """Time the oracle step at all threads (steps_all steps) and at one thread (steps_1 steps)
    on the same work; returns (us per step at all threads, summary dict)."""
    import oracle
    oracle.set_threads(all_threads)
    t_all = [step() for _ in range(steps_all)]
    oracle.set_threads(1)
    t_1 = [step() for _ in range(steps_1)]
    oracle.set_threads(all_threads)
    us_all = statistics.mean(t_all) * 1e6
    us_1 = statistics.mean(t_1) * 1e6
    return us_all, {"threads_all": {"value": us_all, "unit": "us/layer", "threads": all_threads, "steps": steps_all},
                    "threads_1": {"value": us_1, "unit": "us/layer", "threads": 1, "steps": steps_1}}


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    cores = cpu_cores()
    oracle.set_threads(cores)
    step = oracle_step(w)
    for _ in range(max(0, min(args.warmup, 1))):
        step()
    t0 = time.perf_counter()
    times = [step() for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    us = statistics.mean(times) * 1e6
    oracle.set_threads(1)
    t1 = step() * 1e6
    oracle.set_threads(cores)
    sample = (f"the whole workload, unscaled: per step the oracle writes one token to each of the {w.batch} "
              f"sequences and decodes all {w.batch} x {w.heads} heads over every cached token")
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": "us/layer", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(w, 0),
        "timed_wall_s": wall,
        "cpu_baseline": {"value": us, "unit": "us/layer", "cores": cores, "kind": "oracle", "sample": sample,
                         "threads_all": {"value": us, "unit": "us/layer", "threads": cores, "steps": args.steps},
                         "threads_1": {"value": t1, "unit": "us/layer", "threads": 1, "steps": 1}},
        "e2e": {"value": us, "unit": "us/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def config_dict(w, layers):
    return {"workload": w.name, "batch": w.batch, "heads": w.heads, "seq_len": w.seq_len,
            "cache": f"C{w.bits_c}R4", "page": w.page_size, "sink": w.n_sink, "recent": w.n_recent,
            "clip_q": w.clip_q, "layers_rotated": layers,
            "l2": "inputs larger than L2: each step reads a layer cache last touched layers_rotated-1 steps earlier"}


# ------------------------------------------------------------------ GPU arm

EXTRA_WORKLOADS = ("v2lite_c4r4_b32_h16_t32k", "ragged_c2r4_b64_h16_serve", "wide_c2r4_b8_h128_t32k",
                   "long_c4r4_b1_h128_t128k", "tiny_c4r4_b1_h16_t1k")


def run_native(args, w):
    import torch

    import bit_mla_kv_qcache_gb300 as q

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    result = measure_workload(args, replica_workload(w, rank), q, dev, args.steps, args.warmup, args.layers,
                              with_e2e=not args.no_e2e)
    extras = [] if args.extra_workloads == "none" else (
        list(EXTRA_WORKLOADS) if args.extra_workloads == "auto" and w.name == DEFAULT_WORKLOAD else
        [x for x in args.extra_workloads.split(",") if x and x != "auto"])
    if extras:
        result["workloads"] = {}
        for name in extras:
            we = replica_workload(workloads.WORKLOADS[name], rank)
            r = measure_workload(args, we, q, dev, min(args.steps, 10), 3, 0, with_e2e=False)
            result["workloads"][name] = {k: r[k] for k in ("value", "unit", "steps", "decode_us", "write_and_advance_us",
                                                             "packed_cache_gbs", "decode_tflops", "roofline",
                                                             "gpu_launches", "clocks", "config")}
            torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(result))
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def measure_workload(args, w, q, dev, steps, warmup, layers, with_e2e):
    """The timed steps of one workload: layer caches built by the writer, K write+decode steps
    replayed from CUDA graphs over rotated caches, then a decode-only pass for the roofline."""
    import torch
    ws, rank, local = dist_env()
    cfg = q.make_config(**w.config_kwargs())
    B, H = w.batch, w.heads

    # tokens one layer may gain: warm-up, the timed graph replayed twice (warm, timed), the e2e graph twice
    steps_total = warmup + 3 * steps + 40
    inp = workloads.make_inputs(w, extra_pages=math.ceil(steps_total / w.page_size) + 1)
    max_pages = inp.page_table.shape[1]
    per_layer = inp.n_pages * q.page_bytes(cfg)
    NL = layers or max(2, math.ceil(3 * L2_BYTES / per_layer) + 1)

    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else
                                   np.ascontiguousarray(a)).to(dev)
    pt = t(inp.page_table)
    c_all, kr_all, cu_all = t(inp.c), t(inp.kr), t(inp.cu)
    caches = []
    for _ in range(NL):
        cache = q.QuantizedMLACache(cfg, B, max_pages, inp.n_pages, page_table=pt, device=dev)
        cache.write(c_all, kr_all, cu_all, int(inp.seq_lens.max()))
        caches.append(cache)
    del c_all, kr_all
    torch.cuda.synchronize()
    if any(c.error_bits() for c in caches):
        raise RuntimeError("writer reported device errors during prefill")

    # per-step inputs: one new token per sequence, queries (fixed across steps)
    rng = np.random.default_rng(1234)
    c1, k1 = workloads.draw_tokens(rng, B, w.latent_dist, inp.outliers, w.outlier_scale)
    c_new, kr_new = t(c1), t(k1)
    cu1 = torch.arange(B + 1, dtype=torch.int32, device=dev)
    q_lat, q_rope = t(inp.q_lat), t(inp.q_rope)
    out = torch.empty((B, H, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    ws_buf = caches[0].workspace(H)
    stream = torch.cuda.Stream(device=dev)

    # Each layer keeps two length arrays: a step writes the new token with the lengths of one
    # and stores the advanced lengths into the other (one launch), then decodes with those.
    lens_alt = [c.seq_lens.clone() for c in caches]

    def write_step(cache, lens_in, lens_out):
        q.mla_qcache_write_advance(cfg, c_new, kr_new, cu1, lens_in, lens_out, 1, cache.page_table, cache.pool,
                                   cache.sink, cache.ring, cache.err)

    def decode_step(cache, lens):
        q.mla_qcache_decode_attn(cfg, q_lat, q_rope, cache.page_table, lens, cache.pool, cache.sink,
                                 cache.ring, w.softmax_scale, out, lse, ws_buf, cache.err)

    def pending_step(cache, lens_in):
        q.mla_qcache_decode_attn_pending(cfg, q_lat, q_rope, cache.page_table, lens_in, c_new, kr_new, cu1, 1,
                                         cache.pool, cache.sink, cache.ring, w.softmax_scale, out, lse, ws_buf,
                                         cache.err)

    write_stream = torch.cuda.Stream(device=dev)

    def step_body(cache, lens_in, lens_out):
        # the writer forks from the step's start; the decode's node is created first (measured:
        # the writer then delays the decode's one wave of CTAs less); joined before the step ends
        # (the next step's decode reads what this step wrote)
        ev_fork = torch.cuda.Event()
        ev_fork.record(stream)
        pending_step(cache, lens_in)
        write_stream.wait_event(ev_fork)
        with torch.cuda.stream(write_stream):
            write_step(cache, lens_in, lens_out)
        stream.wait_stream(write_stream)

    # Warm-up: two CUDA graphs per layer (write + decode, lengths A -> B and B -> A) replayed
    # alternately. Timed: the K steps, rotating over the layers as a decode iteration over K
    # layers would, captured as one CUDA graph and replayed once (after one untimed replay); the
    # decode-only calls of the roofline likewise, K of them in one graph.
    g_step = []
    with torch.cuda.stream(stream):
        for cache in caches:  # warm the code paths once before capture
            decode_step(cache, cache.seq_lens)
        torch.cuda.synchronize()
        for cache, alt in zip(caches, lens_alt):
            pair = []
            for lens_in, lens_out in ((cache.seq_lens, alt), (alt, cache.seq_lens)):
                gs = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gs, stream=stream):
                    step_body(cache, lens_in, lens_out)
                pair.append(gs)
            g_step.append(pair)
    torch.cuda.synchronize()
    uses = [0] * NL

    def replay_step(k):
        layer = k % NL
        g_step[layer][uses[layer] & 1].replay()
        uses[layer] += 1

    def capture_steps(k0):
        # K consecutive steps from step k0 on, each layer's length arrays in the roles its use
        # count gives (the count advances as the graph is replayed, see run_timed)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream), torch.cuda.graph(g, stream=stream):
            u = list(uses)
            for k in range(steps):
                layer = (k0 + k) % NL
                cache, alt = caches[layer], lens_alt[layer]
                lens_in, lens_out = (cache.seq_lens, alt) if u[layer] % 2 == 0 else (alt, cache.seq_lens)
                u[layer] += 1
                step_body(cache, lens_in, lens_out)
        return g

    def advance_uses(k0):
        for k in range(steps):
            uses[(k0 + k) % NL] += 1

    head_start = torch.empty(int(1.5e9) // 4, dtype=torch.float32, device=dev)  # lets the host queue ahead

    with torch.cuda.stream(stream):
        for k in range(warmup):
            replay_step(k)
        torch.cuda.synchronize()
        g_warm = capture_steps(warmup)  # the same K steps once untimed (graph upload, clocks)
        g_warm.replay()
        advance_uses(warmup)
        torch.cuda.synchronize()
        del g_warm
        k0 = warmup + steps
        g_timed = capture_steps(k0)
        g_dec = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_dec, stream=stream):
            for k in range(steps):
                cache = caches[(k0 + k) % NL]
                decode_step(cache, cache.seq_lens)
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clk:
            head_start.fill_(1.0)
            start.record(stream)
            g_timed.replay()
            end.record(stream)
            torch.cuda.synchronize()
        advance_uses(k0)
        total_ms = start.elapsed_time(end)
        # decode-only pass (same caches, lengths unchanged): K calls in one graph, once warm
        g_dec.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        head_start.fill_(2.0)
        a.record(stream)
        g_dec.replay()
        b.record(stream)
        torch.cuda.synchronize()
        dec_ms = [a.elapsed_time(b) / steps]
    if ws > 1:
        total_ms = max_over_ranks(total_ms, dev)
    if any(c.error_bits() for c in caches):
        raise RuntimeError("device error bits set during the timed region")

    us_step = total_ms * 1e3 / steps
    dec_us = statistics.mean(dec_ms) * 1e3
    # sequence lengths seen by the decode-only pass (after the timed steps)
    mean_T = np.maximum(caches[0].seq_lens.cpu().numpy(), lens_alt[0].cpu().numpy())  # the newer of the two
    bytes_dec = decode_bytes(w, mean_T, H)
    flops_dec = decode_flops(mean_T, H)
    hbm_peak, tensor_peak, peak_kind = peaks()
    achieved = bytes_dec / (dec_us * 1e-6) / 1e9
    tflops = flops_dec / (dec_us * 1e-6) / 1e12
    traffic = profiled_traffic(w.name)
    dec_launches = q.decode_launches(cfg, B, H, max_pages)
    if H % 64 == 0:
        # 64-head blocks run the packed tokens on tcgen05 tensor cores; at ~1000 flops per packed
        # byte the decode is bound by the tensor pipe, not by HBM
        roofline = {"bound": "tensor", "achieved": tflops, "peak": tensor_peak, "unit": "TFLOP/s",
                    "frac": tflops / tensor_peak, "traffic": traffic,
                    "kernel": "mla_qcache_decode_attn (decode_tc_kernel + protected decode_kernel + combine_kernel)",
                    "algorithmic_flops_per_call": flops_dec, "algorithmic_bytes_per_call": bytes_dec,
                    "hbm_frac": achieved / hbm_peak, "peak_kind": peak_kind}
    else:
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved / hbm_peak, "traffic": traffic,
                    "kernel": "mla_qcache_decode_attn (decode_kernel" +
                              (" with the partials merged in place)" if dec_launches == 1 else " + combine_kernel)"),
                    "algorithmic_bytes_per_call": bytes_dec, "peak_kind": peak_kind}
    # the fused write + length update, then the decode's own launches (decode with the merge in
    # place; decode + merge; or protected decode + tensor-core decode + merge)
    launches_per_step = 1 + dec_launches

    result = {
        "metric": METRIC, "value": us_step * 1.0, "unit": "us/layer", "n_gpus": ws, "steps": steps,
        "warmup": warmup, "ms_per_step": us_step / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config_dict(w, NL),
        "decode_us": dec_us, "write_and_advance_us": max(0.0, us_step - dec_us),
        "packed_cache_gbs": achieved, "fraction_of_8tbs": achieved / 8000.0,
        "decode_tflops": tflops,
        "roofline": roofline,
        "gpu_launches": launches_per_step * steps,
        "clocks": clk.summary(),
    }

    if with_e2e:
        result["e2e"] = e2e_measure(args, w, q, caches, lens_alt, uses, cfg, inp, dev, stream)
    del caches, g_step, g_dec, head_start
    return result


def e2e_measure(args, w, q, caches, lens_alt, uses, cfg, inp, dev, stream):
    """The step end to end through the public API: every step copies its new tokens and queries
    from pinned host memory to the device (one copy: staged contiguously, as a serving loop
    would), runs the fused write and the decode on the same rotated layer caches as the timed
    steps, and copies O and LSE back to pinned host memory (one copy). The copies are
    double-buffered on the writer's forked stream: while step k decodes, step k-1's results leave
    and step k+1's inputs arrive, and the step's own join orders them; the whole timed sequence
    of steps is captured once as a CUDA graph and replayed."""
    import torch
    B, H = w.batch, w.heads
    NL = len(caches)
    rng = np.random.default_rng(99)
    c1, k1 = workloads.draw_tokens(rng, B, w.latent_dist, inp.outliers, w.outlier_scale)
    parts = [np.ascontiguousarray(a).view(np.int16).reshape(-1) for a in (c1, k1, inp.q_lat, inp.q_rope)]
    sizes = [x.size for x in parts]
    h_in = torch.from_numpy(np.concatenate(parts)).pin_memory()
    offs = np.cumsum([0] + sizes)
    n_out = B * H * 512
    d_in, d_res, h_res, views = [], [], [], []
    for slot in range(2):
        di = torch.empty_like(h_in, device=dev)
        dr = torch.empty(n_out + B * H, dtype=torch.float32, device=dev)  # O then LSE
        d_in.append(di)
        d_res.append(dr)
        h_res.append(torch.empty_like(dr, device="cpu").pin_memory())
        views.append((di[offs[0]:offs[1]].view(B, 512), di[offs[1]:offs[2]].view(B, 64),
                      di[offs[2]:offs[3]].view(B, H, 512), di[offs[3]:offs[4]].view(B, H, 64),
                      dr[:n_out].view(B, H, 512), dr[n_out:].view(B, H)))
    cu1 = torch.arange(B + 1, dtype=torch.int32, device=dev)
    ws_buf = caches[0].workspace(H)
    s_wr = torch.cuda.Stream(device=dev)
    # steps per graph: whole rounds over the layers, each layer an even number of times, so the
    # two length arrays of every layer are back in their starting roles after each replay
    K = 2 * NL * max(1, math.ceil(max(10, args.steps // 2) / (2 * NL)))
    k0 = sum(uses)

    # The copies ride on the writer's stream, inside the fork and join every step already has:
    # during step k that stream reads back step k-1's results, copies step k+1's inputs into the
    # slot step k-1 used, then runs step k's write, all beside step k's decode; the join at the
    # end of step k therefore also says that step k+1's inputs arrived. No event beyond the step's
    # own fork and join is waited on.
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        s_wr.wait_stream(stream)
        with torch.cuda.stream(s_wr):
            for k in range(min(2, K)):
                d_in[k].copy_(h_in, non_blocking=True)
        stream.wait_stream(s_wr)
        for k in range(K):
            slot = k & 1
            layer = (k0 + k) % NL
            cache, alt = caches[layer], lens_alt[layer]
            lens_in, lens_out = (cache.seq_lens, alt) if uses[layer] % 2 == 0 else (alt, cache.seq_lens)
            uses[layer] += 1
            d_c, d_k, d_ql, d_qr, out, lse = views[slot]
            ev_fork = torch.cuda.Event()
            ev_fork.record(stream)  # the write forks off at the step's start
            q.mla_qcache_decode_attn_pending(cfg, d_ql, d_qr, cache.page_table, lens_in, d_c, d_k, cu1, 1, cache.pool,
                                             cache.sink, cache.ring, w.softmax_scale, out, lse, ws_buf, cache.err,
                                             stream)
            s_wr.wait_event(ev_fork)
            with torch.cuda.stream(s_wr):
                if k >= 1:
                    h_res[slot ^ 1].copy_(d_res[slot ^ 1], non_blocking=True)  # step k-1's O and LSE
                    if k + 1 < K:
                        d_in[slot ^ 1].copy_(h_in, non_blocking=True)  # step k+1's inputs
            q.mla_qcache_write_advance(cfg, d_c, d_k, cu1, lens_in, lens_out, 1, cache.page_table, cache.pool,
                                       cache.sink, cache.ring, cache.err, s_wr)
            stream.wait_stream(s_wr)  # joined: the next step reads what this write stored, and its inputs
        with torch.cuda.stream(s_wr):
            s_wr.wait_stream(stream)
            h_res[(K - 1) & 1].copy_(d_res[(K - 1) & 1], non_blocking=True)  # the last step's results
        stream.wait_stream(s_wr)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        g.replay()  # warm-up replay
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        g.replay()
        e.record(stream)
        torch.cuda.synchronize()
    us = s.elapsed_time(e) * 1e3 / K
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_res[0].numel() * h_res[0].element_size()
    return {"value": us, "unit": "us/layer", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": K,
            "note": "public C ABI calls (fused write with the length update on a forked stream, concurrent with "
                    "the decode of the pending rows) with one H2D copy of the step's inputs and one D2H copy of O "
                    "and LSE per step, double-buffered on the forked stream (during step k: step k-1's results "
                    "back, step k+1's inputs in, then step k's write; the step's join orders them), layer caches "
                    "rotated as in the timed steps; the timed steps form one CUDA graph"}


# ------------------------------------------------------------------ latency sweep against BF16

SWEEP_BATCH_TOKENS = 1 << 23  # largest batch x context swept (bounds device memory and build time)
FLUSH_BYTES = 512 * 1024 * 1024


def flushed_call_us(fn, flush, stream, reps: int = 10, rounds: int = 5) -> float:
    """Device time of one call that reads its inputs from HBM: a CUDA graph of `reps` x (512 MB
    write that evicts L2, call) minus a graph of `reps` x (write), per call; median over
    `rounds` replays of each (the graph launch itself is paid once per replay, not per call)."""
    import torch
    g_all, g_fl = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_all, stream=stream):
        for k in range(reps):
            flush.fill_(float(k))
            fn()
    with torch.cuda.graph(g_fl, stream=stream):
        for k in range(reps):
            flush.fill_(float(k))

    def once(g):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3

    with torch.cuda.stream(stream):
        g_all.replay()
        g_fl.replay()
        torch.cuda.synchronize()
        t_all, t_fl = [], []
        for _ in range(rounds):  # interleaved, so both see the same clocks
            t_all.append(once(g_all))
            t_fl.append(once(g_fl))
    return max(0.0, statistics.median(t_all) - statistics.median(t_fl)) / reps


def bf16_decode_bytes(seq_lens, heads) -> int:
    """Bytes the unquantized decode must move: every token's BF16 row, queries and outputs."""
    B = len(seq_lens)
    return int(sum(int(T) for T in seq_lens)) * 576 * 2 + B * heads * 576 * 2 + B * heads * (512 + 1) * 4


def run_sweep(args):
    """Decode latency of one layer over a C4R4 cache (page 128, sink 4, recent 128) and over an
    unquantized BF16 paged cache (page 64) holding the same tokens, for contexts of 1K..1M tokens
    and batches 1/8/32, as the normalised-latency tables of the low-bit MLA cache pages report:
    delta = t_C4R4 / t_BF16 - 1. A 512 MB write before every call evicts L2, so each call reads
    its cache from HBM (one decode of one layer, whose cache the other layers' calls have
    evicted); per-call device time from CUDA graphs of (write, call) pairs minus graphs of the
    writes alone. Every sequence of a batch holds the same
    synthetic rows (one seeded 1M-token draw; prefixes give the shorter contexts)."""
    import torch

    import bit_mla_kv_qcache_gb300 as q

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    H = args.sweep_heads
    t_max = args.sweep_max_tokens
    batches = [int(x) for x in args.sweep_batches.split(",") if x]
    contexts = [1024 << i for i in range(11) if (1024 << i) <= t_max]
    wq = workloads.Workload("sweep_c4r4", 1, H, max(contexts), 4, 128)
    inp = workloads.make_inputs(wq, extra_pages=0)
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else
                                        np.ascontiguousarray(a)).to(dev)
    c_all, kr_all = to_dev(inp.c), to_dev(inp.kr)
    q1_lat, q1_rope = to_dev(inp.q_lat), to_dev(inp.q_rope)  # [1, H, *]: one query row, every sequence
    cfg = q.make_config(**wq.config_kwargs())
    P_q, P_b = wq.page_size, 64
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    hbm_peak, _, peak_kind = peaks()
    rng = np.random.default_rng(77)
    iters = max(10, args.steps)
    points = []
    with ClockSampler(0) as clk:
        for B in batches:
            q_lat, q_rope = q1_lat.expand(B, H, 512).contiguous(), q1_rope.expand(B, H, 64).contiguous()
            out = torch.empty((B, H, 512), dtype=torch.float32, device=dev)
            lse = torch.empty((B, H), dtype=torch.float32, device=dev)
            for T in contexts:
                if B * T > SWEEP_BATCH_TOKENS:
                    continue
                lens = torch.full((B,), T, dtype=torch.int32, device=dev)
                # C4R4 cache: sequence by sequence through the writer (rows of one sequence only)
                mp_q = math.ceil(T / P_q) + 1
                pt_q, np_q = workloads.page_table_for(rng, B, mp_q, True)
                cache = q.QuantizedMLACache(cfg, B, mp_q, np_q, page_table=to_dev(pt_q), device=dev)
                cu = torch.zeros(B + 1, dtype=torch.int32, device=dev)
                for b in range(B):
                    cu.zero_()
                    cu[b + 1:] = T
                    cache.write(c_all[:T], kr_all[:T], cu, T)
                # BF16 paged cache: the same rows, scattered into 64-token pages
                mp_b = math.ceil(T / P_b) + 1
                pt_b, np_b = workloads.page_table_for(rng, B, mp_b, True)
                d_pt_b = to_dev(pt_b)
                pool = torch.zeros((np_b, P_b, 576), dtype=torch.int16, device=dev)
                rows = torch.cat([c_all[:T], kr_all[:T]], dim=1)
                tok = torch.arange(T, device=dev, dtype=torch.int64)
                for b in range(B):
                    slot = d_pt_b[b].to(torch.int64)[tok // P_b] * P_b + tok % P_b
                    pool.view(-1, 576)[slot] = rows
                del rows, tok
                err = torch.zeros(1, dtype=torch.int32, device=dev)
                ws_q = cache.workspace(H)
                ws_b = torch.zeros(q.bf16_workspace_bytes(B, H, mp_b, P_b), dtype=torch.uint8, device=dev)
                torch.cuda.synchronize()
                if cache.error_bits():
                    raise RuntimeError("writer reported device errors while building the sweep cache")

                def call_q():
                    q.mla_qcache_decode_attn(cfg, q_lat, q_rope, cache.page_table, lens, cache.pool, cache.sink,
                                             cache.ring, wq.softmax_scale, out, lse, ws_q, cache.err)

                def call_b():
                    q.mla_qcache_decode_attn_bf16(q_lat, q_rope, d_pt_b, P_b, lens, pool, wq.softmax_scale, out, lse,
                                                  ws_b, err)

                with torch.cuda.stream(stream):
                    for fn in (call_q, call_b):
                        fn()
                    torch.cuda.synchronize()
                us = [flushed_call_us(call_q, flush, stream, reps=iters, rounds=5),
                      flushed_call_us(call_b, flush, stream, reps=iters, rounds=5)]
                if cache.error_bits() or int(err.item()):
                    raise RuntimeError("device error bits set during the sweep")
                seq = [T] * B
                wb = workloads.Workload("sweep_c4r4", B, H, T, 4, 128)
                bq, bb = decode_bytes(wb, seq, H), bf16_decode_bytes(seq, H)
                bf16_floor_us = bb / (hbm_peak * 1e9) * 1e6  # the comparator at the measured copy bandwidth
                points.append({"batch": B, "T": T, "c4r4_us": us[0], "bf16_us": us[1], "delta": us[0] / us[1] - 1.0,
                               "bf16_roofline_us": bf16_floor_us, "delta_vs_bf16_roofline": us[0] / bf16_floor_us - 1.0,
                               "c4r4_hbm_frac": bq / (us[0] * 1e-6) / 1e9 / hbm_peak,
                               "bf16_hbm_frac": bb / (us[1] * 1e-6) / 1e9 / hbm_peak,
                               "c4r4_bytes": bq, "bf16_bytes": bb})
                del cache, pool, ws_q, ws_b
                torch.cuda.empty_cache()
    print(json.dumps({
        "mode": "latency_sweep", "metric": "decode attention latency per layer, C4R4 vs BF16 paged; "
                                           "delta = t_C4R4 / t_BF16 - 1", "unit": "us", "heads": H,
        "cache": "C4R4 page 128 sink 4 recent 128", "comparator": "BF16 paged cache, page 64 (own kernel)",
        "iters": iters, "statistic": "median of 5 graph replays of iters (flush, call) pairs minus flush-only "
                                     "graphs, per call", "l2": "512 MB write before every timed call",
        "hbm_peak_gbs": hbm_peak, "peak_kind": peak_kind, "data": "synthetic", "points": points,
        "clocks": clk.summary()}))
    return 0


# ------------------------------------------------------------------ latent-transform cost

def run_transform(args):
    """Per-layer cost of the latent transform A_c at decode batches 1..64 over a 2K-token C4R4
    cache (16 heads), in the form of the RAQ-MLA page's appendix Table 9: "standalone" is the
    transform as its own kernel before the cache write, "fused" the extra time of the writer
    that applies it; "share" is the fused cost relative to the transforming write plus the
    decode attention. Each operation is captured 20 times in one CUDA graph and the graph
    replayed (back-to-back calls, caches and A_c L2-resident, as inside a decode step); the
    writes rewrite the same token slot (lengths are not advanced)."""
    import torch

    import bit_mla_kv_qcache_gb300 as q

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    T, H, reps, per_graph = 2048, 16, max(10, args.steps), 20
    stream = torch.cuda.Stream(device=dev)
    rng = np.random.default_rng(2024)
    a_c = torch.from_numpy((rng.standard_normal((512, 512)) / math.sqrt(512)).astype(np.float32)).to(
        torch.bfloat16).view(torch.int16).to(dev)
    rows = []
    with ClockSampler(0) as clk:
        for B in (1, 2, 4, 8, 64):
            w = workloads.Workload("xf_c4r4", B, H, T, 4, 128)
            inp = workloads.make_inputs(w, extra_pages=1)
            to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else
                                                np.ascontiguousarray(a)).to(dev)
            cfg = q.make_config(**w.config_kwargs())
            cache = q.QuantizedMLACache(cfg, B, inp.page_table.shape[1], inp.n_pages,
                                        page_table=to_dev(inp.page_table), device=dev)
            cache.write(to_dev(inp.c), to_dev(inp.kr), to_dev(inp.cu), T)
            c1, k1 = workloads.draw_tokens(rng, B, w.latent_dist, inp.outliers, w.outlier_scale)
            c_new, kr_new = to_dev(c1), to_dev(k1)
            c_t = torch.empty_like(c_new)
            cu1 = torch.arange(B + 1, dtype=torch.int32, device=dev)
            q_lat, q_rope = to_dev(inp.q_lat), to_dev(inp.q_rope)
            out = torch.empty((B, H, 512), dtype=torch.float32, device=dev)
            lse = torch.empty((B, H), dtype=torch.float32, device=dev)
            ws_buf = cache.workspace(H)
            ops = {
                "write": lambda: q.mla_qcache_write(cfg, c_new, kr_new, cu1, cache.seq_lens, 1, cache.page_table,
                                                    cache.pool, cache.sink, cache.ring, cache.err),
                "write_fused": lambda: q.mla_qcache_write_transformed(
                    cfg, c_new, kr_new, cu1, cache.seq_lens, 1, cache.page_table, cache.pool, cache.sink,
                    cache.ring, cache.err, a_c=a_c),
                "transform": lambda: q.mla_qcache_row_transform(c_new, a_c, c_t, cache.err),
                "decode": lambda: q.mla_qcache_decode_attn(cfg, q_lat, q_rope, cache.page_table, cache.seq_lens,
                                                           cache.pool, cache.sink, cache.ring, w.softmax_scale, out,
                                                           lse, ws_buf, cache.err),
            }
            us = {}
            with torch.cuda.stream(stream):
                for name, fn in ops.items():
                    fn()
                    torch.cuda.synchronize()
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        for _ in range(per_graph):
                            fn()
                    for _ in range(3):
                        g.replay()
                    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    s_ev.record(stream)
                    for _ in range(reps):
                        g.replay()
                    e_ev.record(stream)
                    torch.cuda.synchronize()
                    us[name] = s_ev.elapsed_time(e_ev) * 1e3 / (reps * per_graph)
            if cache.error_bits():
                raise RuntimeError("device error bits set in the transform benchmark")
            fused = max(0.0, us["write_fused"] - us["write"])
            rows.append({"batch": B, "standalone_us": us["transform"], "fused_us": fused,
                         "share": fused / (us["write_fused"] + us["decode"]), "write_us": us["write"],
                         "write_fused_us": us["write_fused"], "decode_us": us["decode"]})
            del cache
            torch.cuda.empty_cache()
    print(json.dumps({
        "mode": "latent_transform_cost", "metric": "per-layer cost of the latent transform A_c (512x512 BF16), "
                                                   "standalone kernel vs fused in the writer",
        "unit": "us", "cache": "C4R4 page 128 sink 4 recent 128, 2048 tokens, 16 heads",
        "timing": f"{per_graph} calls per CUDA graph, {reps} replays, L2-resident", "rows": rows,
        "clocks": clk.summary(), "data": "synthetic"}))
    return 0


# ------------------------------------------------------------------ multi-token decode

def run_multi(args):
    """Decode of q_len = 1, 2, 4, 8 new tokens per sequence in one call over the headline cache
    shape (C4R4, 16 heads, batch 32 at 8K tokens, and batch 1 at 128K); L2 flushed before every
    call. At q_len * 16 a multiple of 64 the packed pages are read once for all positions."""
    import torch

    import bit_mla_kv_qcache_gb300 as q

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    hbm_peak, tensor_peak, peak_kind = peaks()
    iters = max(10, args.steps)
    rows = []
    with ClockSampler(0) as clk:
        for B, T in ((32, 8192), (1, 131072)):
            w = workloads.Workload("multi_c4r4", B, 16, T, 4, 128)
            inp = workloads.make_inputs(w, extra_pages=1)
            to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else
                                                np.ascontiguousarray(a)).to(dev)
            cfg = q.make_config(**w.config_kwargs())
            cache = q.QuantizedMLACache(cfg, B, inp.page_table.shape[1], inp.n_pages,
                                        page_table=to_dev(inp.page_table), device=dev)
            cache.write(to_dev(inp.c), to_dev(inp.kr), to_dev(inp.cu), T)
            for q_len in (1, 2, 4, 8):
                R = 16 * q_len
                ql, qr = workloads.draw_queries(np.random.default_rng(q_len), B, R)
                d_ql, d_qr = to_dev(ql), to_dev(qr)
                out = torch.empty((B, R, 512), dtype=torch.float32, device=dev)
                lse = torch.empty((B, R), dtype=torch.float32, device=dev)
                ws = torch.zeros(q.workspace_bytes(cfg, B, R, inp.page_table.shape[1]), dtype=torch.uint8, device=dev)
                fn = lambda: q.mla_qcache_decode_attn_multi(cfg, q_len, d_ql, d_qr, cache.page_table, cache.seq_lens,
                                                            cache.pool, cache.sink, cache.ring, w.softmax_scale, out,
                                                            lse, ws, cache.err)
                with torch.cuda.stream(stream):
                    fn()
                    torch.cuda.synchronize()
                us = flushed_call_us(fn, flush, stream, reps=iters)
                nbytes = decode_bytes(w, [T] * B, R)
                rows.append({"batch": B, "T": T, "q_len": q_len, "rows": R, "us": us, "us_per_token": us / q_len,
                             "hbm_frac": nbytes / (us * 1e-6) / 1e9 / hbm_peak,
                             "tflops": decode_flops([T] * B, R) / (us * 1e-6) / 1e12})
            if cache.error_bits():
                raise RuntimeError("device error bits set in the multi-token benchmark")
            del cache
            torch.cuda.empty_cache()
    print(json.dumps({"mode": "multi_token_decode", "metric": "decode µs per call for q_len new tokens per "
                                                              "sequence (C4R4, 16 heads per position)",
                      "unit": "us", "l2": "512 MB write before every timed call", "iters": iters,
                      "hbm_peak_gbs": hbm_peak, "peak_kind": peak_kind, "rows": rows, "clocks": clk.summary(),
                      "data": "synthetic"}))
    return 0


# ------------------------------------------------------------------ projections either side of attention

def run_proj(args):
    """Query absorption (q_nope W_UK plus the 64 x 64 query-side k_R compensation) and the W_UV
    up-projection of the attention output, per layer at decode batches 1..64, for 16 and 128
    heads (d_nope = d_v = 128). A 512 MB write before every call evicts L2 (a layer's weights
    come from HBM); per-call device time from CUDA graphs of (write, call) pairs minus graphs of
    the writes alone. HBM fraction = (weights + inputs + outputs) / time / measured copy
    bandwidth."""
    import torch

    import bit_mla_kv_qcache_gb300 as q

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    hbm_peak, _, peak_kind = peaks()
    rng = np.random.default_rng(5)
    iters = max(10, args.steps)
    bf = lambda shape, scale: torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32)).to(
        torch.bfloat16).view(torch.int16).to(dev)
    rows = []
    with ClockSampler(0) as clk:
        for H in (16, 128):
            d = dv = 128
            w_uk, w_uv, r_c = bf((H, d, 512), d ** -0.5), bf((H, 512, dv), 512 ** -0.5), bf((64, 64), 0.125)
            for B in (1, 8, 32, 64):
                qn, qr = bf((B, H, d), 1.0), bf((B, H, 64), 1.0)
                ql = torch.empty((B, H, 512), dtype=torch.int16, device=dev)
                qro = torch.empty((B, H, 64), dtype=torch.int16, device=dev)
                o = torch.randn((B, H, 512), dtype=torch.float32, device=dev)
                out = torch.empty((B, H, dv), dtype=torch.float32, device=dev)
                ops = {"absorb": lambda: q.mla_qcache_absorb_query(qn, w_uk, ql, q_rope=qr, r_comp=r_c, q_rope_out=qro),
                       "up_project": lambda: q.mla_qcache_up_project(o, w_uv, out)}
                nbytes = {"absorb": w_uk.numel() * 2 + 8192 + B * H * (d + 64 + 512 + 64) * 2,
                          "up_project": w_uv.numel() * 2 + B * H * (512 + dv) * 4}
                res = {"heads": H, "batch": B}
                with torch.cuda.stream(stream):
                    for fn in ops.values():
                        fn()
                    torch.cuda.synchronize()
                for name, fn in ops.items():
                    us = flushed_call_us(fn, flush, stream, reps=iters)
                    res[f"{name}_us"] = us
                    res[f"{name}_hbm_frac"] = nbytes[name] / (us * 1e-6) / 1e9 / hbm_peak
                rows.append(res)
    print(json.dumps({"mode": "projections", "metric": "per-layer µs of the query absorption and the W_UV "
                                                       "up-projection (d_nope = d_v = 128)",
                      "unit": "us", "l2": "512 MB write before every timed call", "iters": iters,
                      "statistic": "median of 5 graph replays, (flush, call) pairs minus flush-only, per call", "hbm_peak_gbs": hbm_peak, "peak_kind": peak_kind, "rows": rows,
                      "clocks": clk.summary(), "data": "synthetic"}))
    return 0


def cpu_baseline(w):
    """The oracle on the host cores, one full unscaled step of the workload at all threads and
    one at a single thread (the same work)."""
    import oracle
    cores = cpu_cores()
    oracle.set_threads(cores)
    step = oracle_step(w)
    step()  # warm-up
    us_all, d = oracle_threads_summary(step, cores, 1, 1)
    return {"value": us_all, "unit": "us/layer", "cores": cores, "kind": "oracle",
            "sample": f"the whole workload, unscaled: one step (one token written to each of the {w.batch} "
                      f"sequences, then the decode of all {w.batch} x {w.heads} heads over every cached token)",
            **d}


def main():
    args = parse()
    w = workloads.WORKLOADS[args.workload]
    if args.record_traffic:
        regex = args.traffic_kernel or dominant_kernel_regex(w)
        print(json.dumps(record_traffic(args.record_traffic, w.name, regex, args.traffic_command)))
        return 0
    if args.impl == "reference":
        return run_reference(args, w)
    if args.sweep:
        return run_sweep(args)
    if args.transform:
        return run_transform(args)
    if args.proj:
        return run_proj(args)
    if args.multi:
        return run_multi(args)
    return run_native(args, w)


if __name__ == "__main__":
    sys.exit(main())
