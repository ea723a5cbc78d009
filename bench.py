"""Benchmark of the paged decode hot path on GB300.

One step = one pass of the whole hot path over one batch: the workload's
copy-on-write block copies (if any), reshape_and_cache of every sequence's
new token, then paged decode attention over context_lens tokens.  The metric
is KV-read HBM GB/s: the K/V bytes the decode must read (sum over sequences of
ctx * kv_heads * head_dim * element bytes * 2) divided by the step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I]
                  [--impl ours|reference] [--no-cpu-baseline]

Default workload: the long-context split-KV decode (8 sequences, 64 query / 8 kv
heads, head_dim 128, bf16, block size 32, context lengths U[32768, 131072]), the
largest of the five; the same JSON line carries a `per_config` object with every
workload timed the same way (step and decode µs, algorithmic bytes, roofline
fraction against the measured copy bandwidth).
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no exchange step); the value is the bytes of all ranks divided
by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn: KV-read HBM GB/s (% of GB300 peak); µs per decode step"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
DECODE_SOURCES = ["common.cuh", "decode.cuh", "decode_mma.cuh", "decode_launch.cuh",
                  "decode_f32.cu", "decode_f16.cu", "decode_bf16.cu", "tmap.cu", "tmap.cuh",
                  "api.cu"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=3,
                    help="0 tiny MHA fp32, 1 OPT-13B-shaped fp16, 2 GQA bf16, 3 long-context "
                         "split-KV bf16 (default, the largest), 4 FP8 KV + shared prefix")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only --workload (skip the per_config timings of the others)")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="shrink the workload to its first N sequences (profiling captures)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--swap", action="store_true",
                    help="measure pkv_swap_blocks (device pool <-> pinned host pool) instead")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--multi-query", type=int, default=None, metavar="ID",
                    help="measure the multi-query (causal) paged attention on multi-query "
                         "workload ID (1: chunked prefill, 2: prefill, 3: draft-tree "
                         "verification) instead of the decode")
    ap.add_argument("--record-traffic", metavar="CSV", default=None,
                    help="store the DRAM bytes per decode launch of an ncu --csv capture "
                         "(dram__bytes_read.sum, dram__bytes_write.sum of decode_mma / "
                         "decode_simt launches) for --workload in profiles/decode_traffic.json")
    return ap.parse_args(argv)


# ------------------------------------------------------------ distributed --

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return dist


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of x over ranks (identity on one rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(bytes_per_rank: float, seconds_per_rank: float, world: int, device=None):
    """Whole-job throughput: total bytes of all ranks over the slowest rank's time."""
    total = reduce_sum(bytes_per_rank, world, device)
    slowest = reduce_max(seconds_per_rank, world, device)
    return total, slowest, total / slowest / 1e9


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples while the benchmark runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons), "window": "warm-up + timed steps"}


# ------------------------------------------------------------------ peaks --

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if d.get("hbm_gbs"):
            return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json, copy)"
    return FALLBACK_HBM_GBS, "fallback"


def copy_peak_gbs(torch, device, stream) -> float:
    """Same-run device copy bandwidth (read + write bytes), best of 5."""
    n = 1 << 30
    a = torch.empty(n, dtype=torch.uint8, device=device)
    b = torch.empty_like(a)
    best = 0.0
    with torch.cuda.stream(stream):
        for _ in range(6):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            b.copy_(a)
            e1.record(stream)
            e1.synchronize()
            best = max(best, 2 * n / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    del a, b
    return best


MQ_SOURCES = ["common.cuh", "tcgen05.cuh", "mq_attention.cu", "mq_attention.cuh", "tmap.cu",
              "tmap.cuh", "api.cu"]


def decode_source_hash(sources=None) -> str:
    h = hashlib.sha256()
    for fn in sources or DECODE_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_87_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload):
    """DRAM bytes per decode launch from a committed ncu summary, if it matches this code."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(str(workload))
    srcs = MQ_SOURCES if str(workload).startswith("mq") else None
    if not rec or rec.get("source_hash") != decode_source_hash(srcs):
        return None
    return rec.get("dram_bytes_per_launch")


def record_traffic(csv_path: str, workload, kernels=("decode_mma_kernel",
                                                      "decode_simt_kernel")) -> dict:
    """Average DRAM bytes (read + write) per decode launch of an ncu --csv log,
    stored for `workload` with the hash of the decode sources it was taken on."""
    import csv
    rows = list(csv.reader(line for line in open(csv_path) if line.startswith('"')))
    hdr = rows[0]
    ki, mi, vi, ii, ui = (hdr.index(k) for k in ("Kernel Name", "Metric Name", "Metric Value",
                                                  "ID", "Metric Unit"))
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12,
             "KB": 1e3, "MB": 1e6, "GB": 1e9}
    per = {}
    for r in rows[1:]:
        if not any(k in r[ki] for k in kernels):
            continue
        if r[mi] in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            per.setdefault(r[ii], 0.0)
            per[r[ii]] += float(r[vi].replace(",", "")) * scale[r[ui]]
    if not per:
        raise SystemExit(f"no {'/'.join(kernels)} launch with DRAM byte counters in {csv_path}")
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    d = json.load(open(path)) if os.path.exists(path) else {}
    srcs = MQ_SOURCES if str(workload).startswith("mq") else None
    d[str(workload)] = {"dram_bytes_per_launch": sum(per.values()) / len(per),
                        "launches": len(per), "source_hash": decode_source_hash(srcs)}
    with open(path, "w") as f:
        json.dump(d, f, indent=1, sort_keys=True)
        f.write("\n")
    return d[str(workload)]


# ------------------------------------------------------------ CPU baseline --

def oracle_baseline(w, target_s: float, nthreads: int | None = None, seed: int = 0,
                    caches=None):
    """Time the fp64 oracle on whole (sequence, kv head) units of the workload.

    Returns (GB/s of KV read, seconds, bytes, threads, description, single-thread
    GB/s).  The single-thread figure is the calibration run: one (sequence, kv head)
    unit on one thread.  The sample's pool is built (untimed) by the oracle's own
    reshape_and_cache / copy_blocks, or taken from `caches`.
    """
    from tests.helpers import oracle_caches, oracle_decode
    nthreads = nthreads or os.cpu_count() or 1
    G = w.num_q_heads // w.num_kv_heads
    e = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}[w.kv_dtype]
    kc, vc = caches if caches is not None else oracle_caches(w)
    rng = np.random.default_rng(seed)
    order = rng.permutation(w.num_seqs)
    # calibrate on one sequence's kv head 0 group
    s0 = int(order[0])
    sel0 = np.array([[s0, h] for h in range(G)], np.int32)
    t = time.perf_counter()
    oracle_decode(w, kc, vc, sel=sel0, nthreads=1)
    secs0 = time.perf_counter() - t
    per_token_s = secs0 / max(1, int(w.context_lens[s0]))
    single_gbs = int(w.context_lens[s0]) * w.head_dim * e * 2 / max(secs0, 1e-9) / 1e9
    budget_tokens = target_s * nthreads / max(per_token_s, 1e-9)
    units, tokens = [], 0
    for s in order:
        for g in range(w.num_kv_heads):
            units.append((int(s), g))
            tokens += int(w.context_lens[s])
            if tokens >= budget_tokens:
                break
        if tokens >= budget_tokens:
            break
    sel = np.array([[s, g * G + i] for s, g in units for i in range(G)], np.int32)
    t = time.perf_counter()
    oracle_decode(w, kc, vc, sel=sel, nthreads=nthreads)
    secs = time.perf_counter() - t
    nbytes = sum(int(w.context_lens[s]) for s, _ in units) * w.head_dim * e * 2
    desc = (f"{len(units)} (sequence, kv head) units of the workload, {tokens} context tokens, "
            f"{len(sel)} query heads, fp64 oracle on {nthreads} threads")
    return nbytes / secs / 1e9, secs, nbytes, nthreads, desc, single_gbs


# ------------------------------------------------------------------- arms --

def time_decode_steps(torch, st, stream, steps, warmup, flush_buf, world=1, device=None):
    """Warm up, then time `steps` hot-path steps with CUDA events on `stream`.

    Returns (step ms, decode ms) per timed step; the decode events bracket the
    decode call alone (planning + decode (+ merge) kernels).  `flush_buf`, when
    given, is written before every timed step (outside the events) so the step
    starts with a cold L2.  The step's calls are prepared once (arguments
    marshalled), so the host issues each launch with one ctypes call."""
    pre, dec = st.prepare(stream)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            for c in pre:
                c()
            dec()
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize(device)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        for i in range(steps):
            if flush_buf is not None:
                flush_buf.zero_()
            s0, d0, d1, s1 = ev[i]
            s0.record(stream)
            for c in pre:
                c()
            d0.record(stream)
            dec()
            d1.record(stream)
            s1.record(stream)
        stream.synchronize()
        torch.cuda.synchronize(device)
        barrier(world)
    return [e[0].elapsed_time(e[3]) for e in ev], [e[1].elapsed_time(e[2]) for e in ev]


def launches_per_step(w, prefix: bool) -> int:
    """Kernels one hot-path step launches: copy_blocks (if the step has pairs),
    reshape_and_cache, the planning and decode kernels, and for a prefix-aware launch
    on the tensor-core path (16-bit q with K/V of the same type, or e4m3 K/V at
    head_dim 128; at most 8 query heads per kv head) the shared-prefix detection and
    the merge kernel."""
    mma = w.q_dtype in ("f16", "bf16") and (w.kv_dtype == w.q_dtype or
                                             (w.kv_dtype == "e4m3" and w.head_dim == 128))
    grouped = mma and prefix and w.num_q_heads // w.num_kv_heads <= 8
    return (1 if len(w.step_pairs) else 0) + 1 + 2 + (2 if grouped else 0)


def l2_policy(torch, w, device):
    """Flush buffer (2x L2, written before every timed step) when the workload's KV is
    smaller than 4x L2; otherwise None (the inputs are larger than L2)."""
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    if w.unique_kv_bytes < 4 * l2:
        return (torch.empty(2 * l2 // 4 * 4, dtype=torch.uint8, device=device),
                "L2 flushed between steps (write of 2x L2)")
    return None, f"inputs larger than L2 ({w.unique_kv_bytes / 1e9:.2f} GB of distinct KV per step)"


def per_config_entry(w, step_ms, dec_ms, peak, l2_note, prefix) -> dict:
    """One workload's timing: step and decode µs, algorithmic bytes, roofline fraction.

    The roofline's bytes are the unique K/V rows the decode must read (for the
    shared-prefix workload each shared block once per group); the logical bytes
    (every sequence's context) give the KV-read rate, which is not a roofline
    fraction when blocks are shared."""
    dec_s = float(np.mean(dec_ms)) * 1e-3
    step_s = float(np.mean(step_ms)) * 1e-3
    e = {"workload": w.name, "step_us": round(step_s * 1e6, 2), "decode_us": round(dec_s * 1e6, 2),
         "kv_read_bytes": w.kv_read_bytes, "unique_kv_bytes": w.unique_kv_bytes,
         "step_kv_read_gbs": round(w.kv_read_bytes / step_s / 1e9, 1),
         "decode_gbs": round(w.unique_kv_bytes / dec_s / 1e9, 1),
         "frac": round(w.unique_kv_bytes / dec_s / 1e9 / peak, 4),
         "l2": l2_note, "entry": "prefix-aware" if prefix else "plain"}
    if w.unique_kv_bytes != w.kv_read_bytes:
        e["logical_kv_gbs_not_a_roofline"] = round(w.kv_read_bytes / dec_s / 1e9, 1)
    return e


def capture_step(torch, step, stream, h_out):
    """The e2e step (host-to-device copy, the step's launches, device-to-host copy) as a
    CUDA graph, the way a serving loop replays its decode step; returns (graph, label).

    The step runs eagerly once first (its result kept), then once captured and
    replayed: the replay must reproduce the eager result bit for bit.  If capture is
    refused, the eager step is timed instead and the label says why."""
    try:
        with torch.cuda.stream(stream):
            step()
            stream.synchronize()
            eager = h_out.clone()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step()
            h_out.zero_()
            g.replay()
            stream.synchronize()
        if not torch.equal(eager.view(torch.uint8), h_out.view(torch.uint8)):
            return None, "eager launches (the graph replay's output differed)"
        return g, "CUDA graph replay of the copy in, the step's launches and the copy out"
    except Exception as ex:   # capture refused on this stack: time the eager step
        torch.cuda.synchronize()
        return None, f"eager launches (graph capture failed: {type(ex).__name__}: {ex})"[:200]


def run_ours(args, rank, world, local):
    import torch
    from paged_kv_cache_87_gb300 import binding, build, inputs
    from paged_kv_cache_87_gb300.session import DeviceState

    build.build()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    w = inputs.make_config(args.workload, num_seqs=args.num_seqs)
    st = DeviceState(w, device)
    st.run_setup()
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize(device)
    flush_buf, l2_note = l2_policy(torch, w, device)
    peak, peak_src = measured_peak()

    clocks = ClockSampler(local)
    clocks.start()
    step_ms, dec_ms = time_decode_steps(torch, st, stream, args.steps, args.warmup, flush_buf,
                                        world, device)
    clk = clocks.stop()
    assert binding.pkv_get_device_status() == 0, "device status flagged during the benchmark"
    sec_step = float(np.mean(step_ms)) * 1e-3
    total_bytes, slowest, value = aggregate(w.kv_read_bytes, sec_step, world, device)

    # end to end through the public calls: every step, one host-to-device copy of the
    # step's inputs (query, new K/V, slots, context lengths, tables, copy pairs) packed
    # in one pinned buffer, the step, and the output copied back to pinned memory
    h_in, d_in = st.pack_step_inputs()
    h_out = torch.empty_like(st.out, device="cpu").pin_memory()
    h2d, d2h = h_in.numel(), h_out.numel() * h_out.element_size()
    pre, dec = st.prepare(stream)                 # the inputs moved: marshal again

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        for c in pre:
            c()
        dec()
        h_out.copy_(st.out, non_blocking=True)

    graph, e2e_launch = capture_step(torch, e2e_step, stream, h_out)
    e2e_ms = []
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            if flush_buf is not None:
                flush_buf.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            if graph is not None:
                graph.replay()
            else:
                e2e_step()
            b.record(stream)
            b.synchronize()
            if i >= args.warmup:
                e2e_ms.append(a.elapsed_time(b))
    assert binding.pkv_get_device_status() == 0, "device status flagged during the e2e steps"
    _, _, e2e_value = aggregate(w.kv_read_bytes, float(np.mean(e2e_ms)) * 1e-3, world, device)

    head = per_config_entry(w, step_ms, dec_ms, peak, l2_note, st.prefix)
    dec_s = float(np.mean(dec_ms)) * 1e-3
    achieved = w.unique_kv_bytes / dec_s / 1e9
    copy_peak = copy_peak_gbs(torch, device, stream) if rank == 0 else None
    # DRAM bytes of one decode launch from the committed ncu capture (when it was taken
    # on this source)
    traffic = recorded_traffic(args.workload) if args.num_seqs is None else None
    nlaunch = launches_per_step(w, st.prefix)
    del st, d_in, flush_buf
    torch.cuda.empty_cache()

    # the other workloads, each timed the same way (same steps, warm-up and L2 policy)
    per_config = {}
    if not args.no_per_config and args.num_seqs is None:
        for cid in range(len(inputs.CONFIG_NAMES)):
            if cid == args.workload:
                per_config[str(cid)] = head
                continue
            wc = inputs.make_config(cid)
            sc = DeviceState(wc, device)
            sc.run_setup()
            fb, note = l2_policy(torch, wc, device)
            sm, dm = time_decode_steps(torch, sc, stream, args.steps, args.warmup, fb, world,
                                       device)
            assert binding.pkv_get_device_status() == 0, f"device status flagged ({wc.name})"
            per_config[str(cid)] = per_config_entry(wc, sm, dm, peak, note, sc.prefix)
            del sc, fb
            torch.cuda.empty_cache()

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(slowest * 1e3, 5),
        "us_per_step": round(slowest * 1e6, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.q_dtype if w.kv_dtype != "e4m3" else "bf16+e4m3",
        "data": "synthetic (seeded N(0,1) q/K/V; seeded block permutation)",
        "config": {
            "workload": w.name, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "kv_dtype": w.kv_dtype,
            "mean_context": float(w.context_lens.mean()),
            "kv_read_bytes_per_step": w.kv_read_bytes,
            "unique_kv_bytes_per_step": w.unique_kv_bytes,
            "l2": l2_note,
            "step": "copy_blocks (if any) + reshape_and_cache + paged decode",
            "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic,
                     "dram_gbs": round(traffic / dec_s / 1e9, 1) if traffic else None,
                     "algorithmic_bytes": w.unique_kv_bytes,
                     "kernel": "planning + decode kernels (CUDA events around the decode call)",
                     "decode_us": round(dec_s * 1e6, 2)},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(float(np.mean(e2e_ms)), 5),
                "copies_per_step": "one host-to-device (packed inputs), one device-to-host",
                "launch": e2e_launch},
        "gpu_launches": nlaunch * args.steps,
        "clocks": clk,
        "copy_peak_gbs_same_run": round(copy_peak, 1) if copy_peak else None,
    }
    if per_config:
        line["per_config"] = per_config
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, secs, nbytes, threads, desc, single = oracle_baseline(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": threads,
                                "kind": "oracle", "sample": desc,
                                "seconds": round(secs, 2),
                                "single_thread": {"value": round(single, 4), "unit": "GB/s",
                                                  "sample": "one (sequence, kv head) unit"}}
    if rank == 0:
        print(json.dumps(line), flush=True)


MQ_METRIC = "multi-query paged attention (causal or draft tree): TFLOP/s"


def measured_tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if d.get("bf16_tflops"):
            return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json, bf16 burst)"
    return FALLBACK_BF16_TFLOPS, "fallback"


def mq_roofline(w, sec_att: float) -> dict:
    """Roofline of the multi-query attention launch: tensor-bound (TFLOP/s against the
    measured bf16 peak) when the workload's FLOPs per algorithmic byte (every cached K/V
    row once, the queries in, the outputs out) reach the ridge point of the measured
    peaks, HBM-bound (GB/s against the measured copy bandwidth) below it."""
    from paged_kv_cache_87_gb300.inputs import DTYPE_BYTES
    tpeak, tsrc = measured_tensor_peak()
    hpeak, hsrc = measured_peak()
    io_bytes = w.kv_bytes + 2 * w.total_q * w.num_q_heads * w.head_dim * DTYPE_BYTES[w.q_dtype]
    tflops = w.flops / sec_att / 1e12
    gbs = io_bytes / sec_att / 1e9
    intensity = w.flops / io_bytes
    ridge = tpeak * 1e12 / (hpeak * 1e9)
    r = {"flops_per_byte": round(intensity, 1), "ridge_flops_per_byte": round(ridge, 1),
         "algorithmic_bytes": io_bytes}
    if intensity >= ridge:
        r.update(bound="tensor", achieved=round(tflops, 1), peak=tpeak, peak_source=tsrc,
                 unit="TFLOP/s", frac=round(tflops / tpeak, 4),
                 hbm_frac=round(gbs / hpeak, 4))
    else:
        r.update(bound="hbm", achieved=round(gbs, 1), peak=hpeak, peak_source=hsrc,
                 unit="GB/s", frac=round(gbs / hpeak, 4),
                 tensor_frac=round(tflops / tpeak, 4), tflops=round(tflops, 1))
    return r


def mq_oracle_sample(w, target_s: float, nthreads: int, seed: int = 0, caches=None):
    """The oracle on sampled (query row, head) pairs; returns (TFLOP/s, s, flops, desc)."""
    import oracle
    rng = np.random.default_rng(seed)
    if caches is None:
        from paged_kv_cache_87_gb300 import inputs
        kc = inputs.poison_array(w.cache_shape, w.kv_dtype)
        vc = inputs.poison_array(w.cache_shape, w.kv_dtype)
        oracle.reshape_and_cache(w.key, w.value, kc, vc, w.slots, num_kv_heads=w.num_kv_heads,
                                 head_dim=w.head_dim, block_size=w.block_size,
                                 num_blocks=w.num_blocks, src_dtype=w.kv_dtype,
                                 kv_dtype=w.kv_dtype)
    else:
        kc, vc = caches
    seq_of_row = np.repeat(np.arange(w.num_seqs), np.diff(w.query_start))
    pos = (w.context_lens[seq_of_row] - np.diff(w.query_start)[seq_of_row] +
           (np.arange(w.total_q) - w.query_start[seq_of_row]))
    tree = getattr(w, "tree", None)
    if tree is not None:
        # visible keys of a draft-tree row: the prior context, itself, its ancestors
        anc = np.array([bin(int(x)).count("1") for x in tree], dtype=np.int64)
        prior = w.context_lens[seq_of_row] - np.diff(w.query_start)[seq_of_row]
        visible = prior + 1 + anc
    else:
        visible = pos + 1
    args = dict(num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                block_size=w.block_size, num_blocks=w.num_blocks, scale=w.scale,
                q_dtype=w.q_dtype, kv_dtype=w.kv_dtype, nthreads=nthreads)

    def run(k):
        rows = rng.integers(0, w.total_q, size=k)
        heads = rng.integers(0, w.num_q_heads, size=k)
        sel = np.stack([rows, heads], 1).astype(np.int32)
        t = time.perf_counter()
        if tree is not None:
            oracle.paged_tree_attention(w.query, kc, vc, w.block_tables, w.context_lens,
                                        w.query_start, tree, sel=sel, **args)
        else:
            oracle.paged_prefill_attention(w.query, kc, vc, w.block_tables, w.context_lens,
                                           w.query_start, sel=sel, **args)
        dt = time.perf_counter() - t
        return dt, int(4 * w.head_dim * visible[rows].sum())

    dt, fl = run(max(8, nthreads))                         # calibration
    k = int(max(8, nthreads) * max(1.0, target_s / max(dt, 1e-3)))
    dt, fl = run(k)
    return fl / dt / 1e12, dt, fl, (f"{k} random (query row, head) pairs of the workload, "
                                    f"{nthreads} threads")


def run_mq(args, rank, world, local):
    """The multi-query workload: per step, write the queries' own K/V and attend."""
    import torch
    from paged_kv_cache_87_gb300 import binding, build, inputs
    from paged_kv_cache_87_gb300.session import MultiQueryState

    build.build()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    w = inputs.make_multi_query_config(args.multi_query)
    st = MultiQueryState(w, device)
    st.run_setup()
    stream = torch.cuda.Stream(device)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush_buf = torch.empty(2 * l2 // 4 * 4, dtype=torch.uint8, device=device)
    launches_per_step = 3                     # reshape_and_cache, plan, attention
    clocks = ClockSampler(local)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            st.step(stream)
        stream.synchronize()
        barrier(world)
        torch.cuda.synchronize(device)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush_buf.zero_()
            s0, a0, a1, s1 = ev[i]
            s0.record(stream)
            st.append_step(stream)
            a0.record(stream)
            st.attend(stream)
            a1.record(stream)
            s1.record(stream)
        stream.synchronize()
        torch.cuda.synchronize(device)
        barrier(world)
    clk = clocks.stop()
    assert binding.pkv_get_device_status() == 0, "device status flagged during the benchmark"
    sec_step = float(np.mean([e[0].elapsed_time(e[3]) for e in ev])) * 1e-3
    sec_att = float(np.mean([e[1].elapsed_time(e[2]) for e in ev])) * 1e-3
    total, slowest, _ = aggregate(w.flops, sec_step, world, device)
    value = total / slowest / 1e12

    # end to end: one host-to-device copy of the step's inputs packed in one pinned
    # buffer, the step, the output copied back to pinned memory, every step
    h_in, d_in = st.pack_step_inputs()
    h_out = torch.empty_like(st.out, device="cpu").pin_memory()
    h2d, d2h = h_in.numel(), h_out.numel() * h_out.element_size()
    e2e_ms = []
    with torch.cuda.stream(stream):
        for i in range(args.warmup + args.steps):
            flush_buf.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            d_in.copy_(h_in, non_blocking=True)
            st.step(stream)
            h_out.copy_(st.out, non_blocking=True)
            b.record(stream)
            b.synchronize()
            if i >= args.warmup:
                e2e_ms.append(a.elapsed_time(b))
    tot_e, slow_e, _ = aggregate(w.flops, float(np.mean(e2e_ms)) * 1e-3, world, device)

    roof = mq_roofline(w, sec_att)
    traffic = recorded_traffic(f"mq{args.multi_query}")
    line = {
        "metric": MQ_METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(slowest * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.q_dtype,
        "data": "synthetic (seeded N(0,1) q/K/V; seeded block permutation)",
        "config": {"workload": w.name, "num_seqs": w.num_seqs, "total_queries": w.total_q,
                   "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
                   "head_dim": w.head_dim, "block_size": w.block_size,
                   "flops_per_step": w.flops, "kv_bytes": w.kv_bytes,
                   "l2": "L2 flushed between steps (write of 2x L2)",
                   "step": "reshape_and_cache of the queries' tokens + multi-query attention",
                   "parallelism": f"replicas x{world}"},
        "roofline": {**roof, "traffic": traffic,
                     "kernel": "planning + attention kernels (CUDA events around the call)",
                     "attention_us": round(sec_att * 1e6, 2)},
        "e2e": {"value": round(tot_e / slow_e / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(float(np.mean(e2e_ms)), 5)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, secs, fl, desc = mq_oracle_sample(w, args.cpu_seconds, os.cpu_count() or 1)
        line["cpu_baseline"] = {"value": round(v, 6), "unit": "TFLOP/s",
                                "cores": os.cpu_count() or 1, "kind": "oracle", "sample": desc,
                                "seconds": round(secs, 2)}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_mq_reference(args, rank, world, local):
    """The oracle on host cores, each step a bounded sample of the multi-query workload."""
    if rank != 0:
        return
    from paged_kv_cache_87_gb300 import inputs
    import oracle
    oracle.build()
    w = inputs.make_multi_query_config(args.multi_query)
    kc = inputs.poison_array(w.cache_shape, w.kv_dtype)
    vc = inputs.poison_array(w.cache_shape, w.kv_dtype)
    oracle.reshape_and_cache(w.key, w.value, kc, vc, w.slots, num_kv_heads=w.num_kv_heads,
                             head_dim=w.head_dim, block_size=w.block_size,
                             num_blocks=w.num_blocks, src_dtype=w.kv_dtype, kv_dtype=w.kv_dtype)
    threads = os.cpu_count() or 1
    per = max(0.5, args.cpu_seconds / max(1, args.steps + args.warmup))
    res = []
    for i in range(args.warmup + args.steps):
        v, secs, fl, desc = mq_oracle_sample(w, per, threads, seed=i, caches=(kc, vc))
        if i >= args.warmup:
            res.append((v, secs, fl))
    value = sum(r[2] for r in res) / sum(r[1] for r in res) / 1e12
    print(json.dumps({
        "impl": "reference", "metric": MQ_METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(float(np.mean([r[1] for r in res])) * 1e3, 3),
        "higher_is_better": True, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def run_reference(args, rank, world, local):
    """The oracle, as it stands, on host cores: each step a bounded sample of the workload."""
    if rank != 0:
        return
    from paged_kv_cache_87_gb300 import inputs
    import oracle
    oracle.build()
    from tests.helpers import oracle_caches
    w = inputs.make_config(args.workload, num_seqs=args.num_seqs)
    caches = oracle_caches(w)
    per_step = max(0.2, min(4.0, 150.0 / max(1, args.steps + args.warmup)))
    vals, secs, desc, threads = [], [], "", 1
    for i in range(args.warmup + args.steps):
        v, s, _, threads, desc, _ = oracle_baseline(w, per_step, seed=i, caches=caches)
        if i >= args.warmup:
            vals.append(v)
            secs.append(s)
    value = float(np.mean(vals))
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(float(np.mean(secs)) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "block_size": w.block_size, "kv_dtype": w.kv_dtype},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": "per step: " + desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_swap(args, rank, world, local):
    """Swap bandwidth: the workload's used blocks out to pinned host memory and back.

    Beside pkv_swap_blocks, the same number of bytes is moved in the same run by plain
    cudaMemcpyAsync calls (one per pool and direction, between a contiguous device
    range and the pinned pool): the host link's copy-engine rate, which the kernel's
    fraction is reported against."""
    import torch
    from paged_kv_cache_87_gb300 import binding, build, inputs
    from paged_kv_cache_87_gb300.session import DeviceState
    build.build()
    torch.cuda.set_device(local)
    w = inputs.make_config(args.workload, num_seqs=args.num_seqs)
    st = DeviceState(w, torch.device("cuda", local))
    st.run_setup()
    used = np.unique(w.block_tables[w.block_tables >= 0])
    hk = torch.empty((len(used),) + tuple(st.k_cache.shape[1:]), dtype=st.k_cache.dtype
                     ).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    out_pairs = torch.from_numpy(np.stack([used, np.arange(len(used))], 1).astype(np.int32)
                                 ).cuda()
    in_pairs = torch.from_numpy(np.stack([np.arange(len(used)), used], 1).astype(np.int32)
                                ).cuda()
    nbytes = 2 * len(used) * st.k_cache[0].numel() * st.k_cache.element_size()
    dk, dv = st.k_cache[:len(used)], st.v_cache[:len(used)]   # contiguous device ranges
    stream = torch.cuda.Stream()

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.steps):
                fn()
            e1.record(stream)
            e1.synchronize()
        return round(nbytes * args.steps / (e0.elapsed_time(e1) * 1e-3) / 1e9, 1)

    res = {}
    res["swap_out_gbs"] = timed(lambda: binding.pkv_swap_blocks(
        st.k_cache, st.v_cache, hk, hv, out_pairs, stream=stream))
    res["swap_in_gbs"] = timed(lambda: binding.pkv_swap_blocks(
        hk, hv, st.k_cache, st.v_cache, in_pairs, stream=stream))
    assert binding.pkv_get_device_status() == 0
    res["memcpy_d2h_gbs"] = timed(lambda: (hk.copy_(dk, non_blocking=True),
                                           hv.copy_(dv, non_blocking=True)))
    res["memcpy_h2d_gbs"] = timed(lambda: (dk.copy_(hk, non_blocking=True),
                                           dv.copy_(hv, non_blocking=True)))
    res["frac_out"] = round(res["swap_out_gbs"] / res["memcpy_d2h_gbs"], 4)
    res["frac_in"] = round(res["swap_in_gbs"] / res["memcpy_h2d_gbs"], 4)
    if rank == 0:
        print(json.dumps({"metric": "pkv_swap_blocks bandwidth (device pool <-> pinned host)",
                          "unit": "GB/s", **res, "bytes_per_call": nbytes,
                          "blocks": int(len(used)), "steps": args.steps,
                          "peak": {"out": res["memcpy_d2h_gbs"], "in": res["memcpy_h2d_gbs"],
                                   "source": "same-run cudaMemcpyAsync of the same bytes "
                                             "(contiguous device range <-> pinned pool)"},
                          "config": {"workload": w.name}}), flush=True)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.gpus != world and world > 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE {world}", file=sys.stderr)
    if args.record_traffic:
        if args.multi_query is not None:
            rec = record_traffic(args.record_traffic, f"mq{args.multi_query}",
                                 kernels=("mq_attention_kernel",))
        else:
            rec = record_traffic(args.record_traffic, args.workload)
        print(json.dumps(rec))
    elif args.multi_query is not None:
        if args.impl == "reference":
            run_mq_reference(args, rank, world, local)
        else:
            run_mq(args, rank, world, local)
    elif args.swap:
        run_swap(args, rank, world, local)
    elif args.impl == "reference":
        run_reference(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
