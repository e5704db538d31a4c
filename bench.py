"""Benchmark: paged decode attention on GB300.

Default workload: the LLaMA-13B-shaped full decode step — 40 layers x one fused call
(paged_decode_attention_ex: append the new token of each of 48 sequences, then attend
over 48 sequences x 40 heads x 2048 tokens, d 128, fp16 K/V, block size 16), with a
workspace zero-filled once, programmatic dependent launch, early tables and early K/V
tiles (the four launch flags; ``--launch-flags`` and ``--unfused`` select the other
forms).  The pool is
~75 GiB, far larger than L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the float64 oracle on the
host cores instead (the benchmark's reference arm).
"""

from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode-attn achieved HBM GB/s (% of GB300 peak); seq-steps/s"
# kv_decode_args.flags: KV_DECODE_WORKSPACE_ZEROED = 1, KV_DECODE_PDL = 2, KV_DECODE_EARLY_TABLES = 4,
# KV_DECODE_EARLY_POOL = 16
LAUNCH_FLAGS = {"none": 0, "zeroed": 1, "pdl": 3, "early": 7, "earlypool": 23}
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------------------- workloads
def make_workload(name: str):
    import workloads as W
    if name == "llama13b":
        w = W.llama13b()
    elif name == "llama7b":
        w = W.llama7b()
        w.lens = [n + w.steps for n in w.lens]       # context after the last of the 64 steps
    elif name in ("gqa70b", "gqa70b_fp8"):
        w = W.gqa70b()
        if name.endswith("fp8"):
            w.kv = "fp8"
    elif name == "longctx13b":
        w = W.longctx13b()
    elif name.startswith("ragged"):
        # ragged_f16_b16 | ragged_fp8_b8 ...
        _, dt, b = name.split("_")
        w = W.ragged(int(b[1:]))
        w.kv = dt
    else:
        raise SystemExit(f"unknown workload {name}")
    if not hasattr(w, "kv"):
        w.kv = w.dtype
    return w


def apply_overrides(w, args):
    if args.layers:
        w.num_layers = args.layers
    if args.block_size:
        w.block_size = args.block_size
    return w


def algorithmic_bytes(w, window: int = 0) -> int:
    """Bytes one paged_decode_attention call must move at minimum (one layer):
    K+V of every attended token, q, out (fp32), the block-table entries of the attended
    blocks, context_lens, and for FP8 pools the two per-block scales.  With a sliding
    window only the last `window` tokens of each sequence are attended."""
    kv_elem = 1 if w.kv == "fp8" else 2
    H, d, B = w.num_heads, w.head_dim, w.block_size
    Hq = w.q_heads                                   # query heads (grouped-query: > H)
    spans = [(n - min(n, window), n) if window > 0 else (0, n) for n in w.lens]
    nblk = [(-(-hi // B) - lo // B) if hi > lo else 0 for lo, hi in spans]
    kv = sum(hi - lo for lo, hi in spans) * H * d * kv_elem * 2
    q = w.batch * Hq * d * 2
    out = w.batch * Hq * d * 4
    tables = sum(nblk) * 4
    lens = w.batch * 4
    scales = sum(nblk) * 8 if w.kv == "fp8" else 0
    return kv + q + out + tables + lens + scales


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


KERNEL_SRCS = ("attention_kernel.cuh", "kvp_internal.cuh", "decode_attention.cu", "decode_attention_gqa.cu")


def kernel_sources_hash() -> str:
    """sha256 (16 hex digits) of the decode kernel's device and launch code."""
    src = [os.path.join(ROOT, "paged_kv_cache_169_gb300", "csrc", f) for f in KERNEL_SRCS]
    return hashlib.sha256(b"".join(open(f, "rb").read() for f in src)).hexdigest()[:16]


def traffic_record(workload: str):
    """DRAM bytes per launch of the workload's attention kernel from the committed ncu record
    profiles/traffic_<workload>.txt, only if the kernel sources are unchanged since the
    counters were taken (else None)."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    try:
        rec = {}
        for line in open(path):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                rec[k.strip()] = v.strip()
        if rec.get("source_sha256_16") == kernel_sources_hash():
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ----------------------------------------------------------------------------- clocks
def default_launch_flags(workload: str) -> str:
    """All four launch flags on every workload (a parallel-sampling step right after its
    copy-on-write drops the early K/V tiles: the copy kernel wrote rows it reads)."""
    return "earlypool"


class ClockSampler:
    """nvidia-smi samples every 50 ms; stop() keeps those taken between start() (after the
    first sample has arrived) and stop(), by their timestamps, and falls back to all of
    them when none falls inside."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.path = os.path.join("/tmp", f"kvpaged_clocks_{os.getpid()}.csv")
        self.t0 = 0.0

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            deadline = time.time() + 3.0         # the sampler is running before the region starts
            while time.time() < deadline and os.path.getsize(self.path) == 0 and self.proc.poll() is None:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        self.t0 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        t1 = time.time()
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm_mhz, max_mhz = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            active = {n for n, v in zip(names, parts[6:10]) if v.lower().startswith("active")}
            rows.append((ts, sm_mhz, max_mhz, active))
        os.unlink(self.path)
        inside = [r for r in rows if r[0] is not None and self.t0 - 0.06 <= r[0] <= t1 + 0.06]
        rows = inside or rows
        if not rows:
            return None
        sm = sorted(r[1] for r in rows)
        reasons = set().union(*(r[3] for r in rows))
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[2] for r in rows), "reasons": sorted(reasons),
                "samples": len(sm), "interval_ms": 50, "within_region": bool(inside)}


# ----------------------------------------------------------------------------- oracle (CPU)
def _oracle_worker(args):
    """Time the oracle on `units` (sequence, head) decode problems of context n (float64)."""
    units, n, d, seed = args
    import numpy as np
    from oracle import attention as OA
    rng = np.random.default_rng(seed)
    distinct = min(units, 32)                  # bounded host memory; each unit still widens
    data = [(rng.standard_normal(d).astype(np.float16),        # its own fp16 inputs to float64
             rng.standard_normal((n, d), dtype=np.float32).astype(np.float16),
             rng.standard_normal((n, d), dtype=np.float32).astype(np.float16)) for _ in range(distinct)]
    t0 = time.perf_counter()
    for i in range(units):
        q, K, V = data[i % distinct]
        OA.decode_attention_one(q, K, V, 1.0 / math.sqrt(d))
    return time.perf_counter() - t0


def oracle_rate(w, units_total: int):
    """Oracle throughput on a bounded sample of the workload, in the metric's unit (GB/s of
    algorithmic bytes), using every available host core (one single-threaded process each)."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    n = max(w.lens)
    per = [units_total // cores + (1 if i < units_total % cores else 0) for i in range(cores)]
    per = [p for p in per if p > 0]
    env_keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    old = {k: os.environ.get(k) for k in env_keys}
    for k in env_keys:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(len(per)) as pool:
            t0 = time.perf_counter()
            times = pool.map(_oracle_worker, [(p, n, w.head_dim, 1000 + i) for i, p in enumerate(per)])
            wall = time.perf_counter() - t0
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    busy = max(times)
    bytes_per_unit = n * w.head_dim * 2 * 2 + w.head_dim * 2 + w.head_dim * 4
    gbs = units_total * bytes_per_unit / busy / 1e9
    # one process's own rate (single-threaded, while the other cores run theirs)
    one_core = sum(p * bytes_per_unit / t for p, t in zip(per, times)) / len(per) / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": len(per), "kind": "oracle",
            "sample": f"{units_total} (sequence, head) units of context {n}, d {w.head_dim}, "
                      f"fp16 inputs widened to float64; numpy, one single-threaded process per core",
            "one_core_value": one_core, "seconds": busy, "wall_seconds": wall}


# ----------------------------------------------------------------------------- distributed
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, x: float, device: str = "cuda") -> float:
    """Largest value over all ranks (the slowest rank's elapsed time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, bytes_per_step_per_rank: int, steps: int, elapsed_ms_max: float) -> float:
    """Whole-job GB/s: every rank processes its own replica of the workload (weak scaling);
    the job takes as long as the slowest rank."""
    return world * bytes_per_step_per_rank * steps / (elapsed_ms_max / 1e3) / 1e9


# ----------------------------------------------------------------------------- reference arm
def workload_config(w, args) -> dict:
    """The workload keys of a bench line's config (shared by both arms)."""
    return {"workload": args.workload, "layers": w.num_layers, "batch": w.batch, "heads": w.num_heads,
            "q_heads": w.q_heads, "head_dim": w.head_dim, "block_size": w.block_size, "kv_dtype": w.kv,
            "context_mean": sum(w.lens) / len(w.lens), "context_max": max(w.lens),
            "window": args.window or None}


def run_reference(args):
    world, rank, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return 0
    w = make_workload(args.workload)
    units = args.ref_units
    for _ in range(args.warmup):
        oracle_rate(w, max(1, units // 8))
    t0 = time.perf_counter()
    vals = [oracle_rate(w, units) for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    value = sum(v["value"] for v in vals) / len(vals)
    per_step_units = units
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": wall / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(apply_overrides(w, args), args) | {
            "sample_units_per_step": per_step_units,
            "sample": "each step times the oracle on this many (sequence, head) units of the workload"},
        "cpu_baseline": {k: vals[-1][k] for k in ("kind", "cores", "sample")} | {"value": value, "unit": "GB/s"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- our arm
def run_ours(args):
    import numpy as np
    import torch

    import workloads as W
    from paged_kv_cache_169_gb300 import build as B
    from paged_kv_cache_169_gb300.cache import PagedKVCache

    world, rank, local = dist_setup(args.gpus)
    B.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = apply_overrides(make_workload(args.workload), args)
    L, H, d, BS = w.num_layers, w.num_heads, w.head_dim, w.block_size
    nbs = [-(-n // BS) for n in w.lens]
    w.num_blocks = max(w.num_blocks, sum(nbs))
    cache = PagedKVCache(L, w.num_blocks, BS, H, d, w.kv, device=dev)
    for l in range(L):
        if w.kv == "fp8":
            for pool, sc, key in ((cache.k[l], cache.k_scale[l], 0), (cache.v[l], cache.v_scale[l], 1)):
                g = torch.Generator(device=dev)
                g.manual_seed(w.seed * 1000 + 2 * l + key)
                for b0 in range(0, w.num_blocks, 4096):
                    nb = min(4096, w.num_blocks - b0)
                    x = torch.randn((nb, H, BS, d), generator=g, device=dev).half().float()
                    s = (x.abs().amax(dim=(1, 2, 3)).clamp_min(2.0 ** -20 * 448) / 448.0).float()
                    pool[b0:b0 + nb].copy_((x / s.view(-1, 1, 1, 1)).clamp(-448, 448)
                                           .to(torch.float8_e4m3fn).view(torch.uint8))
                    sc[b0:b0 + nb].copy_(s)
        else:
            W.device_fill_normal(cache.k[l], w.seed * 1000 + 2 * l)
            W.device_fill_normal(cache.v[l], w.seed * 1000 + 2 * l + 1)
    tables = W.shuffled_tables(w, nbs)
    slots_h = np.array([int(tables[s, (n - 1) // BS]) * BS + (n - 1) % BS for s, n in enumerate(w.lens)],
                       dtype=np.int64)
    lens_h = np.array(w.lens, dtype=np.int32)
    tdt = torch.float16
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed * 7 + 1)
    Hq = w.q_heads
    q = torch.randn((L, w.batch, Hq, d), generator=g, device=dev).to(tdt)
    k_new = torch.randn((L, w.batch, H, d), generator=g, device=dev).to(tdt)
    v_new = torch.randn((L, w.batch, H, d), generator=g, device=dev).to(tdt)
    bt = torch.from_numpy(tables).to(dev)
    cl = torch.from_numpy(lens_h).to(dev)
    slots = torch.from_numpy(slots_h).to(dev)
    out = torch.empty((L, w.batch, Hq, d), dtype=torch.float32, device=dev)
    max_ctx = max(w.lens)
    grouped = Hq != H
    flags = LAUNCH_FLAGS[args.launch_flags]
    if flags & 1:
        # zero-filled once; every decode launch leaves its counters zero again
        ws = cache.zeroed_workspace(w.batch, max_ctx, args.partition, num_q_heads=Hq, window=args.window)
    elif args.window:
        from paged_kv_cache_169_gb300 import abi as _abi
        xa = _abi.kv_decode_args()
        xa.num_q_heads, xa.batch, xa.max_context = Hq, w.batch, max_ctx
        xa.window, xa.partition_tokens = args.window, args.partition
        ws = torch.empty(_abi.paged_decode_workspace_size_ex(cache.handle, xa), dtype=torch.uint8, device=dev)
    elif grouped:
        from paged_kv_cache_169_gb300 import abi as _abi
        ws = torch.empty(_abi.paged_decode_workspace_size_gqa(cache.handle, w.batch, Hq, max_ctx, args.partition),
                         dtype=torch.uint8, device=dev)
    else:
        ws = cache.workspace(w.batch, max_ctx, args.partition)
    stream = torch.cuda.current_stream(dev)

    from paged_kv_cache_169_gb300 import abi
    # my kernels per layer: the attention kernel (one per 1024 sequences) [+ kv_append]
    launches_per_layer = (1 if args.unfused else 0) + 1 + (w.batch - 1) // 1024

    def layer_call(l, ev=None):
        if args.unfused:
            cache.append(l, k_new[l], v_new[l], slots)
        if ev is not None:
            ev[l][0].record(stream)
        if args.window or flags:
            cache.attention_ex(l, q[l], bt, cl, max_ctx, w.scale, window=args.window,
                               k_new=None if args.unfused else k_new[l],
                               v_new=None if args.unfused else v_new[l], out=out[l],
                               partition_tokens=args.partition, workspace=ws, flags=flags)
        elif grouped:
            cache.attention_gqa(l, q[l], bt, cl, max_ctx, w.scale,
                                k_new=None if args.unfused else k_new[l],
                                v_new=None if args.unfused else v_new[l], out=out[l],
                                partition_tokens=args.partition, workspace=ws)
        elif args.unfused:
            cache.attention(l, q[l], bt, cl, max_ctx, w.scale, out=out[l],
                            partition_tokens=args.partition, workspace=ws)
        else:   # one launch: append each sequence's newest token, then attend
            cache.attention_append(l, q[l], k_new[l], v_new[l], bt, cl, max_ctx, w.scale, out=out[l],
                                   partition_tokens=args.partition, workspace=ws)
        if ev is not None:
            ev[l][1].record(stream)

    def step(ev=None):
        for l in range(L):
            layer_call(l, ev)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if cache.device_error() != 0:
        raise SystemExit("device error during warm-up")

    # ---- device-timed region
    evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in range(L)]
           for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    # Per-call events would sit between consecutive launches and stop programmatic
    # dependent launch from overlapping them, so the timed region holds only the launches:
    # the fused step's one kernel per layer is timed as the region's duration over its
    # calls.  The unfused step (append + attention kernels) records events per call.
    per_call_events = args.unfused
    for i in range(args.steps):
        step(evs[i] if per_call_events else None)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    elapsed_ms = max_over_ranks(world, t_start.elapsed_time(t_end))
    if per_call_events:
        attn_ms = [e[0].elapsed_time(e[1]) for row in evs for e in row]
        attn_ms_mean = sum(attn_ms) / len(attn_ms)
    else:
        attn_ms_mean = t_start.elapsed_time(t_end) / (args.steps * L)

    # ---- end-to-end through the public API with host buffers
    pin = dict(q=torch.empty(q.shape, dtype=tdt).pin_memory(), k=torch.empty(k_new.shape, dtype=tdt).pin_memory(),
               v=torch.empty(v_new.shape, dtype=tdt).pin_memory(), out=torch.empty(out.shape).pin_memory(),
               slots=torch.from_numpy(slots_h).pin_memory(), bt=torch.from_numpy(tables).pin_memory(),
               cl=torch.from_numpy(lens_h).pin_memory())
    pin["q"].copy_(q.cpu())
    pin["k"].copy_(k_new.cpu())
    pin["v"].copy_(v_new.cpu())
    h2d = sum(pin[k].numel() * pin[k].element_size() for k in ("q", "k", "v", "slots", "bt", "cl"))
    d2h = pin["out"].numel() * pin["out"].element_size()

    # The step's copies overlap its layers: tables, lengths and the first `pre` layers'
    # inputs go first on the compute stream; the other layers' inputs follow on a copy
    # stream (layer `pre` waits for them), and the outputs return in chunks on the copy
    # stream while later layers run (only the last layer's output is copied after it).
    # Every event between two launches costs that pair its programmatic-dependent-launch
    # overlap, so there are few: one wait for the inputs, two output chunks, one join.
    copy_stream = torch.cuda.Stream(dev)
    pre = min(L, 2)
    marks = sorted({m for m in (L // 2 - 1, L - 2) if pre <= m < L - 1}) if L >= 4 else []
    ev_start, ev_in, ev_join = (torch.cuda.Event() for _ in range(3))
    ev_out = {m: torch.cuda.Event() for m in marks}

    def e2e_step():
        slots.copy_(pin["slots"], non_blocking=True)
        bt.copy_(pin["bt"], non_blocking=True)
        cl.copy_(pin["cl"], non_blocking=True)
        for dst, key in ((q, "q"), (k_new, "k"), (v_new, "v")):
            dst[:pre].copy_(pin[key][:pre], non_blocking=True)
        ev_start.record(stream)                     # the previous step is done with every buffer
        copy_stream.wait_event(ev_start)
        with torch.cuda.stream(copy_stream):
            for dst, key in ((q, "q"), (k_new, "k"), (v_new, "v")):
                dst[pre:].copy_(pin[key][pre:], non_blocking=True)
            ev_in.record(copy_stream)
        first = 0
        for l in range(L):
            if l == pre:
                stream.wait_event(ev_in)
            layer_call(l)
            if l in ev_out:
                ev_out[l].record(stream)
                copy_stream.wait_event(ev_out[l])
                with torch.cuda.stream(copy_stream):
                    pin["out"][first:l + 1].copy_(out[first:l + 1], non_blocking=True)
                first = l + 1
        pin["out"][first:].copy_(out[first:], non_blocking=True)
        ev_join.record(copy_stream)
        stream.wait_event(ev_join)

    e2e_step()
    torch.cuda.synchronize()
    pin["out"].fill_(float("nan"))                 # every output chunk must come back
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(world, e0.elapsed_time(e1))
    if not torch.equal(pin["out"].view(torch.int32), out.cpu().view(torch.int32)):   # bitwise
        raise SystemExit("end-to-end step: the host copy of the outputs differs from the device's")
    err = cache.device_error()
    if err != 0:
        raise SystemExit(f"device error bits {err}")

    # ---- numbers
    alg = algorithmic_bytes(w, args.window)
    step_bytes = alg * L
    # the timed call's own minimum traffic: the fused call also reads the new K/V and
    # writes them into the pool
    esz = 1 if w.kv == "fp8" else 2
    call_bytes = alg if args.unfused else alg + w.batch * H * d * 2 * (2 + esz)
    ms_per_step = elapsed_ms / args.steps
    value = job_throughput(world, step_bytes, args.steps, elapsed_ms)
    peak, peak_src = measured_peak()
    achieved = call_bytes / (attn_ms_mean / 1e3) / 1e9
    traffic = traffic_record(args.workload) if not (args.window or args.unfused or args.block_size) else None
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = oracle_rate(w, args.cpu_units)
        cpu.pop("wall_seconds", None)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32-accum/" + w.kv, "data": "synthetic",
        "config": workload_config(w, args) | {
                   "pool_gib": round(2 * L * w.num_blocks * H * BS * d * (1 if w.kv == "fp8" else 2) / 2 ** 30, 2),
                   "l2": "no flush: inputs (the KV pool) larger than L2",
                   "partition_tokens": args.partition or "auto", "parallelism": f"replica x{world}",
                   "launch_flags": args.launch_flags,
                   "step": "kv_append + paged_decode_attention" if args.unfused
                           else "paged_decode_attention_append (fused)"},
        "pct_of_peak": 100.0 * value / world / peak,
        "seq_steps_per_s": world * w.batch * args.steps / (elapsed_ms / 1e3),
        "roofline": {"bound": "hbm",
                     "kernel": ("paged_decode_attention" if args.unfused
                                else "paged_decode_attention_append (fused append + attention)"),
                     "achieved": achieved, "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": call_bytes, "mean_call_ms": attn_ms_mean,
                     "call_timing": ("CUDA events around each call" if per_call_events else
                                     "CUDA events around the timed region / calls in it (the only kernel "
                                     "of the step; consecutive launches overlap under PDL)")},
        "cpu_baseline": cpu,
        "e2e": {"value": job_throughput(world, step_bytes, args.steps, e2e_ms), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms / args.steps},
        "gpu_launches": launches_per_layer * L * args.steps,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    cache.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    del abi
    return 0


def run_swap(args):
    """Block-swap bandwidth: one LLaMA-13B-shaped sequence (2048 tokens = 128 blocks, all 40
    layers, K and V: 1.68 GB) moved to pinned host memory and back per step."""
    import numpy as np
    import torch

    import workloads as W
    from paged_kv_cache_169_gb300 import build as B
    from paged_kv_cache_169_gb300.cache import PagedKVCache

    B.build()
    w = W.llama13b()
    L = w.num_layers
    cache = PagedKVCache(L, w.num_blocks, w.block_size, w.num_heads, w.head_dim, "f16")
    for t in cache.k + cache.v:
        t.zero_()
    perm = W.free_order(w)
    out_ids = torch.from_numpy(perm[:128].copy()).cuda()
    in_ids = torch.from_numpy(perm[128:256].copy()).cuda()
    host = cache.swap_out(out_ids)                       # allocates the pinned image
    nbytes = host.numel()
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        cache.swap_out(out_ids, host)
        cache.swap_in(host, in_ids)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    t_out = t_in = 0.0
    for _ in range(args.steps):
        ev[0].record(stream)
        cache.swap_out(out_ids, host)
        ev[1].record(stream)
        cache.swap_in(host, in_ids)
        ev[2].record(stream)
        torch.cuda.synchronize()
        t_out += ev[0].elapsed_time(ev[1])
        t_in += ev[1].elapsed_time(ev[2])
    err = cache.device_error()
    if err:
        raise SystemExit(f"device error bits {err}")
    out_gbs = nbytes * args.steps / (t_out / 1e3) / 1e9
    in_gbs = nbytes * args.steps / (t_in / 1e3) / 1e9
    line = {"metric": "kv block swap GB/s (device <-> pinned host, one 13B-shaped sequence)",
            "value": 2 * nbytes * args.steps / ((t_out + t_in) / 1e3) / 1e9, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": (t_out + t_in) / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": "swap13b", "layers": L, "blocks": 128, "bytes_per_direction": nbytes},
            "swap_out_gbs": out_gbs, "swap_in_gbs": in_gbs, "gpu_launches": 2 * args.steps}
    print(json.dumps(line), flush=True)
    cache.close()
    del np
    return 0



def abi_workspace_bytes(cache, batch, max_ctx, partition, prefix_groups):
    from paged_kv_cache_169_gb300 import abi
    a = abi.kv_decode_args()
    a.batch, a.max_context, a.partition_tokens = batch, max_ctx, partition
    a.num_prefix_groups = 1 if prefix_groups else 0
    return abi.paged_decode_workspace_size_ex(cache.handle, a)


def host_step_loop(cache, alloc, seqs, q_h, k_h, v_h, max_blocks, max_ctx, scale, stream, groups=None,
                   partition=0):
    """The decode loop as a caller runs it, one kv_decode_step call per step, which does:
      1. the host allocator reserves every sequence's next slot (kv_alloc_decode_step),
         planning a block copy where a slot lies in a shared block;
      2. it writes the block tables and lengths into a pinned staging buffer
         (kv_alloc_build_tables), beside the planned block pairs;
      3. that buffer goes to the device in one copy, and the step's q / new K / new V
         (packed in pinned memory) in another;
      4. the planned block copies run (kv_copy_blocks, every layer);
      5. the fused append + attention runs (paged_decode_attention_ex with an argument block
         built once: zeroed workspace and programmatic dependent launch; a host copy precedes
         every call, so no early flags);
      6. the outputs are copied back to pinned host memory.
    q_h, k_h, v_h: host [steps, batch, H, d].  Returns (ms for all steps, H2D bytes, D2H
    bytes, block copies, the pinned outputs)."""
    import ctypes
    import torch
    from paged_kv_cache_169_gb300 import abi

    S, n = q_h.shape[0], q_h.shape[1]
    dev = cache.k[0].device
    per = q_h[0].numel()
    # per step, one pinned row: [tables n*max_blocks | lengths n | block pairs 2n] int32,
    # padding to 256 bytes, then q | k | v; the device copy has the same layout, so the
    # step's inputs travel with its tables in one copy
    width = n * max_blocks + n + 2 * n
    off = (width * 4 + 255) // 256 * 256
    qkv_bytes = 3 * per * q_h.element_size()
    qkv_shape = (3, n) + tuple(q_h.shape[2:])
    pin_rows = torch.empty((S, off + qkv_bytes), dtype=torch.uint8).pin_memory()
    for i in range(S):
        pq = pin_rows[i, off:].view(q_h.dtype).view(qkv_shape)
        pq[0].copy_(q_h[i])
        pq[1].copy_(k_h[i])
        pq[2].copy_(v_h[i])
    pin_out = torch.empty(q_h.shape, dtype=torch.float32).pin_memory()
    d_row = torch.empty(off + qkv_bytes, dtype=torch.uint8, device=dev)
    d_meta = d_row[:width * 4].view(torch.int32)
    d_bt = d_meta[:n * max_blocks].view(n, max_blocks)
    d_cl = d_meta[n * max_blocks:n * max_blocks + n]
    d_qkv = d_row[off:].view(q_h.dtype).view(qkv_shape)
    d_out = torch.empty(q_h.shape[1:], dtype=torch.float32, device=dev)
    ws = cache.zeroed_workspace(n, max_ctx, partition, prefix_groups=groups is not None)
    seq_arr = (ctypes.c_int32 * n)(*seqs)
    a = abi.kv_decode_args()                            # every pointer is fixed over the loop
    a.layer, a.q, a.num_q_heads = 0, d_qkv[0].data_ptr(), 0
    a.k_new, a.v_new, a.in_dtype = d_qkv[1].data_ptr(), d_qkv[2].data_ptr(), abi.KV_F16
    a.out, a.block_tables, a.max_blocks_per_seq = d_out.data_ptr(), d_bt.data_ptr(), max_blocks
    a.context_lens, a.batch, a.max_context = d_cl.data_ptr(), n, max_ctx
    a.scale, a.partition_tokens = float(scale), partition
    a.workspace, a.workspace_bytes = ws.data_ptr(), ws.numel()
    a.stream = stream.cuda_stream
    a.flags = abi.KV_DECODE_WORKSPACE_ZEROED | abi.KV_DECODE_PDL
    if groups is not None:
        a.prefix_groups, a.num_prefix_groups = groups.data_ptr(), groups.shape[0]
    handle = cache.handle
    h2d = d2h = copies = 0
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(S):
            row = pin_rows[i].data_ptr()
            copies += abi.kv_decode_step(alloc.handle, handle, seq_arr, n, max_blocks, row, d_row.data_ptr(),
                                         row + off, d_row.data_ptr() + off, qkv_bytes,
                                         pin_out[i].data_ptr(), per * 4, a)
            h2d += off + qkv_bytes
            d2h += per * 4
        ev[1].record(stream)
    stream.synchronize()
    return ev[0].elapsed_time(ev[1]), h2d, d2h, copies, pin_out


def _flush_l2(buf):
    buf.add_(1)                                         # 256 MB write: evicts the 129 MB L2


def run_decode_steps(args):
    """LLaMA-7B-shaped decode loop: batch 8, contexts 512..2048 before the loop, 64 steps of
    (append one token per sequence + attend) on one layer with the fused call.  The 64 calls
    are captured once in a CUDA graph and replayed (L2 flushed between replays); the same 64
    calls issued eagerly are timed too."""
    import torch

    import workloads as W
    from paged_kv_cache_169_gb300 import build as B
    from paged_kv_cache_169_gb300.cache import PagedKVCache

    B.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = W.llama7b()
    w.kv = w.dtype
    S, H, d, BS = w.steps, w.num_heads, w.head_dim, w.block_size
    init = [n - 1 for n in w.lens]                      # contexts before the first step
    nbs = [-(-(n + S) // BS) for n in init]
    w.num_blocks = max(w.num_blocks, sum(nbs))
    cache = PagedKVCache(1, w.num_blocks, BS, H, d, "f16", device=dev)
    W.device_fill_normal(cache.k[0], w.seed * 1000)
    W.device_fill_normal(cache.v[0], w.seed * 1000 + 1)
    bt = torch.from_numpy(W.shuffled_tables(w, nbs)).to(dev)
    lens = torch.tensor([[n + i + 1 for n in init] for i in range(S)], dtype=torch.int32, device=dev)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed * 7 + 1)
    shape = (S, w.batch, H, d)
    q, kn, vn = (torch.randn(shape, generator=g, device=dev).half() for _ in range(3))
    out = torch.empty(shape, dtype=torch.float32, device=dev)
    max_ctx = max(init) + S
    flags = LAUNCH_FLAGS[args.launch_flags]
    ws = (cache.zeroed_workspace(w.batch, max_ctx, args.partition) if flags & 1
          else cache.workspace(w.batch, max_ctx, args.partition))
    stream = torch.cuda.Stream(dev)

    def loop():
        for i in range(S):
            if flags:
                cache.attention_ex(0, q[i], bt, lens[i], max_ctx, w.scale, k_new=kn[i], v_new=vn[i],
                                   out=out[i], partition_tokens=args.partition, workspace=ws, stream=stream,
                                   flags=flags)
            else:
                cache.attention_append(0, q[i], kn[i], vn[i], bt, lens[i], max_ctx, w.scale, out=out[i],
                                       partition_tokens=args.partition, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            loop()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        loop()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    # algorithmic bytes of the 64 steps (each step's contexts, plus the appended token)
    step_bytes = 0
    for i in range(S):
        w.lens = [n + i + 1 for n in init]
        step_bytes += algorithmic_bytes(w) + w.batch * H * d * 2 * (2 + 2)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed(fn):
        total = 0.0
        for _ in range(args.steps):
            with torch.cuda.stream(stream):
                _flush_l2(flush)
                ev[0].record(stream)
                fn()
                ev[1].record(stream)
            stream.synchronize()
            total += ev[0].elapsed_time(ev[1])
        return total / args.steps

    for _ in range(args.warmup):
        graph.replay()
    stream.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    graph_ms = timed(graph.replay)
    clk = clocks.stop()
    eager_ms = timed(loop)
    # end to end: the 64 steps' q / k / v from pinned host memory, the outputs back, around
    # the replayed graph
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, kn, vn))
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e():
        q.copy_(hq, non_blocking=True)
        kn.copy_(hk, non_blocking=True)
        vn.copy_(hv, non_blocking=True)
        graph.replay()
        hout.copy_(out, non_blocking=True)

    graph_e2e_ms = timed(e2e)
    # end to end with the host step of every decode step (host_step_loop): the host
    # allocator holds the 8 sequences at their lengths before the loop (the prefill, not
    # timed; its tables map the same pool) and reserves one slot per sequence per step
    from paged_kv_cache_169_gb300.cache import BlockAllocator
    runs = []
    for rep in range(1 + max(2, min(args.steps, 5))):
        alloc = BlockAllocator(w.num_blocks, BS, W.free_order(w))
        seqs = [alloc.new_seq() for _ in init]
        for sid, n in zip(seqs, init):
            alloc.append_slots(sid, n)
        with torch.cuda.stream(stream):
            _flush_l2(flush)
        run_ms, h2d, d2h, _, _ = host_step_loop(cache, alloc, seqs, hq, hk, hv, max(nbs), max_ctx, w.scale, stream,
                                                partition=args.partition)
        alloc.close()
        if rep:
            runs.append(run_ms)
    e2e_ms = sum(runs) / len(runs)
    if cache.device_error():
        raise SystemExit("device error during the decode loop")
    peak, peak_src = measured_peak()
    achieved = step_bytes / (graph_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": achieved, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": graph_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32-accum/f16", "data": "synthetic",
        "config": {"workload": "decode7b", "layers": 1, "batch": w.batch, "heads": H, "head_dim": d,
                   "block_size": BS, "decode_steps_per_replay": S, "context_before": [min(init), max(init)],
                   "launch_flags": args.launch_flags,
                   "l2": "flushed (256 MB write) between timed replays", "step": "64 fused calls, one CUDA graph"},
        "seq_steps_per_s": w.batch * S / (graph_ms / 1e3),
        "eager": {"ms_per_64_steps": eager_ms, "GB/s": step_bytes / (eager_ms / 1e3) / 1e9},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic_record("decode7b"),
                     "traffic_note": "DRAM bytes of one launch (one decode step), ncu",
                     "algorithmic_bytes_per_replay": step_bytes},
        "e2e": {"value": step_bytes / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "step": "64 decode steps, one kv_decode_step call each: allocator slot reservation, tables "
                        "into pinned memory, one H2D of tables, lengths, q and new K/V, the fused call, D2H "
                        "of the outputs"},
        "e2e_graph": {"value": step_bytes / (graph_e2e_ms / 1e3) / 1e9, "unit": "GB/s",
                      "h2d_bytes_per_step": 3 * q.numel() * 2, "d2h_bytes_per_step": out.numel() * 4,
                      "ms_per_step": graph_e2e_ms,
                      "step": "the 64 steps' q / new K / new V copied in, the graph replayed, outputs copied out"},
        "gpu_launches": S, "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    cache.close()
    return 0


def run_parallel(args):
    """Parallel sampling: 8 candidates forked from one 1030-token prompt (65 shared blocks,
    the last one partial) decode 128 steps on one LLaMA-13B-shaped layer (40 heads, d 128,
    fp16, B 16).  The first step copies the partial block for 7 candidates (copy-on-write)
    and writes the 8th in place.  A step is (the step's block copies, if any) + one fused
    append + attend call.  The allocator decisions are planned on the host before the
    timed loop.  Logical bytes count every candidate's whole context; unique bytes count
    each physical block once per step (the shared prefix is read from HBM once and then
    from L2), and the roofline fraction uses the unique bytes."""
    import numpy as np
    import torch

    import workloads as W
    from paged_kv_cache_169_gb300 import build as B
    from paged_kv_cache_169_gb300.cache import BlockAllocator, PagedKVCache

    B.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = W.parallel_sampling()
    w.kv = w.dtype
    S, H, d, BS, C = w.steps, w.num_heads, w.head_dim, w.block_size, w.batch
    prompt = W.PROMPT_LEN_PARALLEL
    cache = PagedKVCache(1, w.num_blocks, BS, H, d, "f16", device=dev)
    W.device_fill_normal(cache.k[0], w.seed * 1000)
    W.device_fill_normal(cache.v[0], w.seed * 1000 + 1)
    alloc = BlockAllocator(w.num_blocks, BS, W.free_order(w))
    root = alloc.new_seq()
    alloc.append_slots(root, prompt)
    cands = [root] + [alloc.fork(root) for _ in range(C - 1)]
    max_blocks = -(-(prompt + S) // BS)
    tables, lens, cows, logical, unique = [], [], [], 0, 0
    for i in range(S):
        pairs = []
        for sid in cands:
            _, cow = alloc.append_slots(sid, 1)
            if cow:
                pairs.append(cow)
        tabs, ls = alloc.build_tables(cands, max_blocks)
        tables.append(tabs)
        lens.append(ls)
        cows.append(torch.tensor(pairs, dtype=torch.int32, device=dev).reshape(-1, 2) if pairs else None)
        ctx = ls[0]
        logical += C * ctx * H * d * 2 * 2
        unique += len({b for t in tabs for b in t[: -(-ctx // BS)]}) * H * BS * d * 2 * 2
    n_cow = sum(0 if c is None else c.shape[0] for c in cows)
    bt = torch.tensor(np.array(tables, dtype=np.int32), device=dev)       # [S, C, max_blocks]
    cl = torch.tensor(np.array(lens, dtype=np.int32), device=dev)         # [S, C]
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed * 7 + 1)
    shape = (S, C, H, d)
    q, kn, vn = (torch.randn(shape, generator=g, device=dev).half() for _ in range(3))
    out = torch.empty(shape, dtype=torch.float32, device=dev)
    max_ctx = prompt + S
    flags = LAUNCH_FLAGS[args.launch_flags]
    # the candidates share the prompt's whole blocks (64 of them) for all 128 steps: one
    # prefix group, so each shared (block, head) tile is read once for all 8 query rows
    use_groups = not args.no_prefix_groups
    groups = torch.tensor([[0, C, (prompt // BS) * BS]], dtype=torch.int32, device=dev) if use_groups else None
    if flags & 1:
        ws = cache.zeroed_workspace(C, max_ctx, args.partition, prefix_groups=use_groups)
    else:
        ws = torch.zeros(abi_workspace_bytes(cache, C, max_ctx, args.partition, use_groups), dtype=torch.uint8,
                         device=dev)
    stream = torch.cuda.Stream(dev)

    def loop():
        for i in range(S):
            if cows[i] is not None:
                cache.copy_blocks(cows[i], stream=stream)
            if flags or use_groups:
                # a step after block copies reads rows the copy kernel just wrote: no early pool
                cache.attention_ex(0, q[i], bt[i], cl[i], max_ctx, w.scale, k_new=kn[i], v_new=vn[i],
                                   out=out[i], partition_tokens=args.partition, workspace=ws, stream=stream,
                                   flags=flags if cows[i] is None else flags & ~16, prefix_groups=groups)
            else:
                cache.attention_append(0, q[i], kn[i], vn[i], bt[i], cl[i], max_ctx, w.scale, out=out[i],
                                       partition_tokens=args.partition, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            loop()
    stream.synchronize()
    # the 128 steps are captured once in a CUDA graph and replayed (as a serving loop
    # would); replaying repeats the same copies and appends, so the pool ends identical
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        loop()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed(fn):
        total = 0.0
        for _ in range(args.steps):
            with torch.cuda.stream(stream):
                _flush_l2(flush)
                ev[0].record(stream)
                fn()
                ev[1].record(stream)
            stream.synchronize()
            total += ev[0].elapsed_time(ev[1])
        return total / args.steps

    for _ in range(args.warmup):
        graph.replay()
    stream.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    ms = timed(graph.replay)
    clk = clocks.stop()
    eager_ms = timed(loop)
    if cache.device_error():
        raise SystemExit("device error during parallel sampling")
    # end to end with the host step of every decode step (host_step_loop), from the forked
    # state each time (the fork itself is the prefill, not timed); the first run warms up
    pin_q, pin_k, pin_v = (t.cpu().pin_memory() for t in (q, kn, vn))
    runs = []
    for rep in range(1 + max(2, min(args.steps, 5))):
        a2 = BlockAllocator(w.num_blocks, BS, W.free_order(w))
        r2 = a2.new_seq()
        a2.append_slots(r2, prompt)
        c2 = [r2] + [a2.fork(r2) for _ in range(C - 1)]
        with torch.cuda.stream(stream):
            _flush_l2(flush)
        run_ms, h2d, d2h, n_copies, host_out = host_step_loop(cache, a2, c2, pin_q, pin_k, pin_v, max_blocks, max_ctx,
                                                              w.scale, stream, groups=groups,
                                                              partition=args.partition)
        a2.close()
        if rep:
            runs.append(run_ms)
    e2e_ms = sum(runs) / len(runs)
    # the same decisions and inputs as the timed graph: the same result, bit for bit
    if n_copies != n_cow or not torch.equal(host_out.view(torch.int32), out.cpu().view(torch.int32)):
        raise SystemExit("host-step loop: results differ from the timed loop's")
    if cache.device_error():
        raise SystemExit("device error during parallel sampling")
    peak, peak_src = measured_peak()
    uniq_gbs = unique / (ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": uniq_gbs, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32-accum/f16", "data": "synthetic",
        "config": {"workload": "parallel", "layers": 1, "candidates": C, "prompt": prompt, "decode_steps": S,
                   "heads": H, "head_dim": d, "block_size": BS, "cow_copies": n_cow, "launch_flags": args.launch_flags,
                   "prefix_groups": [[0, C, (prompt // BS) * BS]] if use_groups else None,
                   "blocks_in_use": w.num_blocks - len(alloc.free_list()),
                   "l2": "flushed (256 MB write) before each timed 128-step run",
                   "step": "128 x (block copies + fused append + attention), one CUDA graph per timed step"},
        "seq_steps_per_s": C * S / (ms / 1e3),
        "eager": {"ms_per_128_steps": eager_ms, "unique_GB/s": unique / (eager_ms / 1e3) / 1e9},
        "e2e": {"value": unique / (e2e_ms / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "step": "128 decode steps, one kv_decode_step call each: allocator slot reservation "
                        "(copy-on-write plan), tables into pinned memory, one H2D of tables, lengths, block "
                        "pairs, q and new K/V, kv_copy_blocks when planned, the fused call, D2H of the outputs"},
        "logical_GB/s": logical / (ms / 1e3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": uniq_gbs, "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                     "frac": uniq_gbs / peak, "traffic": traffic_record("parallel"),
                     "traffic_note": "DRAM bytes of one launch (one decode step), ncu",
                     "unique_bytes_per_run": unique,
                     "logical_bytes_per_run": logical},
        "gpu_launches": S + sum(c is not None for c in cows), "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    cache.close()
    alloc.close()
    return 0

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama13b")
    ap.add_argument("--partition", type=int, default=0, help="tokens per partition (0 = library choice)")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling a smaller case)")
    ap.add_argument("--block-size", type=int, default=0, help="override the workload's block size (8, 16 or 32)")
    ap.add_argument("--cpu-units", type=int, default=153600,
                    help="oracle sample size for cpu_baseline ((sequence, head) units; ~4 s on 16 cores)")
    ap.add_argument("--ref-units", type=int, default=768, help="oracle units per reference-arm step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--unfused", action="store_true", help="time kv_append + paged_decode_attention as two calls")
    ap.add_argument("--no-prefix-groups", action="store_true",
                    help="parallel sampling: attend without prefix groups (each candidate reads the shared prompt)")
    ap.add_argument("--window", type=int, default=0, help="sliding-window decode over the last N tokens")
    ap.add_argument("--launch-flags", choices=sorted(LAUNCH_FLAGS), default=None,
                    help="zeroed: a zero-filled workspace kept across calls (no clearing copy per call); "
                         "pdl: zeroed + programmatic dependent launch; early: pdl + tables and lengths "
                         "read before the previous launch ends (they are written before the timed loop); "
                         "earlypool: early + the first K/V tiles fetched before the previous launch ends "
                         "(default)")
    args = ap.parse_args()
    if args.launch_flags is None:
        args.launch_flags = default_launch_flags(args.workload)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "swap13b":
        return run_swap(args)
    if args.workload == "decode7b":
        return run_decode_steps(args)
    if args.workload == "parallel":
        return run_parallel(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
