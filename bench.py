"""Benchmark of split-KV decode attention on GB300.

Default workload (N=1): long-context GQA decode -- batch 1, 32 query heads over
8 KV heads, head_dim 128, 128000 cached tokens, fp16 cache -- over 32 layers
with distinct caches (32 x 524 MB, far larger than L2).  One step is one
decode step through the 32 layers: 32 fd_decode calls (split + combine each)
on one stream.

Printed (one JSON line on rank 0):
  value        KV-read GB/s: K+V bytes of the 32 layers / device time of a step
  us_per_layer device time of one layer's fd_decode
  roofline     fd_split (the dominant kernel): algorithmic bytes per launch /
               its CUDA-event duration, against the measured HBM copy peak
  e2e          the same metric through the public API from pinned host
               buffers: per step, q/K/V/seqlens of one layer copied in, one
               fd_decode, out/lse copied back
  cpu_baseline the fp64 oracle on the host cores on a bounded sample
  clocks       SM clocks and throttle reasons sampled during the timed region
  step_ms      mean / median / min / max of the per-step CUDA-event times
  configs      every configuration of the workloads (tiny MHA with forced
               split counts, the ragged batch, the paged cache, sweep points
               with n_splits = 1 beside the plan, the fp8 cache, the query
               blocks): us per call, K+V GB/s, fraction of the measured HBM
               peak, split and combine kernel times, and the oracle timed on
               sampled rows of the same problem

--impl reference times the oracle (the only reference this method has) on
the same workload, a bounded sample per step.

Multi-GPU: the op has no exchange step, so N GPUs run N independent replicas
(weak scaling); value sums the bytes of all ranks over the max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "long_gqa_128k"
METRIC = "decode-attention µs/layer and KV-read HBM GB/s (% of GB300 peak) at 128K ctx"
PEAK_FALLBACK_GBS = 6800.0


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--layers", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="time the headline only (no per-configuration measurements)")
    ap.add_argument("--eager", action="store_true",
                    help="launch every call from Python instead of replaying a captured CUDA graph")
    ap.add_argument("--cuda-cores", action="store_true",
                    help="use the CUDA-core consumer of fd_split instead of the tensor-core one")
    ap.add_argument("--workload", default=None,
                    choices=["tiny_mha", "long_gqa_128k", "varlen_b16", "paged_b8", "sweep",
                             "query_block_q4", "query_block_g8_q4", "query_block_g8_q8",
                             "query_block_g16_q8", "long_gqa_128k_fp8", "sweep_fp8"],
                    help="time one workload (one JSON line per problem) instead of the default line")
    return ap.parse_args()


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return PEAK_FALLBACK_GBS, "fallback"


class ClockSampler:
    """SM clocks and clock-event (throttle) reasons of the benchmarked GPU,
    sampled in the background: through NVML every 2 ms when libnvidia-ml can
    be loaded, else with nvidia-smi every 50 ms.  The GPU is addressed by its
    UUID, so the samples are of the device CUDA runs on.  mark() brackets the
    timed region; stop() summarises the samples inside it."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # NVML clock-event reason bits (nvml.h)
    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, dev_index: int):
        import torch
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        self.uuid = u if u.startswith("GPU-") else "GPU-" + u
        self.idx = dev_index
        self.samples = []          # (host time, sm MHz, reasons bitmask or names)
        self.window = None
        self.max_mhz = None
        self.source = None
        self._stop = False
        self._thread = None
        self.proc = None
        # the raw nvidia-smi samples go to $FD_BENCH_LOG_DIR (default: the temp directory)
        log_dir = os.environ.get("FD_BENCH_LOG_DIR") or tempfile.gettempdir()
        self.path = os.path.join(log_dir, f"clocks_bench_{os.getpid()}.csv")

    def _nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit")
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByUUID")
        reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        return lib, h, reasons

    def start(self):
        import threading
        try:
            lib, h, reasons = self._nvml()
            import ctypes

            def loop():
                clk, r = ctypes.c_uint(), ctypes.c_ulonglong()
                while not self._stop:
                    if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                            reasons(h, ctypes.byref(r)) == 0:
                        self.samples.append((time.perf_counter(), float(clk.value), int(r.value)))
                    time.sleep(0.002)

            self.source = "nvml, 2 ms"
            self._thread = threading.Thread(target=loop, daemon=True)
            self._thread.start()
            return
        except Exception:
            pass
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi, 50 ms"
            t0 = time.time()
            while time.time() - t0 < 5 and os.path.getsize(self.path) == 0:
                time.sleep(0.05)
        except Exception:
            self.proc = None

    def mark(self, t0: float, t1: float):
        self.window = (t0, t1)

    def stop(self):
        if self._thread is not None:
            time.sleep(0.01)
            self._stop = True
            self._thread.join(timeout=5)
            rows = self.samples
            inside = [x for x in rows if self.window and self.window[0] <= x[0] <= self.window[1]]
            use = inside or rows
            if not use:
                return None
            names = sorted({n for x in use for b, n in self.REASON_BITS.items() if x[2] & b})
            return {"sm_mhz": statistics.median(x[1] for x in use),
                    "sm_max_mhz": self.max_mhz or max(x[1] for x in use), "reasons": names,
                    "samples": len(rows), "samples_in_timed_region": len(inside),
                    "sm_mhz_min": min(x[1] for x in use), "source": self.source}
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9], parts[4]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, s in enumerate(r[2]) if s.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "source": self.source}


def _dist():
    import torch.distributed as dist
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, local, ws


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def aggregate_ranks(ms_local: float, bytes_local: float, ws: int):
    """Whole-job numbers of N replicas: the step time is the slowest rank's,
    the bytes are every rank's.  Works on NCCL (CUDA tensors) and gloo."""
    if ws == 1:
        return ms_local, bytes_local
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms_local], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    b = torch.tensor([bytes_local], dtype=torch.float64, device=dev)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


def _traffic_from_profile(src_hash: str):
    """DRAM bytes per fd_split launch from the committed ncu summary, if it
    was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "fd_split_long_gqa_128k_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("fd_split_cu_sha256") == src_hash:
            return float(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def _code_only(text: str) -> str:
    """C++ source without comments and with whitespace runs collapsed, so that
    a comment-only edit keeps a profile's counters attached to the kernel."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return re.sub(r"\s+", " ", text).strip()


def _kernel_hash():
    h = hashlib.sha256()
    for name in ("fd_split.cu", "fd_device.cuh", "fd_internal.h"):
        with open(os.path.join(ROOT, "split_kv_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


# ---------------------------------------------------------------- CPU oracle legs
def _oracle_layer_time(q_h, k_h, v_h, seqlens_h, n_kv_heads, min_seconds):
    """Time the fp64 oracle over whole layers (all rows) on the host cores."""
    import oracle
    threads = oracle.hardware_threads()
    reps, t_total = 0, 0.0
    while True:
        t0 = time.perf_counter()
        oracle.decode(q_h, k_h, v_h, seqlens_h, dtype="f16", n_kv_heads=n_kv_heads, n_threads=threads)
        t_total += time.perf_counter() - t0
        reps += 1
        if t_total >= min_seconds or reps >= 50:
            break
    return t_total / reps, threads, reps


def _cpu_inputs(c, seed_layer=0):
    import numpy as np

    import fd_inputs
    B, Hq, Hkv, D, T = c["batch"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"], c["ctx"]
    q = fd_inputs.randn((B, Hq, D), c["dtype"], c["seed"] + 7919 * seed_layer)
    k = fd_inputs.randn_chunked((B, Hkv, T, D), c["dtype"], c["seed"] + 10 + 7919 * seed_layer)
    v = fd_inputs.randn_chunked((B, Hkv, T, D), c["dtype"], c["seed"] + 11 + 7919 * seed_layer)
    return q, k, v, np.full(B, T, dtype=np.int32)


def run_reference(args):
    """The oracle as the reference arm.  Each step evaluates a bounded sample
    of the workload's query rows (the same rows every step) on the host
    cores, sized so that warm-up + steps take about a minute; the KV-read rate
    is scaled by the fraction of the layer's rows evaluated."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import fd_inputs
    import oracle
    c = fd_inputs.WORKLOADS[WORKLOAD]
    q, k, v, sl = _cpu_inputs(c)
    threads = oracle.hardware_threads()
    rows_total = c["batch"] * c["n_q_heads"]
    kv_bytes = c["batch"] * c["n_kv_heads"] * c["ctx"] * c["head_dim"] * 2 * 2

    def run(rows):
        oracle.decode(q, k, v, sl, dtype=c["dtype"], n_kv_heads=c["n_kv_heads"],
                      rows=list(range(rows)), n_threads=threads)

    t0 = time.perf_counter()
    run(min(threads, rows_total))
    t_batch = time.perf_counter() - t0                 # one row per thread
    budget = 60.0 / max(1, args.steps + args.warmup)
    rows = max(1, min(rows_total, int(budget / max(t_batch, 1e-6) * min(threads, rows_total))))
    for _ in range(args.warmup):
        run(rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run(rows)
    dt = (time.perf_counter() - t0) / args.steps
    gbs = kv_bytes * rows / rows_total / dt / 1e9
    sample = (f"{rows} of the layer's {rows_total} query rows per step ({c['ctx']} tokens each, fp64), "
              "KV rate scaled by that fraction")
    line = {
        "impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "us_per_layer": dt * 1e6 * rows_total / rows, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic N(0,1), seeded",
        "config": _config(c, None),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(c, S):
    return {"workload": WORKLOAD, "batch": c["batch"], "n_q_heads": c["n_q_heads"],
            "n_kv_heads": c["n_kv_heads"], "head_dim": c["head_dim"], "ctx": c["ctx"],
            "layers": c["layers"], "kv_dtype": c["dtype"], "n_splits": S,
            "l2": "inputs larger than L2: 32 distinct 524 MB layer caches per step",
            "parallelism": "replicas"}


# ---------------------------------------------------------------- GPU arm
def run_gpu(args):
    import numpy as np
    import torch

    import fd_inputs
    import split_kv_gb300 as fd
    from split_kv_gb300 import _build

    rank, local, ws = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _build.build()
    c = fd_inputs.WORKLOADS[WORKLOAD]
    B, Hq, Hkv, D, T = c["batch"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"], c["ctx"]
    n_layers = args.layers or c["layers"]
    sl_h = np.full(B, T, dtype=np.int32)
    S = fd.fd_plan(B, Hq, Hkv, D, sl_h)
    fd.check(S, "fd_plan")

    # inputs resident in HBM: distinct q and K/V per layer
    seqlens = torch.from_numpy(sl_h).to(dev)
    qs, ks, vs = [], [], []
    for i in range(n_layers):
        qs.append(fd_inputs.randn((B, Hq, D), c["dtype"], c["seed"] + 7919 * i, device=dev))
        ks.append(fd_inputs.randn_chunked((B, Hkv, T, D), c["dtype"], c["seed"] + 10 + 7919 * i, device=dev))
        vs.append(fd_inputs.randn_chunked((B, Hkv, T, D), c["dtype"], c["seed"] + 11 + 7919 * i, device=dev))
    desc = fd.make_desc(qs[0], ks[0], vs[0], max_seqlen=T, n_splits=S)
    if args.cuda_cores:
        desc.flags = fd.FD_FLAG_CUDA_CORES
    wsb = fd.fd_workspace_size(desc, S)
    workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    out = torch.empty(n_layers, B, Hq, D, dtype=torch.float32, device=dev)
    lse = torch.empty(n_layers, B, Hq, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream

    def step(handle=sp):
        for i in range(n_layers):
            rc = fd.fd_decode(desc, qs[i], ks[i], vs[i], seqlens, None, out[i], lse[i], workspace,
                              wsb, stream=handle)
            if rc != 0:
                raise fd.FdError(rc, "fd_decode")

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    fd.check(fd.fd_device_status(stream), "device status after warm-up")
    # one step (the 32 fd_decode calls) captured once and replayed: the same
    # kernels with the same arguments, without Python launch overhead
    graph, graph_note = _capture(lambda h: step(h), dev, stream, args.eager)
    run_step = graph.replay if graph is not None else step
    for _ in range(2):
        run_step()
    torch.cuda.synchronize()

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    _barrier(ws)
    torch.cuda.synchronize()
    # an event between consecutive steps: one pair per step, and the whole region
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    t_host0 = time.perf_counter()
    evs[0].record(stream)
    for i in range(args.steps):
        run_step()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    t_host1 = time.perf_counter()
    _barrier(ws)
    if sampler:
        sampler.mark(t_host0, t_host1)
    clocks = sampler.stop() if sampler else None
    ms_local = evs[0].elapsed_time(evs[-1]) / args.steps
    step_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
    fd.check(fd.fd_device_status(stream), "device status after timing")

    kv_bytes_layer = B * Hkv * T * D * 2 * 2
    ms, job_bytes = aggregate_ranks(ms_local, float(n_layers * kv_bytes_layer), ws)
    value = job_bytes / (ms * 1e-3) / 1e9
    us_layer = ms * 1e3 / n_layers

    # ---- roofline of fd_split.  The kernel's time per launch: its n_layers
    # launches back to back, captured in a CUDA graph and replayed between
    # CUDA events on the replay stream (as in the timed step, but without the
    # combine); the combine likewise.  Per-launch events around eager
    # launches, which include each launch's gap, are reported beside it.
    reps = max(3, min(20, args.steps // 10))

    def splits(h):
        for i in range(n_layers):
            fd.check(fd.fd_split_states(desc, qs[i], ks[i], vs[i], seqlens, None, workspace, wsb, stream=h))

    def combines(h):
        for i in range(n_layers):
            fd.check(fd.fd_combine_states(desc, workspace, out[i], lse[i], wsb, stream=h))

    def per_launch_ms(body):
        g, _ = _capture(body, dev, stream, args.eager)
        run = g.replay if g is not None else (lambda: body(sp))
        run()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(reps):
            run()
        a1.record(stream)
        torch.cuda.synchronize()
        return a0.elapsed_time(a1) / (reps * n_layers)

    split_avg_ms = per_launch_ms(splits)
    combine_avg_ms = per_launch_ms(combines)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_layers)]
    split_eager_ms = []
    for rep in range(reps):
        for i in range(n_layers):
            ev[i][0].record(stream)
            fd.check(fd.fd_split_states(desc, qs[i], ks[i], vs[i], seqlens, None, workspace, wsb, stream=sp))
            ev[i][1].record(stream)
            fd.check(fd.fd_combine_states(desc, workspace, out[i], lse[i], wsb, stream=sp))
        torch.cuda.synchronize()
        if rep > 0:   # the first pass warms up
            split_eager_ms += [ev[i][0].elapsed_time(ev[i][1]) for i in range(n_layers)]
    ws_write = B * Hq * S * (D + 2) * 4
    split_alg_bytes = kv_bytes_layer + B * Hq * D * 2 + ws_write + 4 * B
    peak, peak_src = _peaks()
    achieved = split_alg_bytes / (split_avg_ms * 1e-3) / 1e9
    traffic = _traffic_from_profile(_kernel_hash())
    roofline = {"kernel": "fd_split", "bound": "hbm", "achieved": achieved, "peak": peak,
                "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                "peak_source": peak_src, "alg_bytes_per_launch": split_alg_bytes,
                "launch_us": split_avg_ms * 1e3,
                "launch_timing": f"{n_layers} back-to-back launches per replay, {reps} replays",
                "launch_us_eager_events": statistics.mean(split_eager_ms) * 1e3,
                "combine_us": combine_avg_ms * 1e3}

    # ---- e2e: public API from pinned host buffers, one layer per step
    e2e = None
    if rank == 0 or ws > 1:
        hq = qs[0].cpu().pin_memory()
        hk = ks[0].cpu().pin_memory()
        hv = vs[0].cpu().pin_memory()
        hsl = torch.from_numpy(sl_h).pin_memory()
        ho = torch.empty(B, Hq, D, dtype=torch.float32).pin_memory()
        hl = torch.empty(B, Hq, dtype=torch.float32).pin_memory()
        dq, dk, dv, dsl = torch.empty_like(qs[0]), torch.empty_like(ks[0]), torch.empty_like(vs[0]), \
            torch.empty_like(seqlens)
        dout, dl = torch.empty(B, Hq, D, dtype=torch.float32, device=dev), \
            torch.empty(B, Hq, dtype=torch.float32, device=dev)

        def e2e_step():
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            dsl.copy_(hsl, non_blocking=True)
            rc = fd.fd_decode(desc, dq, dk, dv, dsl, None, dout, dl, workspace, wsb, stream=sp)
            if rc != 0:
                raise fd.FdError(rc, "fd_decode")
            ho.copy_(dout, non_blocking=True)
            hl.copy_(dl, non_blocking=True)

        n_e2e = max(3, min(20, args.steps // 10))
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        a1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = a0.elapsed_time(a1) / n_e2e
        h2d = hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2 + hsl.numel() * 4
        d2h = ho.numel() * 4 + hl.numel() * 4
        e2e = {"value": ws * kv_bytes_layer / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms, "step": "one layer: H2D q/K/V/seqlens, fd_decode, D2H out/lse"}

        # serving form: the cache stays resident; per step only q, the new
        # token's K/V row of every KV head and the lengths come from the host
        hk_new = ks[0][:, :, T - 1:T].cpu().pin_memory()
        hv_new = vs[0][:, :, T - 1:T].cpu().pin_memory()
        dk.copy_(ks[0])
        dv.copy_(vs[0])

        def serve_step():
            dq.copy_(hq, non_blocking=True)
            dk[:, :, T - 1:T].copy_(hk_new, non_blocking=True)
            dv[:, :, T - 1:T].copy_(hv_new, non_blocking=True)
            dsl.copy_(hsl, non_blocking=True)
            rc = fd.fd_decode(desc, dq, dk, dv, dsl, None, dout, dl, workspace, wsb, stream=sp)
            if rc != 0:
                raise fd.FdError(rc, "fd_decode")
            ho.copy_(dout, non_blocking=True)
            hl.copy_(dl, non_blocking=True)

        for _ in range(3):
            serve_step()
        torch.cuda.synchronize()
        n_srv = max(10, min(200, args.steps))
        t0 = time.perf_counter()
        a0.record(stream)
        for _ in range(n_srv):
            serve_step()
            stream.synchronize()          # the caller reads the result every step
        a1.record(stream)
        torch.cuda.synchronize()
        srv_ms = a0.elapsed_time(a1) / n_srv
        srv_wall_ms = (time.perf_counter() - t0) * 1e3 / n_srv
        e2e["resident_cache"] = {
            "value": ws * kv_bytes_layer / (srv_wall_ms * 1e-3) / 1e9, "unit": "GB/s",
            "ms_per_step": srv_wall_ms, "device_ms_per_step": srv_ms,
            "h2d_bytes_per_step": hq.numel() * 2 + hk_new.numel() * 2 + hv_new.numel() * 2 + hsl.numel() * 4,
            "d2h_bytes_per_step": d2h,
            "step": "one layer, cache resident: H2D q + new K/V row + seqlens, fd_decode, D2H out/lse, host sync"}

    # ---- CPU baseline: the oracle on the host cores, rank 0 at N=1 only
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        q_h, k_h, v_h = qs[0].cpu(), ks[0].cpu(), vs[0].cpu()
        t_layer, threads, reps = _oracle_layer_time(q_h, k_h, v_h, sl_h, Hkv, min_seconds=10.0)
        cpu = {"value": kv_bytes_layer / t_layer / 1e9, "unit": "GB/s", "cores": threads,
               "kind": "oracle",
               "sample": f"one layer of the workload (all {B * Hq} query rows, {T} tokens) "
                         f"x {reps} repetitions, fp64; {t_layer * 1e6:.0f} us/layer"}

    # ---- every configuration of the workloads, rank 0 at N=1 only (the
    # replicas of N>1 run the headline alone)
    configs = None
    if rank == 0 and ws == 1 and not args.no_configs:
        configs = measure_configs(dev, stream, peak, args.eager, with_cpu=not args.no_cpu_baseline)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "us_per_layer": us_layer,
            "step_ms": {"mean": statistics.mean(step_ms), "median": statistics.median(step_ms),
                        "min": min(step_ms), "max": max(step_ms), "n": len(step_ms),
                        "us_per_layer_median": statistics.median(step_ms) * 1e3 / n_layers},
            "frac_of_hbm_peak": value / peak, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic N(0,1), seeded, fp16 cache",
            "config": _config(c, S), "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "clocks": clocks, "gpu_launches": 2 * n_layers * args.steps,
            "workspace_bytes": wsb, "num_sms": fd.fd_num_sms(),
            "split_compute": "cuda_cores" if args.cuda_cores else "tensor_cores",
            "launch": graph_note,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _capture(body, dev, stream, eager: bool):
    """Capture body(stream_handle) into a CUDA graph (fd_decode allocates and
    synchronises nothing, so it is capturable).  Returns (graph or None, note)."""
    import torch
    if eager:
        return None, "eager"
    try:
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            body(cap.cuda_stream)
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        return g, "cuda_graph"
    except Exception as e:  # report, and time the eager launches instead
        torch.cuda.synchronize()
        return None, f"eager (graph capture failed: {type(e).__name__})"


# ---------------------------------------------------------------- other workloads
def _time_calls(fn, n_sets, iters, warmup, stream, dev, eager):
    """Device time per call; the calls over all input sets are replayed as
    one captured graph unless eager."""
    import torch
    for i in range(warmup):
        fn(i % n_sets, stream.cuda_stream)
    torch.cuda.synchronize()

    def body(h):
        for j in range(n_sets):
            fn(j, h)

    graph, note = _capture(body, dev, stream, eager)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if graph is not None:
        reps = max(2, -(-iters // n_sets))
        graph.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (reps * n_sets), note
    e0.record(stream)
    for i in range(iters):
        fn(i % n_sets, stream.cuda_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters, note


def _problem_sets(name, c, dev, n_sets, batch=None, ctx=None):
    """Distinct input sets of one workload problem (rotated so that the data
    touched between two uses of a set exceeds the L2)."""
    import numpy as np
    import torch

    import fd_inputs
    import split_kv_gb300 as fd
    B = batch or c["batch"]
    Hq, Hkv, D = c["n_q_heads"], c["n_kv_heads"], c["head_dim"]
    T = ctx or c["ctx"]
    dt = c["dtype"]
    seed = c["seed"]
    sets = []
    if name == "varlen_b16":
        sl_h = fd_inputs.varlen_seqlens(seed, B, T)
    else:
        sl_h = np.full(B, T, dtype=np.int32)
    q_len = c.get("q_len", 1)
    bt_h = None
    for j in range(n_sets):
        qshape = (B, q_len, Hq, D) if q_len > 1 else (B, Hq, D)
        q = fd_inputs.randn(qshape, dt, seed + 100 * j, device=dev)
        if name == "paged_b8":
            ps = c["page_size"]
            npp = T // ps
            n_pages = B * npp
            k = fd_inputs.randn_chunked((n_pages, Hkv, ps, D), dt, seed + 100 * j + 1, device=dev)
            v = fd_inputs.randn_chunked((n_pages, Hkv, ps, D), dt, seed + 100 * j + 2, device=dev)
            bt_h = fd_inputs.block_table(seed + 2, B, npp, n_pages)
            bt = torch.from_numpy(bt_h).to(dev)
            desc = fd.make_desc(q, k, v, page_size=ps, max_pages_per_seq=npp, max_seqlen=int(sl_h.max()))
        elif c.get("kv_dtype") == "e4m3":
            gk = c["kv_gain"]
            k = fd_inputs.randn_fp8((B, Hkv, T, D), seed + 100 * j + 1, device=dev, gain=gk)
            v = fd_inputs.randn_fp8((B, Hkv, T, D), seed + 100 * j + 2, device=dev, gain=gk)
            bt = None
            desc = fd.make_desc(q, k, v, max_seqlen=int(sl_h.max()), k_scale=1 / gk, v_scale=1 / gk)
        else:
            k = fd_inputs.randn_chunked((B, Hkv, T, D), dt, seed + 100 * j + 1, device=dev)
            v = fd_inputs.randn_chunked((B, Hkv, T, D), dt, seed + 100 * j + 2, device=dev)
            bt = None
            desc = fd.make_desc(q, k, v, max_seqlen=int(sl_h.max()))
        sets.append((desc, q, k, v, bt))
    return sets, sl_h, bt_h


def _oracle_sample(c, sets, sl_h, bt_h, kv_bytes, target_s):
    """The fp64 oracle, as it stands, on a seeded sample of the problem's query
    rows (set 0) on every host core, sized to about target_s seconds.  The
    KV-read rate counts the fraction of the layer's (row, key) pairs the
    sample covers."""
    import numpy as np

    import oracle
    desc, q, k, v, _ = sets[0]
    B, Hq, Hkv = desc.batch, c["n_q_heads"], c["n_kv_heads"]
    ql = c.get("q_len", 1)
    okw = dict(dtype=c["dtype"], n_kv_heads=Hkv, n_threads=oracle.hardware_threads())
    if c.get("kv_dtype") == "e4m3":
        okw.update(kv_dtype="e4m3", k_scale=desc.k_scale, v_scale=desc.v_scale)
    if bt_h is not None:
        okw.update(page_size=c["page_size"], block_table=bt_h)
    qh, kh, vh = q.cpu(), k.cpu(), v.cpu()
    # row (b*q_len + i)*Hq + h sees the first L_b - q_len + 1 + i keys
    vis = np.array([max(0, int(sl_h[r // (ql * Hq)]) - ql + 1 + (r // Hq) % ql)
                    for r in range(B * ql * Hq)], dtype=np.float64)
    order = np.random.default_rng(7).permutation(B * ql * Hq)
    threads = okw["n_threads"]

    def run(rows):
        t0 = time.perf_counter()
        oracle.decode(qh, kh, vh, sl_h, rows=rows, **okw)
        return time.perf_counter() - t0

    n = min(threads, len(order))
    t = run(np.sort(order[:n]))
    n = int(max(n, min(len(order), n * target_s / max(t, 1e-6))))
    rows = np.sort(order[:n])
    t = run(rows)
    frac = vis[rows].sum() / max(vis.sum(), 1.0)
    return {"value": kv_bytes * frac / t / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "us_per_layer": t / max(frac, 1e-12) * 1e6,
            "sample": f"{n} of the {len(order)} query rows of one layer (seeded), fp64, "
                      f"{t:.2f} s; rate scaled by the sampled fraction of (row, key) pairs"}


def measure_problem(name, c, dev, stream, peak, *, batch=None, ctx=None, forced=(), unsplit=False,
                    eager=False, cuda_cores=False, warmup=3, cpu_seconds=0.0):
    """Device time per fd_decode call of one workload problem (inputs rotated
    across distinct sets larger than the L2, the calls replayed from a CUDA
    graph), at the planned split count and at `forced` ones (and 1 if
    `unsplit`); the split and combine kernels timed alone at the planned
    count; optionally the oracle on sampled rows."""
    import math as _m

    import torch

    import split_kv_gb300 as fd
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    B = batch or c["batch"]
    T = ctx or c["ctx"]
    fp8 = c.get("kv_dtype") == "e4m3"
    esize = 1 if fp8 else 2
    est = B * c["n_kv_heads"] * T * c["head_dim"] * esize * 2
    n_sets = max(1, min(256, _m.ceil(4 * l2 / max(est, 1))))
    sets, sl_h, bt_h = _problem_sets(name, c, dev, n_sets, batch, ctx)
    seqlens = torch.from_numpy(sl_h).to(dev)
    kv_bytes = int(sl_h.sum()) * c["n_kv_heads"] * c["head_dim"] * esize * 2
    ql = c.get("q_len", 1)
    rows = B * ql * c["n_q_heads"]
    d0 = sets[0][0].copy()
    if cuda_cores:
        d0.flags = fd.FD_FLAG_CUDA_CORES
    S_plan = fd.check(fd.fd_plan_desc(d0, sl_h), "fd_plan_desc")
    if ql == 1 and not fp8 and not cuda_cores:
        assert S_plan == fd.fd_plan(B, c["n_q_heads"], c["n_kv_heads"], c["head_dim"], sl_h)
    counts = [S_plan] + [S for S in forced if S != S_plan]
    if unsplit and S_plan != 1 and 1 not in counts:
        counts.append(1)
    iters = max(50, min(2000, int(1e10 / max(kv_bytes, 1))))
    res = {"workload": name, "batch": B, "ctx": T, "q_len": ql, "n_q_heads": c["n_q_heads"],
           "n_kv_heads": c["n_kv_heads"], "kv_dtype": c.get("kv_dtype", c["dtype"]),
           "n_splits": S_plan, "kv_bytes": kv_bytes, "input_sets": n_sets, "peak_gbs": peak}
    by_splits = {}
    for S in counts:
        descs = []
        for (desc, *_rest) in sets:
            d = desc.copy()
            d.n_splits = S
            if cuda_cores:
                d.flags = fd.FD_FLAG_CUDA_CORES
            descs.append(d)
        wsb = fd.fd_workspace_size(descs[0], S)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        out = torch.empty(rows, c["head_dim"], dtype=torch.float32, device=dev)
        lse = torch.empty(rows, dtype=torch.float32, device=dev)

        def call(j, h):
            _, q, k, v, bt = sets[j]
            rc = fd.fd_decode(descs[j], q, k, v, seqlens, bt, out, lse, ws, wsb, stream=h)
            if rc != 0:
                raise fd.FdError(rc, "fd_decode")

        ms, note = _time_calls(call, n_sets, iters, max(3, warmup), stream, dev, eager)
        by_splits[S] = ms * 1e3
        if S == S_plan:
            res["launch"] = note
            if S > 1:
                def split(j, h):
                    _, q, k, v, bt = sets[j]
                    fd.check(fd.fd_split_states(descs[j], q, k, v, seqlens, bt, ws, wsb, stream=h))

                def combine(j, h):
                    fd.check(fd.fd_combine_states(descs[j], ws, out, lse, wsb, stream=h))

                res["split_us"] = _time_calls(split, n_sets, iters, 2, stream, dev, eager)[0] * 1e3
                res["combine_us"] = _time_calls(combine, n_sets, iters, 2, stream, dev, eager)[0] * 1e3
            else:   # one split: the split kernel writes the result, no combine
                res["split_us"], res["combine_us"] = ms * 1e3, 0.0
        del ws
    fd.check(fd.fd_device_status(stream), "device status")
    us = by_splits[S_plan]
    res["us_per_call"] = us
    res["kv_gbs"] = kv_bytes / (us * 1e-6) / 1e9
    res["frac_of_hbm_peak"] = res["kv_gbs"] / peak
    if len(by_splits) > 1:
        res["us_per_call_by_splits"] = {str(S): t for S, t in by_splits.items()}
    if unsplit and 1 in by_splits:
        res["us_per_call_unsplit"] = by_splits[1]
        res["speedup_vs_unsplit"] = by_splits[1] / us
    if cpu_seconds > 0:
        res["cpu_baseline"] = _oracle_sample(c, sets, sl_h, bt_h, kv_bytes, cpu_seconds)
    del sets
    torch.cuda.empty_cache()
    return res


# Every configuration of the method's five workloads (and the next rows'),
# measured on the default bench line beside the headline: (label, workload,
# batch, ctx, forced split counts, time n_splits = 1 too).
CONFIGS = (
    ("tiny_mha", "tiny_mha", None, None, (1, 3, 7), False),
    ("varlen_b16", "varlen_b16", None, None, (), False),
    ("paged_b8", "paged_b8", None, None, (), False),
    ("sweep_b1_8k", "sweep", 1, 8192, (), True),
    ("sweep_b1_128k", "sweep", 1, 131072, (), True),
    ("sweep_b16_8k", "sweep", 16, 8192, (), True),
    ("sweep_b16_128k", "sweep", 16, 131072, (), True),
    ("long_gqa_128k_fp8", "long_gqa_128k_fp8", None, None, (), False),
    ("query_block_q4", "query_block_q4", None, None, (), False),
    ("query_block_g8_q4", "query_block_g8_q4", None, None, (), False),
    ("query_block_g8_q8", "query_block_g8_q8", None, None, (), False),
    ("query_block_g16_q8", "query_block_g16_q8", None, None, (), False),
)


def measure_configs(dev, stream, peak, eager, with_cpu):
    import fd_inputs
    out = {}
    for label, name, batch, ctx, forced, unsplit in CONFIGS:
        c = fd_inputs.WORKLOADS[name]
        out[label] = measure_problem(name, c, dev, stream, peak, batch=batch, ctx=ctx, forced=forced,
                                     unsplit=unsplit, eager=eager,
                                     cpu_seconds=1.0 if with_cpu else 0.0)
    return out


def run_suite(args):
    """One JSON line per problem of a workload: device time per fd_decode call
    (inputs rotated across distinct sets larger than the L2), K+V GB/s and the
    fraction of the measured HBM peak; the sweep also times n_splits = 1."""
    import torch

    import fd_inputs
    from split_kv_gb300 import _build
    _build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peak, peak_src = _peaks()
    name = args.workload
    c = fd_inputs.WORKLOADS[name]
    grid = "batches" in c   # a sweep over batch x context
    probs = [(b, t) for b in c["batches"] for t in c["ctxs"]] if grid else [(None, None)]
    base = dict(c, batch=None, ctx=None) if grid else c
    for batch, ctx in probs:
        line = measure_problem(name, base, dev, stream, peak, batch=batch, ctx=ctx, unsplit=grid,
                               eager=args.eager, cuda_cores=args.cuda_cores, warmup=args.warmup)
        line["peak_source"] = peak_src
        line["split_compute"] = "cuda_cores" if args.cuda_cores else "tensor_cores"
        print(json.dumps(line), flush=True)


def main():
    args = _args()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload is not None:
        run_suite(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
