#!/usr/bin/env python
"""Benchmark of quantized-KV single-query decode attention on GB300.

One step = one qdecode_attn call (split kernel + merge kernel) over the whole synthetic workload, the 8k case by
default: B=1, H=16, Hkv=8, D=256, N=8192, 8-bit affine KV in groups of 32, bf16 q and output. The cache is resident
in HBM; L2 is flushed (a 1 GiB write, at least 2 x L2) before every timed call, outside the call's events. The metric is KV
bytes per call (packed codes + scales + biases of K and V, each read once) over the call's device time.

    python bench.py [--steps K] [--warmup W] [--workload 1..5] [--impl ours|reference] [--no-extra]

Prints one JSON line. Under torchrun (N > 1) every rank runs an independent replica on its own GPU.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

if "reference" in sys.argv:
    # the reference arm times the single-threaded oracle: pin BLAS to one thread before numpy loads
    for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[_v] = "1"

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantized-KV decode attn: KV-bytes GB/s vs HBM peak; µs/call @8k"
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 1 << 30


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=2, help="1-5: the configurations; 6: the D = 128 case")
    ap.add_argument("--no-extra", action="store_true", help="skip the per-workload figures (workloads 3-5, multi-query, compat, GEMV, cache append, graph replay)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def kv_bytes(w, N) -> int:
    rows = w.Hkv * sum(N)
    W, NG = w.D * w.bits // 32, w.D // w.GS
    return 2 * rows * (W * 4 + 2 * NG * 2)


def config_of(w, N, extra=None) -> dict:
    c = {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.Hkv, "D": w.D, "bits": w.bits, "GS": w.GS,
         "N": N if len(N) <= 8 else f"{len(N)} sequences", "dtype_in": w.dtype_in, "dtype_out": w.dtype_out,
         "kv_bytes_per_call": kv_bytes(w, N), "parallelism": "replicas",
         "l2": "flushed before every timed call (a 1 GiB write, >= 2 x L2, outside the call's events)"}
    if extra:
        c.update(extra)
    return c


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def split_kernel_hash() -> str:
    """A digest of the code of every kernel and host source (comments and blank lines left out): recorded traffic
    is used only while the code is unchanged."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_quantized_kv_split_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                code = [re.sub(r"//.*$", "", line).rstrip() for line in fh]
            h.update(f.encode() + b"\0" + "\n".join(line for line in code if line).encode())
    return h.hexdigest()[:16]


def workload_by_index(i: int):
    """1-5: the configurations. 6: the D = 128 case (the most common head dimension of deployed models) on the shape
    of the 32k workload: B1 H32 Hkv8 D128 N32768, 4-bit, GS 64 -- the same 37.7 MB of cache as the 8k workload."""
    from attention_quantized_kv_split_gb300 import synth
    if i == 6:
        return dataclasses.replace(synth.small(B=1, H=32, Hkv=8, D=128, N=(32768,), bits=4, GS=64, seed=20261202 + 128),
                                   name="d128_B1_H32_Hkv8_D128_N32768_4b_GS64_bf16")
    return synth.workload(i)


def recorded_traffic(workload_name: str):
    """DRAM bytes per launch of the split kernel from the committed ncu summary, if it matches this source."""
    path = os.path.join(ROOT, "profiles", "split_kernel_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d.get(workload_name)
        if e and e.get("kernel_hash") == split_kernel_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons every 100 ms, each line stamped on arrival."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for s in self.samples if t0 <= s[0] <= t1 + 0.15]
        if not inside and self.samples:
            inside = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:2]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, p in inside:
            for k, nm in enumerate(names):
                if p[5 + k].lower().startswith("active"):
                    reasons.add(nm)

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for _, p in inside if num(p[1]) is not None]
        mx = [num(p[2]) for _, p in inside if num(p[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(inside),
                "power_w_max": max((num(p[3]) or 0.0) for _, p in inside)}


# --------------------------------------------------------------------------------------------- our arm


def make_workload(w, device):
    import torch
    import attention_quantized_kv_split_gb300 as qda
    from attention_quantized_kv_split_gb300 import synth
    N = synth.lengths(w)
    q = synth.query(w)
    cache = qda.QuantizedKV.empty(N, w.Hkv, w.D, w.GS, w.bits, synth.DT[w.dtype_in], device=device)
    for b in range(w.B):
        for kvh in range(w.Hkv):
            K, V = synth.kv_unit(w, b, kvh, N[b], q=q, device=device)
            cache.quantize_into(b, kvh, K, V)
            del K, V
    torch.cuda.synchronize()
    return N, q.to(device), cache


def time_calls(fn, steps, flush, stream):
    """Per-call device time (ms) with L2 flushed before each call, events on the launching stream."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for k in range(steps):
        flush()
        starts[k].record(stream)
        fn()
        ends[k].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


# the cache arrays shared with the oracle's worker processes (attached once per process, outside the timing)
_SHM = {}


def _shm_arrays(spec):
    from multiprocessing import shared_memory
    import numpy as np
    key = spec["name"]
    if key not in _SHM:
        shm = shared_memory.SharedMemory(name=key)
        arrs = {}
        for nm, (off, shape, dt) in spec["arrays"].items():
            arrs[nm] = np.ndarray(shape, dtype=dt, buffer=shm.buf, offset=off)
        _SHM[key] = (shm, arrs)
    return _SHM[key][1]


def split_time(fn, steps, flush, stream):
    """Mean device time (ms) of the split kernel alone: an event the library records between its split and merge
    launches, on the launching stream, with L2 flushed before each call."""
    import torch
    import attention_quantized_kv_split_gb300 as qda
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        flush()
        a.record(stream)
        b.record(stream)
        qda.qdecode_attn_set_split_event(b)
        fn()
        qda.qdecode_attn_set_split_event(None)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def cpu_oracle_task(args):
    """One (sequence, KV head) unit of the cache with all its query heads, by the oracle as it stands
    (attention_packed: the unit's packed K and V rows dequantized once, then softmax(K q / sqrt(D)) V in fp64 per
    query head)."""
    import oracle as O
    spec, b, kvh = args
    a = _shm_arrays(spec)
    H, Hkv, D = spec["H"], spec["Hkv"], spec["D"]
    nrep = H // Hkv
    q = a["q"].reshape(len(spec["N"]), H, D)
    return O.attention_packed(q, a["kp"], a["ks"], a["kb"], a["vp"], a["vs"], a["vb"], spec["N"], H, Hkv, D,
                              spec["GS"], spec["bits"], heads=[(b, kvh * nrep + j) for j in range(nrep)])


def cpu_baseline(w, N, q, cache, pool, cores):
    """The oracle, unchanged, on the host cores: the whole call as (sequence, KV head) tasks -- each the oracle's
    attention_packed over that unit's query heads -- spread over one single-threaded worker process per core. The
    cache sits in shared memory that every worker attached before the clock starts; only dequantization and
    attention are timed."""
    import numpy as np
    from multiprocessing import shared_memory
    arrs = {"kp": cache.kp.cpu().numpy().view(np.uint32), "ks": cache.ks.float().cpu().numpy(),
            "kb": cache.kb.float().cpu().numpy(), "vp": cache.vp.cpu().numpy().view(np.uint32),
            "vs": cache.vs.float().cpu().numpy(), "vb": cache.vb.float().cpu().numpy(),
            "q": q.double().cpu().numpy().reshape(w.B * w.H, w.D)}
    total = sum((a.nbytes + 63) // 64 * 64 for a in arrs.values())
    shm = shared_memory.SharedMemory(create=True, size=total)
    try:
        spec = {"name": shm.name, "arrays": {}, "D": w.D, "GS": w.GS, "bits": w.bits, "H": w.H, "Hkv": w.Hkv,
                "N": [int(x) for x in N]}
        off = 0
        for nm, a in arrs.items():
            np.ndarray(a.shape, dtype=a.dtype, buffer=shm.buf, offset=off)[...] = a
            spec["arrays"][nm] = (off, a.shape, a.dtype.str)
            off += (a.nbytes + 63) // 64 * 64
        tasks = [(spec, b, kvh) for b in range(w.B) for kvh in range(w.Hkv)]
        # attach and warm up the workers: at least two tasks per worker (not timed)
        pool.map(cpu_oracle_task, tasks * -(-2 * cores // len(tasks)), chunksize=1)
        # whole calls back to back for about five seconds
        rounds = 0
        t0 = time.perf_counter()
        while True:
            pool.map(cpu_oracle_task, tasks, chunksize=1)
            rounds += 1
            dt = time.perf_counter() - t0
            if dt >= 5.0 or rounds >= 200:
                break
    finally:
        shm.close()
        shm.unlink()
    nbytes = kv_bytes(w, N)
    return {"value": rounds * nbytes / dt / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{rounds} whole calls of {w.name} back to back: {len(tasks)} (sequence, KV head) tasks per call, "
                      f"each the oracle's attention_packed over that unit's {w.nrep} query heads (its rows dequantized "
                      f"once, attention in fp64), one single-threaded worker process per core (the cache in shared "
                      f"memory, attached before timing); {min(len(tasks), cores)} of the {cores} workers busy",
            "seconds": round(dt, 3), "ms_per_call": round(dt / rounds * 1e3, 3)}


def cpu_single_thread_c1():
    """SURVEY-style single-thread figure: the oracle on the small workload (B1 H8 Hkv2 D256 N512, 4-bit) in this
    process, one thread."""
    import oracle as O
    from attention_quantized_kv_split_gb300 import synth
    w = synth.workload(1)
    N = synth.lengths(w)
    q = synth.query(w)
    K, V = synth.kv_unit(w, 0, 0, N[0], q=q)
    kp, ks, kb, vp, vs, vb = O.quantize_cache(K.numpy(), V.numpy(), w.GS, w.bits, w.dtype_in)
    qh = q.double().numpy()[0]
    units = w.B * w.Hkv
    best = float("inf")
    for _ in range(3):
        t0 = time.perf_counter()
        for _ in range(units):   # every KV head of the call costs the same as this one
            Kd = O.dequantize(O.unpack(kp, w.bits, w.D), ks, kb, w.GS)
            Vd = O.dequantize(O.unpack(vp, w.bits, w.D), vs, vb, w.GS)
            for j in range(w.nrep):
                O.attention_head(qh[j], Kd, Vd)
        best = min(best, time.perf_counter() - t0)
    return {"workload": w.name, "ms_per_call": round(best * 1e3, 3),
            "GBps": round(kv_bytes(w, N) / best / 1e9, 4), "threads": 1}


def ranks_from_env():
    """(world size, rank, local rank) of this process under torchrun, (1, 0, 0) alone."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest x over the ranks of the default process group (the slowest replica sets the job's time). The
    tensor lives on `device` (a CUDA device for NCCL, the CPU for gloo)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbps(world: int, nbytes: int, steps: int, max_ms_total: float) -> float:
    """Replicas: every rank moves nbytes per step, the job's time is the slowest rank's."""
    return world * nbytes * steps / (max_ms_total * 1e-3) / 1e9


def run_ours(args):
    import torch
    import torch.distributed as dist
    import attention_quantized_kv_split_gb300 as qda
    from attention_quantized_kv_split_gb300 import build, synth

    world, rank, local = ranks_from_env()
    pool = None
    cores = max(1, os.cpu_count() or 1)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle's worker pool (one single-threaded process per host core) is spawned before the first GPU call
        import multiprocessing as mp
        for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[v] = "1"
        ctx = mp.get_context("spawn")
        pool = ctx.Pool(processes=cores)
        pool.map(abs, range(cores))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    build.build()
    qda.lib()
    stream = torch.cuda.current_stream()

    w = workload_by_index(args.workload)
    N, q, cache = make_workload(w, device)
    out = torch.empty((w.B, w.H, w.D), dtype=synth.DT[w.dtype_out], device=device)
    # The flush write evicts L2 (it is at least 2 x L2) and is long enough on the GPU (~1 GiB, ~0.16 ms) that the host
    # enqueues the next call before the GPU reaches it: the call's events then time GPU work, not host latency.
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush_buf = torch.empty(max(2 * l2, FLUSH_BYTES), dtype=torch.uint8, device=device)

    def flush():
        flush_buf.zero_()

    call = qda.bind_decode_attention(q, cache, out, stream)

    plan = qda.qdecode_attn_plan(w.B, w.H, w.Hkv, N, w.D, w.GS, w.bits)
    for _ in range(max(3, args.warmup)):
        flush()
        call()
    torch.cuda.synchronize()

    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.25 if sampler else 0)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    calls_before = qda.qdecode_attn_calls()
    torch.cuda.nvtx.range_push("timed decode calls")
    ms = time_calls(call, args.steps, flush, stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    if world > 1:
        dist.barrier()
    t1 = time.time()
    launches = 2 * (qda.qdecode_attn_calls() - calls_before)
    clocks = sampler.summary(t0, t1) if sampler else None
    if sampler:
        sampler.stop()
    dev_ms_total = max_over_ranks(sum(ms), world, device)
    nbytes = kv_bytes(w, N)
    ms_per_step = dev_ms_total / args.steps
    value = whole_job_gbps(world, nbytes, args.steps, dev_ms_total)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    # dominant kernel: the split kernel, timed alone via an event recorded between the two launches
    rsteps = min(args.steps, 300)
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(rsteps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(rsteps)]
    for k in range(rsteps):
        flush()
        ev0[k].record(stream)
        ev1[k].record(stream)          # marks the event recorded for torch; the library re-records it in the call
        qda.qdecode_attn_set_split_event(ev1[k])
        call()
        qda.qdecode_attn_set_split_event(None)
    torch.cuda.synchronize()
    split_ms = statistics.mean(a.elapsed_time(b) for a, b in zip(ev0, ev1))
    peak, peak_kind = measured_peaks()
    achieved = nbytes / (split_ms * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": recorded_traffic(w.name),
                "kernel": "qda_tc_kernel" if plan["threads"] != 160 else "qda_split2_kernel", "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6800 GB/s",
                "split_kernel_us": round(split_ms * 1e3, 3),
                # the rest of a call (merge kernel, its launch behind the split kernel): the whole call's time minus
                # the split kernel's (an event recorded between the two launches would hold the merge back)
                "call_minus_split_us": round(max(0.0, ms_per_step - split_ms) * 1e3, 3),
                "algorithmic_bytes_per_launch": nbytes}

    # the size floor of this call: the same bytes read once by a plain torch reduction over one contiguous buffer, and
    # a near-empty launch, both timed like the call (L2 flushed first, CUDA events around the launch)
    fbuf = torch.rand(nbytes // 4, dtype=torch.float32, device=device)
    fout = torch.empty((), dtype=torch.float32, device=device)
    tiny = torch.empty(16, dtype=torch.float32, device=device)
    for _ in range(3):
        torch.sum(fbuf, dim=0, out=fout)
    read_ms = statistics.mean(time_calls(lambda: torch.sum(fbuf, dim=0, out=fout), 50, flush, stream))
    launch_ms = statistics.mean(time_calls(lambda: tiny.zero_(), 50, flush, stream))
    del fbuf
    stream_floor = {"read_us": round(read_ms * 1e3, 3), "read_GBps": round(nbytes / (read_ms * 1e-3) / 1e9, 1),
                    "launch_us": round(launch_ms * 1e3, 3), "bytes": nbytes,
                    "how": "torch.sum (dim 0) of one contiguous fp32 buffer of the call's KV bytes, and a 16-element zero_(), "
                           "each after the same L2 flush, CUDA events on the launching stream, mean of 50"}
    roofline["nominal_peak"] = 7900.0
    roofline["frac_of_nominal"] = round(achieved / 7900.0, 4)

    # end to end through the C ABI with host buffers (qdecode_attn_host): every step copies q and the whole cache from
    # pinned host memory to the device, decodes, and copies out back; the library overlaps one step's copies with
    # the previous step's kernels (two staging sets)
    esteps = min(args.steps, 100)
    host = [t.cpu().pin_memory() for t in (q, cache.kp, cache.ks, cache.kb, cache.vp, cache.vs, cache.vb)]
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = hout.numel() * hout.element_size()
    for _ in range(2):   # both staging sets allocated before the timed steps
        qda.qdecode_attn_host(*host, hout, N, w.Hkv, w.GS, w.bits, stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("end-to-end calls (host buffers)")
    e0.record(stream)
    for _ in range(esteps):
        qda.qdecode_attn_host(*host, hout, N, w.Hkv, w.GS, w.bits, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    e2e_ms = e0.elapsed_time(e1) / esteps
    e2e = {"value": round(nbytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4), "steps": esteps}

    extra = {}
    if not args.no_extra:
        # workloads 3-5 and the D = 128 case
        for idx in (3, 4, 5, 6):
            if idx == args.workload:
                continue
            wx = workload_by_index(idx)
            Nx, qx, cx = make_workload(wx, device)
            ox = torch.empty((wx.B, wx.H, wx.D), dtype=synth.DT[wx.dtype_out], device=device)
            fx = qda.bind_decode_attention(qx, cx, ox, stream)
            for _ in range(5):
                fx()
            msx = time_calls(fx, 50, flush, stream)
            bx = kv_bytes(wx, Nx)
            mx = statistics.mean(msx)
            sx = split_time(fx, 50, flush, stream)
            px = qda.qdecode_attn_plan(wx.B, wx.H, wx.Hkv, Nx, wx.D, wx.GS, wx.bits)
            extra[wx.name] = {"us_per_call": round(mx * 1e3, 2), "kv_GBps": round(bx / (mx * 1e-3) / 1e9, 1),
                              "frac_of_peak": round(bx / (mx * 1e-3) / 1e9 / peak, 4), "kv_bytes": bx,
                              "split_kernel_us": round(sx * 1e3, 2),
                              "split_frac_of_peak": round(bx / (sx * 1e-3) / 1e9 / peak, 4),
                              "split_kernel": "qda_tc_kernel" if px["threads"] != 160 else "qda_split2_kernel",
                              "traffic": recorded_traffic(wx.name)}
            del cx, qx, ox
            torch.cuda.empty_cache()
        # the two-pass compat form on this workload's cache (K read in both passes)
        oc = torch.empty_like(out)
        ccall = lambda: qda.qdecode_attn_compat(q, cache.kp, cache.ks, cache.kb, cache.vp, cache.vs, cache.vb, oc,
                                                N, w.Hkv, w.GS, w.bits, stream)
        for _ in range(5):
            ccall()
        mc = statistics.mean(time_calls(ccall, 50, flush, stream))
        extra[f"{w.name}_two_pass_compat"] = {
            "us_per_call": round(mc * 1e3, 2), "kv_GBps": round(nbytes / (mc * 1e-3) / 1e9, 1),
            "frac_of_peak": round(nbytes / (mc * 1e-3) / 1e9 / peak, 4), "kv_bytes": nbytes,
            "note": "K is read in both passes; kv_GBps counts each KV byte once"}
        # the codec under a plain GEMV: an MLP-sized 8-bit matrix (K = 4096, N = 14336, GS = 64) times one vector;
        # random codes, scales and biases (the kernel's time does not depend on their values)
        gK, gN, gGS = 4096, 14336, 64
        gen = torch.Generator(device=device).manual_seed(20261202)
        gw = torch.randint(-2 ** 31, 2 ** 31 - 1, (gN, gK // 4), generator=gen, device=device, dtype=torch.int32)
        gs = (torch.rand(gN, gK // gGS, generator=gen, device=device) * 0.02).to(torch.bfloat16)
        gb = (torch.randn(gN, gK // gGS, generator=gen, device=device)).to(torch.bfloat16)
        gx = torch.randn(1, gK, generator=gen, device=device).to(torch.bfloat16)
        gy = torch.empty(1, gN, dtype=torch.float32, device=device)
        gcall = lambda: qda.qdecode_qgemv(gx, gw, gs, gb, gy, gGS, 8, stream)
        for _ in range(5):
            gcall()
        mg = statistics.mean(time_calls(gcall, 50, flush, stream))
        gbytes = gN * gK + 2 * 2 * gN * (gK // gGS)
        extra["qgemv_8b_K4096_N14336_T1_GS64_bf16"] = {
            "us_per_call": round(mg * 1e3, 2), "GBps": round(gbytes / (mg * 1e-3) / 1e9, 1),
            "frac_of_peak": round(gbytes / (mg * 1e-3) / 1e9 / peak, 4), "weight_bytes": gbytes}
        del gw, gs, gb, gx, gy
        # the step before decode: the next cache, this one's rows plus one new token per (sequence, KV head)
        akn = torch.randn(w.B, w.Hkv, 1, w.D, generator=gen, device=device)
        avn = torch.randn(w.B, w.Hkv, 1, w.D, generator=gen, device=device)
        anext = qda.QuantizedKV.empty([n + 1 for n in N], w.Hkv, w.D, w.GS, w.bits, synth.DT[w.dtype_in], device=device)
        acall = lambda: cache.append(akn, avn, out=anext, stream=stream)
        for _ in range(5):
            acall()
        ma = statistics.mean(time_calls(acall, 50, flush, stream))
        abytes = nbytes + anext.nbytes()   # old cache read once, new cache written once
        extra[f"{w.name}_append_1_token"] = {
            "us_per_call": round(ma * 1e3, 2), "GBps": round(abytes / (ma * 1e-3) / 1e9, 1),
            "frac_of_peak": round(abytes / (ma * 1e-3) / 1e9 / peak, 4), "bytes_moved": abytes}
        del akn, avn, anext
        # this workload's call captured once in a CUDA graph and replayed (split + merge, no host launch work)
        og = torch.empty_like(out)
        gs_ = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gs_):
            with torch.cuda.graph(graph, stream=gs_):
                qda.qdecode_attn(q, cache.kp, cache.ks, cache.kb, cache.vp, cache.vs, cache.vb, og, N, w.Hkv, w.GS,
                                 w.bits, gs_)
        gcall2 = lambda: graph.replay()
        for _ in range(5):
            gcall2()
        torch.cuda.synchronize()
        mgr = statistics.mean(time_calls(gcall2, 50, flush, torch.cuda.current_stream()))
        extra[f"{w.name}_graph_replay"] = {"us_per_call": round(mgr * 1e3, 2),
                                           "kv_GBps": round(nbytes / (mgr * 1e-3) / 1e9, 1),
                                           "frac_of_peak": round(nbytes / (mgr * 1e-3) / 1e9 / peak, 4)}
        del graph, og
        # small-L multi-query decode on this workload's cache: 4 query positions (the last 4 tokens) per sequence
        Lq = 4
        qm = synth.query_multi(w, Lq).to(device)
        om = torch.empty((w.B, Lq, w.H, w.D), dtype=synth.DT[w.dtype_out], device=device)
        mcall = lambda: qda.qdecode_attn_multi(qm, cache.kp, cache.ks, cache.kb, cache.vp, cache.vs, cache.vb, om,
                                               N, w.Hkv, w.GS, w.bits, stream)
        for _ in range(5):
            mcall()
        mm = statistics.mean(time_calls(mcall, 50, flush, stream))
        extra[f"{w.name}_L{Lq}"] = {"us_per_call": round(mm * 1e3, 2), "kv_GBps": round(nbytes / (mm * 1e-3) / 1e9, 1),
                                    "frac_of_peak": round(nbytes / (mm * 1e-3) / 1e9 / peak, 4), "kv_bytes": nbytes,
                                    "query_positions": Lq}

    cpu = None
    if pool is not None:
        cpu = cpu_baseline(w, N, q, cache, pool, cores)
        pool.close()
        cpu["single_thread_small_workload"] = cpu_single_thread_c1()

    line = {"metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "us_per_call": round(ms_per_step * 1e3, 3),
            "us_per_call_median": round(statistics.median(ms) * 1e3, 3),
            "wall_ms_per_step": round((t1 - t0) * 1e3 / args.steps, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 (codes u4/u8, q bf16)"
            if w.dtype_in == "bf16" else "f32 (codes u4/u8, q fp16)",
            "data": "synthetic (seeded generator; K, V ~ N(0,1) fp32 quantized by the library)",
            "config": config_of(w, N, {"plan": plan}), "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches, "clocks": clocks, "stream_floor": stream_floor, "per_workload": extra,
            "impl": "ours"}
    print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


# --------------------------------------------------------------------------------------- reference arm


def run_reference(args):
    """The oracle as it stands, single-threaded on a host core, over a bounded sample of the same workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import torch
    import oracle as O
    from attention_quantized_kv_split_gb300 import synth

    w = workload_by_index(args.workload)
    N = synth.lengths(w)
    q = synth.query(w)
    # one (sequence, KV head) unit, quantized by the oracle itself from the same generator (CPU stream)
    K, V = synth.kv_unit(w, 0, 0, N[0], q=q)
    kp, ks, kb, vp, vs, vb = O.quantize_cache(K.numpy(), V.numpy(), w.GS, w.bits, w.dtype_in)
    qh = q.double().numpy()[0, :w.nrep]
    W, NG = w.D * w.bits // 32, w.D // w.GS
    row_bytes = 2 * (W * 4 + 2 * NG * 2)

    def step(rows):
        Kd = O.dequantize(O.unpack(kp[:rows], w.bits, w.D), ks[:rows], kb[:rows], w.GS)
        Vd = O.dequantize(O.unpack(vp[:rows], w.bits, w.D), vs[:rows], vb[:rows], w.GS)
        for j in range(w.nrep):
            O.attention_head(qh[j], Kd, Vd)

    # size each step so that warm-up + steps take about 90 s in all
    t = time.perf_counter()
    step(N[0])
    per_row = (time.perf_counter() - t) / N[0]
    budget = 90.0 / max(1, args.steps + args.warmup)
    rows = int(max(16, min(N[0], budget / max(per_row, 1e-9))))
    for _ in range(args.warmup):
        step(rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(rows)
    dt = (time.perf_counter() - t0) / args.steps
    value = rows * row_bytes / dt / 1e9
    sample = (f"{rows} rows of one (sequence, KV head) unit of {w.name} with its {w.nrep} query heads per step "
              f"(the full call is {w.B * w.Hkv} units of {N[0] if w.B == 1 else 'ragged'} rows)")
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator)",
            "config": config_of(w, N), "impl": "reference",
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
