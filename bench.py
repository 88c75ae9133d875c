#!/usr/bin/env python3
"""Benchmark of the fused multi-query attention path on GB300.

One step = one decode attention call over the decode workload at 32768
context on a ratio-128 layer (T = 1, 64 heads, D = 512, 128 raw + 256
compressed rows): the split-KV tcgen05 kernel plus the log-sum-exp merge.
Prints ONE JSON line (rank 0).  See ``--help``.

Timing: W eager warm-up steps, then exactly K steps replayed from CUDA graphs
captured over R rotating input sets whose total size is several times the
129 MB L2, bracketed by a barrier and a synchronize, CUDA events on the
launching stream, max over ranks.  ``--gpus N`` under torchrun runs N
independent replicas (the path has no exchange step).
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attn HBM GB/s (% of 8 TB/s); prefill attn TFLOP/s (% fp16 peak)"
L2_BYTES = 129 * 1024 * 1024
SPIN_CYCLES = 200_000  # ~0.1 ms of device spin ahead of a timed region (see run_ours)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ["attn_kernel.cuh", "attn_params.h", "ptx.cuh", "attn.cu"]


# ------------------------------------------------------------------ workload arithmetic

def visible_rows(L: dict, t: int) -> int:
    """Rows token t sees under the structural rule (window + pooled rows)."""
    p = L["q_pos0"] + t
    lo = max(0, p - L["window"] + 1 - L["raw_pos0"])
    hi = min(L["n_raw"], p + 1 - L["raw_pos0"])
    comp = min(L["n_comp"], (p + 1) // L["ratio"]) if L["n_comp"] else 0
    return max(0, hi - lo) + comp


def decode_bytes(L: dict) -> int:
    """Compulsory HBM bytes of one decode call: Q, the visible K and V rows, O."""
    rows = sum(visible_rows(L, t) for t in range(L["T"]))
    return rows * 2 * 1024 + L["T"] * 2 * 64 * 512 * 2


def attn_flops(L: dict, rows_per_token=None) -> float:
    """4 * H * D flops per (token, visible row): QK^T and PV."""
    rows = rows_per_token if rows_per_token is not None else sum(visible_rows(L, t) for t in range(L["T"]))
    return 4.0 * 64 * 512 * rows


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "mqa_flash_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per launch of the attention kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_hash():
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples every 20 ms while running; keeps those inside [t0, t1]."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [r for ts, r in self.rows if t0 <= ts <= t1]
        window = "timed region"
        if not inside and self.rows:
            # a short timed region can fall between two samples: take the nearest ones
            inside = [min(self.rows, key=lambda x: abs(x[0] - (t0 + t1) / 2))[1]]
            window = "nearest sample to the timed region"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "no nvidia-smi"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm, smax, pw = [], [], []
        for r in inside:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                pw.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for i, n in enumerate(names):
                if len(r) > 5 + i and r[5 + i].lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons), "samples": len(inside),
                "window": window}


# ------------------------------------------------------------------ CPU oracle legs

def oracle_leg(workload: str, seconds: float, heads: int | None = None) -> dict:
    """Times the fp64 oracle (as it stands) on this process's host threads."""
    import numpy as np
    import oracle
    from mqa_flash_attention_gb300 import workloads as W
    wl = getattr(W, workload)()
    L = wl.layout
    q = wl.q if heads is None else np.ascontiguousarray(wl.q[:, :heads])
    frac = 1.0 if heads is None else heads / 64.0
    calls, t0 = 0, time.perf_counter()
    while True:
        oracle.attention(L, q, wl.k_raw, wl.v_raw, wl.k_comp, wl.v_comp)
        calls += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    per_call = el / calls
    return {"seconds_per_call": per_call, "calls": calls, "fraction_of_call": frac}


def run_oracle_subprocess(workload: str, seconds: float, heads=None) -> dict:
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--_oracle-leg", workload, "--_seconds", str(seconds)]
    if heads:
        cmd += ["--_heads", str(heads)]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        raise RuntimeError(f"oracle leg failed: {r.stderr[-2000:]}")
    return json.loads(r.stdout.strip().splitlines()[-1])


def run_oracle_all_cores(workload: str, seconds: float) -> dict:
    """The same single-threaded oracle leg in one process per host core, all at
    once: whole-host throughput in calls per second."""
    n = os.cpu_count() or 1
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--_oracle-leg", workload, "--_seconds", str(seconds)]
    procs = [subprocess.Popen(cmd, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for _ in range(n)]
    rate = 0.0
    for pr in procs:
        out, err = pr.communicate(timeout=600)
        if pr.returncode != 0:
            raise RuntimeError(f"oracle leg failed: {err[-2000:]}")
        rate += 1.0 / json.loads(out.strip().splitlines()[-1])["seconds_per_call"]
    return {"calls_per_second": rate, "processes": n}


# ------------------------------------------------------------------ host copies

def cuda_runtime():
    """The toolkit's CUDA runtime library through ctypes, or None.  Its current
    device is set to torch's (this copy of the runtime keeps its own)."""
    import torch
    for name in ("libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
        except OSError:
            continue
        if rt.cudaSetDevice(ctypes.c_int(torch.cuda.current_device())) != 0:
            return None
        return rt
    return None


class RuntimeEvents:
    """cudaEventRecord / cudaStreamWaitEvent without timing, called directly
    (a torch event call costs several microseconds of host time)."""

    def __init__(self, rt, n):
        self.rt = rt
        self.ev = []
        for _ in range(n):
            e = ctypes.c_void_p()
            if rt.cudaEventCreateWithFlags(ctypes.byref(e), 2) != 0:  # cudaEventDisableTiming
                raise RuntimeError("cudaEventCreateWithFlags failed")
            self.ev.append(e)
        rt.cudaEventRecord.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        rt.cudaStreamWaitEvent.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_uint]

    def record(self, i, stream):
        if self.rt.cudaEventRecord(self.ev[i], stream) != 0:
            raise RuntimeError("cudaEventRecord failed")

    def wait(self, stream, i):
        if self.rt.cudaStreamWaitEvent(stream, self.ev[i], 0) != 0:
            raise RuntimeError("cudaStreamWaitEvent failed")

    def close(self):
        for e in self.ev:
            self.rt.cudaEventDestroy(e)


def async_copies(dev_buf, host_buf, host_out, dev_out, stream):
    """Two callables: the host-to-device copy of the packed inputs and the
    device-to-host copy of the output, both on `stream`.  They call the CUDA
    runtime's cudaMemcpyAsync directly when the toolkit's runtime library can
    be loaded, else torch's copy_."""
    import torch
    nin = host_buf.numel() * host_buf.element_size()
    nout = host_out.numel() * host_out.element_size()
    rt = cuda_runtime()
    if rt is not None:
        fn = rt.cudaMemcpyAsync
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p]
        s = ctypes.c_void_p(stream.cuda_stream)
        a_in = (ctypes.c_void_p(dev_buf.data_ptr()), ctypes.c_void_p(host_buf.data_ptr()), nin, 1, s)
        a_out = (ctypes.c_void_p(host_out.data_ptr()), ctypes.c_void_p(dev_out.data_ptr()), nout, 2, s)

        def h2d():
            if fn(*a_in) != 0:
                raise RuntimeError("cudaMemcpyAsync (host to device) failed")

        def d2h():
            if fn(*a_out) != 0:
                raise RuntimeError("cudaMemcpyAsync (device to host) failed")
        return h2d, d2h, "cudaMemcpyAsync from pinned host memory"

    def h2d_t():
        with torch.cuda.stream(stream):
            dev_buf.copy_(host_buf, non_blocking=True)

    def d2h_t():
        with torch.cuda.stream(stream):
            host_out.copy_(dev_out, non_blocking=True)
    return h2d_t, d2h_t, "torch copy_ from pinned host memory"


# ------------------------------------------------------------------ ranks

def max_over_ranks(x: float, device="cpu") -> float:
    """The slowest rank's value (timings are reported as the max over ranks)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_step: float, steps: int, world: int, max_elapsed_s: float) -> float:
    """Units all ranks processed divided by the slowest rank's time (weak scaling:
    every rank runs its own replica of the step)."""
    return units_per_step * steps * world / max_elapsed_s


# ------------------------------------------------------------------ GPU arm

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_ours(args) -> None:
    import numpy as np
    import torch
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from mqa_flash_attention_gb300 import build, ds4a
    from mqa_flash_attention_gb300 import workloads as W
    build.build()
    lib = ds4a.lib()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    wl = W.decode_r128_32k()
    L = wl.layout
    step_bytes = decode_bytes(L)
    set_bytes = sum(a.nbytes for a in (wl.q, wl.k_raw, wl.v_raw, wl.k_comp, wl.v_comp)) + wl.q.nbytes
    R = max(8, math.ceil(4 * L2_BYTES / set_bytes))
    dev = torch.device("cuda", local)

    def to_dev(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    base = [to_dev(a) for a in (wl.q, wl.k_raw, wl.v_raw, wl.k_comp, wl.v_comp)]
    sets = []
    for i in range(R):
        # distinct buffers per set (same values): every step reads memory the previous steps did not touch
        sets.append([b.clone() for b in base] + [torch.empty_like(base[0])])
    n_splits = ds4a.decode_default_splits(L)
    ws = torch.empty(ds4a.decode_workspace_bytes(L, n_splits), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(i):
        q, kr, vr, kc, vc, o = sets[i % R]
        ds4a.attn_decode(L, q, kr, vr, kc, vc, n_splits=n_splits, workspace=ws, out=o, stream=stream)

    def partial_step(i):
        q, kr, vr, kc, vc, _ = sets[i % R]
        ds4a.attn_decode_partials(L, q, kr, vr, kc, vc, n_splits=n_splits, workspace=ws, stream=stream)

    K, Wm = args.steps, args.warmup
    with torch.cuda.stream(stream):
        for i in range(Wm):
            step(i)
    torch.cuda.synchronize()

    def capture(fn, n, offset=0):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                fn(offset + i)
        return g

    g_full = capture(step, min(R, K))
    g_tail = capture(step, K % R) if K > R and K % R else None
    n_full = K // R if K >= R else 1
    with torch.cuda.stream(stream):
        g_full.replay()
        if g_tail is not None:
            g_tail.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.25)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_host0 = time.time()
    with torch.cuda.stream(stream):  # a graph replays on the current stream
        # A short device spin ahead of the start event: the graph launch is queued while the GPU
        # spins, so the timed region holds the K steps and not the host's submission of the graph.
        torch.cuda._sleep(SPIN_CYCLES)
        e0.record(stream)
        for _ in range(n_full):
            g_full.replay()
        if g_tail is not None:
            g_tail.replay()
        e1.record(stream)
    barrier()
    t_host1 = time.time()
    sampler.stop()
    elapsed_ms = max_over_ranks(e0.elapsed_time(e1), dev)
    ms_per_step = elapsed_ms / K
    value = whole_job_rate(step_bytes, K, world, elapsed_ms * 1e-3) / 1e9
    clocks = sampler.summary(t_host0, t_host1)

    # Dominant kernel alone (split-KV attention, no merge): graph of R launches.
    gp = capture(partial_step, R)
    reps = max(1, min(50, 20000 // R))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    with torch.cuda.stream(stream):
        gp.replay()
        torch.cuda.synchronize()
        ev[0].record(stream)
        for i in range(reps):
            gp.replay()
            ev[i + 1].record(stream)
    torch.cuda.synchronize()
    kernel_us = ev[0].elapsed_time(ev[reps]) * 1e3 / (reps * R)
    per_replay = sorted(ev[i].elapsed_time(ev[i + 1]) * 1e3 / R for i in range(reps))
    pk, pk_kind = peaks()
    achieved = step_bytes / (kernel_us * 1e-6) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": ncu_traffic("decode_r128_32k"),
                "kernel": "ds4a::attn_fwd_kernel (split-KV partials)", "kernel_us": round(kernel_us, 3),
                "kernel_us_median": round(per_replay[len(per_replay) // 2], 3),
                "kernel_us_min": round(per_replay[0], 3),
                "kernel_us_note": f"mean, median and min over {reps} graph replays of {R} launches each",
                "peak_kind": f"{pk_kind} hbm_gbs (copy bandwidth)",
                "algorithmic_bytes_per_launch": step_bytes}

    # End to end through the API with host buffers: every step copies its inputs from pinned host
    # memory (Q, K/V raw, K/V compressed packed in one buffer, one transfer), calls the API on
    # device views of that buffer and copies the output back.
    arrays = [np.ascontiguousarray(a) for a in (wl.q, wl.k_raw, wl.v_raw, wl.k_comp, wl.v_comp)]
    offs, total = [], 0
    for a in arrays:
        offs.append(total)
        total += (a.nbytes + 255) // 256 * 256
    host_pack = torch.empty(total, dtype=torch.uint8).pin_memory()
    for a, o in zip(arrays, offs):
        host_pack[o:o + a.nbytes].copy_(torch.from_numpy(a.view(np.uint8).reshape(-1)))
    dev_pack = torch.empty(total, dtype=torch.uint8, device=dev)
    views = [dev_pack[o:o + a.nbytes].view(torch.float16).view(a.shape) for a, o in zip(arrays, offs)]
    host_out = torch.empty(tuple(wl.q.shape), dtype=torch.float16).pin_memory()
    do = torch.empty_like(sets[0][5])
    h2d = total
    d2h = host_out.numel() * host_out.element_size()
    Ke = min(K, 2000)
    # The decode call is prepared once (ctypes arguments built once; every step still calls the
    # C entry point), and copies and events go straight to the CUDA runtime: a torch copy_ costs
    # ~12 us of host time, more than the GPU work of a step.  Steps are pipelined as in a serving
    # loop: three streams and two buffer sets, so the input copy of step i+1 and the read-back of
    # step i-1 overlap step i's kernels; every step still copies its own inputs and output.
    rt = cuda_runtime()
    if rt is not None:
        dev_pack2 = [dev_pack, torch.empty_like(dev_pack)]
        views2 = [views, [dev_pack2[1][o:o + a.nbytes].view(torch.float16).view(a.shape)
                          for a, o in zip(arrays, offs)]]
        dev_out2 = [do, torch.empty_like(do)]
        host_out2 = [host_out, torch.empty_like(host_out).pin_memory()]
        s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        h_in, h_run, h_out = (ctypes.c_void_p(x.cuda_stream) for x in (s_in, stream, s_out))
        calls = [ds4a.prepare_decode(L, *views2[b], n_splits=n_splits, workspace=ws, out=dev_out2[b],
                                     stream=stream) for b in range(2)]
        h2ds = [async_copies(dev_pack2[b], host_pack, host_out2[b], dev_out2[b], s_in)[0] for b in range(2)]
        d2hs = [async_copies(dev_pack2[b], host_pack, host_out2[b], dev_out2[b], s_out)[1] for b in range(2)]
        evs = RuntimeEvents(rt, 6)  # 0,1 inputs copied; 2,3 step done; 4,5 output read back

        def e2e_steps(n):
            for i in range(n):
                b = i & 1
                if i >= 2:
                    evs.wait(h_in, 2 + b)    # step i-2 no longer reads this input buffer
                    evs.wait(h_run, 4 + b)   # and its output buffer has been read back
                h2ds[b]()
                evs.record(b, h_in)
                evs.wait(h_run, b)
                calls[b]()
                evs.record(2 + b, h_run)
                evs.wait(h_out, 2 + b)
                d2hs[b]()
                evs.record(4 + b, h_out)
        e2e_steps(4)
        barrier()
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(s_in)
        s_out.wait_event(x0)
        stream.wait_event(x0)
        e2e_steps(Ke)
        x1.record(s_out)  # after the last read-back, which follows every earlier step
        barrier()
        evs.close()
        e2e_check = host_out2[(Ke - 1) & 1].clone()
        copy_path = "cudaMemcpyAsync from pinned host memory; 3 streams, 2 buffer sets (pipelined steps)"
    else:
        call = ds4a.prepare_decode(L, *views, n_splits=n_splits, workspace=ws, out=do, stream=stream)
        h2d_copy, d2h_copy, copy_path = async_copies(dev_pack, host_pack, host_out, do, stream)
        for _ in range(3):
            h2d_copy()
            call()
            d2h_copy()
        barrier()
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(stream)
        for _ in range(Ke):
            h2d_copy()
            call()
            d2h_copy()
        x1.record(stream)
        barrier()
        e2e_check = host_out.clone()
    e2e_ms = max_over_ranks(x0.elapsed_time(x1), dev) / Ke
    e2e = {"value": round(step_bytes * world / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke, "ms_per_step": round(e2e_ms, 5),
           "api": "ds4a.prepare_decode(...)() each step (the C entry point ds4a_attn_decode)",
           "copies": copy_path}

    # Correctness guard on the timed outputs (decode of set 0 vs the kernel's own eager result), and
    # the end-to-end output against the same call on the workload's own inputs.
    ref = torch.empty_like(sets[0][5])
    ds4a.attn_decode(L, *sets[0][:5], n_splits=n_splits, workspace=ws, out=ref, stream=stream)
    ref_w = torch.empty_like(sets[0][5])
    ds4a.attn_decode(L, *[torch.from_numpy(a).to(dev) for a in arrays], n_splits=n_splits, workspace=ws,
                     out=ref_w, stream=stream)
    torch.cuda.synchronize()
    if not torch.equal(ref, sets[0][5]) or not torch.equal(ref_w.cpu(), e2e_check) or \
            ds4a.device_status() != ds4a.OK:
        raise RuntimeError("timed outputs differ from an eager call or a device wait ran out")

    also = None
    if rank == 0 and not args.no_also:
        also = run_also(torch, ds4a, W, dev, stream, pk, pk_kind)

    cpu = None
    if rank == 0:
        leg = run_oracle_subprocess("decode_r128_32k", args.cpu_seconds)
        allc = run_oracle_all_cores("decode_r128_32k", max(2.0, args.cpu_seconds / 2))
        cpu = {"value": round(step_bytes / leg["seconds_per_call"] / 1e9, 4), "unit": "GB/s", "cores": 1,
               "kind": "oracle",
               "sample": f"full decode call (T=1, 384 rows) x {leg['calls']} calls, "
                         f"{leg['seconds_per_call'] * 1e3:.2f} ms per call, fp64 numpy, 1 thread",
               "all_cores": {"value": round(step_bytes * allc["calls_per_second"] / 1e9, 4), "unit": "GB/s",
                             "cores": allc["processes"],
                             "sample": "the same leg in one single-threaded process per host core, concurrently"}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": Wm, "ms_per_step": round(ms_per_step, 6), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": "decode_ratio128_ctx32768: T=1, 64 q-heads, 1 KV head, D=512, 128 raw + "
                                   "256 compressed rows (all visible), fp16 N(0,1)",
                       "global_batch": world, "seq_len": 32768, "parallelism": f"replicas{world}",
                       "n_splits": n_splits, "rotating_input_sets": R,
                       "l2": f"inputs rotate over {R} sets ({R * set_bytes / 2**20:.0f} MiB > L2)",
                       "timing": "CUDA graphs of the decode call, CUDA events on the launching stream",
                       "step": "ds4a_attn_decode = split-KV tcgen05 attention (in-kernel block selection, "
                               "TMA zero-filled ragged tiles) + LSE merge"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 2 * K, "clocks": clocks,
        }
        if also is not None:
            line["also"] = also
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_also(torch, ds4a, W, dev, stream, pk, pk_kind):
    """The other headline shapes, each timed alone: prefill TFLOP/s, indexed
    TFLOP/s, long decode GB/s, with their roofline fractions."""
    import numpy as np
    out = []

    def timed(fn, n):
        for _ in range(2):
            fn(0)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                fn(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            torch.cuda.synchronize()
            torch.cuda._sleep(SPIN_CYCLES)  # the replay is queued before the start event is reached
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e-3 / n

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def sec_prefill():
        # prefill, raw-only, T = 2048 (two input sets alternate: each is ~270 MB > L2)
        wl = W.prefill_raw_2048()
        sets = [[up(wl.q), up(wl.k_raw), up(wl.v_raw), torch.empty(wl.q.shape, dtype=torch.float16, device=dev)]
                for _ in range(2)]
        sec = timed(lambda i: ds4a.attn_prefill(wl.layout, sets[i % 2][0], sets[i % 2][1], sets[i % 2][2],
                                                out=sets[i % 2][3], stream=stream), 10)
        fl = attn_flops(wl.layout)
        by = 2 * wl.q.nbytes + wl.k_raw.nbytes + wl.v_raw.nbytes
        out.append({"workload": wl.name, "us_per_call": round(sec * 1e6, 2),
                    "tflops": round(fl / sec / 1e12, 1), "frac_tensor": round(fl / sec / 1e12 / pk["bf16_tflops"], 4),
                    "hbm_gbs": round(by / sec / 1e9, 1), "frac_hbm": round(by / sec / 1e9 / pk["hbm_gbs"], 4),
                    "algorithmic_flops": fl, "algorithmic_bytes": by})
        del sets

    def sec_prefill_fp8kv():
        # the same prefill chunk with E4M3 raw rows (codes + one fp32 scale per row)
        wl = W.prefill_raw_2048()
        sets = []
        for _ in range(2):
            kr, vr = up(wl.k_raw), up(wl.v_raw)
            kc, ks = ds4a.quantize_kv_fp8(kr, stream=stream)
            vc, vs = ds4a.quantize_kv_fp8(vr, stream=stream)
            ws = torch.empty(ds4a.prefill_fp8kv_workspace_size(wl.layout), dtype=torch.uint8, device=dev)
            sets.append([up(wl.q), kc, ks, vc, vs, torch.empty(wl.q.shape, dtype=torch.float16, device=dev), ws])
        torch.cuda.synchronize()
        sec = timed(lambda i: ds4a.attn_prefill_fp8kv(wl.layout, sets[i % 2][0], sets[i % 2][1], sets[i % 2][3],
                                                      k_raw_scale=sets[i % 2][2], v_raw_scale=sets[i % 2][4],
                                                      out=sets[i % 2][5], workspace=sets[i % 2][6], stream=stream),
                    10)
        fl = attn_flops(wl.layout)
        n = wl.layout["n_raw"]
        by = 2 * wl.q.nbytes + 2 * n * (512 + 4)
        out.append({"workload": wl.name + "_fp8kv", "us_per_call": round(sec * 1e6, 2),
                    "tflops": round(fl / sec / 1e12, 1), "frac_tensor": round(fl / sec / 1e12 / pk["bf16_tflops"], 4),
                    "hbm_gbs": round(by / sec / 1e9, 1), "frac_hbm": round(by / sec / 1e9 / pk["hbm_gbs"], 4),
                    "algorithmic_flops": fl, "algorithmic_bytes": by,
                    "note": "raw K/V rows as E4M3 codes with per-row scales"})
        del sets

    def sec_indexed():
        # indexed ratio-4, T = 2048, top-512
        wl = W.indexed_r4_2048()
        sets = [[up(wl.q), up(wl.k_raw), up(wl.v_raw), up(wl.k_comp), up(wl.v_comp), up(wl.idx),
                 torch.empty(wl.q.shape, dtype=torch.float16, device=dev)] for _ in range(2)]
        sec = timed(lambda i: ds4a.attn_indexed(wl.layout, *sets[i % 2][:6], out=sets[i % 2][6], stream=stream), 6)
        rows = sum(min(wl.layout["n_raw"], 128) + int((wl.idx[t] >= 0).sum()) for t in range(wl.layout["T"]))
        fl = attn_flops(wl.layout, rows)
        out.append({"workload": wl.name, "us_per_call": round(sec * 1e6, 2),
                    "tflops": round(fl / sec / 1e12, 1), "frac_tensor": round(fl / sec / 1e12 / pk["bf16_tflops"], 4),
                    "algorithmic_flops": fl})
        # the same call with one row serving as K and V (the engine keeps one KV row per position);
        # indexed calls gather K and V apart even then (look-ahead ring order)
        seca = timed(lambda i: ds4a.attn_indexed(wl.layout, sets[i % 2][0], sets[i % 2][1], sets[i % 2][1],
                                                 sets[i % 2][3], sets[i % 2][3], sets[i % 2][5], out=sets[i % 2][6],
                                                 stream=stream), 6)
        out.append({"workload": wl.name + "_kv_shared", "us_per_call": round(seca * 1e6, 2),
                    "tflops": round(fl / seca / 1e12, 1),
                    "frac_tensor": round(fl / seca / 1e12 / pk["bf16_tflops"], 4), "algorithmic_flops": fl,
                    "speedup_vs_separate_kv": round(sec / seca, 2),
                    "note": "K and V are the same rows (k == v), gathered apart as for distinct rows"})
        # the same call with the listed compressed rows (and the raw rows) as E4M3 codes + row scales
        codes = []
        for st in sets:
            kc8, kcs = ds4a.quantize_kv_fp8(st[3], stream=stream)
            vc8, vcs = ds4a.quantize_kv_fp8(st[4], stream=stream)
            kr8, krs = ds4a.quantize_kv_fp8(st[1], stream=stream)
            vr8, vrs = ds4a.quantize_kv_fp8(st[2], stream=stream)
            codes.append((kr8, krs, vr8, vrs, kc8, kcs, vc8, vcs))
        torch.cuda.synchronize()

        def call8(i):
            kr8, krs, vr8, vrs, kc8, kcs, vc8, vcs = codes[i % 2]
            ds4a.attn_indexed_fp8kv(wl.layout, sets[i % 2][0], kr8, vr8, kc8, vc8, sets[i % 2][5], k_comp_scale=kcs,
                                    v_comp_scale=vcs, k_raw_scale=krs, v_raw_scale=vrs, out=sets[i % 2][6],
                                    stream=stream)
        sec8 = timed(call8, 6)
        out.append({"workload": wl.name + "_fp8kv", "us_per_call": round(sec8 * 1e6, 2),
                    "tflops": round(fl / sec8 / 1e12, 1),
                    "frac_tensor": round(fl / sec8 / 1e12 / pk["bf16_tflops"], 4), "algorithmic_flops": fl,
                    "note": "raw and listed compressed rows as E4M3 codes with per-row scales"})
        del sets, codes

    def sec_decode_sweep():
        # long-decode sweep (config 5 at N = 1K, 8K, 64K): input sets rotate so every call reads HBM
        for n_c in (1024, 8192, 65536):
            wl = W.decode_long(n_c)
            base = [up(a) for a in (wl.q, wl.k_raw, wl.v_raw, wl.k_comp, wl.v_comp)]
            sb = sum(t.numel() * t.element_size() for t in base)
            R = min(256, max(2, math.ceil(4 * L2_BYTES / sb)))
            dsets = [[t.clone() for t in base] for _ in range(R)]
            del base
            o = torch.empty(wl.q.shape, dtype=torch.float16, device=dev)
            ws = torch.empty(ds4a.decode_workspace_bytes(wl.layout), dtype=torch.uint8, device=dev)
            sec = timed(lambda i: ds4a.attn_decode(wl.layout, *dsets[i % R], workspace=ws, out=o, stream=stream), R)
            by = decode_bytes(wl.layout)
            out.append({"workload": wl.name, "us_per_call": round(sec * 1e6, 2), "hbm_gbs": round(by / sec / 1e9, 1),
                        "frac_hbm": round(by / sec / 1e9 / pk["hbm_gbs"], 4), "algorithmic_bytes": by,
                        "rotating_input_sets": R})
            del dsets, o, ws

    def sec_decode_256k_fp16_and_fp8():
        # long decode, 262144 compressed rows (537 MB of K/V > L2)
        wl = W.decode_long(262144)
        d = [up(a) for a in (wl.q, wl.k_raw, wl.v_raw, wl.k_comp, wl.v_comp)]
        o = torch.empty(wl.q.shape, dtype=torch.float16, device=dev)
        ws = torch.empty(ds4a.decode_workspace_bytes(wl.layout), dtype=torch.uint8, device=dev)
        sec = timed(lambda i: ds4a.attn_decode(wl.layout, *d, workspace=ws, out=o, stream=stream), 10)
        by = decode_bytes(wl.layout)
        out.append({"workload": wl.name, "us_per_call": round(sec * 1e6, 2), "hbm_gbs": round(by / sec / 1e9, 1),
                    "frac_hbm": round(by / sec / 1e9 / pk["hbm_gbs"], 4), "algorithmic_bytes": by})
        # the same decode with one row serving as K and V (k == v pointers): each row is read once
        seca = timed(lambda i: ds4a.attn_decode(wl.layout, d[0], d[1], d[1], d[3], d[3], workspace=ws, out=o,
                                                stream=stream), 10)
        bya = by - (wl.layout["n_raw"] + wl.layout["n_comp"]) * 1024
        out.append({"workload": wl.name + "_kv_shared", "us_per_call": round(seca * 1e6, 2),
                    "hbm_gbs": round(bya / seca / 1e9, 1), "frac_hbm": round(bya / seca / 1e9 / pk["hbm_gbs"], 4),
                    "algorithmic_bytes": bya, "speedup_vs_fp16": round(sec / seca, 2),
                    "note": "K and V are the same rows (k == v): 1024 bytes per row instead of 2048"})
        # the same decode with E4M3 compressed rows (codes + one fp32 scale per row)
        kc, ks = ds4a.quantize_kv_fp8(d[3], stream=stream)
        vc, vs = ds4a.quantize_kv_fp8(d[4], stream=stream)
        torch.cuda.synchronize()
        sec8 = timed(lambda i: ds4a.attn_decode_fp8(wl.layout, d[0], d[1], d[2], kc, ks, vc, vs, workspace=ws, out=o,
                                                    stream=stream), 10)
        n_c = wl.layout["n_comp"]
        by8 = by - n_c * 2048 + n_c * (1024 + 8)
        out.append({"workload": wl.name + "_fp8kv", "us_per_call": round(sec8 * 1e6, 2), "hbm_gbs": round(by8 / sec8 / 1e9, 1),
                    "frac_hbm": round(by8 / sec8 / 1e9 / pk["hbm_gbs"], 4), "algorithmic_bytes": by8,
                    "speedup_vs_fp16": round(sec / sec8, 2)})
        del d, o, ws, kc, ks, vc, vs

    def sec_decode_batch64():
        # batched decode: 64 sequences, each the ratio-128 32K geometry (128 raw + 256 compressed
        # rows) with its own K/V rows; three input sets rotate (3 x 58.7 MB > L2)
        wl = W.decode_r128_32k()
        B, G = 64, 3
        L = wl.layout
        geo = torch.tensor([[L["q_pos0"], L["n_raw"], L["raw_pos0"], L["n_comp"]]] * B, dtype=torch.int32, device=dev)
        bsets = []
        for gi in range(G):
            gen = torch.Generator(device=dev).manual_seed(90 + gi)
            mk = lambda n: torch.randn((B, n, 512), generator=gen, device=dev).to(torch.float16)  # noqa: E731
            bsets.append([torch.randn((B, 64, 512), generator=gen, device=dev).to(torch.float16),
                          mk(L["n_raw"]), mk(L["n_raw"]), mk(L["n_comp"]), mk(L["n_comp"]),
                          torch.empty((B, 64, 512), dtype=torch.float16, device=dev)])
        b_splits = ds4a.lib().ds4a_attn_decode_batch_default_splits(B, ctypes.byref(ds4a.make_layout(L)), L["n_raw"],
                                                                   L["n_comp"])
        bws = torch.empty(max(256, ds4a.lib().ds4a_attn_decode_batch_workspace_size(B, b_splits)), dtype=torch.uint8,
                          device=dev)
        sec = timed(lambda i: ds4a.attn_decode_batch(L, geo, *bsets[i % G][:5], n_splits=b_splits, workspace=bws,
                                                     out=bsets[i % G][5], stream=stream), 30)
        by = B * decode_bytes(L)
        out.append({"workload": "decode_batch64_ratio128_ctx32768", "us_per_call": round(sec * 1e6, 2),
                    "hbm_gbs": round(by / sec / 1e9, 1), "frac_hbm": round(by / sec / 1e9 / pk["hbm_gbs"], 4),
                    "algorithmic_bytes": by, "n_splits": b_splits,
                    "note": "64 sequences, each 128 raw + 256 compressed rows of its own"})
        del bsets, bws, geo

    def sec_indexer():
        # indexer of the ratio-4 layer: scores (64 heads x 128 dims, max(0, x)) and top-512
        wx = W.indexer_r4_2048()
        L = wx.layout
        qx, kx, wx_w = up(wx.q_idx), up(wx.k_idx), up(wx.w)
        sc = [torch.empty((L["T"], L["n_comp"]), dtype=torch.float32, device=dev) for _ in range(2)]
        sec = timed(lambda i: ds4a.indexer_scores(L, qx, kx, wx_w, scale=wx.scale, relu=True, out=sc[i % 2],
                                                  stream=stream), 10)
        n_cand = sum(min(L["n_comp"], (L["q_pos0"] + t + 1) // L["ratio"]) for t in range(L["T"]))
        n_heads, head_dim = wx.q_idx.shape[1], wx.q_idx.shape[2]
        fl = 2.0 * n_cand * n_heads * head_dim
        out.append({"workload": wx.name + "_scores", "us_per_call": round(sec * 1e6, 2),
                    "tflops": round(fl / sec / 1e12, 1), "frac_tensor": round(fl / sec / 1e12 / pk["bf16_tflops"], 4),
                    "algorithmic_flops": fl, "shape": f"{n_heads} heads x {head_dim} dims, relu"})
        ix_out = torch.empty((L["T"], wx.top_k), dtype=torch.int32, device=dev)
        sec = timed(lambda i: ds4a.indexer_topk(L, sc[i % 2], wx.top_k, out=ix_out, stream=stream), 10)
        by = 4 * n_cand + 4 * L["T"] * wx.top_k
        out.append({"workload": wx.name + "_topk", "us_per_call": round(sec * 1e6, 2),
                    "gbs": round(by / sec / 1e9, 1), "algorithmic_bytes": by,
                    "note": "exact radix select over each token's candidate scores"})

    def sec_compressor_prefill():
        # compressor, one 2048-token prefill chunk of 512-dim rows (fresh state) on a ratio-4 and a
        # ratio-128 layer; 20 input sets rotate (20 x 8 MB > L2)
        for ratio in (4, 128):
            wc = W.compressor_prefill(ratio)
            n, width = wc.kv.shape
            G = 20
            gen = torch.Generator(device=dev).manual_seed(95 + ratio)
            csets = [(torch.randn((n, width), generator=gen, device=dev),
                      2 * torch.randn((n, width), generator=gen, device=dev)) for _ in range(G)]
            st_kv = torch.empty((ratio - 1, width), dtype=torch.float32, device=dev)
            st_s = torch.empty((ratio - 1, width), dtype=torch.float32, device=dev)
            c_out = torch.empty((n // ratio, width), dtype=torch.float16, device=dev)
            sec = timed(lambda i: ds4a.compress_append(csets[i % G][0], csets[i % G][1], st_kv, st_s, 0, ratio,
                                                       out=c_out, stream=stream), 40)
            by = 8 * n * width + 2 * (n // ratio) * width
            out.append({"workload": wc.name, "us_per_call": round(sec * 1e6, 2), "hbm_gbs": round(by / sec / 1e9, 1),
                        "frac_hbm": round(by / sec / 1e9 / pk["hbm_gbs"], 4), "algorithmic_bytes": by,
                        "note": "per-dimension softmax pooling of each ratio span, fp32 in, fp16 out"})
            del csets

    def sec_compressor_decode():
        # compressor decode step at a ratio-128 boundary: 127 positions in the state, one new
        st_kv = torch.randn((127, 512), device=dev)
        st_s = torch.randn((127, 512), device=dev)
        one = [(torch.randn((1, 512), device=dev), torch.randn((1, 512), device=dev)) for _ in range(2)]
        c_out = torch.empty((1, 512), dtype=torch.float16, device=dev)
        sec = timed(lambda i: ds4a.compress_append(one[i % 2][0], one[i % 2][1], st_kv, st_s, 127, 128, out=c_out,
                                                   stream=stream), 40)
        out.append({"workload": "compressor_ratio128_decode_boundary_w512", "us_per_call": round(sec * 1e6, 2),
                    "note": "one token completes a 128-position span (state in L2): latency"})
        del st_kv, st_s, one

    # Each line is measured on its own: a failure (for instance too little memory on a smaller
    # device) becomes an entry with the error instead of losing the benchmark line.
    for sec_fn in (sec_prefill, sec_prefill_fp8kv, sec_indexed, sec_decode_sweep, sec_decode_256k_fp16_and_fp8, sec_decode_batch64,
                   sec_indexer, sec_compressor_prefill, sec_compressor_decode):
        try:
            sec_fn()
        except Exception as e:  # noqa: BLE001 - reported in the line
            out.append({"workload": sec_fn.__name__[4:], "error": repr(e)[:300]})
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    for e in out:
        e["peak_kind"] = pk_kind
    return out


# ------------------------------------------------------------------ profiling cases

CASES = ("tiny", "decode_r128_32k", "prefill_raw_2048", "prefill_raw_2048_fp8kv", "indexed_r4_2048",
         "decode_long_262144", "decode_long_262144_fp8kv", "indexer_r4_2048", "compressor_r4_2048",
         "compressor_r128_2048")


def run_case(name: str, calls: int) -> None:
    """Runs `calls` calls of one workload and exits: the program ncu captures."""
    import numpy as np
    import torch
    from mqa_flash_attention_gb300 import build, ds4a
    from mqa_flash_attention_gb300 import workloads as W
    build.build()
    if name == "indexer_r4_2048":
        wx = W.indexer_r4_2048()
        up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
        qx, kx, w = up(wx.q_idx), up(wx.k_idx), up(wx.w)
        for _ in range(calls):
            s = ds4a.indexer_scores(wx.layout, qx, kx, w, scale=wx.scale, relu=True)
            ds4a.indexer_topk(wx.layout, s, wx.top_k)
        torch.cuda.synchronize()
        if ds4a.device_status() != ds4a.OK:
            raise RuntimeError("device wait ran out")
        print(f"{name}: {calls} calls ok")
        return
    if name.startswith("compressor_r"):
        ratio = int(name[len("compressor_r"):].split("_")[0])
        wc = W.compressor_prefill(ratio)
        up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
        kv, sc = up(wc.kv), up(wc.score)
        st_kv = torch.empty((ratio - 1, kv.shape[1]), dtype=torch.float32, device="cuda")
        st_s = torch.empty_like(st_kv)
        for _ in range(calls):
            ds4a.compress_append(kv, sc, st_kv, st_s, 0, ratio)
        torch.cuda.synchronize()
        print(f"{name}: {calls} calls ok")
        return
    if name == "decode_long_262144_fp8kv":
        # the 262,144-row decode over E4M3 compressed rows (codes + one fp32 scale per row)
        wl = W.decode_long(262144)
        up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
        q, kr, vr = up(wl.q), up(wl.k_raw), up(wl.v_raw)
        kc, ks = ds4a.quantize_kv_fp8(up(wl.k_comp))
        vc, vs = ds4a.quantize_kv_fp8(up(wl.v_comp))
        outs = [torch.empty_like(q) for _ in range(calls)]
        for i in range(calls):
            ds4a.attn_decode_fp8(wl.layout, q, kr, vr, kc, ks, vc, vs, out=outs[i])
        torch.cuda.synchronize()
        if ds4a.device_status() != ds4a.OK:
            raise RuntimeError("device wait ran out")
        print(f"{name}: {calls} calls ok")
        return
    if name == "prefill_raw_2048_fp8kv":
        # the 2048-token raw prefill over E4M3 raw rows: widening pass into the workspace, pair kernel
        wl = W.prefill_raw_2048()
        up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
        q = up(wl.q)
        kc, ks = ds4a.quantize_kv_fp8(up(wl.k_raw))
        vc, vs = ds4a.quantize_kv_fp8(up(wl.v_raw))
        ws = torch.empty(ds4a.prefill_fp8kv_workspace_size(wl.layout), dtype=torch.uint8, device="cuda")
        outs = [torch.empty_like(q) for _ in range(calls)]
        for i in range(calls):
            ds4a.attn_prefill_fp8kv(wl.layout, q, kc, vc, k_raw_scale=ks, v_raw_scale=vs, workspace=ws,
                                    out=outs[i])
        torch.cuda.synchronize()
        if ds4a.device_status() != ds4a.OK:
            raise RuntimeError("device wait ran out")
        print(f"{name}: {calls} calls ok")
        return
    wl = W.decode_long(262144) if name == "decode_long_262144" else getattr(W, name)()
    L = wl.layout

    def up(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    d = [up(a) for a in (wl.q, wl.k_raw, wl.v_raw, wl.k_comp, wl.v_comp)]
    outs = [torch.empty_like(d[0]) for _ in range(calls)]
    for i in range(calls):
        if name == "indexed_r4_2048":
            ds4a.attn_indexed(L, *d, up(wl.idx), out=outs[i])
        elif name.startswith("decode"):
            ds4a.attn_decode(L, *d, out=outs[i])
        else:
            ds4a.attn_prefill(L, *d[:3], *(d[3:] if L["n_comp"] else []), out=outs[i])
    torch.cuda.synchronize()
    if ds4a.device_status() != ds4a.OK:
        raise RuntimeError("device wait ran out")
    print(f"{name}: {calls} calls ok")


# ------------------------------------------------------------------ reference arm

def run_reference(args) -> None:
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    from mqa_flash_attention_gb300 import workloads as W
    wl = W.decode_r128_32k()
    L = wl.layout
    step_bytes = decode_bytes(L)
    probe = oracle_leg("decode_r128_32k", 0.5)
    per_call = probe["seconds_per_call"]
    max_seconds = 90.0  # the whole reference run stays within a few minutes
    heads = None
    if (args.steps + args.warmup) * per_call > max_seconds:
        heads = max(1, min(64, int(64 * max_seconds / ((args.steps + args.warmup) * per_call))))
    import numpy as np  # noqa: F401
    import oracle
    q = wl.q if heads is None else np.ascontiguousarray(wl.q[:, :heads])
    for _ in range(args.warmup):
        oracle.attention(L, q, wl.k_raw, wl.v_raw, wl.k_comp, wl.v_comp)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.attention(L, q, wl.k_raw, wl.v_raw, wl.k_comp, wl.v_comp)
    el = time.perf_counter() - t0
    frac = 1.0 if heads is None else heads / 64.0
    value = step_bytes * frac * args.steps / el / 1e9
    sample = ("full decode call (T=1, 384 rows) per step" if heads is None else
              f"{heads} of 64 heads of the decode call per step (bytes scaled by {frac:.3f})")
    cores = 1
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "decode_ratio128_ctx32768: T=1, 64 q-heads, 1 KV head, D=512, 128 raw + "
                                   "256 compressed rows (all visible), fp16 N(0,1)",
                       "global_batch": 1, "seq_len": 32768, "parallelism": "host"},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-also", action="store_true", help="skip the prefill / indexed / long-decode lines")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="length of the CPU oracle baseline")
    ap.add_argument("--case", choices=CASES, default=None,
                    help="run --calls calls of one workload and exit (the program ncu captures)")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--_oracle-leg", dest="oracle_leg", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--_seconds", dest="leg_seconds", type=float, default=10.0, help=argparse.SUPPRESS)
    ap.add_argument("--_heads", dest="leg_heads", type=int, default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_leg:
        print(json.dumps(oracle_leg(args.oracle_leg, args.leg_seconds, args.leg_heads)))
        return
    if args.case:
        run_case(args.case, args.calls)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    if "--impl" in sys.argv and "reference" in sys.argv:
        for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[v] = "1"
    main()
