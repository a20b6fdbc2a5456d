"""Benchmark of the batch-1 quantized decode GEMVs (fmt=4, fmt=7, MQ4-V2).

One step = one batch-1 pass over the six decode GEMV shapes of the three
formats (fmt=4 int4-g64 2048x7168 and 7168x2048; fmt=7 FP8-e4m3-b128
7168x16384 and 24576x7168; MQ4-V2 5120x17408 and 17408x5120), each a call of
the C ABI on device-resident packed weights.  The metric is weight-GB/s:
(packed weight bytes + scale/header bytes) of the step / step time.  The
step touches 404 MB of weights, more than three times the 129 MB L2, so
every call streams its weights from HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

The batched-prefill dequant-GEMM (fmt=4, M=512 tokens, 7168x7168 and
2048x7168) is measured after the step loop and reported in the same line as
a fraction of the measured bf16 tensor peak ("prefill"): it is compute-bound
and has its own metric, so it is not folded into the GEMV bytes.

Prints one JSON line (rank 0).  With N > 1 (torchrun) every rank runs the
same step on its own GPU (replicas: the GEMVs need no exchange) and the
value is the bytes of all ranks over the slowest rank's time.
``--impl reference`` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "batch-1 quantized GEMV weight-GB/s and % of GB300 HBM peak (fmt4/fmt7/MQ4v2)"
WORKLOAD = ("decode GEMV pass, batch 1: fmt4 int4-g64 2048x7168 + 7168x2048, "
            "fmt7 fp8-e4m3-b128 7168x16384 + 24576x7168, MQ4-V2 5120x17408 + 17408x5120")

# (name, format, O, I, workload tag)
SHAPES = [
    ("fmt4_2048x7168", "i4g", 2048, 7168, 1),
    ("fmt4_7168x2048", "i4g", 7168, 2048, 1),
    ("fmt7_7168x16384", "fp8", 7168, 16384, 2),
    ("fmt7_24576x7168", "fp8", 24576, 7168, 2),
    ("mq4v2_5120x17408", "mq4", 5120, 17408, 3),
    ("mq4v2_17408x5120", "mq4", 17408, 5120, 3),
]
DOMINANT = "fmt7_24576x7168"
DOM_LAUNCHES = 200  # back-to-back launches timed for the dominant kernel's roofline
CPU_RUNS = 5        # oracle timing: median of this many runs per variant
GS = 64


def weight_bytes(fmt, O, I):
    """Algorithmic bytes of one call: packed weights + scales / headers."""
    if fmt == "i4g":
        return O * ((I + 1) // 2) + O * ((I + GS - 1) // GS) * 4
    if fmt == "fp8":
        return O * I + ((O + 127) // 128) * ((I + 127) // 128) * 4
    if fmt == "fp8ue8m0":
        return O * I + ((O + 127) // 128) * ((I + 127) // 128)
    if fmt == "q2_0":
        return O * (I // 64) * 18
    return O * (I // 256) * 136


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001
        return 6800.0, "fallback"


def load_tensor_peak():
    """Dense bf16 TFLOP/s: the measured burst figure (a kernel timed alone)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), "measured (burst)"
    except Exception:  # noqa: BLE001
        return 1900.0, "fallback"


# Sources of the dominant kernel (the staged fmt=7 GEMV); the committed DRAM
# traffic figure is valid only for the build these hash to.
DOMINANT_SOURCES = ("gemv_tma.cuh", "gemv_fp8.cuh", "gemv_fp8b128.cu", "common.cuh", "pipeline.cuh")


def source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "weight_only_quantized_i4g_gb300", "csrc")
    for name in DOMINANT_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def load_traffic():
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, or None when the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        if t.get("source_hash") != source_hash():
            return None
        return t.get(DOMINANT)
    except Exception:  # noqa: BLE001
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:  # noqa: BLE001
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:  # noqa: BLE001
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# inputs (device side: raw values uploaded, packed by the library's encoders)
# ---------------------------------------------------------------------------
def make_raw(name, fmt, O, I, tag):
    if fmt == "i4g":
        w, x = synth.fmt4_raw(O, I, 1, tag)
        return {"w": w, "x": x}
    if fmt == "fp8":
        codes, scales, x = synth.fmt7_raw(O, I, 1, tag)
        return {"codes": codes, "scales": scales, "x": x}
    w, x, d = synth.mq4_raw(O, I, 1, tag)
    return {"w": w, "x": x, "signs": d}


def build_device_call(qg, torch, fmt, O, I, raw, dev, stream):
    """Upload and pack one workload; returns (call(x_ptr, y_ptr), make_call(weights)
    -> the same call on other weight tensors, x, y, the weight tensors, the
    workspace tensor, (workspace pointer, bytes)).
    A shape whose reduction is split across thread blocks gets its workspace
    here, once (allocated outside the timed region, like the weights)."""
    lib = qg._lib
    st = stream.cuda_stream
    nws = qg.qg_workspace_bytes({"i4g": 4, "fp8": 7, "mq4": 44}[fmt], 1, I, O, GS)
    wsb = torch.empty(max(nws, 1), dtype=torch.uint8, device=dev)
    wsp = wsb.data_ptr() if nws else None
    if fmt == "i4g":
        w = torch.from_numpy(raw["w"]).to(dev)
        wq = torch.empty(O * ((I + 1) // 2), dtype=torch.uint8, device=dev)
        sc = torch.empty(O * ((I + GS - 1) // GS), dtype=torch.float32, device=dev)
        qg.check(qg.qg_quantize_i4g(wq, sc, w, O, I, GS, stream=st))
        x = torch.from_numpy(raw["x"]).to(dev)
        y = torch.empty(O, dtype=torch.float32, device=dev)
        del w
        keep = (wq, sc)

        def make_call(k):
            wp, sp = k[0].data_ptr(), k[1].data_ptr()
            return lambda xp, yp: lib.qgemv_i4g(yp, xp, wp, sp, 1, I, O, GS, wsp, nws, st)
    elif fmt == "fp8":
        codes = torch.from_numpy(raw["codes"]).to(dev)
        sc = torch.from_numpy(raw["scales"]).to(dev)
        x = torch.from_numpy(raw["x"].view(np.int16)).to(dev)
        y = torch.empty(O, dtype=torch.float32, device=dev)
        keep = (codes, sc)

        def make_call(k):
            wp, sp = k[0].data_ptr(), k[1].data_ptr()
            return lambda xp, yp: lib.qgemv_fp8b128(yp, xp, wp, sp, 1, I, O, wsp, nws, st)
    else:
        w = torch.from_numpy(raw["w"]).to(dev)
        d = torch.from_numpy(raw["signs"]).to(dev)
        qg.check(qg.qg_fwht256(w, w, d, O * I // 256, stream=st))
        blocks = torch.empty(O * (I // 256) * 136, dtype=torch.uint8, device=dev)
        qg.check(qg.qg_encode_mq4v2(blocks, w, O, I, stream=st))
        xf = torch.from_numpy(raw["x"]).to(dev)
        qg.check(qg.qg_fwht256(xf, xf, d, I // 256, stream=st))
        x = xf.to(torch.bfloat16).view(torch.int16)
        y = torch.empty(O, dtype=torch.float32, device=dev)
        del w
        keep = (blocks,)

        def make_call(k):
            bp = k[0].data_ptr()
            return lambda xp, yp: lib.qgemv_mq4v2(yp, xp, bp, 1, I, O, wsp, nws, st)
    return make_call(keep), make_call, x, y, keep, wsb, (wsp, nws)


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------
def build_oracle_inputs(orc, raws, shapes):
    inputs = []
    for (name, fmt, O, I, _), raw in zip(shapes, raws):
        if fmt == "i4g":
            wq, sc = orc.quantize_i4g(raw["w"], O, I, GS)
            inputs.append((fmt, O, I, (raw["x"], wq, sc)))
        elif fmt == "fp8":
            inputs.append((fmt, O, I, (raw["x"], raw["codes"], raw["scales"])))
        else:
            wr = orc.fwht256(raw["w"], raw["signs"])
            blocks = orc.encode_mq4v2(wr, O, I)
            xb = synth.bf16_bits(orc.fwht256(raw["x"], raw["signs"])).reshape(1, I)
            inputs.append((fmt, O, I, (xb, blocks)))
    return inputs


def oracle_pass(orc, inputs, frac, pool, nthreads):
    """One oracle pass over the first `frac` of every matrix's rows, split
    across host threads; returns the weight bytes processed."""
    jobs = []
    done = 0
    for fmt, O, I, args in inputs:
        rows = max(128, int(O * frac) // 128 * 128) if fmt == "fp8" else max(1, int(O * frac))
        rows = min(rows, O)
        done += weight_bytes(fmt, rows, I)
        step = 128 if fmt == "fp8" else 1
        chunk = max(step, (rows // nthreads + step - 1) // step * step)
        for o0 in range(0, rows, chunk):
            o1 = min(rows, o0 + chunk)
            if fmt == "i4g":
                jobs.append(pool.submit(orc.qgemv_i4g, *args, 1, I, O, GS, rows=(o0, o1)))
            elif fmt == "fp8":
                jobs.append(pool.submit(orc.qgemv_fp8b128, *args, 1, I, O, rows=(o0, o1)))
            else:
                jobs.append(pool.submit(orc.qgemv_mq4v2, *args, 1, I, O, rows=(o0, o1)))
    for j in jobs:
        j.result()
    return done


def cpu_oracle_timing(raws, shapes, steps, warmup, frac, nthreads=None, inputs=None):
    import oracle
    orc = oracle.Oracle()
    if inputs is None:
        inputs = build_oracle_inputs(orc, raws, shapes)
    nthreads = nthreads or os.cpu_count() or 1
    with ThreadPoolExecutor(nthreads) as pool:
        for _ in range(warmup):
            oracle_pass(orc, inputs, frac, pool, nthreads)
        t0 = time.perf_counter()
        nbytes = 0
        for _ in range(steps):
            nbytes += oracle_pass(orc, inputs, frac, pool, nthreads)
        dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, dt, nthreads


def cpu_baseline(raws, shapes):
    """The oracle on one full step (all six matrices, batch 1), single-
    threaded and on every host core (rows split across threads), median of
    CPU_RUNS runs each; the all-core figure is the headline."""
    import oracle
    orc = oracle.Oracle()
    inputs = build_oracle_inputs(orc, raws, shapes)
    cores = os.cpu_count() or 1
    variants = []
    for nthreads in (1, cores):
        runs = []
        for _ in range(CPU_RUNS):
            gbs, dt, _ = cpu_oracle_timing(raws, shapes, 1, 0, 1.0, nthreads=nthreads, inputs=inputs)
            runs.append((gbs, dt))
        runs.sort()
        gbs, dt = runs[len(runs) // 2]
        variants.append({"threads": nthreads, "value": round(gbs, 4), "unit": "GB/s",
                         "median_s_per_step": round(dt, 3), "runs": CPU_RUNS})
    top = variants[-1]
    return {"value": top["value"], "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"one full step (all six matrices, batch 1) per run, rows split across {cores} host threads; "
                      f"median of {CPU_RUNS} runs",
            "variants": variants}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    shapes = selected_shapes(args)
    raws = [make_raw(*s) for s in shapes]
    # bound the CPU work: about 40 full passes' worth over the whole run
    frac = min(1.0, 40.0 / max(1, args.steps + args.warmup))
    gbs, dt, cores = cpu_oracle_timing(raws, shapes, args.steps, args.warmup, frac)
    sample = (f"each step: the first {frac:.3g} of the rows of all six matrices (fp8 in whole "
              f"128-row blocks), batch 1, split by rows across {cores} host threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / max(1, args.steps) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "arm": "CPU oracle (plain C, f64 accumulation)"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(values, world, device=None):
    """Each value's maximum over the ranks of the process group (the slowest
    rank's time); the values themselves at world size 1."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_gbs(bytes_per_rank_step, world, ms_per_step):
    """Weight GB/s of the whole job: every rank streams bytes_per_rank_step
    per step (replicas), all in ms_per_step (the slowest rank's)."""
    return bytes_per_rank_step * world / (ms_per_step * 1e-3) / 1e9


def ours_arm(args):
    import torch
    import weight_only_quantized_i4g_gb300 as qg

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.Stream(device=dev)
    hbm_peak, peak_kind = load_peaks()

    shapes = selected_shapes(args)
    raws = [make_raw(*s) for s in shapes]
    calls = []
    with torch.cuda.stream(stream):
        for (name, fmt, O, I, tag), raw in zip(shapes, raws):
            call, make_call, x, y, keep, wsb, ws = build_device_call(qg, torch, fmt, O, I, raw, dev, stream)
            calls.append({"name": name, "fmt": fmt, "O": O, "I": I, "call": call, "make_call": make_call,
                          "x": x, "y": y, "keep": keep, "wsb": wsb, "ws": ws, "bytes": weight_bytes(fmt, O, I)})
    stream.synchronize()
    for c in calls:
        c["xp"], c["yp"] = c["x"].data_ptr(), c["y"].data_ptr()
    dom = next((i for i, c in enumerate(calls) if c["name"] == DOMINANT), 0)
    nbytes = sum(c["bytes"] for c in calls)

    def step():
        for c in calls:
            rc = c["call"](c["xp"], c["yp"])
            if rc:
                raise qg.QGError(rc)

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # W warm-up steps, then more until at least half a second of GPU work has
    # run: the SM clock of an idle GPU takes a while to reach its maximum.
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        t_warm = time.time()
        while time.time() - t_warm < 0.5:
            for _ in range(50):
                step()
            torch.cuda.synchronize()
    barrier()

    # The timed steps carry no events between calls: an event between two
    # launches stops the next one from starting early (programmatic dependent
    # launch).  The dominant kernel is timed right after them, on the same
    # stream, over DOM_LAUNCHES back-to-back launches alternating between two
    # copies of its weights (352 MB, so every launch streams from HBM).
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    dom_c = calls[dom]
    dom_copy = tuple(t.clone() for t in dom_c["keep"])
    dom_calls = [dom_c["call"], dom_c["make_call"](dom_copy)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)                      # let the sampler take its first reading
    n_launch0 = qg.qg_launch_count()
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for k in range(args.steps):
            step()
        t_end.record(stream)
    barrier()
    launches = qg.qg_launch_count() - n_launch0
    d_start = torch.cuda.Event(enable_timing=True)
    d_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for k in range(8):
            dom_calls[k & 1](dom_c["xp"], dom_c["yp"])
        d_start.record(stream)
        for k in range(DOM_LAUNCHES):
            rc = dom_calls[k & 1](dom_c["xp"], dom_c["yp"])
            if rc:
                raise qg.QGError(rc)
        d_end.record(stream)
    barrier()
    clocks = sampler.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    dom_ms = d_start.elapsed_time(d_end) / DOM_LAUNCHES
    del dom_copy, dom_calls

    # end to end through the C ABI with host buffers: every step copies its
    # activations host->device in one copy from a pinned staging buffer (each
    # call's x at a 256-byte aligned offset), runs the GEMVs on them, and
    # copies all outputs device->host in one copy into pinned memory.  Steps
    # are pipelined as a serving loop would run them: two sets of device
    # buffers, the uploads and the read-backs on their own streams, so that
    # step i+1's upload and step i-1's read-back overlap step i's GEMVs; event
    # waits keep each buffer's reuse in order (an upload waits until the
    # GEMVs two steps back have read its buffer, the GEMVs wait for their
    # upload and for the read-back that last used their output buffer).
    def packed(tensors):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, n

    xoffs, h2d = packed([c["x"] for c in calls])
    yoffs, d2h = packed([c["y"] for c in calls])
    xdev = [torch.empty(h2d, dtype=torch.uint8, device=dev) for _ in range(2)]
    ydev = [torch.zeros(d2h, dtype=torch.uint8, device=dev) for _ in range(2)]
    xhost = torch.empty(h2d, dtype=torch.uint8).pin_memory()
    yhost = [torch.zeros(d2h, dtype=torch.uint8).pin_memory() for _ in range(2)]
    for c, o in zip(calls, xoffs):
        xb = c["x"].contiguous().reshape(-1).view(torch.uint8).cpu()
        xhost[o:o + xb.numel()].copy_(xb)
    e2e_ptrs = [[(xdev[b].data_ptr() + xo, ydev[b].data_ptr() + yo) for xo, yo in zip(xoffs, yoffs)]
                for b in range(2)]
    up_stream, down_stream = torch.cuda.Stream(), torch.cuda.Stream()
    x_ready = [torch.cuda.Event() for _ in range(2)]
    x_read = [torch.cuda.Event() for _ in range(2)]
    y_ready = [torch.cuda.Event() for _ in range(2)]
    y_out = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):          # every buffer starts free
        x_read[b].record(stream)
        y_out[b].record(stream)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, min(args.steps, 2000))

    def e2e_step(i):
        b = i & 1
        up_stream.wait_event(x_read[b])
        with torch.cuda.stream(up_stream):
            xdev[b].copy_(xhost, non_blocking=True)
        x_ready[b].record(up_stream)
        stream.wait_event(x_ready[b])
        stream.wait_event(y_out[b])
        for c, (xp, yp) in zip(calls, e2e_ptrs[b]):
            rc = c["call"](xp, yp)
            if rc:
                raise qg.QGError(rc)
        x_read[b].record(stream)
        y_ready[b].record(stream)
        down_stream.wait_event(y_ready[b])
        with torch.cuda.stream(down_stream):
            yhost[b].copy_(ydev[b], non_blocking=True)
        y_out[b].record(down_stream)

    def drained():
        # the compute stream waits for the last read-backs
        for b in range(2):
            stream.wait_event(y_out[b])

    with torch.cuda.stream(stream):
        for i in range(min(args.warmup, 10)):
            e2e_step(i)
        drained()
        barrier()
        e_start.record(stream)
        up_stream.wait_event(e_start)
        for i in range(e2e_steps):
            e2e_step(i)
        drained()
        e_end.record(stream)
    barrier()
    # the host copies of the outputs must equal the device-timed outputs
    e2e_match = all(
        torch.equal(yhost[b][o:o + c["y"].numel() * c["y"].element_size()],
                    c["y"].contiguous().reshape(-1).view(torch.uint8).cpu())
        for b in range(min(2, e2e_steps)) for c, o in zip(calls, yoffs))
    e2e_ms = e_start.elapsed_time(e_end)

    elapsed_ms, e2e_ms = max_over_ranks([elapsed_ms, e2e_ms], world, dev)

    ms_per_step = elapsed_ms / args.steps
    value = whole_job_gbs(nbytes, world, ms_per_step)
    e2e_value = whole_job_gbs(nbytes, world, e2e_ms / e2e_steps)
    dom_bytes = calls[dom]["bytes"]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9

    per_format = per_format_breakdown(qg, torch, calls, stream, hbm_peak) if args.breakdown else None
    per_shape = None
    if per_format is not None:
        per_format.update(batched_breakdown(qg, torch, calls, stream, hbm_peak, dev))
        per_shape = {k: {"us": v["us_per_call"], "pct_hbm": v["pct_hbm_peak"]} for k, v in per_format.items()}
        if len(shapes) == len(SHAPES):
            per_format.update(one_header_breakdown(qg, torch, stream, hbm_peak, dev))
            per_format.update(moe_breakdown(qg, torch, stream, hbm_peak, dev))
    prefill = prefill_measure(qg, torch, dev, stream) if args.prefill else None
    if prefill is not None and len(shapes) == len(SHAPES):
        prefill["routed_experts"] = moe_prefill_measure(qg, torch, stream, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(raws, shapes)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": WORKLOAD if len(shapes) == len(SHAPES) else
                       "subset: " + ", ".join(c["name"] for c in calls), "batch": 1, "gs": GS,
                       "bytes_per_step": nbytes,
                       "pct_hbm_peak": round(100 * value / world / hbm_peak, 2),
                       "hbm_peak_gbs": hbm_peak, "hbm_peak_kind": peak_kind,
                       "l2": "inputs larger than L2: 404 MB of weights per step (L2 129 MB), "
                             "every call streams from HBM",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "kernel": calls[dom]["name"], "achieved": round(achieved, 2),
                         "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                         "traffic": load_traffic() if calls[dom]["name"] == DOMINANT else None,
                         "algorithmic_bytes": dom_bytes,
                         "avg_launch_us": round(dom_ms * 1e3, 3),
                         "launches_sampled": DOM_LAUNCHES,
                         "timing": f"{DOM_LAUNCHES} back-to-back launches on the launching stream right after "
                                   f"the timed steps, alternating two weight copies (2 x {dom_bytes} B > L2), "
                                   f"one CUDA event pair",
                         "peak_kind": f"{peak_kind} (copy bandwidth)",
                         "per_shape": per_shape,
                         "per_shape_timing": "kernel-only us per call and % of the HBM peak: a CUDA graph of "
                                             "back-to-back calls cycling >= 3x L2 of weight copies, best of 4"},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "copies_per_step": {"h2d": 1, "d2h": 1}, "outputs_match_device_run": e2e_match,
                    "pipelining": "two device buffer sets; each step's upload and read-back run on their "
                                  "own streams, overlapping the neighbouring steps' GEMVs"},
            "gpu_launches": launches,
            "clocks": clocks,
            "per_format": per_format,
            "prefill": prefill,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


PREFILL_M, PREFILL_I = 512, 7168
PREFILL_O = (7168, 2048)


def _time_alone(fn, flush, stream, reps, torch):
    """Median device time (s) of fn() on `stream`, each call after a write
    that flushes L2, bracketed by CUDA events on the same stream."""
    for _ in range(3):
        fn()
    ts = []
    for _ in range(reps):
        flush.fill_(1)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts) * 1e-3


def _prefill_inputs(qg, torch, dev, stream, fmt, O, I, M):
    """Seeded device inputs of one prefill GEMM shape: the decode workloads'
    weight recipes (fmt=4 quantized N(0, 0.02); fmt=7 uniform e4m3 codes
    without the NaN codes and log-uniform [1e-4, 1e-2] block scales (UE8M0:
    exponent bytes uniform in 113..120, the same range in powers of two); the MQ4
    formats (V2, v1, pad) N(0, 0.02) rotated by the seeded sign-FWHT and
    encoded) and bf16 N(0, 1) activations (rotated for MQ4).  Returns the
    weights and X."""
    g = torch.Generator(device=dev)
    g.manual_seed(4000 + O + 7 * I)
    if fmt == "i4g":
        w = torch.randn(O, I, generator=g, device=dev) * 0.02
        wq = torch.empty(O * I // 2, dtype=torch.uint8, device=dev)
        sc = torch.empty(O * (I // GS), dtype=torch.float32, device=dev)
        qg.check(qg.qg_quantize_i4g(wq, sc, w, O, I, GS, stream=stream))
        del w
        weights = (wq, sc)
    elif fmt in ("fp8", "fp8ue8m0"):
        codes = torch.randint(0, 254, (O * I,), generator=g, device=dev, dtype=torch.int32)
        codes = (codes + (codes >= 0x7F).to(torch.int32)).to(torch.uint8)   # skip 0x7F; 0xFF unreachable
        nbo, nbi = -(-O // 128), -(-I // 128)
        if fmt == "fp8":
            u = torch.rand(nbo * nbi, generator=g, device=dev, dtype=torch.float64)
            sc = torch.exp(math.log(1e-4) + u * (math.log(1e-2) - math.log(1e-4))).to(torch.float32)
        else:                                   # UE8M0 bytes 113..120: 2^-14..2^-7
            sc = torch.randint(113, 121, (nbo * nbi,), generator=g, device=dev, dtype=torch.int32).to(torch.uint8)
        weights = (codes, sc)
    else:
        signs = (torch.randint(0, 2, (256,), generator=g, device=dev, dtype=torch.int32) * 2 - 1).to(torch.int8)
        w = torch.randn(O, I, generator=g, device=dev) * 0.02
        qg.check(qg.qg_fwht256(w, w, signs, O * I // 256, stream=stream))
        blocks = torch.empty(O * (I // 256) * 136, dtype=torch.uint8, device=dev)
        qg.check(MQ4_ENCODE[fmt](qg)(blocks, w, O, I, stream=stream))
        del w
        weights = (blocks, signs)
    g.manual_seed(5000 + O + 7 * I)
    x = torch.randn(M, I, generator=g, device=dev)
    if fmt in MQ4_ENCODE:
        qg.check(qg.qg_fwht256(x, x, weights[1], M * I // 256, stream=stream))
    X = x.to(torch.bfloat16).view(torch.int16)
    return weights, X


PREFILL_OTHER = (("fp8", 7168, 16384), ("fp8", 24576, 7168), ("fp8ue8m0", 7168, 16384), ("fp8ue8m0", 24576, 7168),
                 ("mq4", 5120, 17408), ("mq4", 17408, 5120), ("mq4v1", 5120, 17408), ("mq4v1", 17408, 5120),
                 ("mq4c", 5120, 17408), ("mq4c", 17408, 5120))
FMT_ID = {"i4g": 4, "fp8": 7, "fp8ue8m0": 71, "mq4": 44, "mq4v1": 13, "mq4c": 45, "q2_0": 20}
# MQ4 block formats: V2 (a header per 128-weight half), v1 (one f32 header),
# pad (one fp16 header and four zero bytes); 136 bytes per 256 weights each
MQ4_ENCODE = {"mq4": lambda qg: qg.qg_encode_mq4v2, "mq4v1": lambda qg: qg.qg_encode_mq4v1,
              "mq4c": lambda qg: qg.qg_encode_mq4c}
MQ4_GEMV = {"mq4": "qgemv_mq4v2", "mq4v1": "qgemv_mq4v1", "mq4c": "qgemv_mq4c"}
MQ4_GEMM = {"mq4": "qgemm_mq4v2", "mq4v1": "qgemm_mq4v1", "mq4c": "qgemm_mq4c"}


def prefill_measure(qg, torch, dev, stream, reps=20, other=True, shapes=None):
    """The fmt=4 batched-prefill GEMM of the workload's prefill config:
    Y[512, O] = X[512, 7168] . W^T for O = 7168 and 2048, gs = 64, plus the
    fmt=7 and MQ4 (V2, v1, pad) prefill GEMMs at M = 512 on their decode
    shapes ("other_formats").  Weights and activations from seeded generators on
    the device.  Each call is timed alone with CUDA events on its stream
    after a 256 MiB write that flushes L2; median of `reps`.  Returns TFLOP/s
    (2*M*I*O per call) and the fraction of the measured dense bf16 peak.
    `shapes` (fmt, O, I) replaces all of them (profiling runs)."""
    peak, kind = load_tensor_peak()
    M, I = PREFILL_M, PREFILL_I
    out = {"workload": f"fmt4 int4-g64 prefill GEMM, M={M}, I={I}, O in {list(PREFILL_O)}, "
                       f"bf16 activations, f32 out",
           "bound": "tensor", "peak": peak, "unit": "TFLOP/s",
           "peak_kind": f"{kind} bf16 x 1 (the contraction is fp16 x fp16 -> f32; fp16 and bf16 dense rates are "
                        f"equal)", "calls": {}}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    launches = 0

    def run_one(fmt, O, I):
        nonlocal launches
        weights, X = _prefill_inputs(qg, torch, dev, stream, fmt, O, I, M)
        Y = torch.empty(M * O, dtype=torch.float32, device=dev)
        n = qg.qg_gemm_workspace_bytes(FMT_ID[fmt], M, I, O, GS if fmt == "i4g" else 0)
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
        if fmt == "i4g":
            fn = lambda: qg.check(qg.qgemm_i4g(Y, X, weights[0], weights[1], M, I, O, GS, ws, n, stream=stream))
        elif fmt == "fp8":
            fn = lambda: qg.check(qg.qgemm_fp8b128(Y, X, weights[0], weights[1], M, I, O, ws, n, stream=stream))
        elif fmt == "fp8ue8m0":
            fn = lambda: qg.check(qg.qgemm_fp8ue8m0(Y, X, weights[0], weights[1], M, I, O, ws, n, stream=stream))
        else:
            gemm = getattr(qg, MQ4_GEMM[fmt])
            fn = lambda: qg.check(gemm(Y, X, weights[0], M, I, O, ws, n, stream=stream))
        t = _time_alone(fn, flush, stream, reps, torch)
        launches += reps
        tf = 2.0 * M * I * O / t / 1e12
        return {"us": round(t * 1e6, 2), "tflops": round(tf, 1), "frac": round(tf / peak, 4)}

    with torch.cuda.stream(stream):
        if shapes is not None:
            out["calls"] = {f"{fmt} {M}x{O}x{I2}": run_one(fmt, O, I2) for fmt, O, I2 in shapes}
            out["launches_timed"] = launches
            return out
        for O in PREFILL_O:
            out["calls"][f"{M}x{O}x{I}"] = run_one("i4g", O, I)
        if other:
            out["other_formats"] = {f"{fmt} {M}x{O}x{I2}": run_one(fmt, O, I2) for fmt, O, I2 in PREFILL_OTHER}
    tot_flop = sum(2.0 * M * I * O for O in PREFILL_O)
    tot_t = sum(c["us"] for c in out["calls"].values()) * 1e-6
    out["achieved"] = round(tot_flop / tot_t / 1e12, 1)
    out["frac"] = round(out["achieved"] / peak, 4)
    out["launches_timed"] = launches
    return out


def per_format_breakdown(qg, torch, calls, stream, hbm_peak):
    """Kernel-only time per call of each shape: a CUDA graph of back-to-back
    calls cycling through enough copies of the weights (>= 3x L2) that every
    call reads from HBM; mean over the graph, best of 3 replays."""
    out = {}
    l2 = 129 * 2 ** 20
    for c in calls:
        fmt, O, I = c["fmt"], c["O"], c["I"]
        copies = max(1, -(-3 * l2 // c["bytes"]))
        copies = min(copies, 64)
        wcopies = []
        for _ in range(copies - 1):
            wcopies.append(tuple(t.clone() for t in c["keep"]))
        ptrsets = [tuple(t.data_ptr() for t in c["keep"])] + [tuple(t.data_ptr() for t in k) for k in wcopies]
        lib = qg._lib
        st = stream.cuda_stream
        reps = max(copies, 60)
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for r in range(reps):
                ps = ptrsets[r % len(ptrsets)]
                wsp, nws = c["ws"]
                if fmt == "i4g":
                    rc = lib.qgemv_i4g(c["yp"], c["xp"], ps[0], ps[1], 1, I, O, GS, wsp, nws, st)
                elif fmt == "fp8":
                    rc = lib.qgemv_fp8b128(c["yp"], c["xp"], ps[0], ps[1], 1, I, O, wsp, nws, st)
                else:
                    rc = lib.qgemv_mq4v2(c["yp"], c["xp"], ps[0], 1, I, O, wsp, nws, st)
                if rc:
                    raise qg.QGError(rc)
        best = None
        for _ in range(4):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):         # replay runs on the current stream
                a.record(stream)
                g.replay()
                b.record(stream)
            b.synchronize()
            t = a.elapsed_time(b) / reps
            best = t if best is None else min(best, t)
        del g, wcopies
        gbs = c["bytes"] / (best * 1e-3) / 1e9
        out[c["name"]] = {"us_per_call": round(best * 1e3, 3), "weight_gbs": round(gbs, 1),
                          "pct_hbm_peak": round(100 * gbs / hbm_peak, 1), "weight_copies": copies}
    return out


def _graph_per_call(torch, stream, reps, issue):
    """Capture `reps` back-to-back calls (issue(r) launches call r) in a CUDA
    graph on `stream`; returns the mean ms per call, best of 4 replays."""
    gr = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(gr, stream=stream):
        for r in range(reps):
            issue(r)
    best = None
    for _ in range(4):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            gr.replay()
            b.record(stream)
        b.synchronize()
        t = a.elapsed_time(b) / reps
        best = t if best is None else min(best, t)
    del gr
    return best


ONE_HEADER = (("mq4v1", 5120, 17408), ("mq4v1", 17408, 5120), ("mq4c", 5120, 17408), ("mq4c", 17408, 5120),
              ("fp8ue8m0", 7168, 16384), ("fp8ue8m0", 24576, 7168),
              ("q2_0", 2560, 640), ("q2_0", 640, 2560), ("q2_0", 2048, 7168), ("q2_0", 7168, 2048))


def one_header_breakdown(qg, torch, stream, hbm_peak, dev):
    """Kernel-only batch-1 GEMV time of the format variants: the one-header
    MQ4 block formats (v1: f32 scale and zero per 256 weights; pad: fp16 pair
    and four zero bytes) on the MQ4-V2 decode shapes and fmt=7 with UE8M0
    block scales on the fmt=7 decode shapes and the Q2_0 codec (random codes,
    d = 0.01) on the routed-expert shapes of the strata review and of the
    fmt=4 configs; same timing scheme as per_format_breakdown (graph of calls
    over >= 3x L2 of weight copies)."""
    out = {}
    l2 = 129 * 2 ** 20
    lib = qg._lib
    st = stream.cuda_stream
    with torch.cuda.stream(stream):
        for fmt, O, I in ONE_HEADER:
            if fmt == "q2_0":           # random codes, d = fp16 0.01 (no device encoder)
                g = torch.Generator(device=dev)
                g.manual_seed(6000 + O + I)
                blocks = torch.randint(0, 256, (O * (I // 64), 18), generator=g, device=dev,
                                       dtype=torch.int32).to(torch.uint8)
                blocks[:, 0:2] = torch.tensor([0x1F, 0x21], dtype=torch.uint8, device=dev)
                weights = (blocks.reshape(-1),)
                X = torch.randn(1, I, generator=g, device=dev).to(torch.bfloat16).view(torch.int16)
            else:
                weights, X = _prefill_inputs(qg, torch, dev, stream, fmt, O, I, 1)
            y = torch.empty(O, dtype=torch.float32, device=dev)
            nws = qg.qg_workspace_bytes(FMT_ID[fmt], 1, I, O, 0)
            wsb = torch.empty(max(nws, 1), dtype=torch.uint8, device=dev)
            nbytes = weight_bytes(fmt if fmt in ("fp8ue8m0", "q2_0") else "mq4", O, I)
            copies = min(64, max(1, -(-3 * l2 // nbytes)))
            wcopies = [weights[0]] + [weights[0].clone() for _ in range(copies - 1)]

            def issue(r):
                wp = wcopies[r % copies].data_ptr()
                if fmt == "fp8ue8m0":
                    rc = lib.qgemv_fp8ue8m0(y.data_ptr(), X.data_ptr(), wp, weights[1].data_ptr(), 1, I, O,
                                            wsb.data_ptr() if nws else None, nws, st)
                elif fmt == "q2_0":
                    rc = lib.qgemv_q2_0(y.data_ptr(), X.data_ptr(), wp, 1, I, O, wsb.data_ptr() if nws else None, nws,
                                        st)
                else:
                    rc = getattr(lib, MQ4_GEMV[fmt])(y.data_ptr(), X.data_ptr(), wp, 1, I, O,
                                                     wsb.data_ptr() if nws else None, nws, st)
                if rc:
                    raise qg.QGError(rc)
            best = _graph_per_call(torch, stream, max(copies, 60), issue)
            del wcopies
            gbs = nbytes / (best * 1e-3) / 1e9
            out[f"{fmt}_{O}x{I}"] = {"us_per_call": round(best * 1e3, 3), "weight_gbs": round(gbs, 1),
                                     "pct_hbm_peak": round(100 * gbs / hbm_peak, 1), "weight_copies": copies}
    return out


MOE_E, MOE_K = 32, 8     # experts in the table, routed experts per token


def moe_breakdown(qg, torch, stream, hbm_peak, dev):
    """Routed-expert decode at batch 1 on the routed-expert shapes: the gate and
    up projections of K = 8 routed experts (16 slots of 2048x7168 reading the
    token's x) and their down projections (8 slots of 7168x2048, one x each),
    fmt=4 g64 and MQ4-V2, one qgemv_moe launch each.  A table of 32 experts
    (>= 3x L2 of weights); every call routes to a different seeded set of 8,
    so the weights come from HBM.  Kernel-only time per call from a CUDA graph
    of back-to-back calls (best of 4 replays), against the same work as one
    single-matrix launch per slot."""
    out = {}
    lib = qg._lib
    st = stream.cuda_stream
    g = torch.Generator(device=dev)
    sets = 12
    for fmt_name, fmt in (("fmt4", 4), ("mq4v2", 44)):
        for proj, O, I, shared in (("gate_up", 2048, 7168, True), ("down", 7168, 2048, False)):
            per = 2 if proj == "gate_up" else 1            # matrices per expert
            n_tab = MOE_E * per
            g.manual_seed(7000 + O + fmt)
            mats, scs = [], []
            with torch.cuda.stream(stream):
                for _ in range(n_tab):
                    w = torch.randn(O, I, generator=g, device=dev) * 0.02
                    if fmt == 4:
                        wq = torch.empty(O * I // 2, dtype=torch.uint8, device=dev)
                        sc = torch.empty(O * (I // GS), dtype=torch.float32, device=dev)
                        qg.check(qg.qg_quantize_i4g(wq, sc, w, O, I, GS, stream=st))
                        mats.append(wq); scs.append(sc)
                    else:
                        blocks = torch.empty(O * (I // 256) * 136, dtype=torch.uint8, device=dev)
                        qg.check(qg.qg_encode_mq4v2(blocks, w, O, I, stream=st))
                        mats.append(blocks); scs.append(None)
                    del w
            stream.synchronize()
            table = torch.frombuffer(bytearray(qg.expert_table(list(zip(mats, scs)))), dtype=torch.uint8).to(dev)
            n_slots = MOE_K * per
            id_sets = []
            for k in range(sets):
                experts = torch.randperm(MOE_E, generator=torch.Generator().manual_seed(100 * k + O))[:MOE_K]
                ids = torch.stack([experts * per + j for j in range(per)], 1).reshape(-1)
                id_sets.append(ids.to(torch.int32).to(dev))
            n_x = 1 if shared else n_slots
            xs = torch.randn(n_x, I, generator=g, device=dev)
            x = xs if fmt == 4 else xs.to(torch.bfloat16).view(torch.int16)
            y = torch.empty(n_slots * O, dtype=torch.float32, device=dev)
            stride = 0 if shared else I
            nbytes = n_slots * weight_bytes("i4g" if fmt == 4 else "mq4", O, I)

            def issue_moe(r):
                rc = lib.qgemv_moe(fmt, y.data_ptr(), x.data_ptr(), stride, table.data_ptr(), n_tab,
                                   id_sets[r % sets].data_ptr(), n_slots, 1, I, O, GS if fmt == 4 else 0, st)
                if rc:
                    raise qg.QGError(rc)
            host_ids = [s.cpu().tolist() for s in id_sets]
            nws1 = qg.qg_workspace_bytes(fmt, 1, I, O, GS if fmt == 4 else 0)
            ws1 = torch.empty(max(nws1, 1), dtype=torch.uint8, device=dev)
            wsp1 = ws1.data_ptr() if nws1 else None

            def issue_single(r):
                for j, e in enumerate(host_ids[r % sets]):
                    xp = x.data_ptr() + (0 if shared else j * I * x.element_size())
                    yp = y.data_ptr() + j * O * 4
                    if fmt == 4:
                        rc = lib.qgemv_i4g(yp, xp, mats[e].data_ptr(), scs[e].data_ptr(), 1, I, O, GS, wsp1, nws1,
                                           st)
                    else:
                        rc = lib.qgemv_mq4v2(yp, xp, mats[e].data_ptr(), 1, I, O, wsp1, nws1, st)
                    if rc:
                        raise qg.QGError(rc)
            with torch.cuda.stream(stream):             # first launches set kernel attributes, outside capture
                issue_moe(0)
                issue_single(0)
            stream.synchronize()
            reps = 48
            t_moe = _graph_per_call(torch, stream, reps, issue_moe)
            t_one = _graph_per_call(torch, stream, reps, issue_single)
            gbs = nbytes / (t_moe * 1e-3) / 1e9
            out[f"moe_{fmt_name}_{proj}_{n_slots}x{O}x{I}"] = {
                "us_per_call": round(t_moe * 1e3, 3), "weight_gbs": round(gbs, 1),
                "pct_hbm_peak": round(100 * gbs / hbm_peak, 1),
                "single_matrix_launches_us": round(t_one * 1e3, 3), "slots": n_slots,
                "x": "shared" if shared else "per slot"}
            del mats, scs, table
    return out


def moe_prefill_measure(qg, torch, stream, dev, reps=10):
    """Routed-expert prefill: 512 tokens, each routed to 8 of 32 experts
    (seeded), sorted by expert into 4096 rows; the gate projection 2048x7168
    of every expert as one qgemm_moe call (one tensor-core launch over every
    group's tiles).  Timed alone after a 256 MiB write that flushes L2,
    median of `reps`; TFLOP/s over the routed rows (2 * 4096 * 7168 * 2048)."""
    peak, kind = load_tensor_peak()
    out = {"workload": "512 tokens x top-8 of 32 experts, gate projection 2048x7168 per expert, bf16 X, f32 Y",
           "peak": peak, "unit": "TFLOP/s", "calls": {}}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    T, K, E, O, I = 512, 8, 32, 2048, 7168
    gen = torch.Generator().manual_seed(77)
    routes = torch.stack([torch.randperm(E, generator=gen)[:K] for _ in range(T)])     # [T, K]
    counts = torch.bincount(routes.reshape(-1), minlength=E).tolist()
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + c)
    M = offsets[-1]
    g = torch.Generator(device=dev)
    for name, fmt in (("fmt4", 4), ("mq4v2", 44)):
        g.manual_seed(8100 + fmt)
        mats, scs = [], []
        with torch.cuda.stream(stream):
            for _ in range(E):
                w = torch.randn(O, I, generator=g, device=dev) * 0.02
                if fmt == 4:
                    wq = torch.empty(O * I // 2, dtype=torch.uint8, device=dev)
                    sc = torch.empty(O * (I // GS), dtype=torch.float32, device=dev)
                    qg.check(qg.qg_quantize_i4g(wq, sc, w, O, I, GS, stream=stream))
                    mats.append(wq); scs.append(sc)
                else:
                    blocks = torch.empty(O * (I // 256) * 136, dtype=torch.uint8, device=dev)
                    qg.check(qg.qg_encode_mq4v2(blocks, w, O, I, stream=stream))
                    mats.append(blocks); scs.append(None)
                del w
            X = torch.randn(M, I, generator=g, device=dev).to(torch.bfloat16).view(torch.int16)
            Y = torch.empty(M * O, dtype=torch.float32, device=dev)
        stream.synchronize()
        table = qg.expert_table(list(zip(mats, scs)))
        gs = GS if fmt == 4 else 0
        n = qg.qg_moe_gemm_workspace_bytes(fmt, offsets, E, I, O, gs)
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
        fn = lambda: qg.check(qg.qgemm_moe(fmt, Y, X, table, E, list(range(E)), offsets, E, I, O, gs, ws, n,
                                           stream=stream))
        with torch.cuda.stream(stream):
            t = _time_alone(fn, flush, stream, reps, torch)
        tf = 2.0 * M * I * O / t / 1e12
        out["calls"][f"{name} {M} rows"] = {"us": round(t * 1e6, 1), "tflops": round(tf, 1),
                                            "frac": round(tf / peak, 4), "groups": sum(1 for c in counts if c),
                                            "rows_per_group": [min(counts), max(counts)]}
        del mats, scs
    return out


BATCHED = {"i4g": 4, "mq4": 8}     # the configs' batched decode cases: fmt4 at batch 4, MQ4-V2 at 8


def batched_breakdown(qg, torch, calls, stream, hbm_peak, dev):
    """Kernel-only time per call of the batched decode cases (fmt=4 batch 4,
    MQ4-V2 batch 8, on the same two shapes each): as per_format_breakdown,
    a CUDA graph of back-to-back calls cycling through >= 3x L2 of weight
    copies; x ~ N(0, 1) (f32 for fmt=4, bf16 for MQ4-V2), seeded."""
    out = {}
    l2 = 129 * 2 ** 20
    lib = qg._lib
    st = stream.cuda_stream
    for c in calls:
        fmt = next((f for f in BATCHED if c["name"].startswith({"i4g": "fmt4", "mq4": "mq4"}[f])), None)
        if fmt is None:
            continue
        S = BATCHED[fmt]
        O, I = c["O"], c["I"]
        g = torch.Generator(device=dev)
        g.manual_seed(2000 + S)
        xs = torch.randn(S, I, generator=g, device=dev)
        x = xs if fmt == "i4g" else xs.to(torch.bfloat16).view(torch.int16)
        y = torch.empty(S * O, dtype=torch.float32, device=dev)
        n = qg.qg_workspace_bytes(4 if fmt == "i4g" else 44, S, I, O, GS)
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
        copies = min(64, max(1, -(-3 * l2 // c["bytes"])))
        wcopies = [c["keep"]] + [tuple(t.clone() for t in c["keep"]) for _ in range(copies - 1)]
        reps = max(copies, 60)
        gr = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(gr, stream=stream):
            for r in range(reps):
                ps = wcopies[r % len(wcopies)]
                if fmt == "i4g":
                    rc = lib.qgemv_i4g(y.data_ptr(), x.data_ptr(), ps[0].data_ptr(), ps[1].data_ptr(), S, I, O, GS,
                                       ws.data_ptr() if n else None, n, st)
                else:
                    rc = lib.qgemv_mq4v2(y.data_ptr(), x.data_ptr(), ps[0].data_ptr(), S, I, O,
                                         ws.data_ptr() if n else None, n, st)
                if rc:
                    raise qg.QGError(rc)
        best = None
        for _ in range(4):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                gr.replay()
                b.record(stream)
            b.synchronize()
            t = a.elapsed_time(b) / reps
            best = t if best is None else min(best, t)
        del gr, wcopies
        gbs = c["bytes"] / (best * 1e-3) / 1e9
        out[f"{c['name']}_batch{S}"] = {"us_per_call": round(best * 1e3, 3), "weight_gbs": round(gbs, 1),
                                        "pct_hbm_peak": round(100 * gbs / hbm_peak, 1), "batch": S}
    return out


def selected_shapes(args):
    if not args.only:
        return SHAPES
    names = args.only.split(",")
    unknown = set(names) - {s[0] for s in SHAPES}
    if unknown:
        raise SystemExit(f"--only: unknown shape(s) {sorted(unknown)}")
    return [s for s in SHAPES if s[0] in names]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-breakdown", dest="breakdown", action="store_false")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", dest="prefill", action="store_false",
                    help="skip the prefill GEMM measurement")
    ap.add_argument("--only", default="", help="comma-separated subset of the shapes (profiling runs)")
    ap.add_argument("--prefill-only", default="",
                    help="profiling runs: time only these prefill GEMMs (comma-separated fmt:O:I, fmt in "
                         "i4g/fp8/fp8ue8m0/mq4/mq4v1/mq4c, M=512) and print their prefill object")
    ap.add_argument("--prefill-reps", type=int, default=20)
    ap.add_argument("--moe-only", action="store_true", help="profiling runs: print only the routed-expert lines")
    ap.add_argument("--stamps", action="store_true",
                    help="profiling runs: per-block timelines of the batch-1 4-bit GEMVs (stamps build) and the "
                         "launch-chain floor")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = os.environ.get("WORLD_SIZE")
    if world is None and args.gpus > 1:
        # one process per GPU: relaunch this command under torchrun
        import socket
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
        raise SystemExit(subprocess.call(cmd))
    if world is not None and int(world) != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch one process per GPU "
                         f"(torchrun --nproc-per-node {args.gpus}) or pass the matching --gpus")
    if args.stamps:
        stamps_only(args)
    elif args.prefill_only:
        prefill_only(args)
    elif args.moe_only:
        moe_only(args)
    elif args.impl == "reference":
        reference_arm(args)
    else:
        ours_arm(args)


STAMP_SHAPES = (("fmt4_2048x7168", "i4g", 2048, 7168), ("fmt4_7168x2048", "i4g", 7168, 2048),
                ("mq4v2_17408x5120", "mq4", 17408, 5120))
STAMP_PHASES = (("start_to_wait", 0, 1), ("wait_to_x", 1, 2), ("x_to_first_batch", 2, 3),
                ("first_to_last_batch", 3, 4), ("last_batch_to_stored", 4, 5), ("block_total", 0, 5))
FLOOR_GRIDS = ((152, 256), (608, 96), (152, 352))


def stamps_only(args):
    """Per-block timelines of batch-1 decode GEMVs from the stamps build of the
    library (qg_stamps_take), and the floor of a chain of empty
    programmatic-dependent launches (qg_selftest_pdl_chain).  Each shape runs
    as a CUDA graph of back-to-back calls over >= 3x L2 of weight copies (the
    per-shape timing's scheme); the stamps are those of the graph's last call,
    whose predecessor on the stream is the same GEMV.  Prints one JSON line:
    per shape the graph-timed us per call of the stamps build and of
    libqgemv.so, and over the blocks the median and maximum of each phase in
    SM cycles and in us at the median SM clock sampled meanwhile, the spread
    of the blocks' start times (global timer) and the row batches per block;
    per launch shape the floor in us per launch."""
    import ctypes
    import torch
    import weight_only_quantized_i4g_gb300 as qg
    from weight_only_quantized_i4g_gb300 import _build
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream()
    slib = ctypes.CDLL(_build.build_stamps())
    P, I_, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    slib.qgemv_i4g.argtypes = [P, P, P, P, I_, I_, I_, I_, P, Z, P]
    slib.qgemv_i4g.restype = I_
    slib.qgemv_mq4v2.argtypes = [P, P, P, I_, I_, I_, P, Z, P]
    slib.qgemv_mq4v2.restype = I_
    clocks = ClockSampler(0)
    clocks.start()
    l2 = 129 * 2 ** 20
    shapes, raw_stamps = {}, {}
    st = stream.cuda_stream
    for name, fmt, O, I in STAMP_SHAPES:
        raw = make_raw(name, fmt, O, I, 1 if fmt == "i4g" else 3)
        _, _, x, y, keep, wsb, (wsp, nws) = build_device_call(qg, torch, fmt, O, I, raw, dev, stream)
        nbytes = weight_bytes(fmt, O, I)
        copies = min(64, max(1, -(-3 * l2 // nbytes)))
        wsets = [keep] + [tuple(t.clone() for t in keep) for _ in range(copies - 1)]
        xp, yp = x.data_ptr(), y.data_ptr()
        reps = max(copies, 60)

        def issue_with(lib, r):
            k = wsets[r % len(wsets)]
            if fmt == "i4g":
                rc = lib.qgemv_i4g(yp, xp, k[0].data_ptr(), k[1].data_ptr(), 1, I, O, GS, wsp, nws, st)
            else:
                rc = lib.qgemv_mq4v2(yp, xp, k[0].data_ptr(), 1, I, O, wsp, nws, st)
            if rc:
                raise qg.QGError(rc)

        us_normal = _graph_per_call(torch, stream, reps, lambda r: issue_with(qg._lib, r)) * 1e3
        # the stamps build: timed replays of one graph, then one more replay
        # whose last call leaves its stamps
        gr = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(gr, stream=stream):
            for r in range(reps):
                issue_with(slib, r)
        best = None
        for _ in range(4):
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                ev0.record(stream)
                gr.replay()
                ev1.record(stream)
            ev1.synchronize()
            t = ev0.elapsed_time(ev1) / reps
            best = t if best is None else min(best, t)
        us_stamps = best * 1e3
        rc, blocks = qg.qg_stamps_take(qg.STAMP_BLOCKS, lib=slib)      # clear
        qg.check(rc)
        with torch.cuda.stream(stream):
            gr.replay()
        rc, blocks = qg.qg_stamps_take(qg.STAMP_BLOCKS, lib=slib)
        qg.check(rc)
        del gr
        raw_stamps[name] = [b for b in blocks if b[0] != 0]
        shapes[name] = {"us_per_call": round(us_normal, 3), "us_per_call_stamps_build": round(us_stamps, 3),
                        "calls": reps, "weight_copies": copies}
        del wsets, keep, x, y, wsb
        torch.cuda.empty_cache()
    floors = {}
    for blocks_n, threads in FLOOR_GRIDS:
        floors[f"{blocks_n}x{threads}"] = round(
            _graph_per_call(torch, stream, 1, lambda r: qg.check(
                qg.qg_selftest_pdl_chain(blocks_n, threads, 2000, st))) * 1e3 / 2000, 3)
    ck = clocks.stop()
    mhz = ck["sm_mhz"] if ck else 2070.0
    for name, bl in raw_stamps.items():
        d = shapes[name]
        d["blocks"] = len(bl)
        d["batches_per_block"] = sorted({int(b[6]) for b in bl})
        g0 = [b[7] for b in bl]
        d["start_spread_us"] = round((max(g0) - min(g0)) / 1e3, 3) if g0 else None
        for ph, a, b_ in STAMP_PHASES:
            cyc = sorted(int(b[b_]) - int(b[a]) for b in bl if b[b_] and b[a])
            if not cyc:
                continue
            med = cyc[len(cyc) // 2]
            d[ph] = {"median_cycles": med, "max_cycles": cyc[-1], "median_us": round(med / mhz, 3),
                     "max_us": round(cyc[-1] / mhz, 3)}
    print(json.dumps({"stamps": shapes, "pdl_chain_floor_us_per_launch": floors, "clocks": ck,
                      "phases": "per block, SM cycles between: start, wait for the previous kernel returned, "
                                "activations ready, first batch landed (warp-MMA: after the activation setup), "
                                "consumers done with the last batch, last output stored"}), flush=True)


def moe_only(args):
    import torch
    import weight_only_quantized_i4g_gb300 as qg
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream()
    hbm_peak, _ = load_peaks()
    print(json.dumps({"moe": moe_breakdown(qg, torch, stream, hbm_peak, dev),
                      "moe_prefill": moe_prefill_measure(qg, torch, stream, dev)}), flush=True)


def prefill_only(args):
    import torch
    import weight_only_quantized_i4g_gb300 as qg
    shapes = []
    for item in args.prefill_only.split(","):
        fmt, O, I = item.split(":")
        if fmt not in FMT_ID:
            raise SystemExit(f"--prefill-only: unknown format {fmt!r}")
        shapes.append((fmt, int(O), int(I)))
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream()
    out = prefill_measure(qg, torch, dev, stream, reps=args.prefill_reps, shapes=shapes)
    print(json.dumps({"prefill": out}), flush=True)


if __name__ == "__main__":
    main()
