"""Throughput benchmark: causal GQA attention forward + backward on one GB300.

One step = one pass of the whole path over one batch of the GPT-2-small
attention workload (B=8, H=12, Hkv=4, N=1024, d=64, bf16 inputs, fp32 LSE and
accumulation): forward (O, LSE), backward preprocess, backward main kernel,
dQ cast.  Inputs are synthetic (seeded), resident in HBM before the timed
region.  The working set (~70 MB) is smaller than L2, so L2 is flushed
between timed steps, outside each step's events: a 256 MiB buffer is written
and then read back, so that each step starts with none of its data in L2 and
no dirty lines left to write back.

Prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle instead
(on a bounded sample of the same workload, on the host cores).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "causal GQA attention fwd+bwd TFLOP/s and % of GB300 bf16 tensor peak"
WORKLOAD = "gpt2s_bf16"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


DESCR = {"tiny_f32": "tiny fp32 check shape", "gpt2s_bf16": "GPT-2-small shape",
         "gpt2s_f32": "GPT-2-small shape, fp32 inputs (TF32)", "long_bf16": "long context",
         "wide_bf16": "wide head, large logits"}


def workload_config(w, extra=None):
    cfg = {"workload": f"causal GQA attention fwd+bwd, {DESCR.get(w.name, w.name)} "
                       f"B={w.B} H={w.H} Hkv={w.Hkv} N={w.N} d={w.d} {w.dtype}",
           "B": w.B, "H": w.H, "Hkv": w.Hkv, "N": w.N, "d": w.d, "causal": w.causal,
           "scale": w.scale,
           "inputs": f"seeded synthetic (seed 0): Q,K ~ N(0,{w.qk_std:g}^2), V,dO ~ "
                     f"{'U(-1,1)' if w.vdo == 'uniform' else 'N(0,1)'}",
           "l2": "flushed between timed steps (256 MiB write, then read back), outside the step events",
           "parallelism": "replicas"}
    if extra:
        cfg.update(extra)
    return cfg


def kernel_file_hash():
    """Hash of the step kernels' source code with // comments and blank lines
    left out, so that an edit of comments alone keeps the recorded counters."""
    h = hashlib.sha256()
    for f in ("bwd.cu", "fwd.cu", "ptx.cuh"):
        src = open(os.path.join(ROOT, "causal_gqa_flashattention_gb300", "csrc", f)).read()
        for line in src.splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def traffic_for(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernels have changed since the counters were taken or the counters were
    taken on another workload (traffic depends on the shape)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_hash") != kernel_file_hash() or d.get("workload_key") != workload:
        return None
    return d.get("per_launch_bytes", {}).get(kernel)


class ClockSampler:
    """Samples SM clock and clock-event (throttle) reasons while the timed
    region runs: NVML polled from a thread every ~1 ms (the region is a few
    milliseconds long), falling back to `nvidia-smi -lms 100`.  Read-only."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index):
        self.device_index = device_index
        self.samples, self.max_mhz, self.reasons = [], None, set()
        self.proc, self.thread, self.stop = None, None, False
        self.source = "none"

    def _nvml(self):
        import ctypes
        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(self.device_index)
        bus = None
        if hasattr(props, "pci_bus_id"):
            bus = "%08x:%02x:%02x.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                        getattr(props, "pci_device_id", 0))
        if bus is None or lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)):
            if lib.nvmlDeviceGetHandleByIndex_v2(self.device_index, ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
        getr = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        return lib, h, getr

    def __enter__(self):
        import ctypes
        import threading
        try:
            lib, h, getr = self._nvml()
            self.source = "nvml"

            def run():
                clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
                while not self.stop:
                    if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                        self.samples.append(float(clk.value))
                    if getr(h, ctypes.byref(rs)) == 0:
                        for bit, name in self.REASONS.items():
                            if rs.value & bit:
                                self.reasons.add(name)
                    time.sleep(0.001)
            self.thread = threading.Thread(target=run, daemon=True)
            self.thread.start()
        except Exception:
            self.source = "nvidia-smi"
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.device_index),
                     "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
                     "clocks_event_reasons.hw_thermal_slowdown,"
                     "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                     "--format=csv,noheader,nounits", "-lms", "100"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self.proc = None
        return self

    def __exit__(self, *exc):
        self.stop = True
        if self.thread is not None:
            self.thread.join(timeout=2)
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in (out or "").strip().splitlines():
                parts = [p.strip() for p in line.split(",")]
                try:
                    self.samples.append(float(parts[0]))
                    self.max_mhz = float(parts[1])
                except (ValueError, IndexError):
                    continue
                for n, v in zip(names, parts[2:6]):
                    if v.lower().startswith("active"):
                        self.reasons.add(n)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"],
                    "samples": 0, "source": self.source}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons), "samples": len(self.samples),
                "source": self.source}


def dist_setup():
    """Joins the process group when launched as one of several ranks: NCCL,
    one GPU per rank, on a GPU machine; gloo where there is no GPU (host tests)."""
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return ws, rank, local


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, n, port, target, args):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(n),
                      LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    target(args)


def spawn_local_ranks(n, target, args):
    """Runs ``target(args)`` in n local processes, one per GPU, as ranks
    0..n-1 of one job (the same environment torchrun gives each rank).
    Returns the first non-zero exit code, or 0."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, n, port, target, args)) for r in range(n)]
    for p in procs:
        p.start()
    rc = 0
    for p in procs:
        p.join()
        if p.exitcode and not rc:
            rc = p.exitcode
    return rc


def check_gpus(requested, world_size, visible):
    """How --gpus is honoured: 'run' (this process is one of the job's ranks,
    or the job has one GPU), 'spawn' (start that many local ranks), or an
    error message."""
    if requested < 1:
        return "--gpus must be at least 1"
    if world_size is not None:
        if world_size != requested:
            return f"--gpus {requested} but the launcher started {world_size} ranks"
        return "run"
    if requested == 1:
        return "run"
    if visible < requested:
        return f"--gpus {requested} but only {visible} GPU(s) are visible"
    return "spawn"


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws):
    """Largest value over the ranks (the slowest replica sets the step time).
    Uses a CUDA tensor under NCCL and a CPU tensor under gloo."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(flops_per_step, ms_step_max, ws):
    """Whole-job TFLOP/s: every replica runs one step of the workload in
    parallel, so the job does ws * flops per step, timed by the slowest rank."""
    return ws * flops_per_step / (ms_step_max * 1e-3) / 1e12


def run_cuda(args):
    import torch
    from causal_gqa_flashattention_gb300 import nea
    from causal_gqa_flashattention_gb300.workloads import WORKLOADS, make_inputs

    ws, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = WORKLOADS[args.workload]
    nea.lib()
    q, k, v, do = make_inputs(w, seed=0, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    code = nea.NEA_BF16 if w.dtype == "bf16" else nea.NEA_F32
    wsb = nea.bwd_workspace_bytes(w.B, w.H, w.Hkv, w.N, w.d, code)
    wsp = torch.empty(wsb, dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def l2_flush():
        flush.zero_()
        flush.view(torch.float32).sum()  # read-back (no copy): L2 left holding clean lines

    def step(evs=None, st=None):
        st = stream if st is None else st
        if evs:
            evs[0].record(st)
        nea.attn_fwd(q, k, v, causal=True, scale=w.scale, out=o, lse=lse, stream=st)
        nea.attn_bwd_stages(q, k, v, o, do, lse, dq, dk, dv, wsp, causal=True, scale=w.scale,
                            stream=st,
                            between=(lambda i: evs[i + 1].record(st)) if evs else None)

    for _ in range(args.warmup):
        l2_flush()
        step()
    torch.cuda.synchronize()
    if nea.check_status(stream) != nea.NEA_OK:
        raise RuntimeError("kernel status word set during warm-up")

    K = args.steps
    # The step's four kernels captured once as a CUDA graph (the same kernels
    # and arguments; replays skip the per-launch host work and the gaps
    # between dependent launches).  If capture is not possible here, the
    # step is timed as eager launches instead; config.launch says which.
    graph = None
    if not args.no_graph:
        try:
            g_ = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_):
                step(st=torch.cuda.current_stream())
            torch.cuda.synchronize()
            for _ in range(2):
                l2_flush()
                g_.replay()
            torch.cuda.synchronize()
            if nea.check_status(stream) != nea.NEA_OK:
                raise RuntimeError("status word set by a graph replay")
            graph = g_
        except Exception as exc:  # noqa: BLE001 - reported in the JSON line
            graph = None
            graph_error = f"{type(exc).__name__}: {exc}"[:200]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    gev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        for i in range(K):
            l2_flush()
            if graph is not None:
                gev[i][0].record(stream)
                graph.replay()
                gev[i][1].record(stream)
            else:
                step(evs[i])
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    barrier(ws)
    if nea.check_status(stream) != nea.NEA_OK:
        raise RuntimeError("kernel status word set during the timed region")
    # per-kernel times: from the graph-less step (events between the kernels)
    if graph is not None:
        for i in range(K):
            l2_flush()
            step(evs[i])
        torch.cuda.synchronize()
        if nea.check_status(stream) != nea.NEA_OK:
            raise RuntimeError("kernel status word set during the per-kernel timing")
    per = [[evs[i][s].elapsed_time(evs[i][s + 1]) for s in range(4)] for i in range(K)]
    # per[i] = [fwd, bwd_pre, bwd_main, bwd_post] in ms, eager launches (the
    # host work of each launch can land between the events)
    eager_ms = sum(sum(p) for p in per) / K
    # each kernel alone, captured as a CUDA graph and replayed with L2
    # flushed before each replay: device time without host-side gaps
    stage_fns = [
        lambda st: nea.attn_fwd(q, k, v, causal=True, scale=w.scale, out=o, lse=lse, stream=st),
        lambda st: nea.attn_bwd_stages(q, k, v, o, do, lse, dq, dk, dv, wsp, causal=True,
                                       scale=w.scale, stream=st, only={0}),
        lambda st: nea.attn_bwd_stages(q, k, v, o, do, lse, dq, dk, dv, wsp, causal=True,
                                       scale=w.scale, stream=st, only={1}),
        lambda st: nea.attn_bwd_stages(q, k, v, o, do, lse, dq, dk, dv, wsp, causal=True,
                                       scale=w.scale, stream=st, only={2}),
    ]
    alone = [_time_ms(fn, l2_flush, stream, K) for fn in (stage_fns if w.dtype == "bf16"
                                                           else stage_fns[:3])]
    if nea.check_status(stream) != nea.NEA_OK:
        raise RuntimeError("kernel status word set during the per-kernel timing")
    if graph is not None:
        step_ms = [gev[i][0].elapsed_time(gev[i][1]) for i in range(K)]
    else:
        step_ms = [sum(p) for p in per]
    ms_step = max_over_ranks(sum(step_ms) / K, ws)
    flops = w.fwd_flops() + w.bwd_flops()
    value = job_value(flops, ms_step, ws)
    # in-step per-kernel times (eager launches: each kernel finds in L2 what
    # the previous one left there, as inside the step) for the table and the
    # roofline; the isolated replays are reported beside them
    k_ms = [sum(p[s] for p in per) / K for s in range(4)]
    peaks, src = load_peaks()
    peak_tc = float(peaks["bf16_tflops"])
    peak_hbm = float(peaks["hbm_gbs"])

    # end to end through the public calls, with pinned host buffers: H2D of
    # q,k,v,dO, fwd, bwd, D2H of dQ,dK,dV, all inside each step's events
    hin = [t.cpu().pin_memory() for t in (q, k, v, do)]
    hout = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq, dk, dv)]
    dq2, dk2, dv2 = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
    din = [torch.empty_like(t) for t in (q, k, v, do)]
    bi = sum(t.numel() * t.element_size() for t in hin)
    bo = sum(t.numel() * t.element_size() for t in hout)

    side = torch.cuda.Stream(dev)

    def e2e_step(start=None):
        # dO is first needed by the backward: its copy runs on a side stream,
        # after the step's start event, while Q, K, V are copied and the
        # forward runs; the backward waits for it.  The backward runs as its
        # three public stages so that dK and dV can go back to the host while
        # dQ is cast; the step ends when every copy is done.  (Spreading the
        # H2D copies over more streams was slower: they share one link.)
        if start is None:  # order the side stream after the previous step's work
            start = torch.cuda.Event()
            start.record(stream)
        side.wait_event(start)
        with torch.cuda.stream(side):
            din[3].copy_(hin[3], non_blocking=True)
            do_ready = torch.cuda.Event()
            do_ready.record(side)
        with torch.cuda.stream(stream):
            for d_, h_ in zip(din[:3], hin[:3]):
                d_.copy_(h_, non_blocking=True)
            o2, l2 = nea.attn_fwd(din[0], din[1], din[2], causal=True, scale=w.scale,
                                  stream=stream)
            stream.wait_event(do_ready)

            def after_stage(i):
                # dK and dV are final once the main stage is done: they go
                # back on the side stream while the dQ cast runs
                if i == 2 and w.dtype == "bf16":
                    kv_done = torch.cuda.Event()
                    kv_done.record(stream)
                    side.wait_event(kv_done)
                    with torch.cuda.stream(side):
                        hout[1].copy_(dk2, non_blocking=True)
                        hout[2].copy_(dv2, non_blocking=True)

            nea.attn_bwd_stages(din[0], din[1], din[2], o2, din[3], l2, dq2, dk2, dv2, wsp,
                                causal=True, scale=w.scale, stream=stream, between=after_stage)
            hout[0].copy_(dq2, non_blocking=True)
            if w.dtype != "bf16":
                hout[1].copy_(dk2, non_blocking=True)
                hout[2].copy_(dv2, non_blocking=True)
            else:
                back = torch.cuda.Event()
                back.record(side)
                stream.wait_event(back)

    for _ in range(max(args.warmup, 3)):
        e2e_step()
    torch.cuda.synchronize()
    # one step alone, H2D to D2H (latency; reported beside the throughput)
    lat = []
    for _ in range(min(K, 5)):
        l2_flush()
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        e2e_step(a_)
        b_.record(stream)
        b_.synchronize()
        lat.append(a_.elapsed_time(b_))
    e_lat_ms = sum(lat) / len(lat)

    # Throughput: K steps back to back, as a training loop feeds them.  Two
    # sets of device buffers; step i's input copies (own stream) start once
    # step i-2's kernels have read that set, so they overlap step i-1's
    # kernels and output copies; step i's kernels start once its inputs have
    # landed and step i-2's outputs have gone back.  L2 is flushed on the
    # kernel stream before each step.  Every copy of every step lies between
    # the two events.
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sets = [{"din": [torch.empty_like(t) for t in (q, k, v, do)],
             "dout": [torch.empty_like(t) for t in (dq, dk, dv)],
             "hout": [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (dq, dk, dv)]}
            for _ in range(2)]

    def e2e_run(n):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        h2d.wait_event(start)
        d2h.wait_event(start)
        read_done, out_done = [None, None], [None, None]
        for i in range(n):
            S = sets[i % 2]
            with torch.cuda.stream(h2d):
                if read_done[i % 2] is not None:
                    h2d.wait_event(read_done[i % 2])
                for d_, h_ in zip(S["din"], hin):
                    d_.copy_(h_, non_blocking=True)
                in_ready = torch.cuda.Event()
                in_ready.record(h2d)
            with torch.cuda.stream(stream):
                l2_flush()
                stream.wait_event(in_ready)
                if out_done[i % 2] is not None:
                    stream.wait_event(out_done[i % 2])
                d0, d1, d2, d3 = S["din"]
                g0, g1, g2 = S["dout"]
                o3, l3 = nea.attn_fwd(d0, d1, d2, causal=True, scale=w.scale, stream=stream)

                def after_stage(j, S=S):
                    if j == 2 and w.dtype == "bf16":  # dK, dV final: back while dQ is cast
                        kv_done = torch.cuda.Event()
                        kv_done.record(stream)
                        d2h.wait_event(kv_done)
                        with torch.cuda.stream(d2h):
                            S["hout"][1].copy_(S["dout"][1], non_blocking=True)
                            S["hout"][2].copy_(S["dout"][2], non_blocking=True)

                nea.attn_bwd_stages(d0, d1, d2, o3, d3, l3, g0, g1, g2, wsp, causal=True,
                                    scale=w.scale, stream=stream, between=after_stage)
                done = torch.cuda.Event()
                done.record(stream)
                read_done[i % 2] = done
            with torch.cuda.stream(d2h):
                d2h.wait_event(done)
                S["hout"][0].copy_(g0, non_blocking=True)
                if w.dtype != "bf16":
                    S["hout"][1].copy_(g1, non_blocking=True)
                    S["hout"][2].copy_(g2, non_blocking=True)
                back = torch.cuda.Event()
                back.record(d2h)
                out_done[i % 2] = back
        stream.wait_stream(h2d)
        stream.wait_stream(d2h)
        end.record(stream)
        end.synchronize()
        return start.elapsed_time(end) / n

    e2e_run(2)
    e_ms_step = max_over_ranks(e2e_run(K), ws)
    if nea.check_status(stream) != nea.NEA_OK:
        raise RuntimeError("kernel status word set during the end-to-end run")
    # the last step's host results against a device step's (same inputs; the
    # stage-alone timing above left dQ, dK, dV stale)
    step()
    torch.cuda.synchronize()
    for h_, d_ in zip(sets[(K - 1) % 2]["hout"], (dq, dk, dv)):
        ref_ = d_.float().cpu()
        err_ = float((h_.float() - ref_).abs().max()) / max(float(ref_.abs().max()), 1e-30)
        if not err_ <= 1e-2:
            raise RuntimeError(f"end-to-end result differs from the device step: {err_}")

    main_flops = w.bwd_flops()
    main_tf = main_flops / (k_ms[2] * 1e-3) / 1e12
    rows = w.B * w.H * w.N
    # bf16: the preprocess also writes the row-term tiles (32 bytes per row)
    # and clears the fp32 dQ accumulator, which the cast reads back; fp32:
    # the dQ kernel writes dQ directly (no cast)
    acc = rows * w.d * 4 if w.dtype == "bf16" else 0
    fold = 32 * rows if w.dtype == "bf16" else 0
    pre_bytes = 2 * rows * w.d * w.esize + rows * 4 + 2 * rows * 4 + fold + acc
    post_bytes = max(acc + rows * w.d * w.esize if acc else 0, 1)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": ws,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic", "config": workload_config(w),
        "pct_of_peak": round(100.0 * value / ws / peak_tc, 2),
        "pct_of_peak_note": "of the dense bf16 tensor peak" + ("" if w.dtype == "bf16" else
                            "; fp32 inputs run on TF32 tensor cores, whose dense rate is half"),
        "roofline": {"kernel": "bwd_main", "bound": "tensor", "achieved": round(main_tf, 1),
                     "peak": peak_tc, "unit": "TFLOP/s", "frac": round(main_tf / peak_tc, 4),
                     "peak_source": f"bf16_tflops (burst) of {src}",
                     "traffic": traffic_for("bwd_main", w.name)},
        "kernels": {
            "fwd": {"ms": round(k_ms[0], 5),
                    "tflops": round(w.fwd_flops() / (k_ms[0] * 1e-3) / 1e12, 1)},
            "bwd_pre": {"ms": round(k_ms[1], 5),
                        "gbs": round(pre_bytes / (k_ms[1] * 1e-3) / 1e9, 1),
                        "hbm_frac": round(pre_bytes / (k_ms[1] * 1e-3) / 1e9 / peak_hbm, 3)},
            "bwd_main": {"ms": round(k_ms[2], 5), "tflops": round(main_tf, 1)},
            "bwd_post": {"ms": round(k_ms[3], 5),
                         "gbs": round(post_bytes / (k_ms[3] * 1e-3) / 1e9, 1)},
        },
        "e2e": {"value": round(job_value(flops, e_ms_step, ws), 2), "unit": "TFLOP/s",
                "ms_per_step": round(e_ms_step, 4), "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo,
                "how": "K steps back to back through the public calls, pinned host buffers: "
                       "each step copies q,k,v,dO in and dQ,dK,dV out; step i+1's input "
                       "copies overlap step i's kernels and output copies (two buffer sets); "
                       "L2 flushed before each step's kernels",
                "latency_ms_one_step": round(e_lat_ms, 4)},
        "gpu_launches": 4 * K,
        "launch": ("CUDA graph of the step's 4 kernels (replayed per step)" if graph is not None
                   else "eager launches" + (f" (graph capture failed: {graph_error})"
                                            if not args.no_graph else "")),
        "eager_ms_per_step": round(eager_ms, 5),
        "kernel_timing": "kernels: CUDA events between the step's kernels launched eagerly "
                         "(each finds in L2 what the previous one left); kernels_alone_ms: "
                         "each kernel alone as a CUDA graph replay, L2 flushed before each",
        "kernels_alone_ms": {n: round(t, 5) for n, t in zip(("fwd", "bwd_pre", "bwd_main",
                                                             "bwd_post"), alone)},
        "clocks": clk.summary(),
        "wall_s_timed_region": round(wall, 4),
    }
    if not args.no_extras and w.dtype == "bf16":
        line["extras"] = measure_extras(nea, w, q, k, v, do, o, lse, wsp, l2_flush, stream,
                                        peak_hbm, src, reps=max(10, min(K, 50)))
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, seconds=args.cpu_seconds)
    if w.dtype != "bf16":
        del line["kernels"]["bwd_post"]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def _time_ms(fn, l2_flush, stream, reps):
    """Mean device time of fn(st) over reps calls, L2 flushed before each.
    The call is captured once as a CUDA graph and replayed, so that host-side
    launch work does not land inside the events (eager launches if capture
    fails)."""
    import torch
    fn(stream)  # one eager call first (a library's lazily created resources exist before capture)
    torch.cuda.synchronize()
    g = None
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn(torch.cuda.current_stream())
        torch.cuda.synchronize()
    except Exception:  # noqa: BLE001 - eager timing below
        g = None

    def run():
        if g is not None:
            g.replay()
        else:
            fn(stream)
    for _ in range(3):
        l2_flush()
        run()
    ts = []
    for _ in range(reps):
        l2_flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        run()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return sum(ts) / len(ts)


def measure_extras(nea, w, q, k, v, do, o, lse, wsp, l2_flush, stream, peak_hbm, src, reps):
    """The rows beyond the training step: RoPE (rotation pass and the cost of
    the inverse rotation fused into the backward) on this workload, the
    deterministic backward, full attention, the fp32 (TF32) path, and decode
    attention on the decode workloads.  Each is timed alone with CUDA events,
    L2 flushed before every call."""
    import torch
    from causal_gqa_flashattention_gb300.workloads import DECODE_WORKLOADS, make_decode_inputs
    out = {}
    cs = nea.rope_table(w.N, w.d, device=q.device)
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    t_rot = _time_ms(lambda st: nea.rope_qk(q, k, cs, qr=qr, kr=kr, stream=st), l2_flush,
                     stream, reps)
    rot_bytes = 2 * (q.numel() + k.numel()) * q.element_size() + cs.numel() * 4
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    t_b = _time_ms(lambda st: nea.attn_bwd(qr, kr, v, o, do, lse, dq=dq, dk=dk, dv=dv,
                                           workspace=wsp, stream=st), l2_flush, stream, reps)
    t_br = _time_ms(lambda st: nea.attn_bwd(qr, kr, v, o, do, lse, dq=dq, dk=dk, dv=dv,
                                            workspace=wsp, stream=st, rope_cs=cs),
                    l2_flush, stream, reps)
    t_det = _time_ms(lambda st: nea.attn_bwd(qr, kr, v, o, do, lse, dq=dq, dk=dk, dv=dv,
                                             workspace=wsp, stream=st, deterministic=True),
                     l2_flush, stream, reps)
    out["bwd_deterministic"] = {"ms": round(t_det, 5), "ms_default": round(t_b, 5),
                                "tflops": round(w.bwd_flops() / (t_det * 1e-3) / 1e12, 1),
                                "note": "dQ by one CTA per query tile (S and dP recomputed); "
                                        "tflops counts the default path's 5 GEMMs"}
    out["rope_qk"] = {"ms": round(t_rot, 5), "bytes": rot_bytes,
                      "gbs": round(rot_bytes / (t_rot * 1e-3) / 1e9, 1),
                      "hbm_frac": round(rot_bytes / (t_rot * 1e-3) / 1e9 / peak_hbm, 3),
                      "peak_source": f"hbm_gbs of {src}"}
    out["bwd_rope"] = {"ms": round(t_br, 5), "ms_without_rope": round(t_b, 5),
                       "overhead_pct": round(100.0 * (t_br / t_b - 1.0), 2)}
    # Q rotated inside the forward (K by the pass) against the forward on
    # pre-rotated inputs; the pass's Q share is its time times Q's byte share
    of2, lf2 = torch.empty_like(o), torch.empty_like(lse)
    t_fp = _time_ms(lambda st: nea.attn_fwd(qr, kr, v, out=of2, lse=lf2, stream=st), l2_flush,
                    stream, reps)
    t_fq = _time_ms(lambda st: nea.attn_fwd(q, kr, v, out=of2, lse=lf2, stream=st,
                                            rope_q_cs=cs), l2_flush, stream, reps)
    out["fwd_rope_q"] = {"ms": round(t_fq, 5), "ms_pre_rotated": round(t_fp, 5),
                         "overhead_ms": round(t_fq - t_fp, 5),
                         "pass_q_share_ms": round(t_rot * q.numel() / (q.numel() + k.numel()), 5),
                         "note": "forward rotating Q in shared memory vs the forward on Qr; "
                                 "the rotation pass's time for Q alone is its Q byte share"}
    # full (non-causal) attention at the same shape: twice the causal work
    of, lf = torch.empty_like(o), torch.empty_like(lse)
    t_ff = _time_ms(lambda st: nea.attn_fwd(q, k, v, causal=False, out=of, lse=lf, stream=st),
                    l2_flush, stream, reps)
    t_fb = _time_ms(lambda st: nea.attn_bwd(q, k, v, of, do, lf, causal=False, dq=dq, dk=dk,
                                            dv=dv, workspace=wsp, stream=st),
                    l2_flush, stream, reps)
    full_flops = 2.0 * (w.fwd_flops() + w.bwd_flops())
    out["full_attention"] = {"fwd_ms": round(t_ff, 5), "bwd_ms": round(t_fb, 5),
                             "tflops": round(full_flops / ((t_ff + t_fb) * 1e-3) / 1e12, 1),
                             "frac_of_peak": round(full_flops / ((t_ff + t_fb) * 1e-3) / 1e12 /
                                                   float(load_peaks()[0]["bf16_tflops"]), 4)}
    # the fp32 path (TF32 tensor cores) at the GPT-2-small shape: forward and
    # backward, each timed alone; against the TF32 dense peak, taken as the
    # measured bf16 peak times the nominal TF32 / bf16 ratio (1.1 / 2.25)
    from causal_gqa_flashattention_gb300.workloads import WORKLOADS, make_inputs
    wf = WORKLOADS["gpt2s_f32"]
    qf, kf, vf, dof = make_inputs(wf, seed=0, device=q.device)
    of_, lf_ = torch.empty_like(qf), torch.empty((wf.B, wf.H, wf.N), dtype=torch.float32,
                                                   device=q.device)
    dqf, dkf, dvf = torch.empty_like(qf), torch.empty_like(kf), torch.empty_like(vf)
    wsf = torch.empty(nea.bwd_workspace_bytes(wf.B, wf.H, wf.Hkv, wf.N, wf.d, nea.NEA_F32),
                      dtype=torch.uint8, device=q.device)
    t_f32f = _time_ms(lambda st: nea.attn_fwd(qf, kf, vf, causal=True, scale=wf.scale, out=of_,
                                              lse=lf_, stream=st), l2_flush, stream, reps)
    t_f32b = _time_ms(lambda st: nea.attn_bwd(qf, kf, vf, of_, dof, lf_, causal=True,
                                              scale=wf.scale, dq=dqf, dk=dkf, dv=dvf,
                                              workspace=wsf, stream=st), l2_flush, stream, reps)
    peak_tf32 = float(load_peaks()[0]["bf16_tflops"]) * 1.1 / 2.25
    tf_f = wf.fwd_flops() / (t_f32f * 1e-3) / 1e12
    tf_b = wf.bwd_flops() / (t_f32b * 1e-3) / 1e12
    tf_s = (wf.fwd_flops() + wf.bwd_flops()) / ((t_f32f + t_f32b) * 1e-3) / 1e12
    out["fp32_tf32_gpt2s"] = {
        "fwd_ms": round(t_f32f, 5), "bwd_ms": round(t_f32b, 5),
        "fwd_tflops": round(tf_f, 1), "bwd_tflops": round(tf_b, 1), "tflops": round(tf_s, 1),
        "roofline": {"bound": "tensor", "peak": round(peak_tf32, 1), "unit": "TFLOP/s",
                     "frac": round(tf_s / peak_tf32, 4),
                     "peak_source": f"bf16_tflops of {src} x 1.1 / 2.25 (nominal TF32/bf16)"},
        "config": workload_config(wf)}
    for name, dw in DECODE_WORKLOADS.items():
        dq_, kc, vc, lens = make_decode_inputs(dw, seed=0, device=q.device)
        od = torch.empty_like(dq_)
        ld = torch.empty((dw.B, dw.H, dw.nq), dtype=torch.float32, device=q.device)
        wsd = torch.empty(max(nea.decode_workspace_bytes(dw.B, dw.H, dw.Hkv, dw.nq, dw.Lmax,
                                                          dw.d), 1),
                          dtype=torch.uint8, device=q.device)
        t = _time_ms(lambda st: nea.attn_decode(dq_, kc, vc, lens, out=od, lse=ld,
                                                workspace=wsd, stream=st), l2_flush, stream, reps)
        byt = dw.cache_bytes() + 2 * dq_.numel() * dq_.element_size() + ld.numel() * 4
        out[name] = {"ms": round(t, 5), "bytes": byt,
                     "gbs": round(byt / (t * 1e-3) / 1e9, 1),
                     "hbm_frac": round(byt / (t * 1e-3) / 1e9 / peak_hbm, 3),
                     "config": {"B": dw.B, "H": dw.H, "Hkv": dw.Hkv, "nq": dw.nq,
                                "Lmax": dw.Lmax, "d": dw.d, "dtype": dw.dtype},
                     "peak_source": f"hbm_gbs of {src}",
                     "launches": 1 if -(-dw.Lmax // 128) <= 16 else 2}
    return out


def oracle_sample(w, nb):
    """A bounded sample of the workload: the first `nb` batch elements."""
    from causal_gqa_flashattention_gb300.workloads import make_inputs
    q, k, v, do = make_inputs(w, seed=0)
    return q[:nb], k[:nb], v[:nb], do[:nb]


def cpu_baseline(w, seconds=10.0, nb=1):
    import oracle
    q, k, v, do = oracle_sample(w, nb)
    flops = (w.fwd_flops() + w.bwd_flops()) * nb / w.B
    runs = 0
    t0 = time.perf_counter()
    while True:
        oracle.attn_fwd(q, k, v, w.scale, True)
        oracle.attn_bwd(q, k, v, do, w.scale, True)
        runs += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = (time.perf_counter() - t0) / runs
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s",
            "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"batch element(s) 0..{nb - 1} of {w.B} (B={nb}, H={w.H}, Hkv={w.Hkv}, "
                      f"N={w.N}, d={w.d}), fwd+bwd in fp64, {runs} run(s), "
                      f"{dt:.2f} s per run; causal FLOPs counted as on the GPU"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from causal_gqa_flashattention_gb300.workloads import WORKLOADS
    import oracle
    w = WORKLOADS[args.workload]
    nb = 1
    q, k, v, do = oracle_sample(w, nb)
    flops = (w.fwd_flops() + w.bwd_flops()) * nb / w.B
    for _ in range(args.warmup):
        oracle.attn_fwd(q[:, :, :128], k[:, :, :128], v[:, :, :128], w.scale, True)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.attn_fwd(q, k, v, w.scale, True)
        oracle.attn_bwd(q, k, v, do, w.scale, True)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = flops / (ms * 1e-3) / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, {"sample": f"batch element 0 of {w.B} per step"}),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "kind": "oracle",
                             "cores": oracle.num_threads(),
                             "sample": f"B=1 of the B={w.B} workload per step, fp64 oracle"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the step as eager launches instead of a CUDA graph replay")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the RoPE and decode measurements")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(
        ["tiny_f32", "gpt2s_bf16", "gpt2s_f32", "long_bf16", "wide_bf16"]),
        help="default: the GPT-2-small bf16 shape, the headline measurement")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "cuda":
        args.warmup = 3
    ws_env = os.environ.get("WORLD_SIZE")
    if args.impl == "reference":
        # the oracle runs on the host cores of rank 0 only, whatever N is
        run_reference(args)
        return
    import torch
    how = check_gpus(args.gpus, int(ws_env) if ws_env else None,
                     torch.cuda.device_count() if torch.cuda.is_available() else 0)
    if how == "spawn":
        sys.exit(spawn_local_ranks(args.gpus, run_cuda, args))
    if how != "run":
        sys.exit(f"bench.py: {how}")
    run_cuda(args)


if __name__ == "__main__":
    main()
