"""Benchmark of the blr layer's forward+backward step on GB300.

One step = blr_forward + blr_backward over one batch of synthetic tokens (every
kernel of the hot path). Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload small]
  python bench.py --impl reference ...     # the CPU f64 oracle as the reference arm

Timing: W untimed warm-up steps, then K timed steps between a barrier and
cudaDeviceSynchronize on both sides, measured with CUDA events on the launch
stream; max over ranks. L2 (129 MB) is defeated by rotating independent
input/output/workspace sets whose total exceeds twice the L2 size. Kernel-level
durations for the roofline come from the library's event trace over an eager
pass of the same K steps. Steps are timed as CUDA-graph replays (one graph
per buffer set, captured from the same library calls), so host launch cost is
not in the device time; the end-to-end number keeps every host call. Multi-GPU: every rank runs its own batch
(weak scaling); the path needs no collective inside a step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "blr fwd+bwd tokens/sec and TFLOP/s (% of GB300 f16 tensor peak / % HBM BW)"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def kernel_source_hash() -> str:
    """sha256 over the CUDA sources and the C header (what a kernel's DRAM
    traffic depends on), so that stored ncu counters can be matched to them."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "binary_rank_linear_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    with open(os.path.join(ROOT, "include", "blr.h"), "rb") as fh:
        h.update(fh.read())
    return h.hexdigest()


def stored_traffic(workload: str, kernel: str):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of
    `kernel` on `workload` from the committed ncu summary profiles/traffic.json,
    or None when there is none or the kernels changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_sha256") != kernel_source_hash():
        return None
    v = d.get("bytes_per_launch", {}).get(workload, {}).get(kernel)
    return float(v) if v is not None else None


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------- per-kernel work ----
def kernel_work(name: str, M: int, d_in: int, d_out: int, r: int):
    """Algorithmic (flops, bytes) of one launch of a kernel of the step.

    Bytes count each tensor the kernel must read or write once (f32 = 4 B,
    staged f16 = 2 B, bitmaps d*r/8 B); FLOP counts 2 per multiply-add of the
    sign products.
    """
    bits_u = d_out * r / 8
    bits_v = d_in * r / 8
    if name == "fwd_prologue":
        return 0.0, 4.0 * M * d_in + 2.0 * M * d_in + 2 * (bits_u + bits_v)
    if name == "gemm_fwd1":
        return 2.0 * M * r * d_in, 2.0 * M * d_in + bits_v + 4.0 * M * r + 2.0 * M * r
    if name == "gemm_fwd2":
        return 2.0 * M * r * d_out, 2.0 * M * r + bits_u + 4.0 * M * d_out + 2.0 * M * d_out
    if name == "bwd_prologue":
        return 0.0, 4.0 * M * d_out + 2.0 * M * d_out + 2.0 * M * d_out + 2 * (bits_u + bits_v)
    if name == "gemm_bwd1":
        return 2.0 * M * r * d_out, 2.0 * M * d_out + bits_u + 4.0 * M * r + 2.0 * M * r
    if name == "gemm_bwd2":
        return 2.0 * M * r * d_in, 2.0 * M * r + bits_v + 4.0 * M * d_in + 4.0 * M * d_in
    if name == "reduce_partials":
        return 0.0, 4.0 * (d_in + d_out + r) * 2
    if name == "small_fwd":  # fused forward of the small-M path
        parts = [kernel_work(n, M, d_in, d_out, r) for n in ("fwd_prologue", "gemm_fwd1", "gemm_fwd2")]
        return sum(p[0] for p in parts), 4.0 * M * d_in + 4.0 * M * r + 2.0 * M * r + 6.0 * M * d_out + bits_u + bits_v
    if name == "small_bwd":  # fused backward of the small-M path
        parts = [kernel_work(n, M, d_in, d_out, r) for n in ("gemm_bwd1", "gemm_bwd2")]
        return (sum(p[0] for p in parts),
                4.0 * M * d_out + 2.0 * M * d_out + 4.0 * M * r + 2.0 * M * r + 8.0 * M * d_in + bits_u + bits_v)
    return 0.0, 0.0


# --------------------------------------------------------------- clocks -----
class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
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
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------ rank aggregation ---
def max_over_ranks(v: float, device="cpu") -> float:
    """The largest of every rank's `v` (the job's time is its slowest rank's);
    `v` itself when no process group is up."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return float(v)
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank_step: int, steps: int, ms: float) -> float:
    """Whole-job throughput: every rank processes its own batch each step
    (weak scaling), over the slowest rank's time."""
    return world * tokens_per_rank_step * steps / (ms * 1e-3)


def workload_of(args):
    """The named workload, at --tokens tokens when given."""
    from binary_rank_linear_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    return w.with_shape(M=args.tokens) if args.tokens else w


# ---------------------------------------------------------- CPU oracle ------
def cpu_oracle_rate(w, budget_s: float = 12.0, max_reps: int = 1_000_000):
    """tokens/s of the CPU f64 oracle (as it stands) on the workload's batch,
    repeated until ``budget_s`` seconds of CPU work have run. For workloads
    whose batch would exceed the budget, a prefix of the tokens is used."""
    import oracle
    from binary_rank_linear_gb300 import workloads as wl

    sample_M = w.M
    # keep one oracle pass in the seconds range: ~4 f64 GEMMs of 2*M*r*d each
    per_token = 4.0 * w.r * (w.d_in + w.d_out)
    while sample_M > 64 and per_token * sample_M > 3e11:
        sample_M //= 2
    t = wl.make_inputs(w.with_shape(M=sample_M))
    bu, bv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.forward(t["x"], bu, bv, t["g"], t["l"], t["h"])
        oracle.backward(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"])
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= max_reps:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    threads = int(os.environ.get("OPENBLAS_NUM_THREADS", os.environ.get("OMP_NUM_THREADS", cores)))
    return {
        "value": reps * sample_M / el,
        "unit": "tokens/s",
        "cores": min(cores, threads),
        "kind": "oracle",
        "sample": f"{reps} x (forward+backward of {sample_M} tokens of {w.name}) in {el:.1f} s, numpy f64",
    }


# ------------------------------------------------------------ GPU arm -------
def run_gpu(args, rank, world, local_rank):
    import torch

    import binary_rank_linear_gb300 as blr
    from binary_rank_linear_gb300 import workloads as wl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = workload_of(args)
    M, d_in, d_out, r = w.M, w.d_in, w.d_out, w.r
    t = wl.make_inputs(w)

    def d(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    g, l, h = d(t["g"]), d(t["l"]), d(t["h"])
    bu, bv = blr.pack_signs(d(t["su"])), blr.pack_signs(d(t["sv"]))
    x0, dy0 = d(t["x"]), d(t["dy"])
    ws_bytes = blr.workspace_bytes(M, d_in, d_out, r)
    set_bytes = 4 * M * (2 * d_in + 2 * d_out) + ws_bytes
    nsets = max(1, min(64, -(-2 * L2_BYTES // set_bytes) + 1))
    sets = []
    for _ in range(nsets):
        sets.append({
            "x": x0.clone(), "dy": dy0.clone(),
            "y": torch.empty(M, d_out, device=dev), "dx": torch.empty(M, d_in, device=dev),
            "ws": torch.empty(ws_bytes, dtype=torch.uint8, device=dev),
        })
    dg = torch.zeros(d_in, device=dev)
    dl = torch.zeros(r, device=dev)
    dh = torch.zeros(d_out, device=dev)
    stream = torch.cuda.current_stream()

    def step(i):
        s = sets[i % nsets]
        blr.forward(s["x"], bu, bv, g, l, h, s["y"], s["ws"])
        blr.backward(s["x"], s["dy"], bu, bv, g, l, h, s["dx"], dg, dl, dh, s["ws"])

    dist = world > 1
    if dist:
        import torch.distributed as tdist

    def barrier():
        if dist:
            tdist.barrier()
        torch.cuda.synchronize()

    for i in range(max(args.warmup, nsets)):
        step(i)
    status = blr.check_status(sets[0]["ws"])
    if status:
        raise RuntimeError(f"device status {status:#x} after warm-up")

    # one CUDA graph per buffer set: a step is replayed with no host launch cost
    graphs = []
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        for i in range(nsets):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=cap):
                step(i)
            graphs.append(gr)
    stream.wait_stream(cap)
    for i in range(args.warmup):
        graphs[i % nsets].replay()

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        graphs[i % nsets].replay()
    e1.record(stream)
    barrier()
    ms = e0.elapsed_time(e1)
    # kernel-level durations: an eager pass of the same steps with the library's
    # event trace, queued behind a GPU sleep so that host launch gaps do not
    # land inside any kernel's bracket
    t0 = time.perf_counter()
    step(0)
    host_step_s = time.perf_counter() - t0
    barrier()
    blr.trace_begin(capacity=16 * args.steps)
    torch.cuda._sleep(int(min(4e9, 2.5e9 * host_step_s * (args.steps + 2))))
    for i in range(args.steps):
        step(i)
    barrier()
    trace = blr.trace_end()
    clk = clocks.stop()
    for s in sets:
        st = blr.check_status(s["ws"])
        if st:
            raise RuntimeError(f"device status {st:#x}")

    ms = max_over_ranks(ms, dev)

    per = {}
    for name, kms in trace:
        per.setdefault(name, []).append(kms)
    launches_per_step = len(trace) / max(1, args.steps)
    peaks, peak_src = _peaks()
    tc_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    kernels = {}
    for name, lst in per.items():
        avg = sum(lst) / len(lst)
        fl, by = kernel_work(name, M, d_in, d_out, r)
        kernels[name] = {"avg_us": avg * 1e3, "share": sum(lst) / sum(sum(v) for v in per.values()),
                         "tflops": fl / (avg * 1e-3) / 1e12, "gbs": by / (avg * 1e-3) / 1e9}
    dom = max(per, key=lambda n: sum(per[n]))
    fl, by = kernel_work(dom, M, d_in, d_out, r)
    avg_s = kernels[dom]["avg_us"] * 1e-6
    t_tc, t_hbm = fl / (tc_peak * 1e12), by / (hbm_peak * 1e9)
    if t_tc >= t_hbm:
        roof = {"bound": "tensor", "achieved": fl / avg_s / 1e12, "peak": tc_peak, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": by / avg_s / 1e9, "peak": hbm_peak, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = dom
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json: bf16 burst, f16 assumed equal)" \
        if peak_src == "measured" else "fallback"
    # stored counters are for the workloads' own token counts
    roof["traffic"] = stored_traffic(args.workload, dom) if not args.tokens else None

    sign = measure_sign_grads(blr, sets, g, l, args.steps, tc_peak, M, d_in, d_out, r, dev) \
        if not args.no_sign else None
    adam = measure_adam(blr, torch.cat([dg, dl, dh]), args.steps, hbm_peak, dev)
    plane = measure_plane(blr, sets[0], args.steps, tc_peak, M, d_in, d_out, dev) if not args.no_plane else None
    paths = measure_paths(blr, sets[0], bu, bv, g, l, h, args.steps, tc_peak, w, dev) if not args.no_paths else None

    # end-to-end: host buffers through the public API, copies inside the timed
    # region. With a megabyte or more to move per step, steps are pipelined over
    # two device buffer sets on three streams (host->device copies, the layer,
    # device->host copies), as a training loop's data path would be: step i+1's
    # inputs go up and step i-1's results come down while step i computes.
    # Smaller steps run in order on one stream (there the host's launch work,
    # not the copies, sets the pace, and the extra streams only add to it).
    # Every step moves its own inputs and results either way.
    xh = torch.from_numpy(t["x"]).pin_memory()
    dyh = torch.from_numpy(t["dy"]).pin_memory()
    pipelined = 4 * M * (d_in + d_out) >= (1 << 20)
    npipe = 2
    pipe = []
    for b in range(npipe):
        pipe.append({
            "set": sets[b % len(sets)],
            "yh": torch.empty(M, d_out).pin_memory(),
            "dxh": torch.empty(M, d_in).pin_memory(),
            "gh": torch.empty(d_in + r + d_out).pin_memory(),
            "dg": torch.zeros(d_in, device=dev), "dl": torch.zeros(r, device=dev), "dh": torch.zeros(d_out, device=dev),
            "up": torch.cuda.Event(), "done": torch.cuda.Event(), "down": torch.cuda.Event(),
        })
    if pipelined:
        s_up, s_comp, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    else:
        s_up = s_comp = s_down = torch.cuda.current_stream(dev)
    for b in pipe:
        b["down"].record(s_down)  # nothing to wait for yet

    def e2e_step_in_order(i):
        b = pipe[0]
        s0 = b["set"]
        s0["x"].copy_(xh, non_blocking=True)
        s0["dy"].copy_(dyh, non_blocking=True)
        blr.forward(s0["x"], bu, bv, g, l, h, s0["y"], s0["ws"])
        blr.backward(s0["x"], s0["dy"], bu, bv, g, l, h, s0["dx"], b["dg"], b["dl"], b["dh"], s0["ws"])
        b["yh"].copy_(s0["y"], non_blocking=True)
        b["dxh"].copy_(s0["dx"], non_blocking=True)
        b["gh"][:d_in].copy_(b["dg"], non_blocking=True)
        b["gh"][d_in:d_in + r].copy_(b["dl"], non_blocking=True)
        b["gh"][d_in + r:].copy_(b["dh"], non_blocking=True)

    def e2e_step(i):
        if not pipelined:
            e2e_step_in_order(i)
            return
        b = pipe[i % npipe]
        s0 = b["set"]
        # the set's previous results are down (its y/dx and inputs are free again)
        s_up.wait_event(b["down"])
        with torch.cuda.stream(s_up):
            s0["x"].copy_(xh, non_blocking=True)
            s0["dy"].copy_(dyh, non_blocking=True)
        b["up"].record(s_up)
        s_comp.wait_event(b["up"])
        with torch.cuda.stream(s_comp):
            blr.forward(s0["x"], bu, bv, g, l, h, s0["y"], s0["ws"])
            blr.backward(s0["x"], s0["dy"], bu, bv, g, l, h, s0["dx"], b["dg"], b["dl"], b["dh"], s0["ws"])
        b["done"].record(s_comp)
        s_down.wait_event(b["done"])
        with torch.cuda.stream(s_down):
            b["yh"].copy_(s0["y"], non_blocking=True)
            b["dxh"].copy_(s0["dx"], non_blocking=True)
            b["gh"][:d_in].copy_(b["dg"], non_blocking=True)
            b["gh"][d_in:d_in + r].copy_(b["dl"], non_blocking=True)
            b["gh"][d_in + r:].copy_(b["dh"], non_blocking=True)
        b["down"].record(s_down)

    for i in range(max(npipe, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(s_up)
    for i in range(args.steps):
        e2e_step(i)
    s_up.wait_stream(s_down)
    f1.record(s_up)
    torch.cuda.synchronize(dev)
    barrier()
    e2e_ms = f0.elapsed_time(f1)
    e2e_ms = max_over_ranks(e2e_ms, dev)
    for b in pipe:
        st = blr.check_status(b["set"]["ws"])
        if st:
            raise RuntimeError(f"end-to-end pass: device status {st:#x}")

    value = job_tokens_per_s(world, M, args.steps, ms)
    result = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic",
        "config": {
            "workload": f"{w.name}: {w.note}" + (f" (token count set to {M})" if args.tokens else ""),
            "M": M, "d_in": d_in, "d_out": d_out, "r": r,
            "mode": "overwrite y/dx, dynamic per-token gradient scale",
            "small_path": args.small_path,
            "l2": f"{nsets} rotating input/output/workspace sets ({nsets * set_bytes / 2**20:.0f} MiB > 2x L2)",
        },
        "tflops": world * w.flops * args.steps / (ms * 1e-3) / 1e12,
        "tensor_frac": (world * w.flops * args.steps / (ms * 1e-3) / 1e12) / tc_peak,
        "hbm_frac": (w.canonical_bytes * args.steps / (ms * 1e-3) / 1e9) / hbm_peak,
        "roofline": roof,
        "kernels": kernels,
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "clocks": clk,
        "e2e": {"value": job_tokens_per_s(world, M, args.steps, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": 4 * M * (d_in + d_out),
                "d2h_bytes_per_step": 4 * (M * (d_in + d_out) + d_in + r + d_out),
                "copies": "overlapped with the layer on their own streams" if pipelined else "in order on one stream"},
    }
    if sign is not None:
        result["sign_grads"] = sign
    result["adam"] = adam
    if plane is not None:
        result["plane_linear"] = plane
    if paths is not None:
        paths["vs_one_path"] = paths["us_per_step"] / (ms / args.steps * 1e3)
        result["paths"] = paths
    return result


def measure_paths(blr, s, bu, bv, g, l, h, steps, tc_peak, w, dev):
    """A two-path layer (blr_forward_paths + blr_backward_paths) on the
    workload's shape: path 0 with the step's bitmaps, path 1 with random ones;
    its own calls after the step."""
    import torch
    M, d_in, d_out, r = w.M, w.d_in, w.d_out, w.r
    gen = torch.Generator(device=dev).manual_seed(9)
    rb = lambda rows: torch.randint(-2**31, 2**31 - 1, (rows, (r + 31) // 32), dtype=torch.int32, device=dev,  # noqa: E731
                                    generator=gen)
    paths = [{"bu": bu, "bv": bv, "g": g, "l": l, "h": h},
             {"bu": rb(d_out), "bv": rb(d_in), "g": g, "l": l, "h": h}]
    grads = [{"dg": torch.zeros(d_in, device=dev), "dl": torch.zeros(r, device=dev),
              "dh": torch.zeros(d_out, device=dev)} for _ in paths]
    ws = blr.alloc_paths_workspace(2, M, d_in, d_out, r, device=dev)

    def call(i):
        blr.forward_paths(s["x"], paths, s["y"], ws)
        blr.backward_paths(s["x"], s["dy"], paths, s["dx"], grads, ws)

    for i in range(3):
        call(i)
    ms = time_queued(call, steps)
    flops = 2 * w.flops
    return {"what": "two-path layer forward+backward (blr_forward_paths, blr_backward_paths), its own calls",
            "P": 2, "us_per_step": ms * 1e3, "tokens_per_s": M / (ms * 1e-3),
            "tflops": flops / (ms * 1e-3) / 1e12, "tensor_frac": flops / (ms * 1e-3) / 1e12 / tc_peak}


def measure_plane(blr, s, steps, tc_peak, M, d_in, d_out, dev):
    """plane_linear (blr_plane_linear) on the workload's shape as a dense
    frozen f16 linear: y = x P^T with P [d_out][d_in], and its transpose
    dx = dy P; calls of their own after the step (they reuse the step's x, y,
    dy, dx buffers)."""
    import torch
    gen = torch.Generator(device=dev).manual_seed(5)
    P = (torch.randn(d_out, d_in, device=dev, generator=gen) * 0.02).half()
    ws = blr.alloc_plane_workspace(M, d_out, d_in, device=dev)
    flops = 2.0 * M * d_in * d_out
    out = {"what": "dense frozen f16 linear on the workload's shape (not in the step's time)"}
    for name, x, y, tr in (("forward", s["x"], s["y"], False), ("transpose", s["dy"], s["dx"], True)):
        def call(i, x=x, y=y, tr=tr):
            blr.plane_linear(x, P, y, ws, transpose=tr)
        for i in range(3):
            call(i)
        blr.trace_begin(capacity=4 * steps)
        ms = time_queued(call, steps)
        per = {}
        for kname, kms in blr.trace_end():
            per.setdefault(kname, []).append(kms)
        gem = per.get("plane_gemm", [float("nan")])
        g_ms = sum(gem) / len(gem)
        out[name] = {"us_per_call": ms * 1e3, "tflops": flops / (ms * 1e-3) / 1e12,
                     "kernels": {k: {"avg_us": 1e3 * sum(v) / len(v)} for k, v in per.items()},
                     "roofline": {"bound": "tensor", "kernel": "plane_gemm",
                                  "achieved": flops / (g_ms * 1e-3) / 1e12, "peak": tc_peak, "unit": "TFLOP/s",
                                  "frac": flops / (g_ms * 1e-3) / 1e12 / tc_peak}}
    return out


def measure_adam(blr, grad, steps, hbm_peak, dev):
    """One Adam step (blr_adam) over the layer's vectors g | l | h as one
    contiguous array, with this step's dg | dl | dh as the gradient; a call of
    its own after the step."""
    import torch
    n = grad.numel()
    w = torch.ones(n, device=dev)
    m1 = torch.zeros(n, device=dev)
    m2 = torch.zeros(n, device=dev)
    for i in range(3):
        blr.adam(w, grad, m1, m2, step=i + 1, lr=1e-4)
    us = 1e3 * time_queued(lambda i: blr.adam(w, grad, m1, m2, step=i + 4, lr=1e-4), steps)
    by = 28.0 * n  # w, grad, m1, m2 read; w, m1, m2 written (f32)
    return {"what": "Adam step of g | l | h (d_in + r + d_out parameters) after the step (not in its time)",
            "n": n, "us_per_call": us,
            "roofline": {"bound": "hbm", "achieved": by / (us * 1e-6) / 1e9, "peak": hbm_peak, "unit": "GB/s",
                         "frac": by / (us * 1e-6) / 1e9 / hbm_peak},
            "note": "a few hundred KB per call: bound by launch and latency, not bandwidth"}


def time_queued(fn, steps):
    """Device milliseconds per call of `fn` (which queues GPU work on the
    current stream): all calls are queued behind a GPU sleep that outlasts
    their host-side launch cost, then bracketed by two CUDA events, so host
    launch latency stays outside the measurement."""
    import torch
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    fn(0)
    torch.cuda.synchronize()
    host_s = time.perf_counter() - t0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(int(min(4e9, 2.5e9 * host_s * (steps + 2))))
    e0.record(stream)
    for i in range(steps):
        fn(i + 1)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def measure_sign_grads(blr, sets, g, l, steps, tc_peak, M, d_in, d_out, r, dev):
    """The sign gradients G_U, G_V (blr_sign_grads) after the step: a call of
    their own, outside the step's time. Each call reads the tape of one of the
    rotating buffer sets (every set holds a forward+backward by now)."""
    import torch
    sws = blr.alloc_sign_workspace(M, d_in, d_out, r, device=dev)
    gu = torch.empty(d_out, r, device=dev)
    gv = torch.empty(d_in, r, device=dev)
    n = len(sets)

    def call(i):
        s = sets[i % n]
        blr.sign_grads(s["x"], g, l, gu, gv, s["ws"], sws)

    for i in range(max(3, n)):
        call(i)
    ms = time_queued(call, steps)
    blr.trace_begin(capacity=4 * steps)
    time_queued(call, steps)  # the trace brackets each kernel of the queued calls
    per = {}
    for name, kms in blr.trace_end():
        per.setdefault(name, []).append(kms)
    flops = 2.0 * M * r * (d_in + d_out)
    gem = per.get("sign_gemm", [float("nan")])
    g_ms = sum(gem) / len(gem)
    return {
        "what": "G_U = diag(h) dy^T a diag(l), G_V = diag(g) x^T db diag(l) after the step (not in its time)",
        "us_per_call": ms * 1e3,
        "tflops": flops / (ms * 1e-3) / 1e12,
        "kernels": {k: {"avg_us": 1e3 * sum(v) / len(v)} for k, v in per.items()},
        "roofline": {"bound": "tensor", "kernel": "sign_gemm", "achieved": flops / (g_ms * 1e-3) / 1e12,
                     "peak": tc_peak, "unit": "TFLOP/s", "frac": flops / (g_ms * 1e-3) / 1e12 / tc_peak},
        "gpu_launches_per_call": len(sum(per.values(), [])) / (steps + 1),
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="blr", choices=["blr", "reference"])
    ap.add_argument("--workload", default="small")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sign", action="store_true", help="skip the sign-gradient measurement")
    ap.add_argument("--no-plane", action="store_true", help="skip the plane_linear measurement")
    ap.add_argument("--no-paths", action="store_true", help="skip the two-path layer measurement")
    ap.add_argument("--tokens", type=int, default=0,
                    help="run the workload's shapes and distributions at this token count (a smaller case to "
                         "profile); the bench line then is not the workload's")
    ap.add_argument("--small-path", default="general", choices=["general", "fused"],
                    help="kernels for small problems: stand-alone (default) or the fused cooperative pair")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.small_path == "fused":
        os.environ["BLR_SMALL_PATH"] = "fused"  # read by the library at each call

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    from binary_rank_linear_gb300 import workloads as wl

    w = workload_of(args)

    if args.impl == "reference":
        if rank != 0:
            return
        budget = 10.0
        t0 = time.perf_counter()
        for _ in range(args.warmup):  # untimed warm-up passes of the same sample
            cpu_oracle_rate(w, budget_s=0.0, max_reps=1)
        per_step = []
        base = None
        for _ in range(args.steps):
            base = cpu_oracle_rate(w, budget_s=min(budget, 120.0 / max(1, args.steps)), max_reps=1)
            per_step.append(base["value"])
        value = statistics.median(per_step)
        el = time.perf_counter() - t0
        base["value"] = value
        out = {
            "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": w.M / value * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": f"{w.name}: {w.note}", "M": w.M, "d_in": w.d_in,
                                            "d_out": w.d_out, "r": w.r},
            "cpu_baseline": base,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": el,
        }
        print(json.dumps(out))
        return

    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl")
    res = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_oracle_rate(w)
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as tdist
        tdist.barrier()
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
