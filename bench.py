"""Benchmark of the blr layer's forward+backward step on GB300.

One step = blr_forward + blr_backward of every layer of the workload over one
batch of synthetic tokens (every kernel of the hot path); the default workload
is the SwiGLU MLP pair (up 4096 -> 12288 and down 12288 -> 4096, r = 1024,
16384 tokens). Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mlp]
  python bench.py --impl reference ...     # the CPU f64 oracle as the reference arm

Timing: W untimed warm-up steps, then K timed steps between a barrier and
cudaDeviceSynchronize on both sides, measured with CUDA events on the launch
stream; max over ranks. L2 (129 MB) is defeated by rotating independent
input/output/workspace sets whose total exceeds twice the L2 size. Steps are
timed as CUDA-graph replays (one graph per buffer set, captured from the same
library calls), so host launch cost is not in the device time; the
end-to-end number keeps every host call. Kernel-level durations for the
roofline come from the same graphs captured a second time with the library's
event trace on, whose event-record nodes bracket every kernel inside the
replays. Multi-GPU: every rank runs its own batch (weak scaling); the path
needs no collective inside a step.
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
E2E_PIPE = 3  # device buffer sets the end-to-end measurement pipelines over
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
    """(flops, algorithmic bytes, staging bytes) of one launch of a kernel of the step.

    Algorithmic bytes are the tensors the layer itself must move, attributed to
    the kernel that moves them: x (read by the forward and again by the
    dg sums), y, dy, dx, the f32 a tape (written, read), the f16 c tape
    (written, read) and the bitmaps (read once per pass). The staged f16
    operands (x16, dy16, a.l, db.l), the re-laid bitmaps and the partial-sum
    rows are this design's own round trips: they are counted separately as
    staging bytes and never as achieved work. FLOP counts 2 per multiply-add of
    the four sign products.
    """
    words = (r + 31) // 32
    bits_u, bits_v = 4.0 * d_out * words, 4.0 * d_in * words
    relaid_u, relaid_v = 8.0 * sign_rows(d_out) * 2 * ((r + 127) // 128), 8.0 * sign_rows(r) * 2 * ((d_in + 127) // 128)
    relaid_ut = 8.0 * sign_rows(r) * 2 * ((d_out + 127) // 128)
    relaid_vd = 8.0 * sign_rows(d_in) * 2 * ((r + 127) // 128)
    parts = 4.0 * ((M + 127) // 128) * (d_in + d_out + r)  # partial rows, about one per 128 tokens
    table = {
        "fwd_prologue": (0.0, 4.0 * M * d_in + bits_u + bits_v, 2.0 * M * d_in + relaid_u + relaid_v),
        "gemm_fwd1": (2.0 * M * r * d_in, 4.0 * M * r, 2.0 * M * d_in + 2.0 * M * r + relaid_v),
        "gemm_fwd2": (2.0 * M * r * d_out, 6.0 * M * d_out, 2.0 * M * r + relaid_u),
        "bwd_prologue": (0.0, 6.0 * M * d_out + bits_u + bits_v, 2.0 * M * d_out + relaid_ut + relaid_vd),
        "gemm_bwd1": (2.0 * M * r * d_out, 4.0 * M * r, 2.0 * M * d_out + 2.0 * M * r + relaid_ut + parts),
        "gemm_bwd2": (2.0 * M * r * d_in, 8.0 * M * d_in, 2.0 * M * r + relaid_vd + parts),
        "reduce_partials": (0.0, 8.0 * (d_in + d_out + r), parts),
        # a forward whose x staging runs in the a-product: the prologue only
        # re-lays the bitmaps, and the staging product reads x itself and
        # writes the f16 operand it then reads
        "fwd_prep": (0.0, bits_u + bits_v, relaid_u + relaid_v),
        "gemm_fwd1s": (2.0 * M * r * d_in, 4.0 * M * d_in + 4.0 * M * r,
                       4.0 * M * d_in + 2.0 * M * r + relaid_v),
        # a backward whose dy staging runs in the db-product: the scale pass
        # reads dy for the per-token scales; the staging product reads c for
        # the dh sums and reads dy again (a staging round trip, like the f16
        # operand it writes and then reads)
        "bwd_scales": (0.0, 4.0 * M * d_out + bits_u + bits_v, relaid_ut + relaid_vd),
        "gemm_bwd1s": (2.0 * M * r * d_out, 4.0 * M * r + 2.0 * M * d_out,
                       8.0 * M * d_out + 2.0 * M * r + relaid_ut + parts),
    }
    if name == "small_fwd":
        return tuple(sum(table[n][i] for n in ("fwd_prologue", "gemm_fwd1", "gemm_fwd2")) for i in range(3))
    if name == "small_bwd":
        return tuple(sum(table[n][i] for n in ("bwd_prologue", "gemm_bwd1", "gemm_bwd2", "reduce_partials"))
                     for i in range(3))
    return table.get(name, (0.0, 0.0, 0.0))


def sign_rows(n: int) -> int:
    """Rows of a re-laid bitmap (n rounded up to 256)."""
    return (n + 255) // 256 * 256


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


def layers_of(args):
    """The layers one step of the named workload runs (at --tokens tokens when given)."""
    from binary_rank_linear_gb300 import workloads as wl
    return wl.step_layers(args.workload, args.tokens)


def blas_threads():
    """Threads numpy's BLAS may use, from the usual environment variables (None: the library default)."""
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k):
            try:
                return k, int(os.environ[k])
            except ValueError:
                pass
    return None, None


# ---------------------------------------------------------- CPU oracle ------
def cpu_oracle_rate(layers, budget_s: float = 12.0, max_reps: int = 1_000_000):
    """tokens/s of the CPU f64 oracle (as it stands) on the step's layers,
    repeated until ``budget_s`` seconds of CPU work have run. Workloads whose
    batch would exceed the budget run a prefix of their tokens (the seeded
    draws of a prefix are the full batch's first rows)."""
    import oracle
    from binary_rank_linear_gb300 import workloads as wl

    sample_M = layers[0].M
    # keep one oracle pass in the seconds range: ~4 f64 GEMMs of 2*M*r*d each per layer
    per_token = sum(4.0 * w.r * (w.d_in + w.d_out) for w in layers)
    while sample_M > 64 and per_token * sample_M > 3e11:
        sample_M //= 2
    inputs = []
    for w in layers:
        t = wl.make_inputs(w.with_shape(M=sample_M))
        inputs.append((t, oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])))
    reps, t0 = 0, time.perf_counter()
    while True:
        for t, bu, bv in inputs:
            oracle.forward(t["x"], bu, bv, t["g"], t["l"], t["h"])
            oracle.backward(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"])
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= max_reps:
            break
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    env, threads = blas_threads()
    names = "+".join(w.name for w in layers)
    return {
        "value": reps * sample_M / el,
        "unit": "tokens/s",
        "cores": min(cores, threads) if threads else cores,
        "kind": "oracle",
        "sample": f"{reps} x (forward+backward of the first {sample_M} of {layers[0].M} tokens of {names}) in "
                  f"{el:.1f} s, numpy f64",
        "host_cores": cores,
        "blas_threads": {"env": env, "value": threads} if env else "BLAS default (one per available core)",
    }


# ------------------------------------------------------------ GPU arm -------
class Layer:
    """One blr layer of the step on the device: seeded inputs, packed signs,
    rotating buffer sets (x, dy, y, dx, workspace) and gradient vectors."""

    def __init__(self, w, dev, nsets):
        import torch

        import binary_rank_linear_gb300 as blr
        from binary_rank_linear_gb300 import workloads as wl
        self.w, self.dev, self.blr = w, dev, blr
        t = wl.make_inputs(w)
        self.host = t

        def d(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

        M, d_in, d_out, r = w.M, w.d_in, w.d_out, w.r
        self.g, self.l, self.h = d(t["g"]), d(t["l"]), d(t["h"])
        self.bu, self.bv = blr.pack_signs(d(t["su"])), blr.pack_signs(d(t["sv"]))
        x0, dy0 = d(t["x"]), d(t["dy"])
        self.ws_bytes = blr.workspace_bytes(M, d_in, d_out, r)
        self.sets = []
        for _ in range(nsets):
            self.sets.append({
                "x": x0.clone(), "dy": dy0.clone(),
                "y": torch.empty(M, d_out, device=dev), "dx": torch.empty(M, d_in, device=dev),
                "ws": torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev),
            })
        del x0, dy0
        self.dg = torch.zeros(d_in, device=dev)
        self.dl = torch.zeros(r, device=dev)
        self.dh = torch.zeros(d_out, device=dev)

    @staticmethod
    def set_bytes(w, ws_bytes):
        return 4 * w.M * (2 * w.d_in + 2 * w.d_out) + ws_bytes

    def step(self, i, dg=None, dl=None, dh=None):
        s = self.sets[i % len(self.sets)]
        self.blr.forward(s["x"], self.bu, self.bv, self.g, self.l, self.h, s["y"], s["ws"])
        self.blr.backward(s["x"], s["dy"], self.bu, self.bv, self.g, self.l, self.h, s["dx"],
                          self.dg if dg is None else dg, self.dl if dl is None else dl,
                          self.dh if dh is None else dh, s["ws"])

    def check(self, where):
        for s in self.sets:
            st = self.blr.check_status(s["ws"])
            if st:
                raise RuntimeError(f"{where}: {self.w.name}: device status {st:#x}")


def nsets_for(layers_w, blr):
    """Rotating buffer sets: enough that one round of sets exceeds twice the L2,
    and at least E2E_PIPE (the end-to-end pipeline's depth)."""
    total = sum(Layer.set_bytes(w, blr.workspace_bytes(w.M, w.d_in, w.d_out, w.r)) for w in layers_w)
    return max(E2E_PIPE, min(64, -(-2 * L2_BYTES // total) + 1)), total


def label(layers, li, name):
    return name if len(layers) == 1 else f"{layers[li].w.name}/{name}"


def time_step(layers, args, dev, clocks=None):
    """Graph-replayed steps: W warm-up replays, then exactly K timed replays
    between barriers, CUDA events on the launch stream. Returns (ms, graphs)."""
    import torch
    stream = torch.cuda.current_stream()
    nsets = len(layers[0].sets)
    for i in range(max(args.warmup, nsets)):
        for L in layers:
            L.step(i)
    for L in layers:
        L.check("warm-up")
    # one CUDA graph per buffer set: a step is replayed with no host launch cost
    graphs = []
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        for i in range(nsets):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=cap):
                for L in layers:
                    L.step(i)
            graphs.append(gr)
    stream.wait_stream(cap)
    for i in range(args.warmup):
        graphs[i % nsets].replay()
    if clocks is not None:
        # the sampler runs from here to the end of the timed replays; untimed
        # replays for about half a second before them keep the GPU at its
        # loaded clocks, so that the samples describe the timed region
        clocks.start()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(nsets):
            graphs[i].replay()
        torch.cuda.synchronize()
        per = max(1e-6, (time.perf_counter() - t0) / nsets)
        for i in range(min(5000, int(0.5 / per))):
            graphs[i % nsets].replay()
    barrier(args)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        graphs[i % nsets].replay()
    e1.record(stream)
    barrier(args)
    return e0.elapsed_time(e1), graphs


def time_kernels(layers, args, dev):
    """Per-kernel durations of the replayed step: the step is captured once
    more with the library's trace on, which puts a CUDA event-record node
    before and after every kernel of the graph; K replays are timed kernel by
    kernel (and as whole replays). Returns ({label: [ms, ...]}, ms per replay)."""
    import torch

    import binary_rank_linear_gb300 as blr
    stream = torch.cuda.current_stream()
    nsets = len(layers[0].sets)
    blr.trace_begin(capacity=nsets * 16 * len(layers) + 16)
    graphs, ranges = [], []
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(stream)
    try:
        with torch.cuda.stream(cap):
            for i in range(nsets):
                gr = torch.cuda.CUDAGraph()
                rng = []
                with torch.cuda.graph(gr, stream=cap):
                    for li, L in enumerate(layers):
                        a = blr.trace_count()
                        L.step(i)
                        rng.append((li, a, blr.trace_count()))
                graphs.append(gr)
                ranges.append(rng)
    finally:
        blr.trace_end(read=False)
    stream.wait_stream(cap)
    per = {}
    whole = []
    for i in range(max(args.warmup, nsets)):
        graphs[i % nsets].replay()
    torch.cuda.synchronize()
    for i in range(args.steps):
        k = i % nsets
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graphs[k].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        whole.append(e0.elapsed_time(e1))
        for li, a, b in ranges[k]:
            for name, ms in blr.trace_read(a, b):
                per.setdefault(label(layers, li, name), []).append(ms)
    del graphs
    return per, statistics.mean(whole)


def roofline_of(per, layers, tc_peak, hbm_peak, steps):
    """Per-kernel figures and the roofline of the dominant kernel (largest
    total time), from the algorithmic work of each launch."""
    kernels = {}
    tot = sum(sum(v) for v in per.values())
    for name, lst in per.items():
        lname = name.split("/")[-1]
        w = next(L.w for L in layers if len(layers) == 1 or L.w.name == name.split("/")[0])
        fl, alg, stg = kernel_work(lname, w.M, w.d_in, w.d_out, w.r)
        avg_s = sum(lst) / len(lst) * 1e-3
        kernels[name] = {"avg_us": avg_s * 1e6, "launches_per_step": len(lst) / steps, "share": sum(lst) / tot,
                         "tflops": fl / avg_s / 1e12, "alg_gbs": alg / avg_s / 1e9, "staging_gbs": stg / avg_s / 1e9}
    dom = max(per, key=lambda n: sum(per[n]))
    lname = dom.split("/")[-1]
    w = next(L.w for L in layers if len(layers) == 1 or L.w.name == dom.split("/")[0])
    fl, alg, stg = kernel_work(lname, w.M, w.d_in, w.d_out, w.r)
    avg_s = kernels[dom]["avg_us"] * 1e-6
    t_tc, t_hbm = fl / (tc_peak * 1e12), alg / (hbm_peak * 1e9)
    if t_tc >= t_hbm:
        roof = {"bound": "tensor", "achieved": fl / avg_s / 1e12, "peak": tc_peak, "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": alg / avg_s / 1e9, "peak": hbm_peak, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof.update({"kernel": dom, "avg_us": avg_s * 1e6, "flops_per_launch": fl, "alg_bytes_per_launch": alg,
                 "staging_bytes_per_launch": stg})
    return kernels, roof


def barrier(args):
    import torch
    if getattr(args, "_dist", False):
        import torch.distributed as tdist
        tdist.barrier()
    torch.cuda.synchronize()


def measure_config(name, args, dev, tc_peak, hbm_peak):
    """A compact line for one more workload: graph-timed step, per-kernel
    durations and the dominant kernel's roofline (no side measurements)."""
    import torch

    import binary_rank_linear_gb300 as blr
    from binary_rank_linear_gb300 import workloads as wl
    layers_w = wl.step_layers(name)
    nsets, set_bytes = nsets_for(layers_w, blr)
    layers = [Layer(w, dev, nsets) for w in layers_w]
    ms, graphs = time_step(layers, args, dev)
    del graphs
    per, inst_ms = time_kernels(layers, args, dev)
    for L in layers:
        L.check(name)
    kernels, roof = roofline_of(per, layers, tc_peak, hbm_peak, args.steps)
    M = layers_w[0].M
    flops = sum(w.flops for w in layers_w)
    canon = sum(w.canonical_bytes for w in layers_w)
    out = {"workload": f"{name}: {wl.step_note(name)}", "value": M * args.steps / (ms * 1e-3), "unit": "tokens/s",
           "ms_per_step": ms / args.steps, "tflops": flops * args.steps / (ms * 1e-3) / 1e12,
           "tensor_frac": flops * args.steps / (ms * 1e-3) / 1e12 / tc_peak,
           "hbm_frac": canon * args.steps / (ms * 1e-3) / 1e9 / hbm_peak,
           "instrumented_ms_per_step": inst_ms, "roofline": roof,
           "kernels": {k: {"avg_us": v["avg_us"], "share": v["share"]} for k, v in kernels.items()},
           "l2": f"{nsets} rotating input/output/workspace sets ({nsets * set_bytes / 2**20:.0f} MiB > 2x L2)"}
    del layers
    torch.cuda.empty_cache()
    return out


def run_gpu(args, rank, world, local_rank):
    import torch

    import binary_rank_linear_gb300 as blr
    from binary_rank_linear_gb300 import workloads as wl

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    layers_w = layers_of(args)
    nsets, set_bytes = nsets_for(layers_w, blr)
    layers = [Layer(w, dev, nsets) for w in layers_w]
    M = layers_w[0].M
    flops = sum(w.flops for w in layers_w)
    canon = sum(w.canonical_bytes for w in layers_w)

    clocks = ClockSampler(local_rank)
    ms, graphs = time_step(layers, args, dev, clocks)
    clk = clocks.stop()
    del graphs
    for L in layers:
        L.check("timed steps")
    ms = max_over_ranks(ms, dev)

    per, inst_ms = time_kernels(layers, args, dev)
    launches_per_step = sum(len(v) for v in per.values()) / max(1, args.steps)
    peaks, peak_src = _peaks()
    tc_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    kernels, roof = roofline_of(per, layers, tc_peak, hbm_peak, args.steps)
    roof["peak_source"] = (f"{peak_src} (MEASURED_PEAKS.json: burst; bf16 for the f16 products, the same rate "
                           f"on this part)" if peak_src == "measured" else "fallback")
    roof["timing"] = ("CUDA events before and after each kernel, recorded as event nodes of the replayed step "
                      "graph (those replays run the kernels without programmatic overlap)")
    # stored counters are for the workloads' own token counts
    roof["traffic"] = stored_traffic(args.workload, roof["kernel"]) if not args.tokens else None

    L0 = layers[0]
    w0 = L0.w
    sign = measure_sign_grads(blr, L0.sets, L0.g, L0.l, args.steps, tc_peak, w0.M, w0.d_in, w0.d_out, w0.r, dev) \
        if not args.no_sign else None
    adam = measure_adam(blr, torch.cat([L0.dg, L0.dl, L0.dh]), args.steps, hbm_peak, dev)
    plane = measure_plane(blr, L0.sets[0], args.steps, tc_peak, w0.M, w0.d_in, w0.d_out, dev) \
        if not args.no_plane else None
    paths = measure_paths(blr, L0.sets[0], L0.bu, L0.bv, L0.g, L0.l, L0.h, args.steps, tc_peak, w0, dev) \
        if not args.no_paths else None

    e2e_ms, h2d, d2h, pipelined = measure_e2e(layers, args, dev)
    e2e_ms = max_over_ranks(e2e_ms, dev)
    for L in layers:
        L.check("end-to-end pass")

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
        "config": config_of(args, layers_w),
        "small_path": args.small_path,
        "buffer_sets": f"{nsets} rotating input/output/workspace sets ({nsets * set_bytes / 2**20:.0f} MiB)",
        "tflops": world * flops * args.steps / (ms * 1e-3) / 1e12,
        "tensor_frac": (world * flops * args.steps / (ms * 1e-3) / 1e12) / tc_peak,
        "hbm_frac": (world * canon * args.steps / (ms * 1e-3) / 1e9) / hbm_peak,
        "roofline": roof,
        "instrumented_ms_per_step": inst_ms,
        "kernels": kernels,
        "gpu_launches": int(round(launches_per_step * args.steps)),
        "clocks": clk,
        "e2e": {"value": job_tokens_per_s(world, M, args.steps, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": (f"overlapped with the layers on their own streams, {E2E_PIPE} buffer sets in flight"
                           if pipelined else "in order on one stream")},
    }
    if sign is not None:
        result["sign_grads"] = sign
    result["adam"] = adam
    if plane is not None:
        result["plane_linear"] = plane
    if paths is not None:
        paths["vs_one_layer_step"] = paths["us_per_step"] / (ms / args.steps * 1e3 / len(layers))
        result["paths"] = paths
    del layers
    torch.cuda.empty_cache()
    if world == 1 and args.extra:
        result["configs"] = {}
        for name in [n for n in args.extra.split(",") if n and n not in (args.workload, "none")]:
            result["configs"][name] = measure_config(name, args, dev, tc_peak, hbm_peak)
    return result


def measure_e2e(layers, args, dev):
    """End to end through the Python API: every step copies its inputs (x, dy
    of every layer) from pinned host memory and its results (y, dx, dg, dl,
    dh of every layer) back, inside the timed region. With a megabyte or more
    to move per step, steps are pipelined over two device buffer sets on
    three streams (host->device copies, the layers, device->host copies), as
    a training loop's data path would be: step i+1's inputs go up and step
    i-1's results come down while step i computes. Smaller steps run in order
    on one stream (there the host's launch work, not the copies, sets the
    pace). Returns (ms, h2d bytes per step, d2h bytes per step, pipelined).

    Three buffer sets: step i+1's inputs go up into the set whose results
    (step i-2's) came down a step earlier, so the two directions of the host
    link run at the same time; with two sets each upload would wait for the
    previous download of its set, and the copies would take turns."""
    import torch
    npipe = E2E_PIPE
    h2d = sum(4 * L.w.M * (L.w.d_in + L.w.d_out) for L in layers)
    d2h = sum(4 * (L.w.M * (L.w.d_in + L.w.d_out) + L.w.d_in + L.w.r + L.w.d_out) for L in layers)
    pipelined = h2d >= (1 << 20)
    pipe = []
    for b in range(npipe):
        per_layer = []
        for L in layers:
            w = L.w
            per_layer.append({
                "set": L.sets[b % len(L.sets)],
                "xh": torch.from_numpy(L.host["x"]).pin_memory() if b == 0 else None,
                "dyh": torch.from_numpy(L.host["dy"]).pin_memory() if b == 0 else None,
                "yh": torch.empty(w.M, w.d_out).pin_memory(),
                "dxh": torch.empty(w.M, w.d_in).pin_memory(),
                "gh": torch.empty(w.d_in + w.r + w.d_out).pin_memory(),
                "dg": torch.zeros(w.d_in, device=dev), "dl": torch.zeros(w.r, device=dev),
                "dh": torch.zeros(w.d_out, device=dev),
            })
        pipe.append({"layers": per_layer, "up": torch.cuda.Event(), "done": torch.cuda.Event(),
                     "down": torch.cuda.Event()})
    src = pipe[0]["layers"]
    if pipelined:
        s_up, s_comp, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    else:
        s_up = s_comp = s_down = torch.cuda.current_stream(dev)
    for b in pipe:
        b["down"].record(s_down)  # nothing to wait for yet

    def e2e_step(i):
        b = pipe[i % npipe] if pipelined else pipe[0]
        s_up.wait_event(b["down"])  # the set's previous results are down: its buffers are free again
        with torch.cuda.stream(s_up):
            for li, q in enumerate(b["layers"]):
                q["set"]["x"].copy_(src[li]["xh"], non_blocking=True)
                q["set"]["dy"].copy_(src[li]["dyh"], non_blocking=True)
        b["up"].record(s_up)
        s_comp.wait_event(b["up"])
        with torch.cuda.stream(s_comp):
            for L, q in zip(layers, b["layers"]):
                s0 = q["set"]
                L.blr.forward(s0["x"], L.bu, L.bv, L.g, L.l, L.h, s0["y"], s0["ws"])
                L.blr.backward(s0["x"], s0["dy"], L.bu, L.bv, L.g, L.l, L.h, s0["dx"], q["dg"], q["dl"], q["dh"],
                               s0["ws"])
        b["done"].record(s_comp)
        s_down.wait_event(b["done"])
        with torch.cuda.stream(s_down):
            for L, q in zip(layers, b["layers"]):
                w = L.w
                q["yh"].copy_(q["set"]["y"], non_blocking=True)
                q["dxh"].copy_(q["set"]["dx"], non_blocking=True)
                q["gh"][:w.d_in].copy_(q["dg"], non_blocking=True)
                q["gh"][w.d_in:w.d_in + w.r].copy_(q["dl"], non_blocking=True)
                q["gh"][w.d_in + w.r:].copy_(q["dh"], non_blocking=True)
        b["down"].record(s_down)

    for i in range(max(npipe, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(args)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(s_up)
    for i in range(args.steps):
        e2e_step(i)
    s_up.wait_stream(s_down)
    f1.record(s_up)
    torch.cuda.synchronize(dev)
    barrier(args)
    return f0.elapsed_time(f1), h2d, d2h, pipelined


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


def config_of(args, layers_w):
    """The `config` object of both arms' lines (the same keys and values)."""
    from binary_rank_linear_gb300 import workloads as wl
    M = layers_w[0].M
    return {
        "workload": f"{args.workload}: {wl.step_note(args.workload)}" + (f" (token count set to {M})" if args.tokens
                                                                          else ""),
        "layers": [{"name": w.name, "M": w.M, "d_in": w.d_in, "d_out": w.d_out, "r": w.r} for w in layers_w],
        "mode": "overwrite y/dx, dynamic per-token gradient scale",
        "l2": "buffer sets rotated between steps, their total more than twice the 129 MB L2",
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="blr", choices=["blr", "reference"])
    ap.add_argument("--workload", default="mlp",
                    help="mlp (the SwiGLU up+down pair, default), tiny, small, attn, mlp_up, mlp_down, ragged")
    ap.add_argument("--extra", default="tiny,small,attn,ragged",
                    help="workloads measured after the main one (N=1 only), reported under 'configs'; '' or none for none")
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
    layers_w = layers_of(args)
    M = layers_w[0].M

    if args.impl == "reference":
        if rank != 0:
            return
        budget = 10.0
        t0 = time.perf_counter()
        for _ in range(args.warmup):  # untimed warm-up passes of the same sample
            cpu_oracle_rate(layers_w, budget_s=0.0, max_reps=1)
        per_step = []
        base = None
        for _ in range(args.steps):
            base = cpu_oracle_rate(layers_w, budget_s=min(budget, 120.0 / max(1, args.steps)), max_reps=1)
            per_step.append(base["value"])
        value = statistics.median(per_step)
        el = time.perf_counter() - t0
        base["value"] = value
        out = {
            "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": M / value * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(args, layers_w),
            "cpu_baseline": base,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": el,
        }
        print(json.dumps(out))
        return

    args._dist = world > 1
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local_rank)
        tdist.init_process_group("nccl")
    res = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_oracle_rate(layers_w)
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as tdist
        tdist.barrier()
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
