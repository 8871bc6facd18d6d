"""Benchmark: useful TFLOP/s, % of roofline and us per call of the convolution forward pass.

Default workload: the conv1d bf16 frontend sweep at batch 32, the largest configuration
that the metric is quoted on: conv1d 128 -> 1280 k3 s1 p1 on L=3000 + GELU, then conv1d
1280 -> 1280 k3 s2 p1 (L 3000 -> 1500) + GELU, 566 GFLOP per step.  One step runs both
layers through the C-ABI.  Useful FLOPs = 2 x MACs, padded taps counted (the convention of
page "[ET-VK] conv1d runs at ~3% of the GPU's matmul throughput ...", "Measurements").
The same run also measures every other configuration (the 80 -> 384 fp32 conv1d, the
Whisper-tiny frontend in fp32 and bf16, the sweep at batch 1 and 8, the grouped 2D and 3D
layers) and reports each one's us per call and roofline fraction under `per_config`.

Timing: W warm-up steps, then exactly K steps between CUDA events on the launching stream,
bracketed by a barrier and a device synchronise.  A step runs every layer (each conv_fwd
call: the conv kernel, plus the reduction for split plans); the steps are captured in CUDA
graphs, one graph holding R consecutive steps (one per rotation set) that is replayed
K // R times, then one single-step graph for each of the remaining K % R steps.  By default
the plans chain their kernels as programmatic dependents (conv_plan_set_overlap), so each
kernel's set-up and weight loads overlap the previous one, across steps too inside a graph
(--no-overlap turns this off); a graph boundary after every step costs 4-7 us of launch
latency, which a layer inside a larger graph does not pay.  Each layer's device time comes from a second run of the same steps with timing
events recorded inside the graph between the layers (where PyTorch cannot record events
inside a graph, each layer is its own graph and the events sit between them).  Steps
rotate over enough copies of every input, packed weight and output that one rotation
exceeds twice the L2 cache, so no step finds its data in L2.  `eager` times the same
layers called from the host one by one (no graph): each call validates its arguments and
encodes the activation tensor map before it launches.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]
                  [--configs all|none|NAME,...] [--no-overlap] [--serial] [--pass fwd|bwd]
                  [--tune ITERS] [--source-hash]

--tune ITERS lets the measured selector (conv_plan_tune) time every candidate plan of each
layer before the run and keep the fastest; by default the planner's rules choose.  The step's
independent chains (e.g. the fp32 and the bf16 frontend) run one after the other in the
forward pass and as parallel branches of the step graph, each on its own stream, in the
backward pass (--serial / --parallel override).

Under torchrun each rank runs an independent replica on its own GPU (the forward pass
has no exchange step); rank 0 prints the JSON line with the max time over ranks.
--impl reference times the CPU oracle (fp64 direct loops) on the host cores instead, with
the same sampling method as the `cpu_baseline` field of our own line.
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

METRIC = "conv fwd useful TFLOP/s and % of roofline at 1 GB300; µs per call"
L2_BYTES = 129 * 1000 * 1000
FFMA_PER_SM_PER_CLK = 128          # fp32 lanes per SM
SM_COUNT = 152
SM_MAX_MHZ = 2070.0


# ----------------------------------------------------------------------------- workloads
def frontend_workloads(name):
    from convolution_forward_implicit_gb300.workloads import WORKLOADS
    if name == "whisper_frontend":
        return [WORKLOADS["whisper_frontend_f32"], WORKLOADS["whisper_frontend_bf16"]]
    if name == "whisper_mlp":
        return [WORKLOADS["whisper_mlp_f32"], WORKLOADS["whisper_mlp_bf16"]]
    if name in WORKLOADS:
        return [WORKLOADS[name]]
    raise SystemExit(f"unknown workload {name}")


def workload_description(name):
    if name == "whisper_frontend":
        return ("whisper_tiny_conv_frontend: conv1d 80->384 k3 s1 p1 L=3000 +GELU, conv1d 384->384 k3 s2 p1 "
                "(L 3000->1500) +GELU, batch 1, fp32 and bf16 I/O")
    if name == "whisper_mlp":
        return ("whisper_tiny_encoder_mlp as 1x1 convs: 384->1536 +bias +GELU, 1536->384 +bias over 1500 "
                "positions, batch 1, fp32 and bf16 I/O")
    if name.startswith("sweep_bf16_n"):
        n = name[len("sweep_bf16_n"):]
        return (f"conv1d_bf16_frontend_sweep batch {n}: conv1d 128->1280 k3 s1 p1 L=3000 +GELU, conv1d "
                f"1280->1280 k3 s2 p1 (L 3000->1500) +GELU, bf16 I/O")
    from convolution_forward_implicit_gb300.workloads import WORKLOADS
    wl = WORKLOADS.get(name)
    if wl is not None:
        L = wl.layers[0]
        sp = "x".join(str(v) for v in L.spatial)
        fl = "x".join(str(v) for v in L.filter)
        dl = "x".join(str(v) for v in L.dilation)
        return wl.note or (f"{name}: {L.ndim}D grouped conv N={L.N} {sp} G={L.G} C=K={L.C} filter {fl} "
                           f"dilation {dl} {wl.dtype}")
    return name


# every configuration the metric is quoted on (the per_config table of the JSON line)
BASELINE_CONFIGS = ["conv1d_f32_80to384_L3000", "whisper_frontend_f32", "whisper_frontend_bf16", "sweep_bf16_n1",
                    "sweep_bf16_n8", "sweep_bf16_n32", "grouped2d_g8_c64_d1", "grouped2d_g8_c64_d2",
                    "grouped2d_g32_c8_d1", "grouped2d_g32_c8_d2", "grouped3d_g4_c64_d1", "grouped3d_g4_c64_d2"]


# ----------------------------------------------------------------------------- distributed
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(v: float, ws: int, device=None) -> float:
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while running (clocks, power, throttle reasons)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return self.summary()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- our arm
class LayerRun:
    """One layer of one workload: its plan, per-rotation-set buffers and CUDA graphs."""

    def __init__(self, wl, li, layer, R, x_sets, w, b, tune_iters=0):
        import torch
        from convolution_forward_implicit_gb300.binding import ConvPlan
        self.wl, self.li, self.layer = wl, li, layer
        self.plan = ConvPlan(*layer.plan_args(wl.dtype_code))
        tdt = self.plan.torch_dtype()
        if tune_iters:
            # the measured selector: time every candidate plan on these buffers, keep the fastest
            y = torch.empty(self.plan.y_shape(), dtype=tdt, device="cuda")
            self.plan.tune(x_sets[0], w, b if layer.bias_bound is not None else None, y, iters=tune_iters)
            del y
        self.plan.allocate()
        self.x_sets = x_sets
        self.wp_sets, self.b_sets, self.y_sets = [], [], []
        for r in range(R):
            wp = torch.empty_like(self.plan.w_packed)
            self.plan.prepack(w)
            wp.copy_(self.plan.w_packed)
            self.wp_sets.append(wp)
            self.b_sets.append(b.clone() if b is not None else None)
            self.y_sets.append(torch.empty(self.plan.y_shape(), dtype=tdt, device="cuda"))
        self.graphs = []
        fields = dict(kv.split("=", 1) for kv in self.plan.describe().split())
        self.kernels_per_call = 1 + (1 if int(fields.get("splits", "1")) > 1 else 0)   # conv (+ split-K reduction)

    def call(self, r):
        from convolution_forward_implicit_gb300.binding import conv_fwd
        import torch
        b = self.b_sets[r]
        conv_fwd(self.plan.handle, self.x_sets[r].data_ptr(), self.wp_sets[r].data_ptr(),
                 0 if b is None else b.data_ptr(), self.y_sets[r].data_ptr(), torch.cuda.current_stream().cuda_stream)

    def capture(self, R):
        import torch
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for r in range(R):
                self.call(r)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        for r in range(R):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.call(r)
            self.graphs.append(g)

    @property
    def flops(self):
        return self.plan.flops

    def name(self):
        return f"{self.wl.dtype}_L{self.li + 1}"

    def bytes_alg(self):
        L = self.layer
        esz = 2 if self.wl.dtype == "bf16" else 4
        n_out = int(np.prod(self.plan.y_shape()))
        n_x = int(np.prod(L.x_shape()))
        n_w = int(np.prod(L.w_shape()))
        n_b = L.G * L.K if L.bias_bound is not None else 0
        return esz * (n_out + n_x + n_w + n_b)


class BwdRun:
    """Backward data or backward weight of one layer: its plan, per-rotation-set buffers
    (dy, x or the packed weight, and the output dx or dw) and CUDA graphs."""

    def __init__(self, wl, li, layer, R, kind, x_sets, dy_sets, w):
        import torch
        from convolution_forward_implicit_gb300.binding import ConvPlan
        self.wl, self.li, self.layer, self.kind = wl, li, layer, kind
        self.plan = ConvPlan(*layer.plan_args(wl.dtype_code), direction=kind)
        self.plan.allocate()
        tdt = self.plan.torch_dtype()
        self.x_sets, self.dy_sets = x_sets, dy_sets
        self.wp_sets, self.y_sets = [], []
        for r in range(R):
            if kind == "bwd_data":
                wp = torch.empty_like(self.plan.w_packed)
                self.plan.prepack(w)
                wp.copy_(self.plan.w_packed)
                self.wp_sets.append(wp)
                self.y_sets.append(torch.empty(self.plan.x_shape(), dtype=tdt, device="cuda"))
            else:
                self.y_sets.append(torch.empty(self.plan.w_shape(), dtype=tdt, device="cuda"))
        self.graphs = []
        fields = dict(kv.split("=", 1) for kv in self.plan.describe().split())
        self.kernels_per_call = 1 + (1 if int(fields.get("splits", "1")) > 1 and
                                     fields.get("reduce", "kernel") != "cluster" else 0)

    def call(self, r):
        from convolution_forward_implicit_gb300.binding import conv_bwd_data, conv_bwd_weight
        import torch
        s = torch.cuda.current_stream().cuda_stream
        if self.kind == "bwd_data":
            conv_bwd_data(self.plan.handle, self.dy_sets[r].data_ptr(), self.wp_sets[r].data_ptr(),
                          self.y_sets[r].data_ptr(), s)
        else:
            conv_bwd_weight(self.plan.handle, self.x_sets[r].data_ptr(), self.dy_sets[r].data_ptr(),
                            self.y_sets[r].data_ptr(), s)

    capture = LayerRun.capture

    @property
    def flops(self):
        return self.plan.flops

    def name(self):
        return f"{self.wl.dtype}_L{self.li + 1}_{'dx' if self.kind == 'bwd_data' else 'dw'}"

    def bytes_alg(self):
        L = self.layer
        esz = 2 if self.wl.dtype == "bf16" else 4
        n_x = int(np.prod(L.x_shape()))
        n_w = int(np.prod(L.w_shape()))
        n_dy = int(np.prod(self.plan.y_shape()))
        return esz * (n_dy + n_w + n_x)   # dx: dy and w in, dx out; dw: x and dy in, dw out


def to_device(a, dtype):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def setup_layers(wls, R, tune_iters=0):
    """Layers of every workload; layer l+1 of a workload reads layer l's output set."""
    from convolution_forward_implicit_gb300.workloads import gen_inputs
    runs, inputs = [], []
    for wl in wls:
        x, params = gen_inputs(wl)
        xd = to_device(x, wl.dtype)
        x_sets = [xd.clone() for _ in range(R)]
        inputs.append((wl, x, x_sets))
        for li, layer in enumerate(wl.layers):
            w, b = params[li]
            lr = LayerRun(wl, li, layer, R, x_sets, to_device(w, wl.dtype),
                          to_device(b, wl.dtype) if b is not None else None, tune_iters)
            runs.append(lr)
            x_sets = [y.view(-1) for y in lr.y_sets]
    return runs, inputs


def setup_bwd_layers(wls, R):
    """Backward data and backward weight of every layer of every workload, on seeded x, w and
    dy (the gradient of the layer's output); returns (runs, host inputs, output sets)."""
    from convolution_forward_implicit_gb300 import synthetic as syn
    from convolution_forward_implicit_gb300.workloads import gen_inputs
    runs, host_in, outs = [], [], []
    for wl in wls:
        x0, params = gen_inputs(wl)
        for li, layer in enumerate(wl.layers):
            w, _ = params[li]
            x = x0 if li == 0 else syn.gen_normal(7 + li, layer.x_shape(), wl.dtype)
            y_shape = tuple(int(v) for v in np_y_shape(layer))
            dy = syn.gen_normal(20261202 + 1000 * wl.index + 10 * li + 3, y_shape, wl.dtype)
            xd, dyd, wd = to_device(x, wl.dtype), to_device(dy, wl.dtype), to_device(w, wl.dtype)
            x_sets = [xd.clone() for _ in range(R)]
            dy_sets = [dyd.clone() for _ in range(R)]
            host_in += [(x, wl.dtype, x_sets), (dy, wl.dtype, dy_sets)]
            for kind in ("bwd_data", "bwd_weight"):
                br = BwdRun(wl, li, layer, R, kind, x_sets, dy_sets, wd)
                runs.append(br)
                outs.append(br.y_sets)
    return runs, host_in, outs


def np_y_shape(layer):
    """The layer's output shape (N, spatial..., G, K), from the library's own size formula."""
    from convolution_forward_implicit_gb300.binding import (conv_plan_create, conv_plan_destroy,
                                                            conv_plan_output_shape)
    h = conv_plan_create(*layer.plan_args(0))
    try:
        out = conv_plan_output_shape(h, layer.ndim)
    finally:
        conv_plan_destroy(h)
    return (layer.N, *out, layer.G, layer.K)


def rotation_sets(wls, factor=1.0):
    """Copies needed so that one rotation of activations, packed weights and outputs
    exceeds twice the L2 cache (factor scales the bytes of one set)."""
    per_set = 0
    for wl in wls:
        for layer in wl.layers:
            esz = 2 if wl.dtype == "bf16" else 4
            per_set += esz * (int(np.prod(layer.x_shape())) + int(np.prod(layer.w_shape())))
    # outputs are roughly the inputs of the next layer plus the last output
    per_set = int(per_set * 1.6 * factor) + 1
    return max(4, int(np.ceil(2.2 * L2_BYTES / per_set))), per_set


def capture_steps(runs, R, with_events, parallel=False, chain=None):
    """One CUDA graph per rotation set holding every layer of the step.  With with_events,
    timing events are recorded between the layers inside the graph (they give each layer's
    device time, and they also keep consecutive layers from overlapping); returns (graphs,
    events), or None when this PyTorch cannot record events inside a graph.  With parallel,
    the step's independent chains (the layers of each workload) are captured as parallel
    branches on their own streams, joined at the end of the step.  With chain (a list of
    rotation sets), one graph holds one step per listed set, one after the other, so that a
    step's first kernel is launched as a programmatic dependent of the previous step's last
    one, as it would be inside a larger graph, instead of after a graph boundary; returns
    ([graph], None)."""
    import torch
    events = None
    if with_events:
        try:
            events = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(runs) + 1)]
                      for _ in range(R)]
        except TypeError:
            return None
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for r in range(R):
            for lr in runs:
                lr.call(r)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    # the independent chains of the step (one per workload) as parallel branches of the graph
    chains = {}
    for lr in runs:
        chains.setdefault(lr.wl.name, []).append(lr)
    chains = list(chains.values())
    branch = parallel and not events and len(chains) > 1
    side = [torch.cuda.Stream() for _ in range(len(chains) - 1)] if branch else []

    def emit_step(r, cs):
        if branch:
            for ss in side:
                ss.wait_stream(cs)
            for ci, chain_ in enumerate(chains):
                with torch.cuda.stream(cs if ci == 0 else side[ci - 1]):
                    for lr in chain_:
                        lr.call(r)
            for ss in side:
                cs.wait_stream(ss)
        else:
            if events:
                events[r][0].record(cs)
            for j, lr in enumerate(runs):
                lr.call(r)
                if events:
                    events[r][j + 1].record(cs)

    if chain is not None:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream()
            for r in chain:
                emit_step(r, cs)
        return [g], None
    graphs = []
    for r in range(R):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            emit_step(r, torch.cuda.current_stream())
        graphs.append(g)
    return graphs, events


def prepare(args, wls, bwd=False):
    """Plans, rotating buffers and step graphs of the workloads.  Returns a dict with the
    runs, the host inputs and output sets (for the end-to-end leg), the step graphs and the
    graphs (or per-layer graphs) that time each layer."""
    import torch
    R, per_set = rotation_sets(wls, 2.0 if bwd else 1.0)
    if bwd:
        runs, host_in, out_sets = setup_bwd_layers(wls, R)
    else:
        runs, inputs = setup_layers(wls, R, args.tune)
        host_in = [(x, wl.dtype, x_sets) for (wl, x, x_sets) in inputs]
        last = {}
        for lr in runs:
            last[lr.wl.name] = lr
        out_sets = [lr.y_sets for lr in last.values()]
    if args.overlap:
        for lr in runs:
            lr.plan.set_overlap(True)
    # timed steps: graphs with no events inside, so consecutive kernels may overlap; one graph
    # per step, and one holding all R steps in rotation order
    step_graphs, _ = capture_steps(runs, R, with_events=False, parallel=args.parallel)
    chain_graph = capture_steps(runs, R, with_events=False, parallel=args.parallel, chain=list(range(R)))[0][0]
    # per-layer device times: the same steps with events between the layers
    cap = capture_steps(runs, R, with_events=True)
    if cap is not None:
        layer_graphs, gev = cap
        graph_mode = (f"steps timed through one graph of {R} consecutive steps (one per rotation set; all layers"
                      + (", chained as programmatic dependents" if args.overlap else "")
                      + ("; independent workloads as parallel branches" if args.parallel and len(wls) > 1 else "")
                      + "), replayed K // R times, then one graph per step for the remaining K % R; per-layer "
                      "times from a second run of one graph per step with events between the layers")
    else:
        for lr in runs:
            lr.capture(R)
        layer_graphs, gev = None, None
        graph_mode = (f"steps timed through one graph of {R} consecutive steps, replayed K // R times, then one graph "
                      "per step for the remaining K % R; per-layer times from one graph per layer with events between "
                      "graphs")
    torch.cuda.synchronize()
    return {"R": R, "per_set": per_set, "runs": runs, "host_in": host_in, "out_sets": out_sets,
            "step_graphs": step_graphs, "chain_graph": chain_graph, "layer_graphs": layer_graphs, "gev": gev,
            "graph_mode": graph_mode}


def time_steps(st, K, W, stream, ws=1, on_start=None):
    """W warm-up steps, then K steps of the step graphs between CUDA events (barrier and
    synchronise on both sides); returns the total ms (max over ranks by the caller)."""
    import torch
    R, graphs, chain = st["R"], st["step_graphs"], st["chain_graph"]
    for i in range(W):
        graphs[i % R].replay()
    chain.replay()
    torch.cuda.synchronize()
    for lr in st["runs"]:
        lr.plan.check()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if on_start:
        on_start()
    barrier(ws)
    torch.cuda.synchronize()
    # exactly K steps: K // R replays of the R-step graph, then single steps (rotation sets 0..)
    e0.record(stream)
    for i in range(K // R):
        chain.replay()
    for i in range(K % R):
        graphs[i].replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    return e0.elapsed_time(e1)


def time_layers(st, K, W, stream):
    """Per-layer device times (ms) over K steps after W warm-up steps: the mean, and the
    samples behind it (one per step, or the last replay of each rotation set)."""
    import torch
    R, runs, layer_graphs, gev = st["R"], st["runs"], st["layer_graphs"], st["gev"]
    nL = len(runs)
    ev = None if layer_graphs is not None else [[torch.cuda.Event(enable_timing=True) for _ in range(nL + 1)]
                                                for _ in range(K)]
    for i in range(W):
        if layer_graphs is not None:
            layer_graphs[i % R].replay()
    torch.cuda.synchronize()
    for i in range(K):
        if ev is None:
            layer_graphs[i % R].replay()
        else:
            ev[i][0].record(stream)
            for j, lr in enumerate(runs):
                lr.graphs[i % R].replay()
                ev[i][j + 1].record(stream)
    torch.cuda.synchronize()
    if ev is None:
        last = sorted({i % R: i for i in range(K)}.keys())
        samples = [[gev[r][j].elapsed_time(gev[r][j + 1]) for r in last] for j in range(nL)]
    else:
        samples = [[ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K)] for j in range(nL)]
    return [sum(v) / len(v) for v in samples], samples


def time_eager(st, K, W, stream):
    """The layers called from the host, one conv_fwd per layer per step with no graph: the
    device time per step (CUDA events) and the host time per call (Python wall clock around
    the calls: ctypes marshalling, argument checks, the tensor-map encode and the launch)."""
    import torch
    R, runs = st["R"], st["runs"]
    for i in range(W):
        for lr in runs:
            lr.call(i % R)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    t0 = time.perf_counter()
    for i in range(K):
        for lr in runs:
            lr.call(i % R)
    host_s = time.perf_counter() - t0
    e1.record(stream)
    torch.cuda.synchronize()
    for lr in runs:
        lr.plan.check()
    ms = e0.elapsed_time(e1) / K
    return ms, host_s * 1e6 / (K * len(runs))


def release(st):
    import torch
    st.clear()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def per_config_table(args, names, stream, done=None):
    """Every configuration in `names`, each measured the way the headline is (rotating
    buffers larger than twice the L2, graphs of R consecutive steps, per-layer events): us per
    step and per layer, useful TFLOP/s and each layer's roofline fraction."""
    W = max(3, min(args.warmup, 5))
    table = {}
    for name in names:
        if done is not None and name in done:
            table[name] = done[name]
            continue
        st = prepare(args, frontend_workloads(name))
        # about 50 steps (at most --steps), a whole number of R-step graphs
        R = st["R"]
        K = R * max(1, round(min(args.steps, 50) / R))
        ms = time_steps(st, K, W, stream) / K
        per_layer_ms, _ = time_layers(st, K, W, stream)
        runs = st["runs"]
        flops = sum(lr.flops for lr in runs)
        table[name] = config_entry(runs, ms, per_layer_ms, K)
        release(st)
    return table


def config_entry(runs, ms, per_layer_ms, K):
    flops = sum(lr.flops for lr in runs)
    layers = {}
    for lr, t in zip(runs, per_layer_ms):
        roof = roofline_for(lr, t)
        layers[lr.name()] = {"us_per_call": round(t * 1e3, 3), "tflops": round(lr.flops / (t * 1e-3) / 1e12, 2),
                             "roofline_frac": roof["frac"], "bound": roof["bound"], "plan": lr.plan.describe()}
    if len(runs) == 1:
        # one layer per step: the step time is the call's time inside a graph of consecutive
        # calls (no event around it, launched as a programmatic dependent of the previous call)
        roof = roofline_for(runs[0], ms)
        layers[runs[0].name()].update({"us_per_call_chained": round(ms * 1e3, 3), "roofline_frac_chained": roof["frac"]})
    return {"us_per_step": round(ms * 1e3, 3), "tflops": round(flops / (ms * 1e-3) / 1e12, 2),
            "gflop_per_step": round(flops / 1e9, 3), "steps": K, "layers": layers}


def run_ours(args, ws, rank, local):
    import torch
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build()
    wls = frontend_workloads(args.workload)
    bwd = args.pass_ == "bwd"
    stream = torch.cuda.current_stream()
    st = prepare(args, wls, bwd)
    runs, R, per_set = st["runs"], st["R"], st["per_set"]
    K = args.steps
    clocks = ClockSampler(local)
    total_ms = time_steps(st, K, args.warmup, stream, ws, on_start=clocks.start)
    per_layer_ms, samples = time_layers(st, K, args.warmup, stream)
    layer_samples = len(samples[0]) if samples else 0
    layer_spread = {lr.name(): {"median": round(float(np.median(v)) * 1e3, 3),
                                "p10": round(float(np.percentile(v, 10)) * 1e3, 3),
                                "p90": round(float(np.percentile(v, 90)) * 1e3, 3)} for lr, v in zip(runs, samples)}
    # keep sampling clocks over a sustained window of the same steps (at least ~1.5 s)
    t_end = time.time() + 1.5
    i = 0
    while time.time() < t_end:
        for _ in range(50):
            st["step_graphs"][i % R].replay()
            i += 1
        torch.cuda.synchronize()
    clk = clocks.stop()
    for lr in runs:
        lr.plan.check()
    total_ms = max_over_ranks(total_ms, ws, torch.device("cuda", local))

    step_flops = sum(lr.flops for lr in runs)
    ms_per_step = total_ms / K
    value = ws * step_flops / (ms_per_step * 1e-3) / 1e12

    # ---- hot L2 (the same rotation set every step, R steps per graph as in the timed run) and
    # the latency of one isolated step
    g0 = st["step_graphs"][0]
    hot_graph = capture_steps(runs, R, with_events=False, parallel=args.parallel, chain=[0] * R)[0][0]
    for i in range(args.warmup):
        g0.replay()
    hot_graph.replay()
    torch.cuda.synchronize()
    eh0, eh1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    eh0.record(stream)
    for i in range(K // R):
        hot_graph.replay()
    for i in range(K % R):
        g0.replay()
    eh1.record(stream)
    torch.cuda.synchronize()
    hot_ms = eh0.elapsed_time(eh1) / K
    singles = []
    for i in range(20):
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        st["step_graphs"][i % R].replay()
        a1.record(stream)
        torch.cuda.synchronize()
        singles.append(a0.elapsed_time(a1) * 1e3)
    hot = {"ms_per_step": round(hot_ms, 6), "value": round(ws * step_flops / (hot_ms * 1e-3) / 1e12, 4),
           "unit": "TFLOP/s", "note": "one rotation set replayed every step: inputs that fit stay in L2"}
    single = {"median_us": round(float(np.median(singles)), 3), "p10_us": round(float(np.percentile(singles, 10)), 3),
              "p90_us": round(float(np.percentile(singles, 90)), 3), "samples": len(singles),
              "note": "one step between a device synchronize and events: launch latency included"}

    # ---- the same layers called from the host, no graph
    eager = None
    if not bwd:
        e_ms, host_us = time_eager(st, min(K, 50), args.warmup, stream)
        eager = {"us_per_step": round(e_ms * 1e3, 3), "value": round(ws * step_flops / (e_ms * 1e-3) / 1e12, 4),
                 "unit": "TFLOP/s", "host_us_per_call": round(host_us, 3), "steps": min(K, 50),
                 "note": "conv_fwd called from Python per layer per step, no graph: argument checks, the "
                         "activation tensor-map encode and the launch on the host every call"}

    # ---- end to end: pinned host inputs in, final outputs back to pinned host memory
    def step(i):
        st["step_graphs"][i % R].replay()
    e2e = run_e2e(args, runs, st["host_in"], st["out_sets"], R, stream, ws, local, step)

    # ---- roofline of the dominant kernel
    dom = int(np.argmax(per_layer_ms))
    lr = runs[dom]
    roof = roofline_for(lr, per_layer_ms[dom])
    roof["duration_us"] = round(per_layer_ms[dom] * 1e3, 3)
    roof["duration_samples"] = layer_samples

    launches = K * sum(lr.kernels_per_call for lr in runs)
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "TFLOP/s", "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "us_per_call": {lr.name(): round(t * 1e3, 3) for lr, t in zip(runs, per_layer_ms)},
        "us_per_call_spread": layer_spread,
        "useful_gflop_per_step": round(step_flops / 1e9, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "+".join(sorted({wl.dtype for wl in wls}, key=lambda d: d != "f32")),
        "data": "synthetic (seeded N(0,1) inputs, U(+-1/sqrt(C_in*taps)) weights, U(+-0.05) bias)",
        "config": {"workload": workload_description(args.workload) + (
                       "; backward: dx and dw of every layer per step (seeded N(0,1) dy)" if bwd else ""),
                   "pass": "backward (data + weight)" if bwd else "forward",
                   "l2": f"inputs larger than L2: {R} rotating sets of activations, packed weights and outputs "
                         f"(~{R * per_set / 1e6:.0f} MB per rotation, L2 129 MB)",
                   "graphs": st["graph_mode"],
                   "overlap": bool(args.overlap),
                   "selector": (f"measured (conv_plan_tune, {args.tune} timed calls per candidate)" if args.tune
                                else "rules"),
                   "parallelism": "replicas" if ws > 1 else "single GPU",
                   "kernel_sources": kernel_source_hash(),
                   "plans": {lr.name(): lr.plan.describe() for lr in runs}},
        "roofline": roof,
        "hot_l2": hot,
        "single_step": single,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk,
    }
    if eager is not None:
        line["eager"] = eager
    headline = config_entry(runs, ms_per_step, per_layer_ms, K) if not bwd else None
    release(st)
    names = [] if bwd or args.configs == "none" else (
        BASELINE_CONFIGS if args.configs == "all" else [n for n in args.configs.split(",") if n])
    if names:
        clocks_cfg = ClockSampler(local).start()
        done = {args.workload: headline} if args.workload in names else None
        line["per_config"] = per_config_table(args, names, stream, done)
        line["per_config_clocks"] = clocks_cfg.stop()
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline_bwd(wls) if bwd else cpu_baseline(wls)
        print(json.dumps(line), flush=True)


def run_e2e(args, runs, in_specs, out_sets, R, stream, ws, local, step):
    """The same step through the public API with host buffers: each step copies its inputs
    (in_specs: storage array, dtype, device copies) from pinned host memory, runs every layer,
    and copies the results (out_sets: device copies) back to pinned host memory.  The copies
    run on their own streams, pipelined across steps: step i+1's inputs are copied in and
    step i's results copied out while the next step computes, each rotating buffer guarded by
    events (a set is refilled only after the step that last used it has finished and its
    results were read back).  Every byte of every step stays inside the timed region.
    With --e2e-serial the copies and the step run one after the other on one stream."""
    import torch
    host_in, host_out = [], []
    for (a, dtype, sets) in in_specs:
        h = to_device(a, dtype).cpu().pin_memory()
        host_in.append((h, sets))
    for sets in out_sets:
        host_out.append((torch.empty(sets[0].shape, dtype=sets[0].dtype).pin_memory(), sets))
    bi = sum(h.numel() * h.element_size() for h, _ in host_in)
    bo = sum(h.numel() * h.element_size() for h, _ in host_out)
    K = args.steps
    copy_in, copy_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(R)]      # inputs of the set's current step are in
    ev_done = [torch.cuda.Event() for _ in range(R)]    # the set's current step has computed
    ev_out = [torch.cuda.Event() for _ in range(R)]     # the set's results have been read back

    def h2d(i):
        r = i % R
        if i >= R:
            copy_in.wait_event(ev_done[r])               # step i - R, the set's last user, is done
        with torch.cuda.stream(copy_in):
            for h, sets in host_in:
                sets[r].copy_(h, non_blocking=True)
        ev_in[r].record(copy_in)

    def e2e_step(i, last):
        r = i % R
        if args.e2e_serial:
            for h, sets in host_in:
                sets[r].copy_(h, non_blocking=True)
            step(i)
            for h, sets in host_out:
                h.copy_(sets[r], non_blocking=True)
            return
        stream.wait_event(ev_in[r])
        if i >= R:
            stream.wait_event(ev_out[r])                 # step i - R's results were read back
        step(i)
        ev_done[r].record(stream)
        copy_out.wait_event(ev_done[r])
        with torch.cuda.stream(copy_out):
            for h, sets in host_out:
                h.copy_(sets[r], non_blocking=True)
        ev_out[r].record(copy_out)
        if i + 1 < last:
            h2d(i + 1)

    def run(first, count, start_event=None):
        if not args.e2e_serial:
            if start_event is not None:
                copy_in.wait_event(start_event)
            h2d(first)
        for i in range(first, first + count):
            e2e_step(i, first + count)
        if not args.e2e_serial:
            stream.wait_stream(copy_out)

    run(0, args.warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    e0.record(stream)
    run(args.warmup, K, start_event=e0)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    ms = max_over_ranks(e0.elapsed_time(e1), ws, torch.device("cuda", local))
    flops = sum(lr.flops for lr in runs)
    return {"value": round(ws * flops * K / (ms * 1e-3) / 1e12, 4), "unit": "TFLOP/s",
            "ms_per_step": round(ms / K, 6), "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo),
            "copies": ("serial with the step on one stream" if args.e2e_serial else
                       "pinned host buffers; H2D and D2H on their own streams, pipelined across steps")}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def _strip_comments(text):
    """C/C++ source without its comments and blank lines (string literals kept as they are)."""
    import re
    pattern = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\])*"', re.S)
    text = pattern.sub(lambda m: m.group(0) if m.group(0).startswith('"') else "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash():
    """First 16 hex digits of a SHA-256 over the kernel sources and the public header with
    comments removed, so a DRAM traffic figure taken by ncu can be matched to the code it
    was measured on (a change to comments alone keeps the hash)."""
    import glob
    import hashlib
    files = []
    for pat in ("convolution_forward_implicit_gb300/csrc/*.cu", "convolution_forward_implicit_gb300/csrc/*.cuh",
                "convolution_forward_implicit_gb300/csrc/*.h", "include/*.h"):
        files += glob.glob(os.path.join(ROOT, pat))
    h = hashlib.sha256()
    for f in sorted(files):
        h.update(os.path.relpath(f, ROOT).encode())
        with open(f, encoding="utf-8") as fh:
            h.update(_strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(desc):
    """DRAM bytes per launch (read + write) of the kernel a plan runs, from the `traffic:` lines
    of the committed ncu summaries, or None when none matches the plan and the current sources."""
    cur = kernel_source_hash()
    for f in sorted(os.listdir(os.path.join(ROOT, "profiles"))) if os.path.isdir(os.path.join(ROOT, "profiles")) else []:
        if not f.endswith((".md", ".txt")):
            continue
        with open(os.path.join(ROOT, "profiles", f)) as fh:
            for line in fh:
                if not line.startswith("traffic: "):
                    continue
                parts = line[len("traffic: "):].strip().split(" ", 2)
                if len(parts) == 3 and parts[0] == cur and parts[2] == desc:
                    return int(parts[1])
    return None


TRAFFIC_NOTE = ("DRAM bytes read + written while the kernel runs (ncu dram__bytes_read.sum + dram__bytes_write.sum, "
                "one launch); outputs still in L2 when it ends are written back later and are not in this count")


def roofline_for(lr, ms):
    """Roofline of one layer's kernel: the slower of its compute pipe and HBM bytes."""
    peaks, src = measured_peaks()
    flops = lr.flops
    t_s = ms * 1e-3
    byts = lr.bytes_alg()
    desc = lr.plan.describe()
    hbm = peaks["hbm_gbs"] * 1e9
    if "variant=tc_bf16x3" in desc:
        # fp32 split into three bf16 planes: six bf16 products per useful product
        pipe = peaks["bf16_tflops"] / 6.0 * 1e12
        bound_c, unit_peak = "tensor", peaks["bf16_tflops"] / 6.0
        note = f"bf16 dense tensor peak ({src}) / 6 plane products per useful product"
    elif "variant=tc_bf16" in desc:
        pipe = peaks["bf16_tflops"] * 1e12
        bound_c, unit_peak = "tensor", peaks["bf16_tflops"]
        note = f"bf16 dense tensor peak, burst, {src}"
    elif "variant=tc_tf32x3" in desc:
        # TF32 peak = measured bf16 peak x nominal TF32/bf16 (1.1/2.25 PFLOP/s); 3xTF32 issues three
        # TF32 products per useful product, so the useful-flop peak is a third of that
        tf32 = peaks["bf16_tflops"] * (1.1 / 2.25)
        pipe = tf32 / 3.0 * 1e12
        bound_c, unit_peak = "tensor", tf32 / 3.0
        note = f"TF32 dense peak (bf16 {src} x 1.1/2.25) / 3 products per useful product"
    else:
        pipe = SM_COUNT * FFMA_PER_SM_PER_CLK * 2 * SM_MAX_MHZ * 1e6
        bound_c, unit_peak = "alu", pipe / 1e12
        note = "FFMA peak = 152 SMs x 128 fp32 lanes x 2 flop x 2070 MHz (derived)"
    if flops / pipe >= byts / hbm:
        ach = flops / t_s / 1e12
        return {"bound": bound_c, "achieved": round(ach, 4), "peak": round(unit_peak, 2), "unit": "TFLOP/s",
                "frac": round(ach / unit_peak, 4), "traffic": measured_traffic(desc), "traffic_note": TRAFFIC_NOTE,
                "kernel": lr.name(), "plan": desc, "peak_source": note, "algorithmic_flops": flops,
                "algorithmic_bytes": byts}
    ach = byts / t_s / 1e9
    return {"bound": "hbm", "achieved": round(ach, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": measured_traffic(desc), "traffic_note": TRAFFIC_NOTE,
            "kernel": lr.name(), "plan": desc,
            "peak_source": f"HBM copy bandwidth, {src}", "algorithmic_flops": flops, "algorithmic_bytes": byts}


# ----------------------------------------------------------------------------- CPU oracle
def _oracle_layer_sample(wl, layer, x, w, b, nthreads, frac, seed):
    """Time the oracle on a random sample of one layer's output pixels (a fraction frac, at
    least one per thread; every output channel of each sampled pixel, so the sample's rate
    does not depend on its density: a pixel's receptive field is read once for all its
    channels), split over nthreads host threads.  Returns (seconds, useful flops)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    from convolution_forward_implicit_gb300 import synthetic as syn
    from convolution_forward_implicit_gb300.binding import CONV_EPI_BIAS, CONV_EPI_BIAS_GELU, CONV_EPI_GELU
    g = oracle.Geom(layer.N, layer.G, layer.C, layer.K, layer.spatial, layer.filter, layer.stride, layer.pad,
                    layer.dilation)
    gelu = layer.epilogue in (CONV_EPI_BIAS_GELU, CONV_EPI_GELU)
    xf, wf = syn.as_f32(x, wl.dtype), syn.as_f32(w, wl.dtype)
    bf = syn.as_f32(b, wl.dtype) if (b is not None and layer.epilogue in (CONV_EPI_BIAS, CONV_EPI_BIAS_GELU)) else None
    shape = g.y_shape()
    pix_total, per = int(np.prod(shape[:4])), int(shape[4] * shape[5])
    npix = min(pix_total, max(nthreads, int(pix_total * frac)))
    pix = np.sort(np.random.default_rng(seed).choice(pix_total, size=npix, replace=False))
    pc = np.array(np.unravel_index(pix, shape[:4])).T.astype(np.int64)
    gk = np.array(np.unravel_index(np.arange(per), shape[4:])).T.astype(np.int64)
    chunks = [np.concatenate([np.repeat(c, per, axis=0), np.tile(gk, (len(c), 1))], axis=1)
              for c in np.array_split(pc, nthreads) if len(c)]
    n = npix * per
    t = time.perf_counter()
    with ThreadPoolExecutor(len(chunks)) as ex:
        list(ex.map(lambda c: oracle.conv_fwd_points(g, xf, wf, bf, gelu, c), chunks))
    return time.perf_counter() - t, 2.0 * layer.C * layer.taps * n


def oracle_inputs(wls):
    """(workload, layer, x, w, bias) of every layer; layers after the first read a fresh
    N(0,1) draw (the oracle's speed does not depend on the values)."""
    from convolution_forward_implicit_gb300 import synthetic as syn
    from convolution_forward_implicit_gb300.workloads import gen_inputs
    data = []
    for wl in wls:
        x, params = gen_inputs(wl)
        for li, layer in enumerate(wl.layers):
            xin = x if li == 0 else syn.gen_normal(7 + li, layer.x_shape(), wl.dtype)
            data.append((wl, layer, xin, params[li][0], params[li][1]))
    return data


def oracle_step_flops(data):
    import oracle
    total = 0.0
    for (wl, layer, _, _, _) in data:
        g = oracle.Geom(layer.N, layer.G, layer.C, layer.K, layer.spatial, layer.filter, layer.stride, layer.pad,
                        layer.dilation)
        total += 2.0 * g.macs()
    return total


def oracle_sample(data, frac, seed, nthreads):
    """The one CPU-baseline method, used by the cpu_baseline field and by --impl reference:
    the oracle as it stands on a random fraction frac of every layer's outputs, each layer's
    sample split evenly over nthreads threads.  Returns (seconds, useful flops)."""
    secs, flops = 0.0, 0.0
    for li, (wl, layer, x, w, b) in enumerate(data):
        dt, fl = _oracle_layer_sample(wl, layer, x, w, b, nthreads, frac, seed * 100 + li)
        secs += dt
        flops += fl
    return secs, flops


CPU_BASELINE_FLOPS = 150e9      # the cpu_baseline sample: ~5-15 s on 16 cores
REFERENCE_STEP_FLOPS = 3e9      # the least one --impl reference step evaluates


def cpu_baseline(wls):
    """The oracle timed on the host cores, on a bounded random sample of the workload's
    outputs (the method of --impl reference, with a larger sample)."""
    data = oracle_inputs(wls)
    nthreads = os.cpu_count() or 1
    frac = min(1.0, CPU_BASELINE_FLOPS / oracle_step_flops(data))
    secs, flops = oracle_sample(data, frac, 0, nthreads)
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
            "sample": f"every output channel of a random {frac:.2%} of every layer's output pixels, split over "
                      f"{nthreads} threads (fp64 direct loops; the method of --impl reference): {flops / 1e9:.2f} "
                      f"GFLOP in {secs:.2f} s"}


def cpu_baseline_bwd(wls, budget_flops=4e9):
    """The backward oracle on the host cores: a random sample of dx and dw elements of every
    layer (about budget_flops of useful work in all), split over threads."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    from convolution_forward_implicit_gb300 import synthetic as syn
    from convolution_forward_implicit_gb300.workloads import gen_inputs
    nthreads = os.cpu_count() or 1
    total_flops = sum(2.0 * int(np.prod(np_y_shape(l))) * l.C * l.taps for wl in wls for l in wl.layers) * 2
    frac = min(1.0, budget_flops / total_flops)
    secs, flops = 0.0, 0.0
    for wl in wls:
        x0, params = gen_inputs(wl)
        for li, layer in enumerate(wl.layers):
            g = oracle.Geom(layer.N, layer.G, layer.C, layer.K, layer.spatial, layer.filter, layer.stride,
                            layer.pad, layer.dilation)
            w, _ = params[li]
            x = syn.as_f32(x0 if li == 0 else syn.gen_normal(7 + li, layer.x_shape(), wl.dtype), wl.dtype)
            dy = syn.as_f32(syn.gen_normal(3 + li, g.y_shape(), wl.dtype), wl.dtype)
            wf = syn.as_f32(w, wl.dtype)
            layer_flops = 2.0 * int(np.prod(g.y_shape())) * layer.C * layer.taps
            for weight, shape, a, b in ((False, g.x_shape(), dy, wf), (True, g.w_shape(), x, dy)):
                total = int(np.prod(shape))
                n = max(nthreads, int(total * frac))
                n = min(n, total)
                idx = np.random.default_rng(li).choice(total, size=n, replace=False)
                coords = np.array(np.unravel_index(idx, shape)).T.astype(np.int64)
                chunks = np.array_split(coords, nthreads)
                t = time.perf_counter()
                with ThreadPoolExecutor(nthreads) as ex:
                    list(ex.map(lambda c: oracle.conv_bwd_points(g, a, b, weight, c), chunks))
                secs += time.perf_counter() - t
                flops += layer_flops * n / total
    return {"value": round(flops / secs / 1e12, 6), "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
            "sample": f"random dx and dw elements of every layer ({frac:.2%} of each), {flops / 1e9:.2f} "
                      f"GFLOP-equivalent in {secs:.2f} s"}


def run_reference(args, ws, rank, local):
    """The oracle as the reference arm: each step evaluates a fresh random sample of each
    layer's output pixels (3-30 GFLOP of useful work per step, ~1.5 TFLOP over the run) on all
    host cores, by the same method and timing as the cpu_baseline field; throughput counts the
    sampled FLOPs."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    wls = frontend_workloads(args.workload)
    nthreads = os.cpu_count() or 1
    data = oracle_inputs(wls)
    # about 1.5 TFLOP over the whole run (~40 s on 16 host cores), 3-30 GFLOP per step
    step_flops = min(30e9, max(REFERENCE_STEP_FLOPS, 1.5e12 / max(1, args.steps + args.warmup)))
    frac = min(1.0, step_flops / oracle_step_flops(data))
    for i in range(args.warmup):
        oracle_sample(data, frac, 1 + i, nthreads)
    # timed like the cpu_baseline field: the oracle calls only (the sample's index arrays are
    # built before each layer's timer starts)
    tot_f, wall = 0.0, 0.0
    for i in range(args.steps):
        dt, f = oracle_sample(data, frac, 1000 + i, nthreads)
        tot_f += f
        wall += dt
    value = tot_f / wall / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(wall / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "+".join(sorted({wl.dtype for wl in wls}, key=lambda d: d != "f32")),
            "data": "synthetic", "config": {"workload": workload_description(args.workload),
                                            "parallelism": "host threads"},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
                             "sample": f"each step: every output channel of a fresh random {frac:.3%} of every "
                                       f"layer's output pixels, split over {nthreads} threads, fp64 direct loops (the "
                                       "cpu_baseline method)"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="sweep_bf16_n32")
    ap.add_argument("--configs", default="all",
                    help="per_config table: 'all' (every configuration the metric is quoted on), 'none', or a "
                         "comma-separated list of workload names")
    ap.add_argument("--source-hash", action="store_true", help="print the kernel source hash and exit")
    ap.add_argument("--no-overlap", dest="overlap", action="store_false",
                    help="launch each layer only after the previous one completes (no programmatic dependents)")
    ap.add_argument("--serial", dest="parallel", action="store_const", const=False, default=None,
                    help="run the step's independent chains one after the other (the forward default)")
    ap.add_argument("--parallel", dest="parallel", action="store_const", const=True,
                    help="capture the step's independent chains as parallel graph branches (the backward default)")
    ap.add_argument("--e2e-serial", action="store_true",
                    help="end-to-end leg: copy in, step, copy out one after the other instead of pipelined")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="fwd: the forward pass of every layer; bwd: backward data and backward weight of every layer")
    ap.add_argument("--tune", type=int, default=0, metavar="ITERS",
                    help="before timing, let the measured selector time every candidate plan of each layer "
                         "(ITERS calls each) and keep the fastest; 0 = the planner's rules")
    args = ap.parse_args()
    if args.source_hash:
        print(kernel_source_hash())
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.parallel is None:
        # measured: forward layers each fill every SM, so concurrent chains only contend (the
        # Whisper step 51.3 -> 54.6 us); the backward step's long FFMA kernels overlap well
        # (207 -> 189 us)
        args.parallel = args.pass_ == "bwd"
    ws, rank, local = dist_setup()
    if ws > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "ours":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    try:
        if args.impl == "reference":
            run_reference(args, ws, rank, local)
        else:
            run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
