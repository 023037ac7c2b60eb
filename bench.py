"""Benchmark: ConvTranspose GFLOP/s and fraction of roofline per call on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-graph]

One step is one forward pass of a workload (input staging, the tensor-core GEMM with its
fused output stage, and for split-K plans the reduce; every layer of a stack, chained), with
the weight packed beforehand as a deployed layer would have it.

With no --workload the headline is the iSTFT overlap-add as a ConvTranspose1d (4 x 4098 ->
1 channel, 343 frames, kernel 4096, hop 1024, fp32 I/O), the largest of the five
configurations, and the line carries a ``per_config`` block that measures every
configuration the same way: the tiny 16 -> 8 layer, the codec upsampler, the iSTFT, the 2-D
decoder layer and the bf16 vocoder stack (chained), plus the iSTFT by inverse FFTs and the
depthwise layer.  --workload NAME measures one workload only.

Timing: W untimed warm-up steps and a short soak, then exactly K steps bracketed by a
barrier and torch.cuda.synchronize() on both sides, between CUDA events on the launching
stream.  The K timed steps are captured once into one CUDA graph of the library's own
launches and replayed between two events; ``us_per_call_plain`` times the same K steps as
plain library calls (an event pair per step, the median reported), which is what a caller
of ctr_forward sees.  The main kernels' own durations (for the roofline) come from a
further replay of the same K steps with an event pair around each of them, because an event
between two kernels would serialise their programmatic launch.  Consecutive steps rotate
over enough sets of input, packed weight, workspace and output buffers to exceed twice the
L2 size, so no step reads data the previous one left in L2.  The "e2e" figure goes through
the plain public call, with each step's host->device and device->host copies on their own
streams overlapping the forward passes of neighbouring steps.  Under torchrun every rank
runs the same workloads on its own GPU (weak scaling, no collective on the data path); rank
0 prints one JSON line with the maximum times over ranks.

--impl reference times the CPU oracle (double precision, OpenMP on the host cores) on a
bounded sample of the same workload: the reference arm of this benchmark.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "ConvTranspose GFLOP/s and % of roofline (tensor peak vs HBM) per call"
HEADLINE = "istft_f32"
# The five configurations (tiny layer, codec upsampler, iSTFT, 2-D decoder, vocoder stack),
# then the two further workloads: the iSTFT by inverse FFTs and the depthwise layer.
CONFIGS = ["tiny_1d_f32", "codec_upsampler_f32", "istft_f32", "decoder_2d_f32",
           "vocoder_stack_bf16"]
EXTRAS = ["istft_irfft_f32", "depthwise_2d_bf16"]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal dense tensor throughput relative to bf16 (tf32 1.1 vs bf16 2.25 PFLOP/s): the tf32
# peak when it could not be measured in this run.
TF32_OVER_BF16 = 1.1 / 2.25
# The sources of each profiled kernel: a committed ncu summary holds their hash, and its
# DRAM traffic is reported only while they are unchanged.
KERNEL_SOURCES = {
    "gemm_tc": ["transposed_convolution_gb300/csrc/gemm_tc.cu",
                "transposed_convolution_gb300/csrc/gemm_tc_f16.cu",
                "transposed_convolution_gb300/csrc/epilogue.cuh",
                "transposed_convolution_gb300/csrc/ptx.cuh",
                "transposed_convolution_gb300/csrc/gemm_tc.cuh",
                "transposed_convolution_gb300/csrc/gemm_tc_chain.cu"],
    "depthwise": ["transposed_convolution_gb300/csrc/depthwise.cu"],
    "istft": ["transposed_convolution_gb300/csrc/istft.cu"],
    "gather": ["transposed_convolution_gb300/csrc/aux_kernels.cu"],
    "fused_pair": ["transposed_convolution_gb300/csrc/fused_pair.cu",
                   "transposed_convolution_gb300/csrc/epilogue.cuh",
                   "transposed_convolution_gb300/csrc/ptx.cuh"],
}


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(kernel="gemm_tc"):
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload, layer=0, layers=1, kernel="gemm_tc"):
    """Bytes moved per launch of a launch group's main kernel from the committed ncu summary:
    DRAM reads plus the sectors the SMs wrote into L2 (each written line reaches DRAM when
    it is evicted; a partly written sector counts whole, so the write term is an upper
    bound).  None when there is no summary or the kernel sources changed since it was
    taken."""
    path = os.path.join(ROOT, "profiles", "%s_%s.md" % (kernel, workload))
    if kernel not in KERNEL_SOURCES or not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != kernel_source_hash(kernel):
        return None
    key = "dram_bytes_per_launch" if layers == 1 else "dram_bytes_per_launch_layer%d" % layer
    try:
        return int(float(vals[key]))
    except (KeyError, ValueError):
        return None


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the CPU-baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock and throttle-reason samples every 200 ms while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = [s for (t, s) in self.samples if t0 <= t <= t1]
        mhz, maxmhz, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                maxmhz.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not mhz:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(maxmhz),
                "reasons": sorted(reasons), "samples": len(mhz)}


# ------------------------------------------------------------------ our arm

def max_over_ranks(values, device, world):
    """Element-wise maximum of a list of floats over all ranks of the default process group
    (the slowest rank sets the job's time)."""
    if world <= 1:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t]


def barrier(world):
    if world > 1:
        import torch
        torch.distributed.barrier()


def aggregate_rate(world, units_per_rank, ms):
    """Whole-job throughput: the units every rank processed in `ms` milliseconds, in units/s
    divided by 1e9 (GFLOP/s for FLOP units)."""
    return world * units_per_rank / (ms / 1e3) / 1e9


def measure_tf32_peak(dev):
    """Dense tf32 tensor throughput of this GPU in TFLOP/s, measured the way the bf16 peak
    is: torch.matmul of two fp32 8192 x 8192 matrices with TF32 allowed, best of 10, CUDA
    events.  None when the measurement fails."""
    import torch
    old = torch.backends.cuda.matmul.allow_tf32
    try:
        torch.backends.cuda.matmul.allow_tf32 = True
        n = 8192
        a = torch.randn(n, n, device=dev)
        b = torch.randn(n, n, device=dev)
        for _ in range(3):
            torch.matmul(a, b)
        torch.cuda.synchronize(dev)
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b)
            e1.record()
            torch.cuda.synchronize(dev)
            best = min(best, e0.elapsed_time(e1))
        del a, b
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / (best / 1e3) / 1e12
    except Exception:
        return None
    finally:
        torch.backends.cuda.matmul.allow_tf32 = old


def layer_peak(L, peaks, peak_src, tf32_tflops):
    """Tensor peak (TFLOP/s of useful MACs x 2) for a layer and where it comes from."""
    if L.dtype == "bf16":
        return peaks["bf16_tflops"], "bf16 dense, %s burst" % peak_src
    # fp32 I/O: every useful MAC costs one tf32 MAC (hi*hi) and two bf16 MACs (the cross
    # products), so the peak is 1 / (1/P_tf32 + 2/P_bf16).
    if tf32_tflops:
        return (split_peak(tf32_tflops, peaks["bf16_tflops"]),
                "fp32 split: 1/(1/P_tf32 + 2/P_bf16), P_tf32 measured in this run "
                "(torch.matmul fp32 8192^3, TF32, best of 10), P_bf16 %s burst" % peak_src)
    return (split_peak(peaks["bf16_tflops"] * TF32_OVER_BF16, peaks["bf16_tflops"]),
            "fp32 split: 1/(1/P_tf32 + 2/P_bf16), P_bf16 %s burst, P_tf32 = P_bf16 x nominal "
            "tf32/bf16 (1.1/2.25)" % peak_src)


def split_peak(p_tf32, p_bf16):
    """Useful-MAC throughput of the fp32 split (one tf32 and two bf16 MACs per MAC)."""
    return 1.0 / (1.0 / p_tf32 + 2.0 / p_bf16)


def measure_workload(name, args, env, headline):
    """Time one workload on this rank's GPU: graph-replayed steps, plain calls, main-kernel
    durations, end to end through the public API, and parity against the oracle.  Returns
    the raw figures (times already the maximum over ranks)."""
    import torch
    import transposed_convolution_gb300 as ctr

    dev, world, rank = env["dev"], env["world"], env["rank"]
    layers = workloads.make_workload(name)
    Ls = [li.layer for li in layers]
    tdts = [torch.bfloat16 if L.dtype == "bf16" else torch.float32 for L in Ls]

    def t(a, tdt):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev).to(tdt)

    l2 = env["l2"]
    w_dev = [t(li.w, tdt) for li, tdt in zip(layers, tdts)]
    b_dev = [t(li.bias, tdt) for li, tdt in zip(layers, tdts)]
    x_dev = t(layers[0].x, tdts[0])

    def make_plans():
        plans = [ctr.Istft(L.B, L.kernel[0], L.stride[0], L.in_sp[0], L.padding[0],
                           L.output_padding[0], device=dev) if L.kind == "istft" else
                 ctr.Plan(L.B, L.C_in, L.C_out, L.in_sp, L.kernel, L.stride, L.padding,
                          L.output_padding, dtype=tdt, negative_slope=L.act_slope, device=dev,
                          groups=L.groups)
                 for L, tdt in zip(Ls, tdts)]
        # A stack of layers runs chained (each layer's output stage writes the next layer's
        # staged input) where the library allows it; --no-chain keeps every tensor in the
        # torch layout.
        for a, b in zip(plans[:-1], plans[1:]):
            if args.chain:
                try:
                    a.chain(b)
                except ctr.CtrError:
                    pass
        return plans

    probe = make_plans()
    set_bytes = x_dev.numel() * Ls[0].elem_bytes
    for p, L in zip(probe, Ls):
        set_bytes += p.packed_bytes + p.workspace_bytes
        if p.next_plan is None:   # a chained layer's y is never written
            set_bytes += int(np.prod(p.out_shape)) * L.elem_bytes
    # Launch groups: a chained pair the library can run as one kernel (ctr_forward_fused)
    # runs fused unless --no-fuse; every other layer is a group of its own.
    groups, i = [], 0
    while i < len(probe):
        p = probe[i]
        if (args.fuse and p.next_plan is not None and i + 1 < len(probe)
                and p.next_plan is probe[i + 1] and p.fusable):
            groups.append((i, i + 1))
            i += 2
        else:
            groups.append((i,))
            i += 1
    for p in probe:
        p.close()
    nsets = max(2, int(math.ceil(2.0 * l2 / set_bytes)) + 1)
    sets = []
    for _ in range(nsets):
        plans = make_plans()
        for p, w in zip(plans, w_dev):
            p.prepack(w)
        ys = [torch.empty(p.out_shape, dtype=tdt, device=dev) for p, tdt in zip(plans, tdts)]
        sets.append({"plans": plans, "x": x_dev.clone(), "y": ys,
                     "b": [None if b is None else b.clone() for b in b_dev]})
    torch.cuda.synchronize()

    # Prepack time of the whole workload (reported separately; not part of a step).
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for p, w in zip(sets[0]["plans"], w_dev):
        p.prepack(w)
    e1.record()
    torch.cuda.synchronize()
    prepack_ms = e0.elapsed_time(e1)

    def run_set(s, x=None, kevs=None):
        inp = s["x"] if x is None else x
        for gi, grp in enumerate(groups):
            li_idx = grp[0]
            p = s["plans"][li_idx]
            if kevs is not None:
                p.set_timing_events(kevs[gi][0].cuda_event, kevs[gi][1].cuda_event)
            if len(grp) == 2:
                last = grp[1]
                nxt = s["plans"][last]
                if nxt.next_plan is not None:
                    raise RuntimeError("a fused pair ends a chain")
                p.forward_fused(inp, s["b"][li_idx], s["b"][last], y=s["y"][last])
                inp = s["y"][last]
            elif p.next_plan is not None:
                p.forward(inp, s["b"][li_idx])
                inp = None
            else:
                p.forward(inp, s["b"][li_idx], y=s["y"][li_idx])
                inp = s["y"][li_idx]
            if kevs is not None:
                p.set_timing_events(None, None)
        return inp

    for i in range(args.warmup):
        run_set(sets[i % nsets])
    torch.cuda.synchronize()
    for s in sets:
        for p in s["plans"]:
            p.check()

    K = args.steps
    nl = len(groups)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    kev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(nl)] for _ in range(K)]
    for row in kev:       # create the driver events before handing them to the library
        for a, b in row:
            a.record()
            b.record()
    torch.cuda.synchronize()

    # The K steps (rotating over the buffer sets) captured once, untimed, into one CUDA graph
    # of the library's launches (and again with each main kernel between its own events,
    # recorded as external event nodes).
    launches0 = ctr.ctr_launch_count()
    graph = graph_k = None
    launches = 0
    if args.graph:
        cap = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cap):
            for k in range(K):
                run_set(sets[k % nsets])
        launches = ctr.ctr_launch_count() - launches0
        graph_k = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_k, stream=cap):
            for k in range(K):
                run_set(sets[k % nsets], kevs=kev[k])
        graph.replay()            # first replays upload the graphs (untimed)
        graph_k.replay()
        torch.cuda.synchronize()

    def plain_steps(kernel_events=False):
        for k in range(K):
            if not kernel_events:
                ev[k][0].record()
            run_set(sets[k % nsets], kevs=kev[k] if kernel_events else None)
            if not kernel_events:
                ev[k][1].record()

    soak = args.soak if headline else min(args.soak, 0.3)
    soak_t0 = time.time()
    while time.time() - soak_t0 < soak:
        if graph is not None:
            graph.replay()
        else:
            plain_steps()
        torch.cuda.synchronize()

    # Timed region: exactly K steps.
    barrier(world)
    torch.cuda.synchronize()
    launches0 = ctr.ctr_launch_count()
    t_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    wall0 = time.time()
    t_ev[0].record()
    if graph is not None:
        graph.replay()
    else:
        plain_steps()
    t_ev[1].record()
    torch.cuda.synchronize()
    wall1 = time.time()
    if graph is None:
        launches = ctr.ctr_launch_count() - launches0
    barrier(world)
    total_ms = t_ev[0].elapsed_time(t_ev[1])
    # Plain calls: the same K steps without the graph, an event pair per step.
    if graph is not None:
        plain_steps()
        torch.cuda.synchronize()
    plain_ms = sorted(a.elapsed_time(b) for a, b in ev)
    plain_median = plain_ms[len(plain_ms) // 2]
    barrier(world)
    # Kernel durations: the same K steps again, each main kernel between its own events.
    if graph_k is not None:
        graph_k.replay()
    else:
        plain_steps(kernel_events=True)
    torch.cuda.synchronize()
    barrier(world)
    for s in sets:
        for p in s["plans"]:
            p.check()
    kern_ms = [sum(kev[k][j][0].elapsed_time(kev[k][j][1]) for k in range(K)) / K
               for j in range(nl)]
    total_ms, plain_median, *kern_ms = max_over_ranks([total_ms, plain_median] + kern_ms,
                                                       dev, world)

    # End to end through the public API, as a streaming caller runs it: every step copies
    # its x from pinned host memory, runs the forward passes (Plan.forward, no graph) and
    # copies its y back to pinned host memory.  The copies run on their own streams, so step
    # k's upload and step k-1's download overlap the forward passes; events order each
    # buffer's reuse (a set's x is overwritten only after its previous forward read it, its
    # y only after its previous download).  Time per step = whole run / steps.
    n_e2e = max(3, min(K, 50 if headline else 20))
    x_hosts = [torch.from_numpy(np.ascontiguousarray(layers[0].x)).to(tdts[0]).pin_memory()
               for _ in range(2)]
    y_hosts = [torch.empty(sets[0]["y"][-1].shape, dtype=tdts[-1]).pin_memory() for _ in range(2)]
    main_stream = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(n_e2e)]
    ev_done = [torch.cuda.Event() for _ in range(n_e2e)]
    ev_out = [torch.cuda.Event() for _ in range(n_e2e)]
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(main_stream)
    s_in.wait_event(e_start)
    for k in range(n_e2e):
        s = sets[k % nsets]
        with torch.cuda.stream(s_in):
            if k >= nsets:
                s_in.wait_event(ev_done[k - nsets])      # that set's x no longer read
            s["x"].copy_(x_hosts[k % 2], non_blocking=True)
            ev_in[k].record(s_in)
        main_stream.wait_event(ev_in[k])
        if k >= nsets:
            main_stream.wait_event(ev_out[k - nsets])    # that set's y already downloaded
        out = run_set(s)
        ev_done[k].record(main_stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[k])
            y_hosts[k % 2].copy_(out, non_blocking=True)
            ev_out[k].record(s_out)
    main_stream.wait_event(ev_out[n_e2e - 1])
    e_end.record(main_stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks([e_start.elapsed_time(e_end) / n_e2e], dev, world)[0]

    # Parity of this run's output against the oracle, layer by layer (computed after
    # timing).  An unchained layer takes the library's own previous output as input; through
    # a chain (no intermediate y) the oracle carries on from its own output rounded to the
    # I/O type, and the chain's last layer is compared.
    parity = None
    if rank == 0 and args.parity:
        import oracle
        s = sets[(K - 1) % nsets]
        xin = layers[0].x
        errs = []
        for j, (li, L) in enumerate(zip(layers, Ls)):
            ref = oracle.conv_transpose(xin, oracle_weight(li), li.bias, L.stride, L.padding,
                                        L.output_padding, groups=L.groups)
            if L.act_slope is not None:
                ref = oracle.leaky_relu(ref, L.act_slope)
            if s["plans"][j].next_plan is not None:
                xin = oracle.round_bf16(ref) if L.dtype == "bf16" else oracle.round_f32(ref)
                continue
            got = s["y"][j].float().cpu().numpy()
            errs.append(oracle.rel_l2(got, ref))
            xin = got
        parity = max(errs)

    paths = [sets[0]["plans"][g[0]].path for g in groups]
    describe = [p.describe() for p in sets[0]["plans"]]
    chained = sum(p.next_plan is not None for p in sets[0]["plans"])
    h2d = int(x_hosts[0].numel() * x_hosts[0].element_size())
    d2h = int(y_hosts[0].numel() * y_hosts[0].element_size())
    for s in sets:
        for p in s["plans"]:
            p.close()
    del sets, w_dev, b_dev, x_dev, x_hosts, y_hosts
    graph = graph_k = None
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return {
        "name": name, "Ls": Ls, "K": K, "ms_per_step": total_ms / K,
        "plain_ms": plain_median, "kern_ms": kern_ms, "e2e_ms": e2e_ms, "n_e2e": n_e2e,
        "h2d": h2d, "d2h": d2h, "parity": parity, "paths": paths, "describe": describe,
        "chained": chained, "nsets": nsets, "set_bytes": set_bytes, "prepack_ms": prepack_ms,
        "groups": groups,
        "launches": int(launches), "window": (soak_t0, wall1), "wall_timed": wall1 - wall0,
    }


def summarize(m, env):
    """Roofline, GFLOP/s and kernel figures of one measured workload."""
    import transposed_convolution_gb300 as ctr
    peaks, peak_src, tf32 = env["peaks"], env["peak_src"], env["tf32_tflops"]
    Ls = m["Ls"]
    is_fft = any(L.kind == "istft" for L in Ls)
    flops = sum(2.0 * L.useful_macs for L in Ls)
    bytes_c = sum(L.compulsory_bytes for L in Ls)
    step_s = m["ms_per_step"] / 1e3

    def t_tensor(L, pk):
        # The FFT path's arithmetic is far below the dense contraction it replaces: bytes only.
        return 0.0 if L.kind == "istft" else 2.0 * L.useful_macs / (pk * 1e12)

    t_roof = 0.0
    for L in Ls:
        pk, _ = layer_peak(L, peaks, peak_src, tf32)
        t_roof += max(t_tensor(L, pk), L.compulsory_bytes / (peaks["hbm_gbs"] * 1e9))
    # The dominant launch group (one kernel: a layer, or a fused pair of layers).  A fused
    # pair's algorithmic bytes are its first layer's input, both weights and biases and its
    # last layer's output: the intermediate is not moved.
    groups = m["groups"]
    j = max(range(len(groups)), key=lambda q: m["kern_ms"][q])
    grp = groups[j]
    L = Ls[grp[0]]
    g_layers = [Ls[i] for i in grp]
    g_macs = sum(x.useful_macs for x in g_layers)
    g_bytes = (sum(x.compulsory_bytes for x in g_layers)
               - sum(x.out_bytes for x in g_layers[:-1]) - sum(x.in_bytes for x in g_layers[1:]))
    pk, peak_note = layer_peak(L, peaks, peak_src, tf32)
    tt = 0.0 if L.kind == "istft" else 2.0 * g_macs / (pk * 1e12)
    th = g_bytes / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if tt >= th else "hbm"
    kern_s = m["kern_ms"][j] / 1e3
    if bound == "tensor":
        achieved, peak, unit = 2.0 * g_macs / kern_s / 1e12, pk, "TFLOP/s"
        nominal = (split_peak(peaks["bf16_tflops"] * TF32_OVER_BF16, peaks["bf16_tflops"])
                   if L.dtype == "f32" else pk)
    else:
        achieved, peak, unit = g_bytes / kern_s / 1e9, peaks["hbm_gbs"], "GB/s"
        peak_note = "HBM copy bandwidth, %s" % peak_src
        nominal = peak
    path = m["paths"][j]
    kname = {ctr.CTR_PATH_GATHER: "gather_kernel", ctr.CTR_PATH_DEPTHWISE: "depthwise_kernel",
             -1: "spectrum_rows_kernel+irfft_frames_kernel+istft_ola_kernel"}.get(
                 path, "gemm_tc_kernel")
    kfile = {ctr.CTR_PATH_GATHER: "gather", ctr.CTR_PATH_DEPTHWISE: "depthwise",
             -1: "istft"}.get(path, "gemm_tc")
    if len(grp) > 1:
        kfile = "fused_pair"
    traffic = profiled_traffic(m["name"], j, len(groups), kfile)
    roof = {"bound": bound, "achieved": round(achieved, 2), "peak": round(peak, 2),
            "unit": unit, "frac": round(achieved / peak, 4), "traffic": traffic,
            "kernel": kname if len(grp) == 1 else "fused_pair_kernel",
            "layer": list(grp) if len(grp) > 1 else grp[0],
            "kernel_us": round(m["kern_ms"][j] * 1e3, 3),
            "peak_source": peak_note + (", of measured" if peak_src == "measured" else
                                        ", of fallback")}
    if bound == "tensor" and L.dtype == "f32":
        roof["frac_vs_nominal_tf32_ratio"] = round(achieved / nominal, 4)
    out = {
        "us_per_call": round(m["ms_per_step"] * 1e3, 3),
        "us_per_call_plain": round(m["plain_ms"] * 1e3, 3),
        "gflops": None if is_fft else round(flops / step_s / 1e9, 1),
        "pct_of_roofline": round(100.0 * t_roof / step_s, 2),
        "roofline_us": round(t_roof * 1e6, 3),
        "roofline": roof,
        "layer_kernel_us": [round(v * 1e3, 3) for v in m["kern_ms"]],
        "launch_groups": [list(g) for g in groups],
        "parity_rel_l2": m["parity"],
        "parity_tolerance": 1e-2 if Ls[-1].dtype == "bf16" else 1e-5,
        "e2e_us_per_call": round(m["e2e_ms"] * 1e3, 3),
        "prepack_us": round(m["prepack_ms"] * 1e3, 2),
        "launches_per_step": m["launches"] / m["K"],
        "shape": "; ".join(x.describe() for x in Ls),
        "plan": " | ".join(m["describe"]),
    }
    if is_fft:
        out["hbm_frac_step"] = round(bytes_c / step_s / 1e9 / peaks["hbm_gbs"], 4)
        out["note"] = ("inverse real FFTs: the dense contraction's flops are not performed, so "
                       "no GFLOP/s; the roofline is the compulsory bytes at the HBM bandwidth")
    if m["chained"]:
        out["chained_layers"] = m["chained"]
    return out, flops, bytes_c


# ------------------------------------------------------------------ oracle (CPU) arm

def oracle_weight(li):
    """The ConvTranspose weight the oracle takes: the layer's own, or for an inverse-FFT
    layer the windowed inverse real-DFT basis its window implies."""
    L = li.layer
    return workloads.istft_basis(L.kernel[0], li.w) if L.kind == "istft" else li.w


def _oracle_call(x, li, w):
    import oracle
    L = li.layer
    oracle.conv_transpose(x, w, li.bias, L.stride, L.padding, L.output_padding, groups=L.groups)


def oracle_sample(name, budget_s, start_len=None):
    """A bounded sample of the workload for the oracle: its first layer on a prefix of the
    input positions (all of them when one call fits budget_s / 3 seconds).  Returns (seconds
    per call, useful flops per call, sample description, (x, layer inputs, weight))."""
    li = workloads.make_workload(name)[0]
    L = li.layer
    w = oracle_weight(li)
    x = li.x
    if start_len is not None and start_len < x.shape[-1]:
        x = x[..., : max(8, int(start_len))]
    for _ in range(16):
        t0 = time.time()
        _oracle_call(x, li, w)
        dt = time.time() - t0
        if dt <= budget_s / 3 or x.shape[-1] <= 8:
            break
        x = x[..., : max(8, x.shape[-1] // 2)]
    desc = ("first layer, " if len(workloads.WORKLOADS[name]) > 1 else "") + (
        "full layer" if x.shape[-1] == L.in_sp[-1]
        else "input prefix %d of %d positions" % (x.shape[-1], L.in_sp[-1]))
    macs = L.B * L.C_in * (L.C_out // L.groups) * int(np.prod(L.kernel))
    macs *= int(np.prod(x.shape[2:]))
    return dt, 2.0 * macs, desc, (x, li, w)


def time_oracle(name, budget_s, threads=0, start_len=None):
    """Oracle GFLOP/s on a bounded sample of the workload (threads <= 0: all host cores)."""
    import oracle
    oracle.set_threads(threads)
    try:
        dt, flops, desc, (x, li, w) = oracle_sample(name, budget_s, start_len)
        reps, total = 0, 0.0
        while total < budget_s and reps < 50:
            t0 = time.time()
            _oracle_call(x, li, w)
            total += time.time() - t0
            reps += 1
        sec = total / reps
        return {"value": round(flops / sec / 1e9, 3), "unit": "GFLOP/s",
                "cores": oracle.threads(), "kind": "oracle",
                "sample": "%s of %s, %d calls, %.3f s each" % (desc, name, reps, sec),
                "sample_len": int(x.shape[-1]), "sec_per_call": sec}
    finally:
        oracle.set_threads(0)


def cpu_baseline(name, budget_s):
    """The oracle on all host cores and on one core, with the host's core count and CPU."""
    allc = time_oracle(name, budget_s)
    # One core takes about `cores` times longer: start from a prefix that keeps a call
    # within a third of the budget.
    shrink = allc["sec_per_call"] * allc["cores"] / (budget_s / 3)
    start = allc["sample_len"] if shrink <= 1 else max(8, int(allc["sample_len"] / shrink))
    one = time_oracle(name, budget_s, threads=1, start_len=start)
    out = {k: allc[k] for k in ("value", "unit", "cores", "kind", "sample")}
    out["one_core"] = {k: one[k] for k in ("value", "unit", "cores", "sample")}
    out["nproc"] = os.cpu_count()
    out["cpu_model"] = cpu_model()
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return None
    K, W = args.steps, args.warmup
    name = args.workload or HEADLINE
    _, flops, desc, (x, li, w) = oracle_sample(name, 8.0)
    L = li.layer
    for _ in range(min(W, 1)):
        _oracle_call(x, li, w)
    times = []
    for _ in range(K):
        t0 = time.time()
        _oracle_call(x, li, w)
        times.append(time.time() - t0)
        if sum(times) > 120:
            break
    sec = sum(times) / len(times)
    v = round(flops / sec / 1e9, 3)
    import oracle
    return {
        "impl": "reference", "metric": METRIC,
        "value": v, "unit": "GFLOP/s", "n_gpus": world, "steps": len(times), "warmup": W,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded; workloads.py)",
        "config": {"workload": name, "shape": L.describe(), "sample": desc},
        "cpu_baseline": {"value": v, "unit": "GFLOP/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": desc, "nproc": os.cpu_count(),
                         "cpu_model": cpu_model()},
        "e2e": {"value": v, "unit": "GFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ main

def run_ours(args, rank, world, local_rank):
    import torch
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    props = torch.cuda.get_device_properties(dev)
    peaks, peak_src = load_peaks()
    env = {"dev": dev, "world": world, "rank": rank,
           "l2": getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20,
           "peaks": peaks, "peak_src": peak_src}
    names = [args.workload] if args.workload else CONFIGS + EXTRAS
    head = args.workload or HEADLINE
    env["tf32_tflops"] = (measure_tf32_peak(dev)
                          if any(L.dtype == "f32" for n in names
                                 for L in workloads.WORKLOADS[n]) else None)
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    measured = {}
    # The headline first (with the full soak), then every other workload.
    for name in [head] + [n for n in names if n != head]:
        measured[name] = measure_workload(name, args, env, headline=(name == head))
    time.sleep(0.25)
    sampler.stop()

    m = measured[head]
    summ, flops, bytes_c = summarize(m, env)
    Ls = m["Ls"]
    clocks = sampler.summary(*m["window"])
    result = {
        "metric": METRIC,
        "value": round(aggregate_rate(world, flops, m["ms_per_step"]), 1),
        "unit": "GFLOP/s",
        "n_gpus": world,
        "steps": m["K"],
        "warmup": args.warmup,
        "ms_per_step": round(m["ms_per_step"], 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32 I/O, tf32 + bf16 split products, fp32 accumulate" if Ls[0].dtype == "f32"
                 else "bf16 I/O, bf16 products, fp32 accumulate",
        "data": "synthetic (seeded; workloads.py)",
        "config": {"workload": head, "shape": summ["shape"],
                   "l2": "rotating %d buffer sets, %.0f MB > 2x L2 (%.0f MB)"
                         % (m["nsets"], m["nsets"] * m["set_bytes"] / 1e6, env["l2"] / 1e6),
                   "parallelism": "replica per GPU" if world > 1 else "single GPU",
                   "chained_layers": m["chained"],
                   "launch": ("one CUDA graph of the K steps" if args.graph else "plain calls")
                             + "; kernel times from a further K-step run",
                   "plan": summ["plan"]},
        "us_per_call": summ["us_per_call"],
        "us_per_call_plain": summ["us_per_call_plain"],
        "pct_of_roofline": summ["pct_of_roofline"],
        "roofline_us": summ["roofline_us"],
        "roofline": summ["roofline"],
        "layer_kernel_us": summ["layer_kernel_us"],
        "e2e": {"value": round(aggregate_rate(world, flops, m["e2e_ms"]), 1), "unit": "GFLOP/s",
                "h2d_bytes_per_step": m["h2d"], "d2h_bytes_per_step": m["d2h"],
                "ms_per_step": round(m["e2e_ms"], 5), "steps": m["n_e2e"],
                "copies": "own streams, overlapping the forward passes"},
        "gpu_launches": m["launches"],
        "launches_per_step": m["launches"] / m["K"],
        "clocks": clocks,
        "prepack_ms": round(m["prepack_ms"], 4),
        "parity_rel_l2": m["parity"],
        "compulsory_bytes": bytes_c,
        "wall_s_timed": round(m["wall_timed"], 4),
        "tf32_tflops_measured": (round(env["tf32_tflops"], 1) if env["tf32_tflops"] else None),
    }
    if len(measured) > 1:
        per = {}
        for name in names:
            s, _, _ = summarize(measured[name], env)
            s["clocks"] = sampler.summary(*measured[name]["window"])
            per[name] = s
        result["per_config"] = per
    return result


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, choices=workloads.WORKLOAD_ORDER,
                    help="measure one workload only (default: the iSTFT headline plus every "
                         "configuration in per_config)")
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of untimed load before timing")
    ap.add_argument("--no-parity", dest="parity", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-chain", dest="chain", action="store_false",
                    help="run a stack's layers unchained (every intermediate in torch layout)")
    ap.add_argument("--no-fuse", dest="fuse", action="store_false",
                    help="run a fusable chained pair as two launches instead of one")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="time plain library calls instead of CUDA-graph replays of them")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return

    if world > 1:
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend=backend)
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if args.cpu_baseline and world == 1:
            head = args.workload or HEADLINE
            res["cpu_baseline"] = cpu_baseline(head, 6.0)
            for name, entry in res.get("per_config", {}).items():
                entry["cpu_baseline"] = (res["cpu_baseline"] if name == head
                                         else cpu_baseline(name, 2.0))
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
