"""Benchmark of the deformable convolution forward pass on GB300.

One step = one full forward pass through dcn_forward (weight pack + fused
sampling/contraction/epilogue kernel) over the 7x7, C = O = 64, 256 x 256
ASPP workload, inputs already resident in device memory.  The fused kernel
alone is timed in a second loop (dcn_pack_weight and dcn_forward_packed
with events between them) for the roofline figures.  L2 is flushed (a 256 MiB write, twice
the 129 MB L2) before every step, outside the timed events.  Every step is
timed with CUDA events on the stream the kernels run on; ms_per_step is
the mean, the maximum over ranks when several run (weak scaling: every rank
runs the same workload, no collective on the data path).

Also reported, outside the headline value: the same call without the L2
flush (warm_l2_mean), the host-buffer entry end to end (e2e), the backward
pass, the MSDA forward and backward, single-scale deformable sampling
(DCNv3) forward and backward, and the forward on the decoder 3x3, backbone 3x3 and boundary 5x5
configurations (other_configs).

Prints one JSON line.  --impl reference times the CPU oracle instead.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "deform-conv fwd effective TFLOP/s & out-pixels/s on 1 GB300; % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
L2_NOTE = f"flushed before every step ({L2_FLUSH_BYTES >> 20} MiB write), outside the timed events"
MAIN_KERNEL = "dcn_tc_kernel"
TC_SOURCES = ["dcn_tc.cu", "dcn_device.cuh", "dcn_sampling.cuh", "dcn_kernels.h"]


# ----------------------------------------------------------- host helpers

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def reduce_max(value, world):
    """Maximum of a float over all ranks (identity for one rank)."""
    if world == 1:
        return float(value)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, max_seconds):
    """Weak scaling: every rank processes units_per_rank; the job's rate is
    all units over the slowest rank's time."""
    return units_per_rank * world / max_seconds


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured (MEASURED_PEAKS.json)"
    return dict(FALLBACK_PEAKS), "fallback (profiling recipe)"


def algorithmic_bytes(wl):
    """x, offset, mask, weight, bias and out, each moved once."""
    es = 2 if wl.dtype == "bf16" else 4
    return (wl.B * wl.H * wl.W * wl.C * es + wl.B * 2 * wl.taps * wl.Ho * wl.Wo * 4
            + (wl.B * wl.taps * wl.Ho * wl.Wo * 4 if wl.mask != "none" else 0)
            + wl.O * wl.C * wl.taps * es + (wl.O * 4 if wl.bias_std > 0 else 0)
            + wl.pixels * wl.O * es)


def tc_source_hash():
    h = hashlib.sha256()
    for name in TC_SOURCES:
        with open(os.path.join(ROOT, "deformable_convolution_vision_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def dram_traffic(workload):
    """DRAM bytes per launch of the main kernel from the committed ncu
    summary, or None if none was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        d = json.load(fh)
    e = d.get(workload)
    if not e or e.get("source_hash") != tc_source_hash():
        return None
    return float(e["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.device_index = device_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.device_index), "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, flag in zip(names, r[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- CPU oracle

def time_oracle(wl, inp, seconds, seed=0):
    """Run the oracle on batches of random output pixels (all O channels each)
    until `seconds` have passed.  Returns (pixels, elapsed s, threads)."""
    import numpy as np
    import oracle
    orc = oracle.get()
    threads = orc.max_threads()
    rng = np.random.default_rng(seed)
    batch = max(threads * 4, 16)
    done, t0 = 0, time.perf_counter()
    while True:
        flat = rng.integers(0, wl.pixels, size=batch)
        pts = np.stack([flat // (wl.Ho * wl.Wo), (flat // wl.Wo) % wl.Ho, flat % wl.Wo], 1)
        orc.forward_points(inp["x"], inp["offset"], inp["mask"], inp["weight"], inp["bias"],
                           wl.pad, pts)
        done += batch
        el = time.perf_counter() - t0
        if el >= seconds:
            return done, el, threads


def cpu_baseline(wl, inp, seconds):
    px, el, threads = time_oracle(wl, inp, seconds)
    flops = 2.0 * px * wl.O * wl.taps * wl.C
    return {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{px} random output pixels x all {wl.O} channels of {wl.name} "
                      f"({el:.1f} s, fp64 C oracle, OpenMP over pixels)",
            "out_pixels_per_s": px / el}


# ------------------------------------------------------------------- arms

def reference_step_seconds(args):
    """Oracle seconds per reference step: each step is a sample of the
    workload sized so that the whole run (warm-up steps at a quarter of a
    step) stays within the budget -- at most reference_step_seconds a step,
    less when there are many steps."""
    return min(args.reference_step_seconds,
               args.reference_budget_seconds / max(args.steps + 0.25 * args.warmup, 1.0))


def run_reference(args, wl, rank, world):
    """The oracle, timed on the host cores: each step is a bounded sample."""
    if rank != 0:
        return
    from deformable_convolution_vision_gb300.inputs import make_inputs
    inp = make_inputs(wl)
    per_step = reference_step_seconds(args)
    for _ in range(args.warmup):
        time_oracle(wl, inp, per_step * 0.25)
    steps = []
    for k in range(args.steps):
        px, el, threads = time_oracle(wl, inp, per_step, seed=k + 1)
        steps.append((px, el))
    px = sum(s[0] for s in steps)
    el = sum(s[1] for s in steps)
    flops = 2.0 * px * wl.O * wl.taps * wl.C
    value = flops / el / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        # the same workload description as the GPU arm (the oracle runs on
        # the host; the flush note of the GPU arm does not apply to it)
        "config": config_dict(wl, L2_NOTE),
        "out_pixels_per_s": px / el,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{px} random output pixels x all {wl.O} channels over "
                                   f"{args.steps} steps of ~{per_step:.3g} s"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(wl, l2):
    return {"workload": f"{wl.name}: B={wl.B} C={wl.C} O={wl.O} H={wl.H} W={wl.W} "
                        f"{wl.kh}x{wl.kw} pad={wl.pad} {wl.dtype} offsets~N(0,{wl.offset_std}) "
                        f"mask {wl.mask}",
            "B": wl.B, "C": wl.C, "O": wl.O, "H": wl.H, "W": wl.W, "kh": wl.kh, "kw": wl.kw,
            "pad": wl.pad, "out_pixels": wl.pixels, "flops_per_step": wl.flops, "l2": l2}


def fp32_fma_peak_tflops(sm_count, sm_mhz):
    """fp32 CUDA-core peak: 128 FFMA lanes per SM, 2 FLOP each, per clock."""
    return sm_count * 128 * 2 * sm_mhz * 1e6 / 1e12


def time_backward(args, wl, dcn, torch, dev, stream, h, x, off, m, w, flush, code):
    """The backward pass (all five gradients) on the same workload: CUDA
    events around each dcn_backward call, L2 flushed before each."""
    if args.no_backward:
        return None
    g = torch.Generator().manual_seed(7)
    gout = torch.randn(wl.B, wl.O, wl.Ho, wl.Wo, generator=g).to(x.dtype).to(dev) \
        .contiguous(memory_format=torch.channels_last)
    f32 = dict(dtype=torch.float32, device=dev)
    gx = torch.empty(x.shape, memory_format=torch.channels_last, **f32)
    goff = torch.empty(off.shape, **f32)
    gm = None if m is None else torch.empty(m.shape, **f32)
    gw = torch.empty(w.shape, **f32)
    gb = torch.empty((wl.O,), **f32)
    dims = (wl.B, wl.C, wl.H, wl.W, wl.O, wl.kh, wl.kw, wl.pad, code)

    def call():
        dcn.dcn_backward(h.h, x, off, m, w, gout, gx, goff, gm, gw, gb, *dims, stream)

    for _ in range(max(3, min(args.warmup, 5))):
        flush.fill_(2)
        call()
    n = max(3, min(args.steps, args.backward_steps))
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    for k in range(n):
        flush.fill_(k & 0xFF)
        ev[k][0].record(stream)
        call()
        ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    if dcn.dcn_sync_status(h.h, stream) != 0:
        raise RuntimeError("device status set during the backward timing")
    ms = statistics.fmean(e[0].elapsed_time(e[1]) for e in ev)
    flops = 2 * wl.flops   # the column-gradient and weight-gradient contractions
    props = torch.cuda.get_device_properties(dev)
    peak = fp32_fma_peak_tflops(props.multi_processor_count, 2070.0)
    achieved = flops / (ms * 1e-3) / 1e12
    return {"ms_per_call": ms, "value": achieved, "unit": "TFLOP/s",
            "flops_per_call": flops, "calls": n,
            "gradients": "x, offset, mask, weight, bias (fp32)",
            "roofline": {"bound": "fma", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak,
                         "peak_source": f"{props.multi_processor_count} SMs x 128 fp32 FMA lanes x 2 FLOP "
                                        f"x 2070 MHz (the SM clock maximum)",
                         "scope": "whole dcn_backward call"}}


def msda_bytes(m, es):
    """Algorithmic HBM bytes of one MSDA call: value, locations, weights and
    out, each moved once."""
    return (m.B * m.S * m.G * m.D * es + m.B * m.Q * m.G * m.L * m.K * 2 * 4
            + m.B * m.Q * m.G * m.L * m.K * 4 + m.B * m.Q * m.G * m.D * es)


def time_msda(args, dcn, torch, dev, stream, flush, pk):
    """Multi-scale deformable attention forward on the encoder-scale
    workloads: CUDA events around each call, L2 flushed before each."""
    if args.no_msda:
        return None
    from deformable_convolution_vision_gb300.inputs import MSDA_WORKLOADS, make_msda_inputs
    res = {}
    for name in ("msda_encoder", "msda_encoder_22k"):
        m = MSDA_WORKLOADS[name]
        inp = make_msda_inputs(m)
        v = inp["value"].to(dev)
        loc = inp["locations"].to(dev)
        w = inp["weights"].to(dev)
        out = torch.empty((m.B, m.Q, m.G, m.D), dtype=v.dtype, device=dev)
        call = lambda: dcn.msda(v, m.shapes, m.starts, loc, w, method="softmax", out=out, stream=stream)
        for _ in range(5):
            flush.fill_(3)
            call()
        n = max(3, min(args.steps, 200))
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for k in range(n):
            flush.fill_(k & 0xFF)
            ev[k][0].record(stream)
            call()
            ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        us = statistics.fmean(e[0].elapsed_time(e[1]) for e in ev) * 1e3
        es = v.element_size()
        nbytes = msda_bytes(m, es)
        samples = m.B * m.Q * m.G * m.L * m.K
        achieved = nbytes / (us * 1e-6) / 1e9
        res[name] = {
            "config": f"B={m.B} G={m.G} D={m.D} levels={list(m.shapes)} Q={m.Q} K={m.K} "
                      f"{m.dtype} softmax",
            "us_per_call": us, "queries_per_s": m.B * m.Q / (us * 1e-6),
            "samples_per_s": samples / (us * 1e-6), "calls": n,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / pk["hbm_gbs"], "algorithmic_bytes": nbytes,
                         "corner_bytes_on_chip": samples * 4 * m.D * es,
                         "scope": "whole dcn_msda_forward call (one kernel)"}}
    return res


def time_other_configs(args, dcn, torch, dev, stream, flush, pk):
    """The forward on the other synthetic configurations (decoder 3x3,
    backbone 3x3, boundary 5x5): the public dcn_forward call, L2 flushed
    before each, against the same roofline as the headline workload."""
    if args.no_other_configs:
        return None
    from deformable_convolution_vision_gb300.inputs import WORKLOADS, make_inputs
    res = {}
    for name in ("decoder3x3", "backbone3x3", "boundary5x5"):
        wl = WORKLOADS[name]
        inp = make_inputs(wl)
        x = inp["x"].to(dev).contiguous(memory_format=torch.channels_last)
        off = inp["offset"].to(dev)
        m = None if inp["mask"] is None else inp["mask"].to(dev)
        w = inp["weight"].to(dev).contiguous()
        b = None if inp["bias"] is None else inp["bias"].to(dev)
        out = torch.empty((wl.B, wl.O, wl.Ho, wl.Wo), dtype=x.dtype, device=dev,
                          memory_format=torch.channels_last)
        dims = (wl.B, wl.C, wl.H, wl.W, wl.O, wl.kh, wl.kw, wl.pad,
                dcn.DCN_BF16 if wl.dtype == "bf16" else dcn.DCN_F32)
        with dcn.Handle() as h:
            call = lambda: dcn.dcn_forward(h.h, x, off, m, w, b, out, *dims, stream)
            for _ in range(5):
                flush.fill_(3)
                call()
            n = max(3, min(args.steps, 200))
            ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
            for k in range(n):
                flush.fill_(k & 0xFF)
                ev[k][0].record(stream)
                call()
                ev[k][1].record(stream)
            torch.cuda.synchronize(dev)
            if dcn.dcn_sync_status(h.h, stream) != 0:
                raise RuntimeError(f"device status set on {name}")
            path = dcn.dcn_last_path(h.h)
        us = statistics.fmean(e[0].elapsed_time(e[1]) for e in ev) * 1e3
        t_tc = wl.flops / (pk["bf16_tflops"] * 1e12)
        t_hbm = algorithmic_bytes(wl) / (pk["hbm_gbs"] * 1e9)
        res[name] = {
            "config": config_dict(wl, "flushed before every call")["workload"],
            "us_per_call": us, "tflops": wl.flops / (us * 1e-6) / 1e12,
            "out_pixels_per_s": wl.pixels / (us * 1e-6), "calls": n,
            "path": "tensor cores" if path == dcn.DCN_PATH_TC else "CUDA cores",
            "roofline": {"bound": "tensor" if t_tc >= t_hbm else "hbm",
                         "frac": max(t_tc, t_hbm) / (us * 1e-6),
                         "t_tensor_us": t_tc * 1e6, "t_hbm_us": t_hbm * 1e6,
                         "scope": "whole dcn_forward call (weight pack + fused kernel)"}}
    return res


def msda_backward_bytes(m, es):
    """Algorithmic HBM bytes of one MSDA backward call: value, grad_out,
    locations and weights read once; the fp32 value gradient (zeroed, then
    written), location and weight gradients written once."""
    pts = m.B * m.Q * m.G * m.L * m.K
    return (m.B * m.S * m.G * m.D * (es + 2 * 4) + m.B * m.Q * m.G * m.D * es
            + pts * 2 * 4 * 2 + pts * 4 * 2)


def time_msda_backward(args, dcn, torch, dev, stream, flush, pk):
    """The MSDA backward on the encoder-scale workloads: whole
    dcn_msda_backward calls (the zeroing of grad_value included), CUDA
    events, L2 flushed before each."""
    if args.no_msda:
        return None
    from deformable_convolution_vision_gb300.inputs import (MSDA_WORKLOADS, make_msda_grad_out,
                                                            make_msda_inputs)
    res = {}
    for name in ("msda_encoder", "msda_encoder_22k"):
        m = MSDA_WORKLOADS[name]
        inp = make_msda_inputs(m)
        v = inp["value"].to(dev)
        loc = inp["locations"].to(dev)
        w = inp["weights"].to(dev)
        go = make_msda_grad_out(m).to(dev)
        gv = torch.empty((m.B, m.S, m.G, m.D), dtype=torch.float32, device=dev)
        gl = torch.empty((m.B, m.Q, m.G, m.L, m.K, 2), dtype=torch.float32, device=dev)
        gw = torch.empty((m.B, m.Q, m.G, m.L * m.K), dtype=torch.float32, device=dev)
        code = {torch.bfloat16: dcn.DCN_BF16, torch.float16: dcn.DCN_F16}.get(v.dtype, dcn.DCN_F32)
        call = lambda: dcn.dcn_msda_backward(v, m.shapes, m.starts, loc, w, go, gv, gl, gw, m.B,
                                             m.S, m.G, m.D, m.Q, m.K, True, code, stream)
        for _ in range(5):
            flush.fill_(3)
            call()
        n = max(3, min(args.steps, 200))
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for k in range(n):
            flush.fill_(k & 0xFF)
            ev[k][0].record(stream)
            call()
            ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        us = statistics.fmean(e[0].elapsed_time(e[1]) for e in ev) * 1e3
        nbytes = msda_backward_bytes(m, v.element_size())
        samples = m.B * m.Q * m.G * m.L * m.K
        achieved = nbytes / (us * 1e-6) / 1e9
        res[name] = {
            "config": f"B={m.B} G={m.G} D={m.D} levels={list(m.shapes)} Q={m.Q} K={m.K} "
                      f"{m.dtype} softmax",
            "us_per_call": us, "queries_per_s": m.B * m.Q / (us * 1e-6), "calls": n,
            "gradients": "value, locations, weights (fp32)",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / pk["hbm_gbs"], "algorithmic_bytes": nbytes,
                         "fp32_reduction_bytes_on_chip": samples * 4 * m.D * 4,
                         "scope": "whole dcn_msda_backward call (memset + one kernel)"}}
    return res


def attn_bytes(a, es):
    """Algorithmic HBM bytes of one single-scale sampling call: value,
    offsets, weights and out, each moved once."""
    Ho, Wo = a.out_size()
    rows = a.B * Ho * Wo * a.G
    return a.B * a.H * a.W * a.G * a.D * es + rows * a.K * (2 * 4 + 4) + rows * a.D * es


def time_attn(args, dcn, torch, dev, stream, flush, pk):
    """Single-scale deformable sampling (DCNv3) forward: CUDA events around
    each call, L2 flushed before each."""
    if args.no_msda:
        return None
    from deformable_convolution_vision_gb300.inputs import ATTN_WORKLOADS, make_attn_inputs
    res = {}
    for name in ("attn_page", "attn_stage1_1024"):
        a = ATTN_WORKLOADS[name]
        inp = make_attn_inputs(a)
        v = inp["value"].to(dev)
        off = inp["offsets"].to(dev)
        w = inp["weights"].to(dev)
        Ho, Wo = a.out_size()
        out = torch.empty((a.B, Ho, Wo, a.G, a.D), dtype=v.dtype, device=dev)
        call = lambda: dcn.attn(v, off, w, a.kernel, a.stride, a.padding, a.dilation,
                                method="softmax", out=out, stream=stream)
        for _ in range(5):
            flush.fill_(3)
            call()
        n = max(3, min(args.steps, 200))
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for k in range(n):
            flush.fill_(k & 0xFF)
            ev[k][0].record(stream)
            call()
            ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        us = statistics.fmean(e[0].elapsed_time(e[1]) for e in ev) * 1e3
        nbytes = attn_bytes(a, v.element_size())
        samples = a.B * Ho * Wo * a.G * a.K
        achieved = nbytes / (us * 1e-6) / 1e9
        res[name] = {
            "config": f"B={a.B} {a.H}x{a.W} G={a.G} D={a.D} {a.kernel[0]}x{a.kernel[1]} "
                      f"pad={a.padding[0]} {a.dtype} softmax",
            "us_per_call": us, "out_pixels_per_s": a.B * Ho * Wo / (us * 1e-6),
            "samples_per_s": samples / (us * 1e-6), "calls": n,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / pk["hbm_gbs"], "algorithmic_bytes": nbytes,
                         "corner_bytes_on_chip": samples * 4 * a.D * v.element_size(),
                         "scope": "whole dcn_attn_forward call (one kernel)"}}
    return res


def attn_backward_bytes(a, es):
    """Algorithmic HBM bytes of one single-scale backward call: value,
    grad_out, offsets and weights read once; the fp32 value gradient
    (zeroed, then written), offset and weight gradients written once."""
    Ho, Wo = a.out_size()
    rows = a.B * Ho * Wo * a.G
    return (a.B * a.H * a.W * a.G * a.D * (es + 2 * 4) + rows * a.D * es
            + rows * a.K * (2 * 4 + 4) * 2)


def time_attn_backward(args, dcn, torch, dev, stream, flush, pk):
    """The single-scale sampling backward: whole dcn_attn_backward calls
    (the zeroing of grad_value included), CUDA events, L2 flushed before
    each."""
    if args.no_msda:
        return None
    from deformable_convolution_vision_gb300.inputs import (ATTN_WORKLOADS, make_attn_grad_out,
                                                            make_attn_inputs)
    res = {}
    for name in ("attn_page", "attn_stage1_1024"):
        a = ATTN_WORKLOADS[name]
        inp = make_attn_inputs(a)
        v = inp["value"].to(dev)
        off = inp["offsets"].to(dev)
        w = inp["weights"].to(dev)
        go = make_attn_grad_out(a).to(dev)
        Ho, Wo = a.out_size()
        gv = torch.empty((a.B, a.H, a.W, a.G, a.D), dtype=torch.float32, device=dev)
        gof = torch.empty((a.B, Ho, Wo, a.G, a.K, 2), dtype=torch.float32, device=dev)
        gw = torch.empty((a.B, Ho, Wo, a.G, a.K), dtype=torch.float32, device=dev)
        code = {torch.bfloat16: dcn.DCN_BF16, torch.float16: dcn.DCN_F16}.get(v.dtype, dcn.DCN_F32)
        call = lambda: dcn.dcn_attn_backward(v, off, w, go, gv, gof, gw, a.B, a.H, a.W, a.G, a.D,
                                             a.kernel[0], a.kernel[1], a.stride[0], a.stride[1],
                                             a.padding[0], a.padding[1], a.dilation[0],
                                             a.dilation[1], True, code, stream)
        for _ in range(5):
            flush.fill_(3)
            call()
        n = max(3, min(args.steps, 200))
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        for k in range(n):
            flush.fill_(k & 0xFF)
            ev[k][0].record(stream)
            call()
            ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        us = statistics.fmean(e[0].elapsed_time(e[1]) for e in ev) * 1e3
        nbytes = attn_backward_bytes(a, v.element_size())
        samples = a.B * Ho * Wo * a.G * a.K
        achieved = nbytes / (us * 1e-6) / 1e9
        res[name] = {
            "config": f"B={a.B} {a.H}x{a.W} G={a.G} D={a.D} {a.kernel[0]}x{a.kernel[1]} "
                      f"pad={a.padding[0]} {a.dtype} softmax",
            "us_per_call": us, "out_pixels_per_s": a.B * Ho * Wo / (us * 1e-6), "calls": n,
            "gradients": "value, offsets, weights (fp32)",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / pk["hbm_gbs"], "algorithmic_bytes": nbytes,
                         "fp32_reduction_bytes_on_chip": samples * 4 * a.D * 4,
                         "scope": "whole dcn_attn_backward call (memset + one kernel)"}}
    return res


def run_ours(args, wl, rank, local_rank, world):
    import torch
    import deformable_convolution_vision_gb300 as dcn
    from deformable_convolution_vision_gb300.inputs import make_inputs

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp = make_inputs(wl)
    x = inp["x"].to(dev).contiguous(memory_format=torch.channels_last)
    off = inp["offset"].to(dev)
    m = None if inp["mask"] is None else inp["mask"].to(dev)
    w = inp["weight"].to(dev).contiguous()
    b = None if inp["bias"] is None else inp["bias"].to(dev)
    out = torch.empty((wl.B, wl.O, wl.Ho, wl.Wo), dtype=x.dtype, device=dev,
                      memory_format=torch.channels_last)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    code = dcn.DCN_BF16 if wl.dtype == "bf16" else dcn.DCN_F32
    dims = (wl.B, wl.C, wl.H, wl.W, wl.O, wl.kh, wl.kw, wl.pad, code)
    h = dcn.Handle()
    stream = torch.cuda.current_stream(dev)

    def step():
        # the public call: weight pack, then the fused kernel, which starts
        # while the pack runs (programmatic dependent launch)
        dcn.dcn_forward(h.h, x, off, m, w, b, out, *dims, stream)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize(dev)
    if dcn.dcn_sync_status(h.h, stream) != 0:
        raise RuntimeError("device status set during warm-up")
    path_taken = dcn.dcn_last_path(h.h)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for k in range(args.steps):
        flush.fill_(k & 0xFF)
        ev[k][0].record(stream)
        step()
        ev[k][1].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler else None
    if dcn.dcn_sync_status(h.h, stream) != 0:
        raise RuntimeError("device status set during the timed region")
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]

    # The dominant kernel on its own, for the roofline: the same steps with
    # the two halves of the call timed apart (events between them, so the
    # fused kernel does not overlap the pack here).
    n_split = min(args.steps, 500)
    ev3 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_split)]
    for k in range(n_split):
        flush.fill_(k & 0xFF)
        ev3[k][0].record(stream)
        dcn.dcn_pack_weight(h.h, w, wl.O, wl.C, wl.kh, wl.kw, code, stream)
        ev3[k][1].record(stream)
        dcn.dcn_forward_packed(h.h, x, off, m, b, out, *dims, stream)
        ev3[k][2].record(stream)
    torch.cuda.synchronize(dev)
    if dcn.dcn_sync_status(h.h, stream) != 0:
        raise RuntimeError("device status set during the split timing")
    main_ms = [e[1].elapsed_time(e[2]) for e in ev3]
    pack_ms = [e[0].elapsed_time(e[1]) for e in ev3]

    # The fused kernel with the fp32 bilinear combine (the sampled value
    # summed in fp32 and rounded once to the operand type, instead of the
    # input-dtype combine of the page's routine): same flush and events.
    main_f32 = None
    if code != dcn.DCN_F32:
        with dcn.Handle(sample=dcn.DCN_SAMPLE_F32) as hf:
            dcn.dcn_pack_weight(hf.h, w, wl.O, wl.C, wl.kh, wl.kw, code, stream)
            for _ in range(3):
                flush.fill_(3)
                dcn.dcn_forward_packed(hf.h, x, off, m, b, out, *dims, stream)
            evf = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_split)]
            for k in range(n_split):
                flush.fill_(k & 0xFF)
                evf[k][0].record(stream)
                dcn.dcn_forward_packed(hf.h, x, off, m, b, out, *dims, stream)
                evf[k][1].record(stream)
            torch.cuda.synchronize(dev)
            if dcn.dcn_sync_status(hf.h, stream) != 0:
                raise RuntimeError("device status set during the fp32-combine timing")
            main_f32 = statistics.fmean(e[0].elapsed_time(e[1]) for e in evf)
    ms = statistics.fmean(step_ms)
    ms_max = reduce_max(ms, world)
    main_mean = statistics.fmean(main_ms)

    # the same call with no flush between steps (inputs left in L2 by the
    # previous step), reported apart and labelled as such
    n_warm = min(args.steps, 500)
    evw = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n_warm)]
    for k in range(n_warm):
        evw[k][0].record(stream)
        step()
        evw[k][1].record(stream)
    torch.cuda.synchronize(dev)
    warm_ms = statistics.fmean(e[0].elapsed_time(e[1]) for e in evw)

    # end to end through the host-buffer entry point: pinned host inputs in,
    # pinned host output back, copies inside the timed region
    hx = inp["x"].permute(0, 2, 3, 1).contiguous().pin_memory()
    hoff = inp["offset"].pin_memory()
    hm = None if inp["mask"] is None else inp["mask"].pin_memory()
    hw = inp["weight"].contiguous().pin_memory()
    hb = None if inp["bias"] is None else inp["bias"].pin_memory()
    hout = torch.empty((wl.B, wl.Ho, wl.Wo, wl.O), dtype=x.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hx, hoff, hm, hw, hb) if t is not None)
    d2h = hout.numel() * hout.element_size()
    e2e_steps = max(3, min(args.steps, 50))
    for _ in range(max(args.warmup, 3)):
        dcn.dcn_forward_host(h.h, hx, hoff, hm, hw, hb, hout, *dims, stream)
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        dcn.dcn_forward_host(h.h, hx, hoff, hm, hw, hb, hout, *dims, stream)
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    e2e_max = reduce_max(e2e_s, world)
    backward = time_backward(args, wl, dcn, torch, dev, stream, h, x, off, m, w, flush, code)
    msda = time_msda(args, dcn, torch, dev, stream, flush, peaks()[0])
    msda_bwd = time_msda_backward(args, dcn, torch, dev, stream, flush, peaks()[0])
    attn = time_attn(args, dcn, torch, dev, stream, flush, peaks()[0])
    attn_bwd = time_attn_backward(args, dcn, torch, dev, stream, flush, peaks()[0])
    others = time_other_configs(args, dcn, torch, dev, stream, flush, peaks()[0])
    h.close()

    if rank != 0:
        return
    pk, pk_src = peaks()
    achieved = wl.flops / (main_mean * 1e-3) / 1e12
    value = whole_job_rate(wl.flops, world, ms_max * 1e-3) / 1e12
    t_tc = wl.flops / (pk["bf16_tflops"] * 1e12)
    t_hbm = algorithmic_bytes(wl) / (pk["hbm_gbs"] * 1e9)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
        "data": "synthetic",
        "config": config_dict(wl, L2_NOTE),
        "out_pixels_per_s": whole_job_rate(wl.pixels, world, ms_max * 1e-3),
        "roofline_frac_step": max(t_tc, t_hbm) / (ms_max * 1e-3),
        "step_ms": {"mean": ms, "min": min(step_ms), "median": statistics.median(step_ms),
                    "pack_mean": statistics.fmean(pack_ms), "main_mean": main_mean,
                    "main_min": min(main_ms),
                    "main_mean_f32_combine": main_f32,
                    "main_f32_combine_note": "the fused kernel alone with the fp32 bilinear combine "
                                             "(DCN_SAMPLE_F32); the headline uses the input-dtype combine",
                    "warm_l2_mean": warm_ms,
                    "warm_l2_note": "no flush between steps; not the reported value"},
        "roofline": {"bound": "tensor" if t_tc >= t_hbm else "hbm", "achieved": achieved,
                     "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / pk["bf16_tflops"], "traffic": dram_traffic(wl.name),
                     "kernel": MAIN_KERNEL if path_taken == dcn.DCN_PATH_TC else "dcn_simt_kernel",
                     "peak_source": pk_src + ", bf16 dense burst",
                     "t_tensor_us": t_tc * 1e6, "t_hbm_us": t_hbm * 1e6,
                     "algorithmic_bytes": algorithmic_bytes(wl)},
        "e2e": {"value": whole_job_rate(wl.flops, world, e2e_max) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_max * 1e3, "api": "dcn_forward_host (pinned host buffers)"},
        "clocks": clocks,
        "gpu_launches": 2 * args.steps,   # per step: the weight pack and the fused kernel
        "wall_s_timed_region": wall,
    }
    if backward is not None:
        line["backward"] = backward
    if msda is not None:
        line["msda"] = msda
    if msda_bwd is not None:
        line["msda_backward"] = msda_bwd
    if attn is not None:
        line["single_scale_sampling"] = attn
    if attn_bwd is not None:
        line["single_scale_sampling_backward"] = attn_bwd
    if others is not None:
        line["other_configs"] = others
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, inp, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="aspp7x7")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--reference-step-seconds", type=float, default=2.0)
    ap.add_argument("--reference-budget-seconds", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--backward-steps", type=int, default=50)
    ap.add_argument("--no-msda", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    from deformable_convolution_vision_gb300.inputs import WORKLOADS
    wl = WORKLOADS[args.workload]
    rank, local_rank, world = dist_env()
    if args.impl == "reference":
        # the oracle runs on rank 0's host cores only
        run_reference(args, wl, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_ours(args, wl, rank, local_rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
