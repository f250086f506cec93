#!/usr/bin/env python
"""Benchmark of the normalization-fused Conv1d blocks on one GB300 per rank.

Default workload: the full-size fp32 pre-norm residual block
out = x + Conv1d(ReLU(BatchNorm1d_eval(x))), N=32 C=256 L=4096, k=3,
dilation=padding=128 (x is 134 MB, 51.5 GFLOP per call).  One step = one call
of the library's C ABI entry point (weight repack + fused implicit GEMM).

Prints ONE JSON line (rank 0).  `value` is whole-job throughput in TFLOP/s of
the block's algorithmic FLOPs (2*N*L*C_out*C_in*3) with inputs resident in
HBM; `e2e` is the same metric through the public Python API with pinned host
buffers (host->device copies of every input and the device->host copy of the
output inside the timed region).  L2 is flushed (256 MB write, untimed)
between timed steps.  The K timed steps run twice: untraced for `value` (as a
caller runs the library), then with the library's launch trace on for the
dominant kernel's CUDA-event duration (`roofline`).  `graph` reports the same
call captured once in a CUDA graph and replayed: device time per replay (L2
flushed between replays) and the host's enqueue cost per call, eager against
replay.  Multi-GPU (torchrun) runs independent replicas: the
blocks have no exchange step, so the work is weak-scaled with no collective
on the data path; the barrier and the max-over-ranks timing use the process
group only around the timed region.

--impl reference times the fp64 CPU oracle (the checker of the library, not a
tuned CPU implementation) on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused norm+Conv1d block ms/call, TFLOP/s, % of roofline on 1 GB300"
DEFAULT_WORKLOAD = "prenorm_block_f32"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TF32_PER_BF16 = 1.1 / 2.25        # nominal dense tf32 : bf16 tensor rate on GB300
L2_FLUSH_BYTES = 256 << 20

# DRAM traffic (read + write bytes) of one launch of the dominant kernel, from
# one ncu capture of that workload, keyed by workload; valid only while the
# sources that define that kernel (its translation unit and the shared
# headers) hash to the recorded value, else the line reports null.
NCU_TRAFFIC = {
    "prenorm_block_f32": {"bytes": 135219200 + 86754048, "src_hash": "2d03b6983ae13010"},
    "linear_bn_swish_f32": {"bytes": 335566336 + 23069184, "src_hash": "4154b4a9fd0a1a11"},
    "linear_bn_swish_eval_f32": {"bytes": 335696128 + 22748928, "src_hash": "4154b4a9fd0a1a11"},
    "prenorm_block_train_f32": {"bytes": 135193856 + 86392320, "src_hash": "2d03b6983ae13010"},
    "conv1d_groupnorm_f32": {"bytes": 8897792 + 0, "src_hash": "2d03b6983ae13010"},
    "prenorm_block_bf16_C256_d1": {"bytes": 67612672 + 22260992, "src_hash": "2d03b6983ae13010"},
    "prenorm_block_bf16_C256_d512": {"bytes": 67597824 + 22804992, "src_hash": "2d03b6983ae13010"},
    "prenorm_block_bf16_C512_d1": {"bytes": 135956736 + 90289664, "src_hash": "2d03b6983ae13010"},
    "prenorm_block_bf16_C512_d512": {"bytes": 135947264 + 91842560, "src_hash": "2d03b6983ae13010"},
}
KERNEL_TU = {"block": "conv_blocks.cu", "block_train": "conv_blocks.cu",
             "conv_gn": "conv_blocks.cu", "linear": "linear_bn_swish.cu"}
TRAIN_MOMENTUM = 0.1


def kernel_source_hash(workload: str) -> str:
    """Hash of the translation unit defining the workload's kernels plus the
    shared headers (nrc_*.cuh, nrc_host.h)."""
    from normalization_convolution_blocks_gb300 import synthetic as syn
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "normalization_convolution_blocks_gb300", "csrc")
    tu = KERNEL_TU[syn.WORKLOADS[workload].kind]
    for name in sorted(os.listdir(csrc)):
        if name == tu or name.endswith((".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------
# Workload accounting
# ---------------------------------------------------------------------------
def workload_info(name):
    """FLOPs and minimal bytes per call, dtype, and how the tensor peak is taken."""
    from normalization_convolution_blocks_gb300 import synthetic as syn
    wl = syn.WORKLOADS[name]
    p = wl.params
    if wl.kind in ("block", "block_train"):
        esz = 2 if p.get("dtype") == "bf16" else 4
        N, C, L = p["N"], p["C"], p["L"]
        flops = 2.0 * N * L * C * C * 3
        min_bytes = esz * (2 * N * C * L + 3 * C * C + C) + 4 * 4 * C
        cfg = dict(workload=name, N=N, C=C, L=L, kernel_size=3, dilation=p["dilation"],
                   padding=p["dilation"], storage=p.get("dtype", "f32"))
        if wl.kind == "block_train":
            # min_bytes stays the GEMM's own; the statistics pass before it reads
            # x once more (reported on its own, see stats_kernel)
            cfg.update(bn="training", momentum=TRAIN_MOMENTUM)
        dtype = "bf16" if esz == 2 else "f32"
        main = "prenorm_block_gemm"
    elif wl.kind == "conv_gn":
        N, Cin, Cout, T = p["N"], p["Cin"], p["Cout"], p["T"]
        flops = 2.0 * N * T * Cout * Cin * 3
        min_bytes = 4 * (N * Cin * T + N * Cout * T + 3 * Cout * Cin + 2 * Cout)
        cfg = dict(workload=name, N=N, C_in=Cin, C_out=Cout, T=T, kernel_size=3, padding=1,
                   num_groups=p["G"], storage="f32")
        dtype = "f32"
        main = "conv_gn_gemm"
    else:
        B, IN, OUT = p["B"], p["IN"], p["OUT"]
        flops = 2.0 * B * IN * OUT
        min_bytes = 4 * (B * IN + OUT * IN + B * OUT + 5 * OUT)
        cfg = dict(workload=name, B=B, in_features=IN, out_features=OUT,
                   bn="training" if p.get("training", True) else "eval", storage="f32")
        dtype = "f32"
        main = "linear_gemm"
    if wl.kind in ("block", "block_train"):
        largest = ("x", esz * N * C * L)
    elif wl.kind == "conv_gn":
        largest = ("out", 4 * N * Cout * T)
    else:
        largest = ("W", 4 * OUT * IN)
    return dict(flops=flops, min_bytes=min_bytes, config=cfg, dtype=dtype, main_kernel=main,
                kind=wl.kind, largest_tensor=largest)


L2_BYTES = 129 * 1000 * 1000      # GB300 L2 (126 MiB)


def l2_note(info):
    name, nbytes = info["largest_tensor"]
    note = f"flushed between steps ({L2_FLUSH_BYTES >> 20} MB write, untimed)"
    if nbytes > L2_BYTES:
        return note + f"; {name} alone ({nbytes / 1e6:.0f} MB) exceeds L2 on this workload"
    return note + f"; the largest tensor ({name}, {nbytes / 1e6:.1f} MB) fits in L2, so the flush " \
                  "is what keeps the steps cold"


def roofline_peaks(info, peaks):
    """Tensor peak of the contraction's own dtype: bf16 storage -> bf16; fp32
    storage -> tf32 (the fp32 input type of the tensor cores), derived from the
    measured bf16 peak by the nominal tf32:bf16 ratio."""
    bf16 = peaks["bf16_tflops"]
    if info["dtype"] == "bf16":
        return bf16, "bf16 (measured burst)"
    return bf16 * TF32_PER_BF16, "tf32 = measured bf16 burst x nominal 1.1/2.25"


def roofline_of(info, main_ms, peaks):
    """The dominant kernel's roofline: whichever of the tensor and HBM bounds
    is longer for the workload, the kernel's achieved rate against it, and the
    effective fraction (fp32: the three TF32 products per term that 3xTF32
    compensation issues)."""
    tensor_peak, tensor_note = roofline_peaks(info, peaks)
    hbm_peak = peaks["hbm_gbs"]
    t_tensor = info["flops"] / (tensor_peak * 1e12)
    t_hbm = info["min_bytes"] / (hbm_peak * 1e9)
    if t_tensor >= t_hbm:
        achieved = info["flops"] / (main_ms * 1e-3) / 1e12
        roof = dict(bound="tensor", achieved=round(achieved, 2), peak=round(tensor_peak, 1),
                    unit="TFLOP/s", frac=round(achieved / tensor_peak, 4))
    else:
        achieved = info["min_bytes"] / (main_ms * 1e-3) / 1e9
        roof = dict(bound="hbm", achieved=round(achieved, 1), peak=round(hbm_peak, 1),
                    unit="GB/s", frac=round(achieved / hbm_peak, 4))
    roof["roofline_ms"] = round(max(t_tensor, t_hbm) * 1e3, 5)
    if info["dtype"] == "f32" and roof["bound"] == "tensor":
        t_eff = max(3 * t_tensor, t_hbm)
        roof["roofline_ms_effective"] = round(t_eff * 1e3, 5)
        roof["frac_effective"] = round(t_eff / (main_ms * 1e-3), 4)
    else:
        roof["roofline_ms_effective"] = roof["roofline_ms"]
        roof["frac_effective"] = roof["frac"]
    return roof, tensor_note


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
CLOCK_FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device_index):
        self.proc = None
        self.t0 = self.t1 = None
        self.device_index = device_index

    def start(self):
        try:
            import torch
            sel = []
            try:
                uuid = str(torch.cuda.get_device_properties(self.device_index).uuid)
                sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
            except Exception:
                pass
            self.proc = subprocess.Popen(
                ["nvidia-smi", *sel, f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def mark(self, which):
        if which == "begin":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"samples": 0, "note": "nvidia-smi unavailable"}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for row in csv.reader(io.StringIO(out)):
            if len(row) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(row[0].strip().split(".")[0],
                                               "%Y/%m/%d %H:%M:%S"))
                frac = float("0." + row[0].strip().split(".")[1]) if "." in row[0] else 0.0
                rows.append(dict(t=ts + frac, sm=float(row[1]), smax=float(row[2]),
                                 power=float(row[3]) if row[3].strip() not in ("[N/A]", "") else None,
                                 active=row[4].strip(),
                                 hw=row[5].strip(), hwt=row[6].strip(), swt=row[7].strip(),
                                 swp=row[8].strip()))
            except (ValueError, IndexError):
                continue
        window = [r for r in rows if self.t0 is not None and self.t1 is not None
                  and self.t0 - 0.15 <= r["t"] <= self.t1 + 0.15]
        used = window if window else rows
        if not used:
            return {"samples": 0}
        reasons = set()
        for r in used:
            for key, label in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                               ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(label)
        return {"sm_mhz": statistics.median(r["sm"] for r in used),
                "sm_max_mhz": max(r["smax"] for r in used),
                "reasons": sorted(reasons),
                "samples": len(used),
                "in_window": bool(window),
                "power_w_max": max((r["power"] for r in used if r["power"] is not None),
                                   default=None)}


# ---------------------------------------------------------------------------
# Distributed plumbing (replicas: barrier + max-over-ranks timing only)
# ---------------------------------------------------------------------------
def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_tflops(world, flops_per_rank_step, ms_per_step):
    """Weak scaling: every rank processes its own copy of the workload each step,
    so the job's throughput is world x the per-rank work over the slowest rank's
    step time."""
    return world * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def max_over_ranks(world, value, device=None):
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# The GPU arm
# ---------------------------------------------------------------------------
def make_call(name, dev, host=False):
    """Inputs of the workload (device-resident, or pinned host tensors) and a
    closure running one call of the library on them."""
    import torch

    from normalization_convolution_blocks_gb300 import api
    from normalization_convolution_blocks_gb300 import synthetic as syn
    wl = syn.WORKLOADS[name]
    inp = wl.make(seed=0)

    def place(t):
        if t is None:
            return None
        return t.pin_memory() if host else t.to(dev)

    if wl.kind == "block":
        x, rm, rv, g, b, w, bias = map(place, (inp.x, inp.running_mean, inp.running_var,
                                              inp.gamma, inp.beta, inp.weight, inp.bias))
        # host buffers: the output is pinned and the workspace allocated once, as
        # a caller running the block repeatedly would hold them
        out = torch.empty(x.shape, dtype=x.dtype, pin_memory=True) if host else \
            torch.empty_like(x)
        ws_bytes = api.prenorm_dilconv_residual_host_workspace_size(*x.shape, x.dtype) if host \
            else api.prenorm_dilconv_residual_workspace_size(x.shape[1], x.dtype)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        tensors_in = (x, rm, rv, g, b, w, bias)

        def call():
            return api.prenorm_dilconv_residual(x, rm, rv, g, b, inp.eps, w, bias,
                                                inp.dilation, out=out, workspace=ws)
        out_shape = (x.shape, x.dtype)
    elif wl.kind == "block_train":
        x, g, b, w, bias = map(place, (inp.x, inp.gamma, inp.beta, inp.weight, inp.bias))
        rm, rv = inp.running_mean.to(dev), inp.running_var.to(dev)
        nbt = torch.zeros(1, dtype=torch.int64, device=dev)
        # host buffers: the output is pinned and the workspace allocated once
        out = torch.empty(x.shape, dtype=x.dtype, pin_memory=True) if host else \
            torch.empty_like(x)
        ws_bytes = api.prenorm_dilconv_residual_train_host_workspace_size(*x.shape, x.dtype) \
            if host else api.prenorm_dilconv_residual_train_workspace_size(*x.shape, x.dtype)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        tensors_in = (x, g, b, w, bias)

        def call():
            return api.prenorm_dilconv_residual_train(x, rm, rv, g, b, inp.eps, TRAIN_MOMENTUM,
                                                      w, bias, inp.dilation,
                                                      num_batches_tracked=nbt, out=out,
                                                      workspace=ws)
        out_shape = (x.shape, x.dtype)
    elif wl.kind == "conv_gn":
        x, w, g, b = map(place, (inp.x, inp.weight, inp.gamma, inp.beta))
        N, Cin, T = x.shape
        Cout = w.shape[0]
        # host buffers: the output is pinned and the workspace allocated once
        out = torch.empty((N, Cout, T), pin_memory=True) if host else \
            torch.empty((N, Cout, T), device=dev)
        ws_bytes = api.conv1d_groupnorm_host_workspace_size(N, Cin, Cout, T, inp.num_groups) \
            if host else api.conv1d_groupnorm_workspace_size(N, Cin, Cout, T, inp.num_groups)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        tensors_in = (x, w, g, b)

        def call():
            return api.conv1d_groupnorm(x, w, None, inp.num_groups, g, b, inp.eps, out=out,
                                        workspace=ws)
        out_shape = ((N, Cout, T), torch.float32)
    else:
        x, w, lb, g, b, ab = map(place, (inp.x, inp.weight, inp.lin_bias, inp.gamma,
                                         inp.beta, inp.add_bias))
        rm, rv = inp.running_mean.to(dev), inp.running_var.to(dev)
        nbt = torch.zeros(1, dtype=torch.int64, device=dev)
        B, IN = x.shape
        OUT = w.shape[0]
        # host buffers: the output is pinned and the workspace allocated once
        out = torch.empty((B, OUT), pin_memory=True) if host else \
            torch.empty((B, OUT), device=dev)
        ws_bytes = api.linear_bn_swish_host_workspace_size(B, IN, OUT) if host else \
            api.linear_bn_swish_workspace_size(B, IN, OUT)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        tensors_in = (x, w, lb, g, b, ab)

        training = wl.params.get("training", True)

        def call():
            return api.linear_bn_swish(x, w, lb, g, b, rm, rv, ab, inp.divide_value, inp.eps,
                                       inp.momentum, training, nbt, out=out, workspace=ws)
        out_shape = ((B, OUT), torch.float32)
    h2d = sum(t.numel() * t.element_size() for t in tensors_in if t is not None)
    d2h = math.prod(out_shape[0]) * (2 if out_shape[1] == torch.bfloat16 else 4)
    return call, h2d, d2h


def gpu_arm(args, world, rank, local):
    import torch

    from normalization_convolution_blocks_gb300 import api
    from normalization_convolution_blocks_gb300 import build as nbuild
    nbuild.build()
    api.load()
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    info = workload_info(args.workload)
    call, _, _ = make_call(args.workload, dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        call()
        flush.fill_(1.0)
    torch.cuda.synchronize()
    if api.query_status() != api.NRC_OK:
        raise RuntimeError("device status error during warm-up")

    steps = args.steps
    if steps is None:   # aim at ~2 s of timed work so the clock sampler sees it
        t0 = time.perf_counter()
        for _ in range(5):
            call()
            flush.fill_(1.0)
        torch.cuda.synchronize()
        per = (time.perf_counter() - t0) / 5
        steps = int(min(20000, max(20, 2.0 / max(per, 1e-6))))

    sampler = ClockSampler(dev.index) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.3)

    def timed_pass(traced):
        """K steps, each bracketed by CUDA events on the launch stream, with an
        untimed L2 flush between steps; returns the per-step ms."""
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        api.trace_enable(traced)
        barrier(world)
        torch.cuda.synchronize()
        for i in range(steps):
            starts[i].record(stream)
            call()
            ends[i].record(stream)
            flush.fill_(1.0)      # untimed: evict x/out/weights from L2 between steps
        torch.cuda.synchronize()
        barrier(world)
        api.trace_enable(False)
        if api.query_status() != api.NRC_OK:
            raise RuntimeError("device status error in the timed region")
        return [s.elapsed_time(e) for s, e in zip(starts, ends)]

    if sampler:
        sampler.mark("begin")
    # The step time is measured untraced, as a caller runs the library; the
    # per-kernel durations (roofline) come from a second pass of the same K
    # steps with the library's launch trace on.  The trace puts CUDA events
    # between launches, which also serialises a GEMM with the repack before it.
    step_ms = timed_pass(False)
    trace_step_ms = timed_pass(True)
    if sampler:
        sampler.mark("end")
    clocks = sampler.stop() if sampler else None
    total_ms = max_over_ranks(world, sum(step_ms), dev)
    recs = api.trace_records()
    launches = len(recs)
    per_kernel = {}
    for name, ms in recs:
        per_kernel.setdefault(name, []).append(ms)
    main = info["main_kernel"]
    main_ms = statistics.mean(per_kernel[main])

    ms_per_step = total_ms / steps
    value = whole_job_tflops(world, info["flops"], ms_per_step)
    peaks, peaks_src = load_peaks()
    hbm_peak = peaks["hbm_gbs"]
    roof, tensor_note = roofline_of(info, main_ms, peaks)
    tr = NCU_TRAFFIC.get(args.workload)
    roof["traffic"] = (tr["bytes"] if tr and tr["src_hash"] == kernel_source_hash(args.workload)
                       else None)
    roof["kernel"] = main
    roof["kernel_ms"] = round(main_ms, 5)
    roof["peak_source"] = f"{peaks_src}: {tensor_note if roof['bound'] == 'tensor' else 'hbm_gbs'}"
    if info["dtype"] == "f32":
        # executed work: three bf16 products per term, against the bf16 peak
        roof["executed_bf16_frac"] = round(3 * info["flops"] / (main_ms * 1e-3) / 1e12
                                           / peaks["bf16_tflops"], 4)
    kernels = {k: dict(launches=len(v), mean_ms=round(statistics.mean(v), 5),
                       share=round(sum(v) / sum(sum(x) for x in per_kernel.values()), 4))
               for k, v in per_kernel.items()}
    if "bn_row_stats" in per_kernel:
        # the training-mode statistics pass: x read once, HBM-bound
        st_ms = statistics.mean(per_kernel["bn_row_stats"])
        cfg = info["config"]
        x_bytes = cfg["N"] * cfg["C"] * cfg["L"] * (2 if info["dtype"] == "bf16" else 4)
        roof["stats_kernel"] = dict(kernel="bn_row_stats", ms=round(st_ms, 5),
                                    achieved_gbs=round(x_bytes / (st_ms * 1e-3) / 1e9, 1),
                                    frac_of_hbm=round(x_bytes / (st_ms * 1e-3) / 1e9 / hbm_peak, 4))
    roof["kernel_timing"] = ("CUDA events around each launch, in a second timed pass of the "
                             f"same {steps} steps with the launch trace on "
                             f"({round(statistics.mean(trace_step_ms), 5)} ms/step traced)")
    result = dict(value=value, ms_per_step=ms_per_step, steps=steps, roofline=roof,
                  launches=launches, kernels=kernels, clocks=clocks, info=info,
                  step_ms_p10=sorted(step_ms)[len(step_ms) // 10],
                  step_ms_median=statistics.median(step_ms),
                  step_ms_p90=sorted(step_ms)[(9 * len(step_ms)) // 10])

    # end to end through the public API with pinned host buffers
    hcall, h2d, d2h = make_call(args.workload, dev, host=True)
    hcall()
    torch.cuda.synchronize()
    n_e2e = max(3, min(steps, args.e2e_steps))
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        hcall()                   # copies inputs in, runs, copies the output back (blocking)
    torch.cuda.synchronize()
    barrier(world)
    e2e_s = max_over_ranks(world, (time.perf_counter() - t0) / n_e2e, dev)
    result["e2e"] = dict(value=world * info["flops"] / e2e_s / 1e12, unit="TFLOP/s",
                         h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h,
                         ms_per_step=e2e_s * 1e3, steps=n_e2e)
    result["graph"] = graph_leg(call, flush, stream, min(steps, 200))
    if world == 1 and not args.no_other_workloads:
        del call
        torch.cuda.empty_cache()
        try:
            result["workloads"] = other_workloads(args.workload, dev, flush, stream, peaks)
        except Exception as e:
            result["workloads"] = dict(error=f"{type(e).__name__}: {e}"[:200])
    return result


def measure_briefly(name, dev, flush, stream, peaks, steps):
    """One workload: 3 warm-up calls, `steps` untraced calls (median ms) and
    `steps` traced calls (the dominant kernel's mean CUDA-event ms)."""
    import torch

    from normalization_convolution_blocks_gb300 import api
    info = workload_info(name)
    call, _, _ = make_call(name, dev)
    for _ in range(3):
        call()
        flush.fill_(1.0)
    torch.cuda.synchronize()
    times = {}
    for traced in (False, True):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        api.trace_enable(traced)
        for i in range(steps):
            starts[i].record(stream)
            call()
            ends[i].record(stream)
            flush.fill_(1.0)
        torch.cuda.synchronize()
        api.trace_enable(False)
        times[traced] = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    if api.query_status() != api.NRC_OK:
        raise RuntimeError("device status error")
    main = info["main_kernel"]
    main_ms = statistics.mean(ms for n, ms in api.trace_records() if n == main)
    roof, _ = roofline_of(info, main_ms, peaks)
    med = statistics.median(times[False])
    return dict(ms_per_call_median=round(med, 5),
                tflops=round(info["flops"] / (med * 1e-3) / 1e12, 2),
                kernel=main, kernel_ms=round(main_ms, 5), bound=roof["bound"],
                frac=roof["frac"], frac_effective=roof["frac_effective"])


def other_workloads(skip, dev, flush, stream, peaks, steps=30):
    """Every other workload of the library, measured the same way as the
    headline one but briefly: 3 warm-up calls, then `steps` timed calls
    untraced (ms/call, median) and `steps` traced (the dominant kernel's
    CUDA-event time and its roofline fraction), L2 flushed between calls.
    One clock record covers the whole pass."""
    import torch

    from normalization_convolution_blocks_gb300 import api
    from normalization_convolution_blocks_gb300 import synthetic as syn
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    sampler.mark("begin")
    res = {}
    for name in syn.WORKLOADS:
        if name == skip:
            continue
        try:
            res[name] = measure_briefly(name, dev, flush, stream, peaks, steps)
        except Exception as e:      # a secondary figure must not cost the headline line
            res[name] = dict(error=f"{type(e).__name__}: {e}"[:200])
            try:
                torch.cuda.synchronize()
                api.query_status()  # reads and clears the device status word
            except Exception:
                break
        torch.cuda.empty_cache()
    sampler.mark("end")
    res["clocks"] = sampler.stop()
    res["note"] = (f"{steps} untraced and {steps} traced calls each after 3 warm-up calls, "
                   "L2 flushed between calls; frac as in roofline")
    return res


def graph_leg(call, flush, stream, n):
    """The device-buffer call captured once in a CUDA graph (after a warm-up
    call on a side stream) and replayed n times: device ms per replay (CUDA
    events, L2 flushed between replays); then, over 50 back-to-back calls (no
    flush), the host's enqueue cost per call and the wall time per call until
    the GPU has finished, eager calls against replays."""
    import torch
    from normalization_convolution_blocks_gb300 import api
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        call()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for i in range(n):
        starts[i].record(stream)
        graph.replay()
        ends[i].record(stream)
        flush.fill_(1.0)
    torch.cuda.synchronize()
    replay_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    m = 50
    host, wall = {}, {}
    for kind, fn in (("eager", call), ("graph", graph.replay)):
        fn()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(m):
            fn()
        host[kind] = (time.perf_counter() - t0) / m * 1e6
        torch.cuda.synchronize()
        wall[kind] = (time.perf_counter() - t0) / m * 1e6
    if api.query_status() != api.NRC_OK:
        raise RuntimeError("device status error in the graph replays")
    return dict(ms_per_call_median=round(statistics.median(replay_ms), 5),
                ms_per_call_p10=round(sorted(replay_ms)[n // 10], 5), replays=n,
                host_us_per_call_eager=round(host["eager"], 1),
                host_us_per_call_graph=round(host["graph"], 1),
                back_to_back_us_per_call_eager=round(wall["eager"], 1),
                back_to_back_us_per_call_graph=round(wall["graph"], 1))


# ---------------------------------------------------------------------------
# The oracle, timed on the host cores (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------
def oracle_sampler(name):
    """Returns (run(n_units) -> flops done, unit description, total units)."""
    import numpy as np

    import oracle
    from normalization_convolution_blocks_gb300 import synthetic as syn
    wl = syn.WORKLOADS[name]
    inp = wl.make(seed=0)
    rng = np.random.default_rng(0)
    if wl.kind == "block":
        N, C, L = inp.x.shape
        args = [t.double().numpy() for t in (inp.x, inp.running_mean, inp.running_var,
                                             inp.gamma, inp.beta)]
        w, b = inp.weight.double().numpy(), inp.bias.double().numpy()

        def run(k):
            rn, ro = rng.integers(0, N, k), rng.integers(0, C, k)
            oracle.prenorm_block_rows(args[0], args[1], args[2], args[3], args[4], inp.eps, w, b,
                                      inp.dilation, rn, ro)
            return 2.0 * C * 3 * L * k
        return run, "output rows (n, o, all L)", N * C
    if wl.kind == "block_train":
        N, C, L = inp.x.shape
        x = inp.x.double().numpy()
        w, b = inp.weight.double().numpy(), inp.bias.double().numpy()

        def run(k):
            # every sample repeats the whole statistics pass over x
            oracle.prenorm_block_train(x, inp.running_mean, inp.running_var, inp.gamma,
                                       inp.beta, inp.eps, TRAIN_MOMENTUM, w, b, inp.dilation,
                                       rows_n=rng.integers(0, N, k), rows_o=rng.integers(0, C, k))
            return 2.0 * C * 3 * L * k
        return run, "output rows (n, o, all L) after the batch statistics", N * C
    if wl.kind == "conv_gn":
        N, Cin, T = inp.x.shape
        Cout, G = inp.weight.shape[0], inp.num_groups
        x, w = inp.x.double().numpy(), inp.weight.double().numpy()

        def run(k):
            oracle.conv_groupnorm_groups(x, w, None, G, inp.gamma, inp.beta, inp.eps,
                                         rng.integers(0, N, k), rng.integers(0, G, k))
            return 2.0 * (Cout // G) * T * Cin * 3 * k
        return run, "GroupNorm groups (n, g)", N * G
    B, IN = inp.x.shape
    OUT = inp.weight.shape[0]
    x, w = inp.x.double().numpy(), inp.weight.double().numpy()
    training = wl.params.get("training", True)

    def run(k):
        oracle.linear_bn_swish(x, w, inp.lin_bias, inp.gamma, inp.beta, inp.running_mean,
                               inp.running_var, inp.eps, inp.momentum, training,
                               float(inp.add_bias[0]), inp.divide_value,
                               cols=rng.integers(0, OUT, k))
        return 2.0 * B * IN * k
    return run, ("output columns (all batch rows, BN over the batch)" if training else
                 "output columns (all batch rows, BN with the running statistics)"), OUT


def size_sample(run, seconds):
    """Units per sample so that one sample takes about `seconds`."""
    k = 2
    while True:
        t0 = time.perf_counter()
        run(k)
        dt = time.perf_counter() - t0
        if dt > 0.2 or k >= 1 << 20:
            return max(1, int(k * seconds / max(dt, 1e-9)))
        k *= 4


def cpu_baseline(name, seconds=15.0):
    import oracle
    run, unit, total = oracle_sampler(name)
    k = min(total, size_sample(run, seconds))
    t0 = time.perf_counter()
    flops = run(k)
    dt = time.perf_counter() - t0
    return dict(value=flops / dt / 1e12, unit="TFLOP/s", cores=oracle.max_threads(),
                kind="oracle", sample=f"{k} of {total} {unit}, seed 0, {dt:.1f} s",
                ms_per_call_equiv=dt * total / k * 1e3)


def reference_arm(args):
    import oracle
    info = workload_info(args.workload)
    run, unit, total = oracle_sampler(args.workload)
    steps = args.steps if args.steps is not None else 5
    budget = 150.0 / max(1, steps + args.warmup)       # whole run within a few minutes
    k = min(total, size_sample(run, min(budget, 20.0)))
    for _ in range(args.warmup):
        run(k)
    times, flops = [], 0.0
    for _ in range(steps):
        t0 = time.perf_counter()
        flops = run(k)
        times.append(time.perf_counter() - t0)
    per = statistics.mean(times)
    value = flops / per / 1e12
    sample = f"{k} of {total} {unit} per step, seed 0"
    line = dict(impl="reference", metric=METRIC, value=value, unit="TFLOP/s", n_gpus=args.gpus,
                steps=steps, warmup=args.warmup, ms_per_step=per * 1e3,
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
                data="synthetic", config=dict(info["config"], l2="n/a (CPU)"),
                cpu_baseline=dict(value=value, unit="TFLOP/s", cores=oracle.max_threads(),
                                  kind="oracle", sample=sample),
                e2e=dict(value=value, unit="TFLOP/s", h2d_bytes_per_step=0,
                         d2h_bytes_per_step=0),
                ms_per_call_equiv=per * total / k * 1e3)
    return line


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the brief pass over the library's other workloads")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_setup(args.gpus) if args.impl == "ours" else (
        int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0)
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args)), flush=True)
        return

    r = gpu_arm(args, world, rank, local)
    if rank != 0:
        return
    info = r["info"]
    line = dict(
        metric=METRIC, value=round(r["value"], 3), unit="TFLOP/s", n_gpus=world,
        steps=r["steps"], warmup=args.warmup, ms_per_step=round(r["ms_per_step"], 5),
        higher_is_better=True, scaling="weak", vs_baseline=None, dtype=info["dtype"],
        data="synthetic",
        config=dict(info["config"], l2=l2_note(info),
                    parallelism="replicas" if world > 1 else "single GPU",
                    arithmetic=("bf16 tensor products, fp32 accumulate" if info["dtype"] == "bf16"
                                else "3 bf16 tensor products per term (hi/lo split), "
                                     "fp32 accumulate")),
        roofline=r["roofline"], e2e=r["e2e"], gpu_launches=r["launches"],
        clocks=r["clocks"], graph=r["graph"],
        ms_per_call_median=round(r["step_ms_median"], 5),
        ms_per_call_p10=round(r["step_ms_p10"], 5), ms_per_call_p90=round(r["step_ms_p90"], 5),
        kernels=r["kernels"],
        bandwidth=dict(value=round(world * info["min_bytes"] / (r["ms_per_step"] * 1e-3) / 1e9, 1),
                       unit="GB/s", bytes_per_call=info["min_bytes"],
                       note="the call's algorithmic bytes (inputs read once, output written "
                            "once) over its untraced time"),
    )
    if "workloads" in r:
        line["workloads"] = r["workloads"]
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
